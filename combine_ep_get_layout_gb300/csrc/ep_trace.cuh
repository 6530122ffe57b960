// Per-block timeline marks for diagnosing kernel boundaries (fill, drain,
// the wait for the kernel ahead).  Compiled in only when EP_TRACE is
// defined (the trace build of the library, see build.py --trace); in the
// product build every mark expands to nothing.
//
// A mark stores %globaltimer (ns) into a per-kernel array at
// [blockIdx.x][slot] (EP_TRACE_VALUE stores a count instead); the caller
// decides which thread marks.  Each translation unit that marks defines its own array
// with EP_TRACE_ARRAY and exports a reader with EP_TRACE_READER.  A
// launch overwrites the slots its blocks reach, so the arrays hold the last
// launch of each kernel (a slot no block reached keeps an older value:
// readers compare with the entry slot).
#pragma once

#include <cstdint>

namespace ep {

constexpr int kTraceBlocks = 4096;  // blocks traced per kernel (higher indices are not)
constexpr int kTraceSlots = 8;

}  // namespace ep

#ifdef EP_TRACE
#define EP_TRACE_ARRAY(name) __device__ unsigned long long name[ep::kTraceBlocks * ep::kTraceSlots]
#define EP_TRACE_MARK(name, slot)                                                           \
  do {                                                                                      \
    if (blockIdx.x < (unsigned)ep::kTraceBlocks)                                            \
      name[blockIdx.x * ep::kTraceSlots + (slot)] = ep::global_timer_ns();                  \
  } while (0)
#define EP_TRACE_VALUE(name, slot, value)                                                   \
  do {                                                                                      \
    if (blockIdx.x < (unsigned)ep::kTraceBlocks)                                            \
      name[blockIdx.x * ep::kTraceSlots + (slot)] = (unsigned long long)(value);            \
  } while (0)
// extern "C" int fn(unsigned long long *host_dst, int blocks): copies the
// first `blocks` blocks' slots to the host; returns a cudaError_t.
#define EP_TRACE_READER(fn, name)                                                           \
  extern "C" int fn(unsigned long long *host_dst, int blocks) {                             \
    if (blocks < 0 || blocks > ep::kTraceBlocks) return (int)cudaErrorInvalidValue;         \
    return (int)cudaMemcpyFromSymbol(host_dst, name,                                        \
                                     (size_t)blocks * ep::kTraceSlots * sizeof(unsigned long long)); \
  }
#else
#define EP_TRACE_ARRAY(name) static_assert(true, "")
#define EP_TRACE_MARK(name, slot) \
  do {                            \
  } while (0)
#define EP_TRACE_VALUE(name, slot, value) \
  do {                                    \
  } while (0)
#define EP_TRACE_READER(fn, name) static_assert(true, "")
#endif
