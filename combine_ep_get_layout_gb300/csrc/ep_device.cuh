// Device-side helpers shared by the layout, dispatch and combine kernels:
// hand-written PTX for mbarriers and bulk (TMA 1D) copies, bounded waits,
// and bf16 / e4m3 conversions.  sm_103a only.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "ep_internal.h"

namespace ep {

// A device wait that has not finished after this long gives up, sets
// EP_ERRBIT_TIMEOUT and lets the kernel return.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Plain arrival (release semantics at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete; false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// ------------------------------------------------------- bulk (TMA 1D) copy
// Sizes and both addresses must be multiples of 16 bytes.

// A hint that `bytes` of global memory at src (both multiples of 16) will be
// read soon: the lines are brought into L2.  No value is returned, so it is
// safe on memory another kernel may still be writing (L2 is where its writes
// land).
__device__ __forceinline__ void bulk_prefetch_l2(const void *src_gmem, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src_gmem), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Same, with an L2 eviction-priority policy (from createpolicy).
__device__ __forceinline__ void bulk_load_hint(void *dst_smem, const void *src_gmem,
                                               uint32_t bytes, uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_store(void *dst_gmem, const void *src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst_gmem),
               "r"(smem_addr(src_smem)), "r"(bytes)
               : "memory");
}

// Same, with an L2 eviction-priority policy (from createpolicy).
__device__ __forceinline__ void bulk_store_hint(void *dst_gmem, const void *src_smem, uint32_t bytes,
                                                uint64_t policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst_gmem),
               "r"(smem_addr(src_smem)), "r"(bytes), "l"(policy)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until at most N of this thread's bulk groups are still in flight.
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------ global memory

__device__ __forceinline__ int4 ld_stream_v4(const void *p) {
  int4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream_v4(void *p, int4 v) {
  asm volatile("st.global.cs.v4.s32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------- formats

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two floats -> packed bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Two floats -> packed e4m3x2 (lo in the low byte), round to nearest even,
// saturating to the largest finite magnitude (448).
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Hardware reciprocal approximation (PTX rcp.approx.f32, at most 1 ulp off
// over the normal range; subnormal inputs are not flushed).
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// (a * c, b * c), rounded to nearest even, as one packed f32x2 multiply.
__device__ __forceinline__ void mul2_rn(float a, float b, float c, float &ac, float &bc) {
  asm("{\n\t.reg .b64 t, k, u;\n\tmov.b64 t, {%2, %3};\n\tmov.b64 k, {%4, %4};\n\t"
      "mul.rn.f32x2 u, t, k;\n\tmov.b64 {%0, %1}, u;\n\t}"
      : "=f"(ac), "=f"(bc)
      : "f"(a), "f"(b), "f"(c));
}

// (a0 + y0, a1 + y1) as one packed f32x2 add, rounded to nearest even.
__device__ __forceinline__ void add2_rn(float &a0, float &a1, float y0, float y1) {
  asm("{\n\t.reg .b64 y, a;\n\tmov.b64 y, {%2, %3};\n\tmov.b64 a, {%0, %1};\n\t"
      "add.rn.f32x2 a, a, y;\n\tmov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(y0), "f"(y1));
}

// ------------------------------------------------------------- grid barrier
// For cooperative launches (all blocks co-resident).  The two words live in
// caller-zeroed global memory; the last block out resets them, so the next
// launch finds them zero again.

struct GridBarrierWords {
  uint32_t arrive;
  uint32_t depart;
};

// Every thread of every block calls it.  Returns false (in every thread of
// the block) if the wait gave up after kWaitLimitNs.  `s_flag` is a shared
// int the block uses to broadcast the outcome.
__device__ __forceinline__ bool grid_barrier(GridBarrierWords *bar, int *s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&bar->arrive, 1u);
    int ok = 1;
    const uint64_t t0 = global_timer_ns();
    while (ld_acquire_gpu(&bar->arrive) < gridDim.x) {
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

// Called once per block, after the block's last use of the barrier.
__device__ __forceinline__ void grid_barrier_exit(GridBarrierWords *bar) {
  if (threadIdx.x == 0) {
    const uint32_t prev = atomicAdd(&bar->depart, 1u);
    if (prev == gridDim.x - 1u) {
      atomicExch(&bar->arrive, 0u);
      atomicExch(&bar->depart, 0u);
    }
  }
}

// ------------------------------------------------------------- token source
// The order in which the blocks of a dispatch or combine grid take tokens:
// a fixed stripe per block (token blockIdx.x + i * gridDim.x), or tickets
// from a grid-wide counter (`ticket` given), so that a block that starts
// late or draws heavy tokens takes fewer.  One thread per block draws.
// `done` counts the blocks that will draw no more; the last of them puts
// both words back to zero for the next grid that uses them.

struct TokenSource {
  uint32_t *ticket;  // nullptr: fixed stripes
  uint32_t *done;
  int T;
};

// The drawing thread's block takes no more tokens (idempotent).
__device__ __forceinline__ void retire_tokens(const TokenSource &ts, bool &drained) {
  if (drained) return;
  drained = true;
  if (ts.ticket != nullptr && atomicAdd(ts.done, 1u) == gridDim.x - 1u) {
    atomicExch(ts.ticket, 0u);
    atomicExch(ts.done, 0u);
  }
}

// The block's i-th token, or -1 once the tokens are exhausted (from then
// on without touching the counter).  With a counter every token is drawn,
// the first too: a block that starts late (its SM still busy with the
// previous kernel) then owns no token yet.  `drained`: the drawing thread's
// state, false at the start.
//
// `head` > 0 (ticket mode): the block's first `head` tokens are its own
// stripe (blockIdx.x + i * gridDim.x, i < head) and tickets number the
// tokens after head * gridDim.x, so those first draws touch no counter.
__device__ __forceinline__ int draw_token(const TokenSource &ts, int i, bool &drained, int head = 0) {
  if (drained) return -1;
  const int t = (ts.ticket == nullptr || i < head) ? (int)blockIdx.x + i * (int)gridDim.x
                                                   : head * (int)gridDim.x + (int)atomicAdd(ts.ticket, 1u);
  if (t < ts.T) return t;
  retire_tokens(ts, drained);
  return -1;
}

// ------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialization may start before
// the kernel ahead of it in the stream has finished; it must wait here before
// its first access to global memory.  The trigger lets the kernel after it
// launch early (its blocks then wait in griddep_wait for this one to end).

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Warp-collective: whether a token's set of ranks under its routing (expert
// id `e` in lanes k < K, -1 in the other lanes) is exactly its set of ranks
// with a slot (`slot_lo` = slot of rank `lane`, `slot_hi` = of rank
// lane + 32, -1 where absent).  A layout depends on nothing else, so this
// detects a layout computed for another routing.
__device__ __forceinline__ bool ranks_agree(int64_t e, int E, int epr, int R, int slot_lo, int slot_hi,
                                            int lane) {
  const uint64_t bit = (e >= 0 && e < E) ? (1ull << (static_cast<int>(e) / epr)) : 0ull;
  const uint64_t mask = (uint64_t)__reduce_or_sync(0xffffffffu, (uint32_t)bit) |
                        ((uint64_t)__reduce_or_sync(0xffffffffu, (uint32_t)(bit >> 32)) << 32);
  bool ok = true;
  if (lane < R) ok = (((mask >> lane) & 1ull) != 0) == (slot_lo >= 0);
  if (lane + 32 < R) ok = ok && ((((mask >> (lane + 32)) & 1ull) != 0) == (slot_hi >= 0));
  return __all_sync(0xffffffffu, ok);
}

// Warp-collective, expanded layouts: whether each lane k < K holds a row
// (`slot` >= 0) exactly when expert id `e` is valid and not named by a lower
// lane (lanes >= K hold e = -1).  Detects a layout of another routing.
__device__ __forceinline__ bool choices_agree(int64_t e, int E, int K, int slot, int lane) {
  const uint32_t peers = __match_any_sync(0xffffffffu, (unsigned long long)e);
  const bool first = e >= 0 && e < E && (peers & ((1u << lane) - 1u)) == 0u;
  const bool ok = lane >= K || first == (slot >= 0);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void set_error(uint32_t *word, uint32_t bits) {
  if (word != nullptr) atomicOr(word, bits);
}

// Host side: launches a kernel on `stream` with programmatic stream
// serialization (when kUsePdl) and, if asked, as a cooperative grid.
template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kernel)(Params...), int grid, int block, size_t smem, cudaStream_t stream,
                          bool cooperative, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (kUsePdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cooperative) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace ep
