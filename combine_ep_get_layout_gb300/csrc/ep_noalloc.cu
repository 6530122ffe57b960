// ep_get_layout_noalloc: the layout entry point for callers that cannot
// allocate device memory at call time (for example a plugin inside another
// runtime's enqueue callback, which owns all device memory, or a serving
// loop that must not risk the device-wide synchronisation a cudaMalloc or
// cudaFree can cause).  Instead of a caller-supplied workspace it uses the
// static device array below; it calls no cudaMalloc, cudaFree or other
// allocating routine.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "ep_internal.h"

namespace ep {
namespace {

// Scratch of the layout kernels (the per-block rank totals they exchange).
// Zero at module load; every GPU that loads the library holds it until exit.
__device__ __align__(256) unsigned char g_layout_scratch[EP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Host code cannot use g_layout_scratch's name as a device address: look the
// address up once per device, with that device current, and keep it for the
// life of the process (a cudaDeviceReset of the device would invalidate it,
// as it does the library's other per-device set-up).
ep_status_t scratch_address(void **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(EP_ERR_UNSUPPORTED, "ep_get_layout_noalloc: device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> g(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_layout_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(g_layout_scratch)");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return EP_OK;
}

}  // namespace
}  // namespace ep

extern "C" ep_status_t ep_get_layout_noalloc(const int64_t *topk_idx, int num_tokens, int num_topk,
                                             int num_experts, int num_ranks, const ep_layout_t *layout,
                                             ep_stream_t stream) {
  using namespace ep;
  static const char *fn = "ep_get_layout_noalloc";
  clear_error();
  // The same checks as ep_get_layout, short of the workspace.
  if (num_tokens < 0) return fail(EP_ERR_INVALID_ARG, "%s: num_tokens=%d < 0", fn, num_tokens);
  ep_status_t s = check_routing_sizes(fn, num_topk, num_experts, num_ranks);
  const bool any = num_tokens > 0;
  if (s == EP_OK) s = check_ptr(fn, "topk_idx", topk_idx, 8, any);
  if (s != EP_OK) return s;
  if (layout == nullptr) return fail(EP_ERR_INVALID_ARG, "%s: layout is NULL", fn);
  const struct {
    const char *name;
    const void *p;
    size_t align;
    bool required;
  } members[] = {
      {"layout.num_tokens_per_expert", layout->num_tokens_per_expert, 4, true},
      {"layout.num_tokens_per_rank", layout->num_tokens_per_rank, 4, true},
      {"layout.rank_prefix", layout->rank_prefix, 4, true},
      {"layout.is_token_in_rank", layout->is_token_in_rank, 16, any},
      {"layout.token_slot", layout->token_slot, 16, any},
      {"layout.error_word", layout->error_word, 4, true},
      {"layout.work_counters", layout->work_counters, 16, false},
  };
  for (const auto &m : members)
    if ((s = check_ptr(fn, m.name, m.p, m.align, m.required)) != EP_OK) return s;
  // The layout kernels' grid is capped, so they touch at most this much.
  const size_t need = layout_workspace_bytes_used(num_tokens, num_ranks);
  if (need > EP_NOALLOC_SCRATCH_BYTES)
    return fail(EP_ERR_UNSUPPORTED,
                "%s: %d tokens over %d ranks need %zu bytes of scratch; the static scratch holds %u "
                "(use ep_get_layout with a workspace)",
                fn, num_tokens, num_ranks, need, (unsigned)EP_NOALLOC_SCRATCH_BYTES);
  void *scratch = nullptr;
  if ((s = scratch_address(&scratch)) != EP_OK) return s;
  // The array keeps the previous call's contents: clear what this call uses.
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(scratch, 0, need, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(scratch)");
  return launch_layout(topk_idx, num_tokens, num_topk, num_experts, num_ranks, *layout, scratch, st);
}
