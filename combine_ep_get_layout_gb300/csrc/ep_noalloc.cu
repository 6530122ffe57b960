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

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Host code cannot use g_layout_scratch's name as a device address: look the
// address up once per device, with that device current.
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
  if (num_tokens < 0) return fail(EP_ERR_INVALID_ARG, "%s: num_tokens=%d < 0", fn, num_tokens);
  if (num_topk < 1 || num_topk > EP_MAX_TOPK)
    return fail(num_topk < 1 ? EP_ERR_INVALID_ARG : EP_ERR_UNSUPPORTED, "%s: num_topk=%d not in [1, %d]", fn,
                num_topk, EP_MAX_TOPK);
  if (num_ranks < 1 || num_ranks > EP_MAX_RANKS)
    return fail(num_ranks < 1 ? EP_ERR_INVALID_ARG : EP_ERR_UNSUPPORTED, "%s: num_ranks=%d not in [1, %d]", fn,
                num_ranks, EP_MAX_RANKS);
  if (num_experts < num_ranks || num_experts > EP_MAX_EXPERTS || num_experts % num_ranks != 0)
    return fail(num_experts > EP_MAX_EXPERTS ? EP_ERR_UNSUPPORTED : EP_ERR_INVALID_ARG,
                "%s: num_experts=%d must be a multiple of num_ranks=%d and at most %d", fn, num_experts,
                num_ranks, EP_MAX_EXPERTS);
  const bool any = num_tokens > 0;
  if (any && (topk_idx == nullptr || !aligned(topk_idx, 8)))
    return fail(EP_ERR_INVALID_ARG, "%s: topk_idx is NULL or not 8-byte aligned", fn);
  if (layout == nullptr || layout->num_tokens_per_expert == nullptr || layout->num_tokens_per_rank == nullptr ||
      layout->rank_prefix == nullptr || layout->error_word == nullptr ||
      (any && (layout->is_token_in_rank == nullptr || layout->token_slot == nullptr)))
    return fail(EP_ERR_INVALID_ARG, "%s: layout or one of its arrays is NULL", fn);
  if (!aligned(layout->num_tokens_per_expert, 4) || !aligned(layout->num_tokens_per_rank, 4) ||
      !aligned(layout->rank_prefix, 4) || !aligned(layout->error_word, 4) ||
      !aligned(layout->is_token_in_rank, 16) || !aligned(layout->token_slot, 16) ||
      !aligned(layout->work_counters, 16))
    return fail(EP_ERR_INVALID_ARG, "%s: a layout array is misaligned", fn);
  const size_t need = layout_workspace_bytes(num_tokens, num_experts, num_ranks);
  if (need > EP_NOALLOC_SCRATCH_BYTES)
    return fail(EP_ERR_UNSUPPORTED,
                "%s: %d tokens over %d ranks need %zu bytes of scratch; the static scratch holds %u "
                "(use ep_get_layout with a workspace)",
                fn, num_tokens, num_ranks, need, (unsigned)EP_NOALLOC_SCRATCH_BYTES);
  void *scratch = nullptr;
  const ep_status_t s = scratch_address(&scratch);
  if (s != EP_OK) return s;
  // The array keeps the previous call's contents: clear what this call uses.
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(scratch, 0, need, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(scratch)");
  return launch_layout(topk_idx, num_tokens, num_topk, num_experts, num_ranks, *layout, scratch, st);
}
