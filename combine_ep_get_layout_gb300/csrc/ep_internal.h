// Host-side internals shared by the C ABI (ep_api.cu) and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "ep_gb300.h"

namespace ep {

constexpr int kWarpSize = 32;

// Kernels are launched with programmatic stream serialization: each may be
// scheduled while the kernel ahead of it drains, and waits (griddep_wait)
// before touching global memory.
constexpr bool kUsePdl = true;

// Properties of the current device, queried once per device.
struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  size_t max_smem_per_block_optin = 0;
  size_t smem_per_sm = 0;
};

// The current device's properties; nullptr (and a message) on failure.
const DeviceInfo *current_device_info();

// Record a detail message for ep_last_error() and return the status.
ep_status_t fail(ep_status_t status, const char *fmt, ...);
ep_status_t cuda_fail(cudaError_t err, const char *what);
// Empty the calling thread's detail message (every entry point does first).
void clear_error();

// Host-side argument checks shared by the entry points: K, E and R within
// the limits with E % R == 0; a pointer non-null when `required` and aligned
// to `align` bytes when given.
ep_status_t check_routing_sizes(const char *fn, int num_topk, int num_experts, int num_ranks);
ep_status_t check_ptr(const char *fn, const char *name, const void *p, size_t align, bool required);

// ---- layout (ep_layout.cu)
size_t layout_workspace_bytes(int num_tokens, int num_experts, int num_ranks);
// The bytes of the workspace that launch_layout touches (its grid is capped,
// so at most this much of a larger workspace is used).
size_t layout_workspace_bytes_used(int num_tokens, int num_ranks);
ep_status_t launch_layout(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                          int num_ranks, const ep_layout_t &layout, void *workspace,
                          cudaStream_t stream);

// The first half of a layout whose slots the dispatch finishes
// (ep_get_layout_and_dispatch): one launch writes is_token_in_rank, each
// (token, rank)'s slot relative to its 256-token block into token_slot, and
// in the workspace (*local_base, [G*R], G = ceil(T / 256)) either each
// block's per-rank totals (*table_blocks = G > 0: G*R <= kBaseTableMax; the
// dispatch scans them itself and writes rank_prefix and
// num_tokens_per_rank), or, for larger layouts (*table_blocks = 0), each
// block's first slot in each rank, with rank_prefix and num_tokens_per_rank
// final.  The dispatch adds the block's base to each slot, writes it back
// and counts num_tokens_per_expert and bad ids.  Applies to
// 0 < T <= local_layout_max_tokens().
int local_layout_max_tokens();
constexpr int kLocalTokensPerBlock = 256;
constexpr int kBaseTableMax = 1024;  // block totals the dispatch scans itself (G * R)
ep_status_t launch_layout_local(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                                int num_ranks, const ep_layout_t &layout, void *workspace, cudaStream_t stream,
                                const int32_t **local_base, int *table_blocks);

// ---- expanded layout (ep_layout_expanded.cu)
size_t expanded_layout_workspace_bytes(int num_tokens, int num_experts);
ep_status_t launch_layout_expanded(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                                   int expert_alignment, const ep_expanded_layout_t &layout, void *workspace,
                                   cudaStream_t stream);

// ---- dispatch (ep_dispatch.cu)
// Bytes of a packed fp8 row: codes, scales, zero padding to 16 bytes, or to
// 512 when that adds under 5% to the unpadded row.
inline size_t fp8_packed_row_bytes(int hidden) {
  const size_t raw = (size_t)hidden + (size_t)(hidden / EP_FP8_GROUP) * 4;
  const size_t pad16 = (raw + 15) / 16 * 16;
  const size_t pad512 = (raw + 511) / 512 * 512;
  return (pad512 - raw) * 20 < raw ? pad512 : pad16;
}

struct DispatchArgs {
  const uint16_t *x;
  int num_tokens, hidden, num_topk, num_experts, num_ranks;
  const int64_t *topk_idx;
  const float *topk_weights;
  const int32_t *token_slot;  // [T * D]: rank layout D = R, expanded D = K
  uint32_t *error_word;
  bool expanded;
  const int32_t *expert_offset;        // expanded: [E+1]
  const int32_t *num_rows_per_expert;  // expanded: [E]
  bool zero_padding;                   // expanded: write the padding rows
  bool fp8;
  int packed_row_bytes;  // > 0: packed fp8 rows of this many bytes
  uint32_t *work_counters;  // 2 words (ticket, done) or null: fixed token stripes
  void *recv_x;
  float *recv_x_scales;
  int32_t *recv_src_idx;
  int32_t *recv_topk_idx;
  float *recv_topk_weights;
  int recv_capacity;
  uint32_t *recv_stats;  // [E] or null
  // warp-specialised kernels: tokens per block loaded (and for fp8 cast)
  // before the wait for the previous kernel on the stream; only when that
  // kernel writes none of x
  int early_rows = 0;
  // after launch_layout_local: token_slot holds slots relative to each
  // 256-token block; the dispatch adds the block's base, writes the slot back
  // to token_slot_out and counts num_tokens_per_expert.  The base is
  // local_base[b * R + r], or with local_table_blocks = G > 0 it is derived
  // from the per-block totals at local_base by the dispatch itself, which
  // then also writes rank_prefix and num_tokens_per_rank.
  const int32_t *local_base = nullptr;
  int local_table_blocks = 0;
  int32_t *token_slot_out = nullptr;
  int32_t *num_tokens_per_expert = nullptr;
  int32_t *rank_prefix = nullptr;
  int32_t *num_tokens_per_rank = nullptr;
};
// early_rows of ep_get_layout_and_dispatch (the input stages and the output
// buffers of the warp-specialised kernel hold up to 4 tokens)
constexpr int kEarlyRows = 3;
// bf16 rows of the rank path through the warp-specialised kernel (else the
// ring kernel); the one-launch layout of ep_get_layout_and_dispatch needs it
constexpr bool kBf16WarpSpecialised = true;
ep_status_t launch_dispatch(const DispatchArgs &a, cudaStream_t stream);

// ---- combine (ep_combine.cu)
struct CombineArgs {
  const uint16_t *y;
  int recv_capacity, hidden, num_tokens, num_ranks, num_topk, num_experts;
  bool expanded;              // token_slot is [T * K] of an expanded layout
  const int32_t *token_slot;
  uint32_t *error_word;
  const int64_t *topk_idx;
  const float *topk_weights;
  const uint16_t *bias0, *bias1;  // [T*H] or null
  uint16_t *out;
  uint32_t *work_counters;  // 2 words (ticket, done) or null: fixed token stripes
};
ep_status_t launch_combine(const CombineArgs &a, cudaStream_t stream);

}  // namespace ep
