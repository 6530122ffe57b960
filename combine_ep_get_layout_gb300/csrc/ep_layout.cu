// Layout kernel: the count phase and the count exchange of TileScale PR #68
// ("[Example] EP v2 intranode dispatch/combine", README section "Design"),
// on one GPU where the expert-parallel ranks are logical partitions of the
// expert set.
//
//   phase 1  each block owns a contiguous range of tokens.  Per token it
//            validates the K expert ids, counts them in a shared-memory
//            histogram (shared atomics) and ORs rank bits into a 64-bit mask,
//            so a token is in a rank once however many of its experts live
//            there (the pages' per-(token, destination) dedup).  Warp ballots
//            turn the masks into per-rank block totals.
//   exchange the block totals go to global memory; a bounded grid barrier
//            (cooperative launch: all blocks are co-resident) stands in for
//            the pages' count exchange between ranks.
//   phase 2  every block scans the totals of the blocks before it, which
//            gives rank_prefix (the pages' send_base[d]) plus this block's
//            first slot in each rank; warp ballots and a shared scan over
//            warps then give each (token, rank) its slot in ascending token
//            order (a stable scatter).
#include <algorithm>
#include <mutex>

#include "ep_device.cuh"

namespace ep {
namespace {

constexpr int kLayoutThreads = 256;  // one token per thread per chunk
constexpr int kLayoutWarps = kLayoutThreads / kWarpSize;
constexpr size_t kPartialOffset = 256;  // bytes: barrier words come first

struct LayoutParams {
  const int64_t *topk_idx;
  int num_tokens, num_topk, num_experts, num_ranks, experts_per_rank;
  int tokens_per_block;
  ep_layout_t out;
  GridBarrierWords *bar;
  int32_t *partial;  // [gridDim.x * R] per-block, per-rank token counts
};

size_t layout_smem_bytes(int tokens_per_block, int E, int R) {
  // masks[tpb] u64, hist[E], blk_cnt[R], warp_off[W*R], chunk_tot[R],
  // tot[R], before[R], base[R+1], run[R], flags[2], scan_all[T], scan_before[T]
  size_t ints = (size_t)E + R + (size_t)kLayoutWarps * R + R + R + R + (R + 1) + R + 3 + 2 * kLayoutThreads;
  return (size_t)tokens_per_block * sizeof(uint64_t) + ints * sizeof(int32_t);
}

// KMAX bounds the unrolled index loads: all K ids of a token are requested
// before the first is used.
template <int KMAX>
__global__ void __launch_bounds__(kLayoutThreads) layout_kernel(LayoutParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x;
  const int lane = tid & (kWarpSize - 1);
  const int warp = tid / kWarpSize;
  const int G = gridDim.x;
  const int b = blockIdx.x;
  const int R = p.num_ranks, E = p.num_experts, K = p.num_topk;

  uint64_t *masks = reinterpret_cast<uint64_t *>(smem);
  int *hist = reinterpret_cast<int *>(masks + p.tokens_per_block);
  int *blk_cnt = hist + E;
  int *warp_off = blk_cnt + R;  // [kLayoutWarps][R]
  int *chunk_tot = warp_off + kLayoutWarps * R;
  int *tot = chunk_tot + R;
  int *before = tot + R;
  int *base = before + R;  // [R + 1]
  int *run = base + R + 1;
  int *flags = run + R;  // [0] bad index seen, [1] barrier timed out, [2] barrier scratch
  int *scan_all = flags + 3;                  // [kLayoutThreads]
  int *scan_before = scan_all + kLayoutThreads;  // [kLayoutThreads]

  for (int i = tid; i < E; i += kLayoutThreads) hist[i] = 0;
  for (int i = tid; i < R; i += kLayoutThreads) blk_cnt[i] = 0;
  if (tid < 2) flags[tid] = 0;
  griddep_wait();
  griddep_launch_dependents();
  if (b == 0) {
    // Cleared before the barrier; every block adds into them after it.
    for (int i = tid; i < E; i += kLayoutThreads) p.out.num_tokens_per_expert[i] = 0;
    if (tid == 0) *p.out.error_word = 0u;
    if (tid < EP_WORK_COUNTER_WORDS && p.out.work_counters != nullptr) p.out.work_counters[tid] = 0u;
  }
  __syncthreads();

  const int begin = min(b * p.tokens_per_block, p.num_tokens);
  const int end = min(begin + p.tokens_per_block, p.num_tokens);

  // ---- phase 1: count
  bool bad = false;
  for (int c0 = begin; c0 < end; c0 += kLayoutThreads) {
    const int t = c0 + tid;
    uint64_t mask = 0;
    if (t < end) {
      const int64_t *row = p.topk_idx + (size_t)t * K;
      int64_t ids[KMAX];
#pragma unroll
      for (int k = 0; k < KMAX; ++k) ids[k] = k < K ? __ldg(row + k) : -1;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        const int64_t e = ids[k];
        if (e == -1) continue;
        if (e < 0 || e >= E) {
          bad = true;
          continue;
        }
        const int ei = static_cast<int>(e);
        atomicAdd(&hist[ei], 1);
        mask |= 1ull << (ei / p.experts_per_rank);
      }
      masks[t - begin] = mask;
    }
    for (int r = 0; r < R; ++r) {
      const uint32_t bal = __ballot_sync(0xffffffffu, (mask >> r) & 1ull);
      if (lane == 0 && bal != 0u) atomicAdd(&blk_cnt[r], __popc(bal));
    }
  }
  if (bad) flags[0] = 1;
  __syncthreads();
  for (int r = tid; r < R; r += kLayoutThreads) p.partial[(size_t)b * R + r] = blk_cnt[r];

  // ---- exchange: bounded grid barrier (all blocks co-resident)
  __threadfence();
  if (!grid_barrier(p.bar, &flags[2]) && tid == 0) flags[1] = 1;

  // ---- phase 2: bases (exclusive scan over ranks and over earlier blocks);
  // the block totals are summed by kLayoutThreads / R threads per rank
  const int per_rank = kLayoutThreads / R;  // >= 2 since R <= 64
  if (tid < per_rank * R) {
    const int r = tid % R;
    int all = 0, earlier = 0;
    for (int bb = tid / R; bb < G; bb += per_rank) {
      const int v = __ldcg(&p.partial[(size_t)bb * R + r]);
      all += v;
      if (bb < b) earlier += v;
    }
    scan_all[tid] = all;
    scan_before[tid] = earlier;
  }
  __syncthreads();
  for (int r = tid; r < R; r += kLayoutThreads) {
    int all = 0, earlier = 0;
    for (int q = 0; q < per_rank; ++q) {
      all += scan_all[q * R + r];
      earlier += scan_before[q * R + r];
    }
    tot[r] = all;
    before[r] = earlier;
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int r = 0; r < R; ++r) {
      base[r] = acc;
      acc += tot[r];
    }
    base[R] = acc;
  }
  __syncthreads();
  if (b == 0) {
    for (int r = tid; r <= R; r += kLayoutThreads) {
      p.out.rank_prefix[r] = base[r];
      if (r < R) p.out.num_tokens_per_rank[r] = tot[r];
    }
  }
  for (int e = tid; e < E; e += kLayoutThreads)
    if (hist[e] != 0) atomicAdd(&p.out.num_tokens_per_expert[e], hist[e]);
  if (tid == 0) {
    const uint32_t bits = (flags[0] ? EP_ERRBIT_BAD_INDEX : 0u) | (flags[1] ? EP_ERRBIT_TIMEOUT : 0u);
    if (bits) atomicOr(p.out.error_word, bits);
  }
  for (int r = tid; r < R; r += kLayoutThreads) run[r] = base[r] + before[r];
  __syncthreads();

  // ---- phase 2: slots, in ascending token order within each rank
  const uint32_t lanes_below = (1u << lane) - 1u;
  const bool vec4 = (R % 4) == 0;
  for (int c0 = begin; c0 < end; c0 += kLayoutThreads) {
    const int t = c0 + tid;
    const uint64_t mask = (t < end) ? masks[t - begin] : 0ull;
    for (int r = 0; r < R; ++r) {
      const uint32_t bal = __ballot_sync(0xffffffffu, (mask >> r) & 1ull);
      if (lane == 0) warp_off[warp * R + r] = __popc(bal);
    }
    __syncthreads();
    for (int r = tid; r < R; r += kLayoutThreads) {
      int acc = 0;
      for (int w = 0; w < kLayoutWarps; ++w) {
        const int c = warp_off[w * R + r];
        warp_off[w * R + r] = acc;
        acc += c;
      }
      chunk_tot[r] = acc;
    }
    __syncthreads();
    int32_t *slot_row = p.out.token_slot + (size_t)t * R;
    uint8_t *in_row = p.out.is_token_in_rank + (size_t)t * R;
    for (int r0 = 0; r0 < R; r0 += 4) {
      int s[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = r0 + q;
        s[q] = -1;
        if (r < R) {  // uniform across the warp
          const bool in = (mask >> r) & 1ull;
          const uint32_t bal = __ballot_sync(0xffffffffu, in);
          if (in) s[q] = run[r] + warp_off[warp * R + r] + __popc(bal & lanes_below);
        }
      }
      if (t < end) {
        if (vec4) {
          *reinterpret_cast<int4 *>(slot_row + r0) = make_int4(s[0], s[1], s[2], s[3]);
          const uint32_t bytes = (s[0] >= 0 ? 1u : 0u) | (s[1] >= 0 ? 1u << 8 : 0u) |
                                 (s[2] >= 0 ? 1u << 16 : 0u) | (s[3] >= 0 ? 1u << 24 : 0u);
          *reinterpret_cast<uint32_t *>(in_row + r0) = bytes;
        } else {
          for (int q = 0; q < 4 && r0 + q < R; ++q) {
            slot_row[r0 + q] = s[q];
            in_row[r0 + q] = s[q] >= 0 ? 1 : 0;
          }
        }
      }
    }
    __syncthreads();
    for (int r = tid; r < R; r += kLayoutThreads) run[r] += chunk_tot[r];
    __syncthreads();
  }

  // ---- exit: the last block out resets the barrier words for the next call
  grid_barrier_exit(p.bar);
}

int max_layout_blocks(int num_tokens) {
  return std::max(1, (num_tokens + kLayoutThreads - 1) / kLayoutThreads);
}

}  // namespace

size_t layout_workspace_bytes(int num_tokens, int num_experts, int num_ranks) {
  (void)num_experts;
  const size_t partial = (size_t)max_layout_blocks(num_tokens) * (size_t)num_ranks * sizeof(int32_t);
  return kPartialOffset + ((partial + 255) / 256) * 256;
}

ep_status_t launch_layout(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                          int num_ranks, const ep_layout_t &layout, void *workspace,
                          cudaStream_t stream) {
  const DeviceInfo *di = current_device_info();
  if (di == nullptr) return EP_ERR_CUDA;

  const auto kernel = num_topk <= 8 ? layout_kernel<8> : layout_kernel<EP_MAX_TOPK>;
  static std::mutex mu;
  static bool configured[64] = {};
  {
    std::lock_guard<std::mutex> g(mu);
    if (di->device < 64 && !configured[di->device]) {
      for (auto k : {layout_kernel<8>, layout_kernel<EP_MAX_TOPK>}) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)di->max_smem_per_block_optin);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(layout_kernel)");
      }
      configured[di->device] = true;
    }
  }

  // Grid: one block per 256 tokens, capped at what can be co-resident.
  int grid = max_layout_blocks(num_tokens);
  size_t smem = 0;
  for (int iter = 0;; ++iter) {
    const int tpb = (num_tokens + grid - 1) / grid;
    smem = layout_smem_bytes(tpb, num_experts, num_ranks);
    if (smem > di->max_smem_per_block_optin)
      return fail(EP_ERR_UNSUPPORTED,
                  "ep_get_layout: %d tokens need %zu bytes of shared memory per block (max %zu)",
                  num_tokens, smem, di->max_smem_per_block_optin);
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kLayoutThreads, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(layout)");
    const int cap = per_sm * di->num_sms;
    if (cap <= 0) return fail(EP_ERR_UNSUPPORTED, "ep_get_layout: layout kernel cannot be resident");
    if (grid <= cap) break;
    if (iter > 8) return fail(EP_ERR_UNSUPPORTED, "ep_get_layout: no co-resident grid found");
    grid = cap;
  }

  LayoutParams p;
  p.topk_idx = topk_idx;
  p.num_tokens = num_tokens;
  p.num_topk = num_topk;
  p.num_experts = num_experts;
  p.num_ranks = num_ranks;
  p.experts_per_rank = num_experts / num_ranks;
  p.tokens_per_block = (num_tokens + grid - 1) / grid;
  p.out = layout;
  p.bar = static_cast<GridBarrierWords *>(workspace);
  p.partial = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(workspace) + kPartialOffset);

  cudaError_t e = launch_kernel(kernel, grid, kLayoutThreads, smem, stream, true, p);
  if (e != cudaSuccess) return cuda_fail(e, "launch layout_kernel");
  return EP_OK;
}

}  // namespace ep
