// Layout kernels: the count phase and the count exchange of TileScale PR
// #68 ("[Example] EP v2 intranode dispatch/combine", README section
// "Design"), on one GPU where the expert-parallel ranks are logical
// partitions of the expert set.  Two ordinary launches, the kernel boundary
// standing in for the pages' count exchange between ranks:
//
//   layout_count_kernel  each block owns a contiguous range of tokens.  Per
//            token it validates the K expert ids and ORs rank bits into a
//            64-bit mask, so a token is in a rank once however many of its
//            experts live there (the pages' per-(token, destination) dedup).
//            Warp ballots turn the masks into per-rank block totals, written
//            to the workspace.
//   layout_slot_kernel   every block re-reads its tokens' ids (from L2),
//            rebuilds the masks and counts the ids in a shared-memory
//            histogram (shared atomics), scans the block totals of all
//            blocks (rank_prefix, the pages' send_base[d], plus this block's
//            first slot in each rank), then warp ballots and a shared scan
//            over warps give each (token, rank) its slot in ascending token
//            order (a stable scatter).
//
// layout_local_kernel is the one-launch layout of ep_get_layout_and_dispatch:
// slots relative to each 256-token block and the blocks' per-rank totals,
// which the dispatch scans itself (up to kBaseTableMax totals) or the last
// block to finish turns into bases; the dispatch adds the bases.
#include <algorithm>

#include "ep_device.cuh"
#include "ep_trace.cuh"

namespace ep {
namespace {

constexpr int kLayoutThreads = 256;  // one token per thread per chunk
constexpr int kLayoutWarps = kLayoutThreads / kWarpSize;
constexpr size_t kPartialOffset = 256;  // workspace header (the local layout's ticket word), then the totals
constexpr int kMaxLayoutBlocks = 2048;  // more tokens per block beyond this

// Trace build only: 0 entry, 1 the wait for the kernel ahead done, 2 ids
// loaded, 3 totals published, 5 slots written, 6 (last block) totals read,
// 7 (last block) bases written.
EP_TRACE_ARRAY(g_trace_layout);

struct LayoutParams {
  const int64_t *topk_idx;
  int num_tokens, num_topk, num_experts, num_ranks, experts_per_rank;
  int tokens_per_block;
  ep_layout_t out;
  int32_t *partial;  // [gridDim.x * R] per-block, per-rank token counts
};

// The rank mask of a token whose ids are `ids`; counts each valid id in
// `hist` (shared; null to skip) and sets `bad` for an id outside [-1, E).
template <int KMAX>
__device__ __forceinline__ uint64_t rank_mask(const int64_t (&ids)[KMAX], int K, int E, int epr, int *hist,
                                              bool &bad) {
  uint64_t mask = 0;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    const int64_t e = ids[k];
    if (k >= K || e == -1) continue;
    if (e < 0 || e >= E) {
      bad = true;
      continue;
    }
    const int ei = static_cast<int>(e);
    if (hist != nullptr) atomicAdd(&hist[ei], 1);
    mask |= 1ull << (ei / epr);
  }
  return mask;
}

// Brings the ids of tokens [t0, t0 + n) into L2 without reading them (safe
// before the wait for the kernel ahead, which may be the one writing them:
// L2 is where its writes land): one prefetch per 128-byte line, the first
// kPrefetchIdBytes of the range at most.
constexpr size_t kPrefetchIdBytes = 64 * 1024;
__device__ __forceinline__ void prefetch_ids(const LayoutParams &p, int t0, int n) {
  if (n <= 0) return;
  const char *base = reinterpret_cast<const char *>(p.topk_idx + (size_t)t0 * p.num_topk);
  const size_t bytes = min((size_t)n * p.num_topk * sizeof(int64_t), kPrefetchIdBytes);
  for (size_t off = (size_t)threadIdx.x * 128; off < bytes; off += (size_t)blockDim.x * 128) prefetch_l2(base + off);
  if (threadIdx.x == 0) prefetch_l2(base + bytes - 1);  // the last line, when base is not line-aligned
}

// The K ids of token t, all requested before the first is used; -1 past K
// and for t >= end.
template <int KMAX>
__device__ __forceinline__ void load_ids(const LayoutParams &p, int t, int end, int64_t (&ids)[KMAX]) {
  const int64_t *row = p.topk_idx + (size_t)t * p.num_topk;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) ids[k] = (t < end && k < p.num_topk) ? __ldg(row + k) : -1;
}

template <int KMAX>
__global__ void __launch_bounds__(kLayoutThreads) layout_count_kernel(LayoutParams p) {
  __shared__ int blk_cnt[EP_MAX_RANKS];
  const int tid = threadIdx.x;
  const int lane = tid & (kWarpSize - 1);
  const int b = blockIdx.x;
  const int R = p.num_ranks, E = p.num_experts;
  for (int r = tid; r < R; r += kLayoutThreads) blk_cnt[r] = 0;
  const int begin = min(b * p.tokens_per_block, p.num_tokens);
  const int end = min(begin + p.tokens_per_block, p.num_tokens);
  prefetch_ids(p, begin, end - begin);
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();
  if (b == 0) {  // the slot kernel adds into them, after this kernel
    for (int i = tid; i < E; i += kLayoutThreads) p.out.num_tokens_per_expert[i] = 0;
    if (tid == 0) *p.out.error_word = 0u;
    if (tid < EP_WORK_COUNTER_WORDS && p.out.work_counters != nullptr) p.out.work_counters[tid] = 0u;
  }
  bool bad = false;
  for (int c0 = begin; c0 < end; c0 += kLayoutThreads) {
    int64_t ids[KMAX];
    load_ids(p, c0 + tid, end, ids);
    const uint64_t mask = rank_mask(ids, p.num_topk, E, p.experts_per_rank, nullptr, bad);
    for (int r = 0; r < R; ++r) {
      const uint32_t bal = __ballot_sync(0xffffffffu, (mask >> r) & 1ull);
      if (lane == 0 && bal != 0u) atomicAdd(&blk_cnt[r], __popc(bal));
    }
  }
  __syncthreads();
  for (int r = tid; r < R; r += kLayoutThreads) p.partial[(size_t)b * R + r] = blk_cnt[r];
}

size_t slot_smem_bytes(int E, int R) {
  // hist[E], warp_off[W*R], chunk_tot[R], tot[R], before[R], base[R+1], run[R],
  // flags[1], scan_all[T], scan_before[T]
  return ((size_t)E + (size_t)kLayoutWarps * R + 4 * (size_t)R + (R + 1) + 1 + 2 * kLayoutThreads) * sizeof(int32_t);
}

template <int KMAX>
__global__ void __launch_bounds__(kLayoutThreads) layout_slot_kernel(LayoutParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x;
  const int lane = tid & (kWarpSize - 1);
  const int warp = tid / kWarpSize;
  const int G = gridDim.x;
  const int b = blockIdx.x;
  const int R = p.num_ranks, E = p.num_experts;
  int *hist = reinterpret_cast<int *>(smem);
  int *warp_off = hist + E;  // [kLayoutWarps][R]
  int *chunk_tot = warp_off + kLayoutWarps * R;
  int *tot = chunk_tot + R;
  int *before = tot + R;
  int *base = before + R;  // [R + 1]
  int *run = base + R + 1;
  int *flags = run + R;  // [0] bad index seen
  int *scan_all = flags + 1;                     // [kLayoutThreads]
  int *scan_before = scan_all + kLayoutThreads;  // [kLayoutThreads]
  for (int i = tid; i < E; i += kLayoutThreads) hist[i] = 0;
  if (tid == 0) flags[0] = 0;
  __syncthreads();
  // The kernel after this one waits for it to complete (and so for the count
  // kernel too) before it reads the layout: it may start early.
  griddep_launch_dependents();
  griddep_wait();

  const int begin = min(b * p.tokens_per_block, p.num_tokens);
  const int end = min(begin + p.tokens_per_block, p.num_tokens);
  int64_t ids[KMAX];
  load_ids(p, begin + tid, end, ids);  // in flight during the scan

  // bases: exclusive scan over ranks and over earlier blocks
  const int per_rank = kLayoutThreads / R;  // >= 4 since R <= 64
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
  for (int r = tid; r < R; r += kLayoutThreads) run[r] = base[r] + before[r];
  __syncthreads();

  // slots, in ascending token order within each rank
  const uint32_t lanes_below = (1u << lane) - 1u;
  const bool vec4 = (R % 4) == 0;
  bool bad = false;
  for (int c0 = begin; c0 < end; c0 += kLayoutThreads) {
    const int t = c0 + tid;
    if (c0 != begin) load_ids(p, t, end, ids);
    const uint64_t mask = rank_mask(ids, p.num_topk, E, p.experts_per_rank, hist, bad);
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
      int sl[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = r0 + q;
        sl[q] = -1;
        if (r < R) {  // uniform across the warp
          const bool in = (mask >> r) & 1ull;
          const uint32_t bal = __ballot_sync(0xffffffffu, in);
          if (in) sl[q] = run[r] + warp_off[warp * R + r] + __popc(bal & lanes_below);
        }
      }
      if (t < end) {
        if (vec4) {
          *reinterpret_cast<int4 *>(slot_row + r0) = make_int4(sl[0], sl[1], sl[2], sl[3]);
          const uint32_t bytes = (sl[0] >= 0 ? 1u : 0u) | (sl[1] >= 0 ? 1u << 8 : 0u) |
                                 (sl[2] >= 0 ? 1u << 16 : 0u) | (sl[3] >= 0 ? 1u << 24 : 0u);
          *reinterpret_cast<uint32_t *>(in_row + r0) = bytes;
        } else {
          for (int q = 0; q < 4 && r0 + q < R; ++q) {
            slot_row[r0 + q] = sl[q];
            in_row[r0 + q] = sl[q] >= 0 ? 1 : 0;
          }
        }
      }
    }
    __syncthreads();
    for (int r = tid; r < R; r += kLayoutThreads) run[r] += chunk_tot[r];
    __syncthreads();
  }
  if (bad) flags[0] = 1;
  __syncthreads();
  for (int e = tid; e < E; e += kLayoutThreads)
    if (hist[e] != 0) atomicAdd(&p.out.num_tokens_per_expert[e], hist[e]);
  if (tid == 0 && flags[0]) atomicOr(p.out.error_word, EP_ERRBIT_BAD_INDEX);
}

// ------------------------------------------------------------------------
// The first half of a layout that the dispatch finishes (see
// launch_layout_local).  One block per 256 tokens (one per thread): the rank
// masks, each (token, rank)'s slot relative to the block (ballot prefix plus
// a shared scan over warps, ascending token order), is_token_in_rank, and
// the block's totals.  The ids are prefetched into L2 before the wait for
// the kernel ahead.
//   SCAN = false: that is all; the dispatch, once this kernel has
//     completed, scans the totals itself (a small table: G * R entries).
//   SCAN = true: the totals go out first, then a ticket on `done` (after a
//     fence); the last block to take one turns the totals into each block's
//     first slot in each rank, in place, and writes rank_prefix and
//     num_tokens_per_rank, while the other blocks write their slots.  It
//     leaves `done` at zero for the next call.
template <int KMAX, bool SCAN>
__global__ void __launch_bounds__(kLayoutThreads) layout_local_kernel(LayoutParams p, uint32_t *done) {
  __shared__ int warp_off[kLayoutWarps * EP_MAX_RANKS];
  __shared__ int seg_sum[kLayoutThreads];
  __shared__ int tot[EP_MAX_RANKS];
  __shared__ int base[EP_MAX_RANKS + 1];
  __shared__ int s_last;
  const int tid = threadIdx.x;
  const int lane = tid & (kWarpSize - 1);
  const int warp = tid / kWarpSize;
  const int G = gridDim.x;
  const int b = blockIdx.x;
  const int R = p.num_ranks, E = p.num_experts;
  if (tid == 0) EP_TRACE_MARK(g_trace_layout, 0);
  prefetch_ids(p, b * kLayoutThreads, min(kLayoutThreads, p.num_tokens - b * kLayoutThreads));
  griddep_wait();
  griddep_launch_dependents();
  if (tid == 0) EP_TRACE_MARK(g_trace_layout, 1);
  if (b == 0) {  // the dispatch adds into them, after this kernel
    for (int i = tid; i < E; i += kLayoutThreads) p.out.num_tokens_per_expert[i] = 0;
    if (tid == 0) *p.out.error_word = 0u;
    if (tid < EP_WORK_COUNTER_WORDS && p.out.work_counters != nullptr) p.out.work_counters[tid] = 0u;
  }
  const int t = b * kLayoutThreads + tid;
  int64_t ids[KMAX];
  load_ids(p, t, p.num_tokens, ids);
  bool bad = false;  // the dispatch reports bad ids
  const uint64_t mask = rank_mask(ids, p.num_topk, E, p.experts_per_rank, nullptr, bad);
  if (tid == 0 && mask != ~0ull) EP_TRACE_MARK(g_trace_layout, 2);  // once the ids are in
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
    p.partial[(size_t)b * R + r] = acc;
  }
  // With SCAN the totals are visible before the ticket; the slots are
  // written after it (the dispatch reads them once this kernel has
  // completed), so the last block's pass overlaps the other blocks' slot
  // writes.
  if constexpr (SCAN) __threadfence();
  __syncthreads();
  if (tid == 0) EP_TRACE_MARK(g_trace_layout, 3);
  if (SCAN && tid == 0) s_last = atomicAdd(done, 1u) == (uint32_t)G - 1u;
  const uint32_t lanes_below = (1u << lane) - 1u;
  const bool vec4 = (R % 4) == 0;
  int32_t *slot_row = p.out.token_slot + (size_t)t * R;
  uint8_t *in_row = p.out.is_token_in_rank + (size_t)t * R;
  for (int r0 = 0; r0 < R; r0 += 4) {
    int sl[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = r0 + q;
      sl[q] = -1;
      if (r < R) {  // uniform across the warp
        const bool in = (mask >> r) & 1ull;
        const uint32_t bal = __ballot_sync(0xffffffffu, in);
        if (in) sl[q] = warp_off[warp * R + r] + __popc(bal & lanes_below);
      }
    }
    if (t < p.num_tokens) {
      if (vec4) {
        *reinterpret_cast<int4 *>(slot_row + r0) = make_int4(sl[0], sl[1], sl[2], sl[3]);
        const uint32_t bytes = (sl[0] >= 0 ? 1u : 0u) | (sl[1] >= 0 ? 1u << 8 : 0u) |
                               (sl[2] >= 0 ? 1u << 16 : 0u) | (sl[3] >= 0 ? 1u << 24 : 0u);
        *reinterpret_cast<uint32_t *>(in_row + r0) = bytes;
      } else {
        for (int q = 0; q < 4 && r0 + q < R; ++q) {
          slot_row[r0 + q] = sl[q];
          in_row[r0 + q] = sl[q] >= 0 ? 1 : 0;
        }
      }
    }
  }
  if (tid == 0) EP_TRACE_MARK(g_trace_layout, 5);
  if constexpr (!SCAN) return;

  // The last block: bases.  Thread (q, r) owns a contiguous run of blocks
  // for rank r; run sums, then their exclusive scan, then the running bases.
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int per_rank = kLayoutThreads / R;  // >= 4 since R <= 64
  const int run_len = (G + per_rank - 1) / per_rank;
  const int q = tid / R, r = tid % R;
  const bool owner = tid < per_rank * R;
  const int b0 = min(q * run_len, G), b1 = min(b0 + run_len, G);
  if (owner) {
    int sum = 0;
    for (int bb = b0; bb < b1; ++bb) sum += __ldcg(&p.partial[(size_t)bb * R + r]);
    seg_sum[tid] = sum;
  }
  __syncthreads();
  if (tid == 0) EP_TRACE_MARK(g_trace_layout, 6);
  for (int rr = tid; rr < R; rr += kLayoutThreads) {
    int all = 0;
    for (int qq = 0; qq < per_rank; ++qq) all += seg_sum[qq * R + rr];
    tot[rr] = all;
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int rr = 0; rr < R; ++rr) {
      base[rr] = acc;
      acc += tot[rr];
    }
    base[R] = acc;
  }
  __syncthreads();
  for (int rr = tid; rr <= R; rr += kLayoutThreads) {
    p.out.rank_prefix[rr] = base[rr];
    if (rr < R) p.out.num_tokens_per_rank[rr] = tot[rr];
  }
  if (owner) {
    int run = base[r];
    for (int qq = 0; qq < q; ++qq) run += seg_sum[qq * R + r];
    for (int bb = b0; bb < b1; ++bb) {
      const int v = __ldcg(&p.partial[(size_t)bb * R + r]);
      p.partial[(size_t)bb * R + r] = run;
      run += v;
    }
  }
  if (tid == 0) *done = 0u;
  if (tid == 0) EP_TRACE_MARK(g_trace_layout, 7);
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

size_t layout_workspace_bytes_used(int num_tokens, int num_ranks) {
  const int grid = std::min(max_layout_blocks(num_tokens), kMaxLayoutBlocks);
  const size_t partial = (size_t)grid * (size_t)num_ranks * sizeof(int32_t);
  return kPartialOffset + ((partial + 255) / 256) * 256;
}

ep_status_t launch_layout(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                          int num_ranks, const ep_layout_t &layout, void *workspace,
                          cudaStream_t stream) {
  // One block per 256 tokens, at most kMaxLayoutBlocks (then more tokens per
  // block): every slot block scans all blocks' totals.
  LayoutParams p;
  const int grid = std::min(max_layout_blocks(num_tokens), kMaxLayoutBlocks);
  p.topk_idx = topk_idx;
  p.num_tokens = num_tokens;
  p.num_topk = num_topk;
  p.num_experts = num_experts;
  p.num_ranks = num_ranks;
  p.experts_per_rank = num_experts / num_ranks;
  p.tokens_per_block = (num_tokens + grid - 1) / grid;
  p.out = layout;
  p.partial = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(workspace) + kPartialOffset);
  const bool wide = num_topk > 8;
  cudaError_t e = wide ? launch_kernel(layout_count_kernel<EP_MAX_TOPK>, grid, kLayoutThreads, 0, stream, false, p)
                       : launch_kernel(layout_count_kernel<8>, grid, kLayoutThreads, 0, stream, false, p);
  if (e != cudaSuccess) return cuda_fail(e, "launch layout_count_kernel");
  const size_t smem = slot_smem_bytes(num_experts, num_ranks);
  e = wide ? launch_kernel(layout_slot_kernel<EP_MAX_TOPK>, grid, kLayoutThreads, smem, stream, false, p)
           : launch_kernel(layout_slot_kernel<8>, grid, kLayoutThreads, smem, stream, false, p);
  if (e != cudaSuccess) return cuda_fail(e, "launch layout_slot_kernel");
  return EP_OK;
}

int local_layout_max_tokens() { return kMaxLayoutBlocks * kLocalTokensPerBlock; }

ep_status_t launch_layout_local(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                                int num_ranks, const ep_layout_t &layout, void *workspace, cudaStream_t stream,
                                const int32_t **local_base, int *table_blocks) {
  static_assert(kLocalTokensPerBlock == kLayoutThreads, "one token per thread");
  LayoutParams p;
  const int grid = (num_tokens + kLocalTokensPerBlock - 1) / kLocalTokensPerBlock;
  p.topk_idx = topk_idx;
  p.num_tokens = num_tokens;
  p.num_topk = num_topk;
  p.num_experts = num_experts;
  p.num_ranks = num_ranks;
  p.experts_per_rank = num_experts / num_ranks;
  p.tokens_per_block = kLocalTokensPerBlock;
  p.out = layout;
  p.partial = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(workspace) + kPartialOffset);
  uint32_t *done = static_cast<uint32_t *>(workspace);  // zero between calls
  // A small table of block totals is scanned by the dispatch itself: no
  // fence, ticket or last-block pass on the path the dispatch waits for.
  const bool table = (size_t)grid * (size_t)num_ranks <= (size_t)kBaseTableMax;
  const bool wide = num_topk > 8;
  cudaError_t e;
  if (table)
    e = wide ? launch_kernel(layout_local_kernel<EP_MAX_TOPK, false>, grid, kLayoutThreads, 0, stream, false, p, done)
             : launch_kernel(layout_local_kernel<8, false>, grid, kLayoutThreads, 0, stream, false, p, done);
  else
    e = wide ? launch_kernel(layout_local_kernel<EP_MAX_TOPK, true>, grid, kLayoutThreads, 0, stream, false, p, done)
             : launch_kernel(layout_local_kernel<8, true>, grid, kLayoutThreads, 0, stream, false, p, done);
  if (e != cudaSuccess) return cuda_fail(e, "launch layout_local_kernel");
  *local_base = p.partial;
  *table_blocks = table ? grid : 0;
  return EP_OK;
}

}  // namespace ep

EP_TRACE_READER(ep_trace_read_layout, ep::g_trace_layout);
