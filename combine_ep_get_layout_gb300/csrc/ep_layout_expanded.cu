// Expanded layout kernel: one received row per (token, expert) selection,
// grouped by expert, each expert's segment rounded up to expert_alignment
// rows -- DeepEP's do_expand as TileScale PR #68 ("[Example] EP v2 intranode
// dispatch/combine", commit message on do_expand) builds it: phase 1 tallies
// per destination, phase 2 turns tallies into a base (the exclusive prefix
// sum of aligned counts), phase 3 adds a locally claimed slot -- with the
// destination redefined from rank to expert.
//
//   phase 1  a block owns a contiguous range of tokens, one token per thread
//            per chunk.  A thread keeps the first occurrence of each expert of
//            its token (a repeat sets EP_ERRBIT_DUP_EXPERT and gets no row)
//            and sets its lane's bit in its warp's 32-bit token mask of that
//            expert (shared memory).  The row's rank inside the block is the
//            block's running count of the expert, plus the popcounts of the
//            lower warps' masks, plus the popcount of the lower lanes of its
//            own: ascending (token, k) order.  It is parked in token_slot.
//   exchange per-block expert totals go to global memory; a bounded grid
//            barrier (cooperative launch) lets every block read them all.
//   phase 2  per expert: the earlier blocks' rows and the total; the aligned
//            totals are scanned (block-wide) into the segment starts; every
//            parked rank becomes start + earlier rows + rank.
#include <algorithm>
#include <mutex>

#include "ep_device.cuh"

namespace ep {
namespace {

constexpr int kXThreads = 256;
constexpr int kXWarps = kXThreads / kWarpSize;
constexpr size_t kXPartialOffset = 256;

struct XLayoutParams {
  const int64_t *topk_idx;
  int T, K, E, align;
  int tokens_per_block;
  ep_expanded_layout_t out;
  GridBarrierWords *bar;
  int32_t *partial;  // [gridDim.x * E]
};

size_t xlayout_smem_bytes(int E) {
  // wmask[W][E] u32, run[E], before[E], start[E+1], scan[kXThreads], flags[4]
  return ((size_t)kXWarps * E + E + E + (E + 1) + kXThreads + 4) * sizeof(int32_t);
}

template <int KMAX>
__global__ void __launch_bounds__(kXThreads) layout_expanded_kernel(XLayoutParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x;
  const int lane = tid & (kWarpSize - 1);
  const int warp = tid / kWarpSize;
  const int G = gridDim.x;
  const int b = blockIdx.x;
  const int E = p.E, K = p.K;

  uint32_t *wmask = reinterpret_cast<uint32_t *>(smem);  // [kXWarps][E]
  int *run = reinterpret_cast<int *>(wmask + (size_t)kXWarps * E);
  int *before = run + E;
  int *start = before + E;  // [E + 1]
  int *scan = start + E + 1;  // [kXThreads]
  int *flags = scan + kXThreads;  // [0] bad id, [1] repeat, [2] timeout, [3] barrier scratch

  for (int i = tid; i < kXWarps * E; i += kXThreads) wmask[i] = 0u;
  for (int i = tid; i < E; i += kXThreads) run[i] = 0;
  if (tid < 4) flags[tid] = 0;
  griddep_wait();
  griddep_launch_dependents();
  if (b == 0 && tid == 0) *p.out.error_word = 0u;
  if (b == 0 && tid < EP_WORK_COUNTER_WORDS && p.out.work_counters != nullptr) p.out.work_counters[tid] = 0u;
  __syncthreads();

  const int begin = min(b * p.tokens_per_block, p.T);
  const int end = min(begin + p.tokens_per_block, p.T);
  const uint32_t lanes_below = (1u << lane) - 1u;
  bool bad = false, repeat = false;

  // ---- phase 1: ranks inside the block
  for (int c0 = begin; c0 < end; c0 += kXThreads) {
    const int t = c0 + tid;
    int64_t ids[KMAX];
    bool first[KMAX];
    if (t < end) {
      const int64_t *row = p.topk_idx + (size_t)t * K;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) ids[k] = k < K ? __ldg(row + k) : -1;
    } else {
#pragma unroll
      for (int k = 0; k < KMAX; ++k) ids[k] = -1;
    }
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      const int64_t e = ids[k];
      bool f = e >= 0 && e < E;
      if (e != -1 && !f) bad = true;
#pragma unroll
      for (int j = 0; j < k; ++j)
        if (f && ids[j] == e) f = false;
      if (e >= 0 && e < E && !f) repeat = true;
      first[k] = f;
      if (f) atomicOr(&wmask[(size_t)warp * E + (int)e], 1u << lane);
    }
    __syncthreads();
    if (t < end) {
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k >= K) break;
        int rank = -1;
        if (first[k]) {
          const int e = static_cast<int>(ids[k]);
          rank = run[e] + __popc(wmask[(size_t)warp * E + e] & lanes_below);
          for (int w = 0; w < warp; ++w) rank += __popc(wmask[(size_t)w * E + e]);
        }
        p.out.token_slot[(size_t)t * K + k] = rank;  // parked: the rank inside the block
      }
    }
    __syncthreads();
    for (int e = tid; e < E; e += kXThreads) {
      int cnt = 0;
      for (int w = 0; w < kXWarps; ++w) {
        cnt += __popc(wmask[(size_t)w * E + e]);
        wmask[(size_t)w * E + e] = 0u;
      }
      run[e] += cnt;
    }
    __syncthreads();
  }
  if (bad) flags[0] = 1;
  if (repeat) flags[1] = 1;
  for (int e = tid; e < E; e += kXThreads) p.partial[(size_t)b * E + e] = run[e];

  // ---- exchange
  __threadfence();
  if (!grid_barrier(p.bar, &flags[3]) && tid == 0) flags[2] = 1;

  // ---- phase 2: totals, earlier blocks' rows, aligned segment starts
  for (int e = tid; e < E; e += kXThreads) {
    int all = 0, earlier = 0;
#pragma unroll 8
    for (int bb = 0; bb < G; ++bb) {
      const int v = __ldcg(&p.partial[(size_t)bb * E + e]);
      all += v;
      earlier += bb < b ? v : 0;
    }
    run[e] = all;  // now: the expert's total
    before[e] = earlier;
  }
  __syncthreads();
  // exclusive scan of the aligned totals: each thread a contiguous run of
  // experts, then a scan of the per-thread sums
  const int per = (E + kXThreads - 1) / kXThreads;
  const int e0 = min(tid * per, E), e1 = min(e0 + per, E);
  int mine = 0;
  for (int e = e0; e < e1; ++e) mine += (run[e] + p.align - 1) / p.align * p.align;
  int incl = mine;  // inclusive scan inside the warp, then over the warps' totals
#pragma unroll
  for (int off = 1; off < kWarpSize; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == kWarpSize - 1) scan[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int w = 0; w < kXWarps; ++w) {
      const int v = scan[w];
      scan[w] = acc;
      acc += v;
    }
    start[E] = acc;
  }
  __syncthreads();
  {
    int acc = scan[warp] + incl - mine;
    for (int e = e0; e < e1; ++e) {
      start[e] = acc;
      acc += (run[e] + p.align - 1) / p.align * p.align;
    }
  }
  __syncthreads();
  if (b == 0) {
    for (int e = tid; e <= E; e += kXThreads) {
      p.out.expert_offset[e] = start[e];
      if (e < E) p.out.num_rows_per_expert[e] = run[e];
    }
  }
  if (tid == 0) {
    const uint32_t bits = (flags[0] ? EP_ERRBIT_BAD_INDEX : 0u) | (flags[1] ? EP_ERRBIT_DUP_EXPERT : 0u) |
                          (flags[2] ? EP_ERRBIT_TIMEOUT : 0u);
    if (bits) atomicOr(p.out.error_word, bits);
  }
  for (int e = tid; e < E; e += kXThreads) before[e] += start[e];  // the block's first row of e
  __syncthreads();

  // ---- phase 2: final slots
  for (int c0 = begin; c0 < end; c0 += kXThreads) {
    const int t = c0 + tid;
    if (t >= end) continue;
    for (int k = 0; k < K; ++k) {
      int32_t *slot = p.out.token_slot + (size_t)t * K + k;
      const int rank = *slot;
      if (rank >= 0) *slot = before[static_cast<int>(__ldg(p.topk_idx + (size_t)t * K + k))] + rank;
    }
  }
  grid_barrier_exit(p.bar);
}

int max_xlayout_blocks(int num_tokens) { return std::max(1, (num_tokens + kXThreads - 1) / kXThreads); }

}  // namespace

size_t expanded_layout_workspace_bytes(int num_tokens, int num_experts) {
  const size_t partial = (size_t)max_xlayout_blocks(num_tokens) * (size_t)num_experts * sizeof(int32_t);
  return kXPartialOffset + ((partial + 255) / 256) * 256;
}

ep_status_t launch_layout_expanded(const int64_t *topk_idx, int num_tokens, int num_topk, int num_experts,
                                   int expert_alignment, const ep_expanded_layout_t &layout, void *workspace,
                                   cudaStream_t stream) {
  const DeviceInfo *di = current_device_info();
  if (di == nullptr) return EP_ERR_CUDA;
  const auto kernel = num_topk <= 8 ? layout_expanded_kernel<8> : layout_expanded_kernel<EP_MAX_TOPK>;
  static std::mutex mu;
  static bool configured[64] = {};
  {
    std::lock_guard<std::mutex> g(mu);
    if (di->device < 64 && !configured[di->device]) {
      for (auto k : {layout_expanded_kernel<8>, layout_expanded_kernel<EP_MAX_TOPK>}) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)di->max_smem_per_block_optin);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(layout_expanded_kernel)");
      }
      configured[di->device] = true;
    }
  }
  const size_t smem = xlayout_smem_bytes(num_experts);
  if (smem > di->max_smem_per_block_optin)
    return fail(EP_ERR_UNSUPPORTED, "ep_get_layout_expanded: %d experts need %zu bytes of shared memory",
                num_experts, smem);
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kXThreads, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(layout_expanded)");
  if (per_sm <= 0) return fail(EP_ERR_UNSUPPORTED, "ep_get_layout_expanded: kernel cannot be resident");
  const int grid = std::min(max_xlayout_blocks(num_tokens), per_sm * di->num_sms);

  XLayoutParams p;
  p.topk_idx = topk_idx;
  p.T = num_tokens;
  p.K = num_topk;
  p.E = num_experts;
  p.align = expert_alignment;
  p.tokens_per_block = (num_tokens + grid - 1) / grid;
  p.out = layout;
  p.bar = static_cast<GridBarrierWords *>(workspace);
  p.partial = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(workspace) + kXPartialOffset);
  e = launch_kernel(kernel, grid, kXThreads, smem, stream, true, p);
  if (e != cudaSuccess) return cuda_fail(e, "launch layout_expanded_kernel");
  return EP_OK;
}

}  // namespace ep
