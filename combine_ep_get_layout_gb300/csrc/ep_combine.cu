// Combine kernel: the local reduce of TileScale PR #68 ("[Example] EP v2
// intranode dispatch/combine", PR summary: one block per source token reduces
// the rows stored back for it).  On one GPU the store-back slot
// comm_x[rank][src_token] is the received row token_slot[t][r] itself, so the
// kernel gathers straight from the expert stage's output y.
//
// A CTA takes tokens t = blockIdx.x + i * gridDim.x.  Warp 0 compacts the
// token's valid (rank, slot) pairs in ascending rank order into shared memory
// together with the rank's coefficient (1, or the fp32 sum in k order of the
// token's gate weights on that rank).  Then every thread owns 16-byte columns
// of the row: it issues the loads of up to 8 rank rows at once and only then
// accumulates them, in ascending rank order, in fp32 with separate multiply
// and add, and stores the bf16 result rounded to nearest even.
#include <algorithm>

#include "ep_device.cuh"

namespace ep {
namespace {

constexpr int kCombineThreads = 128;
constexpr int kRowsPerBatch = 8;

struct CombineParams {
  const uint16_t *y;
  int cap, H, T, R, K, E, epr;
  const int32_t *token_slot;
  uint32_t *error_word;
  const int64_t *topk_idx;
  const float *topk_weights;
  uint16_t *out;
};

template <bool WEIGHTED>
__device__ __forceinline__ void accumulate(float (&acc)[8], int4 v, float c) {
  const uint32_t w[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float lo = bf16_lo(w[q]);
    const float hi = bf16_hi(w[q]);
    if constexpr (WEIGHTED) {
      acc[2 * q] = __fadd_rn(acc[2 * q], __fmul_rn(c, lo));
      acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], __fmul_rn(c, hi));
    } else {
      acc[2 * q] = __fadd_rn(acc[2 * q], lo);
      acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], hi);
    }
  }
}

template <bool WEIGHTED>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineParams p) {
  __shared__ int32_t s_slot[2][EP_MAX_RANKS];
  __shared__ float s_coef[2][EP_MAX_RANKS];
  __shared__ int s_n[2];

  const int tid = threadIdx.x;
  const int lane = tid & (kWarpSize - 1);
  const int warp = tid / kWarpSize;
  const int ncol = p.H / 8;  // 16-byte columns
  const uint32_t lanes_below = (1u << lane) - 1u;

  int i = 0;
  for (int t = blockIdx.x; t < p.T; t += gridDim.x, ++i) {
    const int b = i & 1;
    if (warp == 0) {
      int count = 0;
      for (int r0 = 0; r0 < p.R; r0 += kWarpSize) {
        const int r = r0 + lane;
        int slot = -1;
        float c = 1.0f;
        if (r < p.R) {
          slot = __ldg(p.token_slot + (size_t)t * p.R + r);
          if (slot >= p.cap) {
            set_error(p.error_word, EP_ERRBIT_CAPACITY);
            slot = -1;
          }
          if (WEIGHTED && slot >= 0) {
            c = 0.0f;
            for (int k = 0; k < p.K; ++k) {
              const int64_t e = __ldg(p.topk_idx + (size_t)t * p.K + k);
              if (e >= 0 && e < p.E && static_cast<int>(e) / p.epr == r)
                c = __fadd_rn(c, __ldg(p.topk_weights + (size_t)t * p.K + k));
            }
          }
        }
        const uint32_t bal = __ballot_sync(0xffffffffu, slot >= 0);
        if (slot >= 0) {
          const int pos = count + __popc(bal & lanes_below);
          s_slot[b][pos] = slot;
          s_coef[b][pos] = c;
        }
        count += __popc(bal);
      }
      if (lane == 0) s_n[b] = count;
    }
    __syncthreads();

    const int n = s_n[b];
    uint16_t *out_row = p.out + (size_t)t * p.H;
    for (int col = tid; col < ncol; col += kCombineThreads) {
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
      for (int j0 = 0; j0 < n; j0 += kRowsPerBatch) {
        int4 v[kRowsPerBatch];
#pragma unroll
        for (int q = 0; q < kRowsPerBatch; ++q)
          if (j0 + q < n) v[q] = ld_stream_v4(p.y + (size_t)s_slot[b][j0 + q] * p.H + (size_t)col * 8);
#pragma unroll
        for (int q = 0; q < kRowsPerBatch; ++q)
          if (j0 + q < n) accumulate<WEIGHTED>(acc, v[q], s_coef[b][j0 + q]);
      }
      int4 o;
      o.x = (int)pack_bf16x2(acc[0], acc[1]);
      o.y = (int)pack_bf16x2(acc[2], acc[3]);
      o.z = (int)pack_bf16x2(acc[4], acc[5]);
      o.w = (int)pack_bf16x2(acc[6], acc[7]);
      st_stream_v4(out_row + (size_t)col * 8, o);
    }
    // s_slot[b] is rewritten two tokens later, after the next barrier.
  }
}

template <bool WEIGHTED>
ep_status_t launch_impl(const CombineParams &p, const DeviceInfo &di, cudaStream_t stream) {
  int per_sm = 0;
  cudaError_t e =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel<WEIGHTED>, kCombineThreads, 0);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(combine)");
  if (per_sm <= 0) return fail(EP_ERR_UNSUPPORTED, "ep_combine: kernel cannot be resident");
  const int grid = std::min(p.T, per_sm * di.num_sms);
  combine_kernel<WEIGHTED><<<grid, kCombineThreads, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch combine_kernel");
  return EP_OK;
}

}  // namespace

ep_status_t launch_combine(const CombineArgs &a, cudaStream_t stream) {
  if (a.num_tokens == 0) return EP_OK;
  const DeviceInfo *di = current_device_info();
  if (di == nullptr) return EP_ERR_CUDA;
  CombineParams p;
  p.y = a.y;
  p.cap = a.recv_capacity;
  p.H = a.hidden;
  p.T = a.num_tokens;
  p.R = a.num_ranks;
  p.K = a.num_topk;
  p.E = a.num_experts;
  p.epr = (a.topk_weights != nullptr) ? a.num_experts / a.num_ranks : 1;
  p.token_slot = a.token_slot;
  p.error_word = a.error_word;
  p.topk_idx = a.topk_idx;
  p.topk_weights = a.topk_weights;
  p.out = a.out;
  return a.topk_weights != nullptr ? launch_impl<true>(p, *di, stream) : launch_impl<false>(p, *di, stream);
}

}  // namespace ep
