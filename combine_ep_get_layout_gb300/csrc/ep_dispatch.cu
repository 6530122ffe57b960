// Dispatch kernel: the scatter phase of TileScale PR #68 ("[Example] EP v2
// intranode dispatch/combine", PR summary: rows go straight to their final
// compact index, no copy epilogue), with the per-token, per-128-element fp8
// cast fused into the same pass (same page, commit message on packing the
// fp8 row; DeepEP's per_token_cast_to_fp8 layout).
//
// One CTA works through its tokens (t = blockIdx.x + i * gridDim.x) with a
// ring of `stages` shared-memory row buffers:
//   - a bulk (TMA 1D) copy brings token i's bf16 row into its stage, signalled
//     on an mbarrier; loads run `stages - 1` tokens ahead;
//   - bf16: warp 0 issues one bulk store of the stage per destination rank,
//     straight to recv_x[token_slot[t][r]];
//   - fp8: every warp casts 128-element groups (amax by warp shuffles,
//     scale = amax / 448, e4m3 round-to-nearest-even with saturation) into a
//     double-buffered output row, then warp 0 bulk-stores it per destination;
//   - the other warps write the received metadata (source token, local expert
//     ids, gate weights) and, for fp8, the scales.
// Each row of x is read from HBM once and written once per destination rank.
#include <algorithm>
#include <mutex>

#include "ep_device.cuh"

namespace ep {
namespace {

constexpr int kDispatchThreads = 256;
constexpr int kDispatchWarps = kDispatchThreads / kWarpSize;
constexpr int kMaxStages = 8;
constexpr int kHeaderBytes = 1024;  // mbarriers, flags, slot buffers
constexpr size_t kSmemBudget = 80 * 1024;  // per CTA: aims at >= 2-3 CTAs per SM

struct DispatchParams {
  const uint16_t *x;
  int T, H, K, E, R, epr, groups;
  const int64_t *topk_idx;
  const float *topk_weights;
  const int32_t *token_slot;
  uint32_t *error_word;
  void *recv_x;
  float *recv_x_scales;
  int32_t *recv_src_idx;
  int32_t *recv_topk_idx;
  float *recv_topk_weights;
  int cap;
  int stages;
  uint32_t row_in_bytes;   // 2H
  uint32_t row_out_bytes;  // 2H (bf16) or H (fp8)
  uint32_t stage_stride;   // row_in_bytes rounded up to 128
  uint32_t out_stride;     // fp8 output row, H rounded up to 128
  uint32_t scale_stride;   // fp8 scales of one row, groups*4 rounded up to 16
};

__device__ __forceinline__ void issue_row_load(const DispatchParams &p, unsigned char *stages,
                                               uint64_t *full, int i, uint64_t policy) {
  const int t = blockIdx.x + i * gridDim.x;
  const int s = i % p.stages;
  mbar_arrive_expect_tx(&full[s], p.row_in_bytes);
  bulk_load_hint(stages + (size_t)s * p.stage_stride, p.x + (size_t)t * p.H, p.row_in_bytes,
                 &full[s], policy);
}

// Received metadata of token t, by threads [32, blockDim): source token,
// local expert ids and gate weights of every row the token is sent as, and
// for fp8 the row's scales.
template <bool FP8>
__device__ __forceinline__ void write_metadata(const DispatchParams &p, int t,
                                               const int32_t *slots, const float *scales) {
  const int mt = threadIdx.x - kWarpSize;
  const int nt = kDispatchThreads - kWarpSize;
  if (p.recv_src_idx != nullptr) {
    for (int j = mt; j < p.R; j += nt) {
      const int slot = slots[j];
      if (slot >= 0 && slot < p.cap) p.recv_src_idx[slot] = t;
    }
  }
  if (p.recv_topk_idx != nullptr || p.recv_topk_weights != nullptr) {
    const int RK = p.R * p.K;
    for (int q = mt; q < RK; q += nt) {
      const int j = q / p.K;
      const int k = q - j * p.K;
      const int slot = slots[j];
      if (slot < 0 || slot >= p.cap) continue;
      const int64_t e = __ldg(p.topk_idx + (size_t)t * p.K + k);
      const bool here = e >= 0 && e < p.E && static_cast<int>(e) / p.epr == j;
      if (p.recv_topk_idx != nullptr)
        p.recv_topk_idx[(size_t)slot * p.K + k] = here ? static_cast<int>(e) - j * p.epr : -1;
      if (p.recv_topk_weights != nullptr)
        p.recv_topk_weights[(size_t)slot * p.K + k] =
            here ? __ldg(p.topk_weights + (size_t)t * p.K + k) : 0.0f;
    }
  }
  if constexpr (FP8) {
    const int RG = p.R * p.groups;
    for (int q = mt; q < RG; q += nt) {
      const int j = q / p.groups;
      const int g = q - j * p.groups;
      const int slot = slots[j];
      if (slot >= 0 && slot < p.cap) p.recv_x_scales[(size_t)slot * p.groups + g] = scales[g];
    }
  }
}

template <bool FP8>
__global__ void __launch_bounds__(kDispatchThreads) dispatch_kernel(DispatchParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);               // [kMaxStages]
  int *s_abort = reinterpret_cast<int *>(smem + 64);
  int32_t *s_slot = reinterpret_cast<int32_t *>(smem + 128);         // [2][EP_MAX_RANKS]
  unsigned char *stages = smem + kHeaderBytes;
  unsigned char *obuf = stages + (size_t)p.stages * p.stage_stride;  // fp8: [2][out_stride]
  float *sbuf = reinterpret_cast<float *>(obuf + 2 * (size_t)p.out_stride);  // fp8: [2][groups]

  const int tid = threadIdx.x;
  const int warp = tid / kWarpSize;
  const int lane = tid & (kWarpSize - 1);
  const int S = p.stages;
  const int n = (p.T > (int)blockIdx.x) ? (p.T - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const uint64_t policy = policy_evict_first();  // x is read exactly once
  int loads_issued = 0;                           // meaningful in thread 0 only
  if (tid == 0)
    for (; loads_issued < min(S, n); ++loads_issued) issue_row_load(p, stages, full, loads_issued, policy);

  int i = 0;
  for (; i < n; ++i) {
    const int t = blockIdx.x + i * gridDim.x;
    const int s = i % S;
    const uint32_t parity = (uint32_t)(i / S) & 1u;
    const int b = i & 1;
    int32_t *slots = s_slot + b * EP_MAX_RANKS;
    unsigned char *stage = stages + (size_t)s * p.stage_stride;

    if (tid < p.R) slots[tid] = __ldg(p.token_slot + (size_t)t * p.R + tid);
    if constexpr (FP8) {
      // the stores of token i-2 read obuf[b]: let them finish reading it
      if (warp == 0) bulk_wait_read<1>();
    }
    __syncthreads();
    if (*s_abort) break;

    if constexpr (FP8) {
      if (!mbar_wait_bounded(&full[s], parity)) {
        *s_abort = 1;
        if (lane == 0) set_error(p.error_word, EP_ERRBIT_TIMEOUT);
      }
      unsigned char *orow = obuf + (size_t)b * p.out_stride;
      float *srow = sbuf + (size_t)b * (p.scale_stride / 4);
      for (int g = warp; g < p.groups; g += kDispatchWarps) {
        const uint2 raw = *reinterpret_cast<const uint2 *>(stage + (size_t)g * 256 + lane * 8);
        const float v0 = bf16_lo(raw.x), v1 = bf16_hi(raw.x);
        const float v2 = bf16_lo(raw.y), v3 = bf16_hi(raw.y);
        float a = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        const float scale = __fdiv_rn(a, 448.0f);
        const bool nz = a > 0.0f;  // an all-zero group keeps each zero's sign
        const float u0 = nz ? __fdiv_rn(v0, scale) : v0;
        const float u1 = nz ? __fdiv_rn(v1, scale) : v1;
        const float u2 = nz ? __fdiv_rn(v2, scale) : v2;
        const float u3 = nz ? __fdiv_rn(v3, scale) : v3;
        *reinterpret_cast<uint32_t *>(orow + (size_t)g * 128 + lane * 4) =
            pack_e4m3x2(u0, u1) | (pack_e4m3x2(u2, u3) << 16);
        if (lane == 0) srow[g] = scale;
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (*s_abort) break;
      if (warp == 0) {
        if (lane == 0 && i + S < n) issue_row_load(p, stages, full, loads_issued++, policy);
        for (int j = lane; j < p.R; j += kWarpSize) {
          const int slot = slots[j];
          if (slot < 0) continue;
          if (slot < p.cap)
            bulk_store(static_cast<unsigned char *>(p.recv_x) + (size_t)slot * p.row_out_bytes, orow,
                       p.row_out_bytes);
          else
            set_error(p.error_word, EP_ERRBIT_CAPACITY);
        }
        bulk_commit();
      } else {
        write_metadata<true>(p, t, slots, srow);
      }
    } else {
      if (warp == 0) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], parity));
        if (!ok) {
          if (lane == 0) {
            *s_abort = 1;
            set_error(p.error_word, EP_ERRBIT_TIMEOUT);
          }
        } else {
          for (int j = lane; j < p.R; j += kWarpSize) {
            const int slot = slots[j];
            if (slot < 0) continue;
            if (slot < p.cap)
              bulk_store(static_cast<unsigned char *>(p.recv_x) + (size_t)slot * p.row_out_bytes,
                         stage, p.row_out_bytes);
            else
              set_error(p.error_word, EP_ERRBIT_CAPACITY);
          }
          bulk_commit();
          // the stores of token i-1 have read their stage: reload it
          bulk_wait_read<1>();
          __syncwarp();
          if (lane == 0 && i >= 1 && i - 1 + S < n) issue_row_load(p, stages, full, loads_issued++, policy);
        }
      } else {
        write_metadata<false>(p, t, slots, nullptr);
      }
    }
  }

  // Drain: stores must finish reading shared memory before the CTA exits;
  // after an abort, loads still in flight are waited for (bounded).
  if (warp == 0) bulk_wait<0>();
  __syncthreads();
  if (*s_abort && tid == 0) {
    for (int m = i; m < loads_issued; ++m) (void)mbar_wait_bounded(&full[m % S], (uint32_t)(m / S) & 1u);
  }
}

size_t dispatch_smem_bytes(const DispatchParams &p, bool fp8) {
  size_t bytes = kHeaderBytes + (size_t)p.stages * p.stage_stride;
  if (fp8) bytes += 2 * (size_t)p.out_stride + 2 * (size_t)p.scale_stride;
  return bytes;
}

template <bool FP8>
ep_status_t launch_impl(DispatchParams &p, const DeviceInfo &di, cudaStream_t stream) {
  static std::mutex mu;
  static bool configured[64] = {};
  {
    std::lock_guard<std::mutex> g(mu);
    if (di.device < 64 && !configured[di.device]) {
      cudaError_t e = cudaFuncSetAttribute(dispatch_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)di.max_smem_per_block_optin);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(dispatch_kernel)");
      configured[di.device] = true;
    }
  }
  // Deepest ring that keeps the CTA within budget (at least 2 stages).
  p.stages = kMaxStages > 4 ? 4 : kMaxStages;
  while (p.stages > 2 && dispatch_smem_bytes(p, FP8) > kSmemBudget) --p.stages;
  const size_t smem = dispatch_smem_bytes(p, FP8);
  if (smem > di.max_smem_per_block_optin)
    return fail(EP_ERR_UNSUPPORTED, "ep_dispatch: hidden %d needs %zu bytes of shared memory", p.H, smem);
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_kernel<FP8>,
                                                                kDispatchThreads, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(dispatch)");
  if (per_sm <= 0) return fail(EP_ERR_UNSUPPORTED, "ep_dispatch: kernel cannot be resident");
  const int grid = std::min(p.T, per_sm * di.num_sms);
  dispatch_kernel<FP8><<<grid, kDispatchThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch dispatch_kernel");
  return EP_OK;
}

}  // namespace

ep_status_t launch_dispatch(const DispatchArgs &a, cudaStream_t stream) {
  if (a.num_tokens == 0) return EP_OK;
  const DeviceInfo *di = current_device_info();
  if (di == nullptr) return EP_ERR_CUDA;
  DispatchParams p = {};
  p.x = a.x;
  p.T = a.num_tokens;
  p.H = a.hidden;
  p.K = a.num_topk;
  p.E = a.num_experts;
  p.R = a.num_ranks;
  p.epr = a.num_experts / a.num_ranks;
  p.groups = a.fp8 ? a.hidden / EP_FP8_GROUP : 0;
  p.topk_idx = a.topk_idx;
  p.topk_weights = a.topk_weights;
  p.token_slot = a.token_slot;
  p.error_word = a.error_word;
  p.recv_x = a.recv_x;
  p.recv_x_scales = a.recv_x_scales;
  p.recv_src_idx = a.recv_src_idx;
  p.recv_topk_idx = a.recv_topk_idx;
  p.recv_topk_weights = a.recv_topk_weights;
  p.cap = a.recv_capacity;
  p.row_in_bytes = 2u * (uint32_t)a.hidden;
  p.row_out_bytes = a.fp8 ? (uint32_t)a.hidden : 2u * (uint32_t)a.hidden;
  p.stage_stride = (p.row_in_bytes + 127u) / 128u * 128u;
  p.out_stride = a.fp8 ? ((uint32_t)a.hidden + 127u) / 128u * 128u : 0u;
  p.scale_stride = a.fp8 ? ((uint32_t)p.groups * 4u + 15u) / 16u * 16u : 0u;
  return a.fp8 ? launch_impl<true>(p, *di, stream) : launch_impl<false>(p, *di, stream);
}

}  // namespace ep
