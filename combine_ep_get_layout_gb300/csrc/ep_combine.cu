// Combine kernel: the local reduce of TileScale PR #68 ("[Example] EP v2
// intranode dispatch/combine", PR summary: one block per source token reduces
// the rows stored back for it).  On one GPU the store-back slot
// comm_x[rank][src_token] is the received row token_slot[t][r] itself, so the
// kernel gathers straight from the expert stage's output y.
//
// Two kernels: combine_ws_kernel (below, R <= 8) and combine_kernel, the
// register kernel, used for more ranks.
//
// combine_kernel: a CTA takes tokens t = blockIdx.x + i * gridDim.x.  Warp 0 compacts the
// token's valid (rank, slot) pairs in ascending rank order into shared memory
// together with the rank's coefficient (1, or the fp32 sum in k order of the
// token's gate weights on that rank).  Then every thread owns 16-byte columns
// of the row: it issues the loads of up to 8 rank rows at once and only then
// accumulates them, in ascending rank order, in fp32 with separate multiply
// and add, and stores the bf16 result rounded to nearest even.
#include <algorithm>
#include <mutex>

#include "ep_device.cuh"
#include "ep_trace.cuh"

namespace ep {
namespace {

constexpr int kCombineThreads = 128;
constexpr int kRowsPerBatch = 8;
constexpr int kCombineCols = 1;  // 16-byte columns per thread per pass

struct CombineParams {
  const uint16_t *y;
  int cap, H, T, R, K, E, epr;
  int D;          // destinations per token: R ranks, or K rows (expanded)
  bool expanded;  // token_slot is [T * K]: one row per (token, expert)
  const int32_t *token_slot;  // [T * D]
  uint32_t *error_word;
  const int64_t *topk_idx;
  const float *topk_weights;
  const uint16_t *bias0, *bias1;  // [T*H] or null: seed the accumulator
  uint16_t *out;
  TokenSource tokens;  // the order in which blocks take tokens (warp-specialised kernel)
};

// acc = bias0 (or 0), then acc = acc + bias1, for 8 consecutive elements.
__device__ __forceinline__ void seed(float (&acc)[8], const CombineParams &p, int4 b0, int4 b1) {
  const uint32_t w0[4] = {(uint32_t)b0.x, (uint32_t)b0.y, (uint32_t)b0.z, (uint32_t)b0.w};
  const uint32_t w1[4] = {(uint32_t)b1.x, (uint32_t)b1.y, (uint32_t)b1.z, (uint32_t)b1.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] = p.bias0 != nullptr ? bf16_lo(w0[q]) : 0.0f;
    acc[2 * q + 1] = p.bias0 != nullptr ? bf16_hi(w0[q]) : 0.0f;
    if (p.bias1 != nullptr) {
      acc[2 * q] = __fadd_rn(acc[2 * q], bf16_lo(w1[q]));
      acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], bf16_hi(w1[q]));
    }
  }
}

// PACKED: the adds as packed f32x2 adds (the same roundings, fewer issues).
template <bool WEIGHTED, bool PACKED = false>
__device__ __forceinline__ void accumulate(float (&acc)[8], int4 v, float c) {
  const uint32_t w[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float lo = bf16_lo(w[q]);
    const float hi = bf16_hi(w[q]);
    if constexpr (PACKED) {
      // The products stay scalar: a packed multiply feeding a packed add was
      // contracted into a fused multiply-add by the assembler (one rounding
      // instead of two; 603 of 16.8 M outputs differed by an ulp).
      if constexpr (WEIGHTED) add2_rn(acc[2 * q], acc[2 * q + 1], __fmul_rn(c, lo), __fmul_rn(c, hi));
      else add2_rn(acc[2 * q], acc[2 * q + 1], lo, hi);
    } else if constexpr (WEIGHTED) {
      acc[2 * q] = __fadd_rn(acc[2 * q], __fmul_rn(c, lo));
      acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], __fmul_rn(c, hi));
    } else {
      acc[2 * q] = __fadd_rn(acc[2 * q], lo);
      acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], hi);
    }
  }
}

// Warp-collective: the layout holds exactly this routing's rows (lane j:
// the slot of destination j; e: the expert of top-k slot lane, -1 past K).
__device__ __forceinline__ bool layout_agrees(const CombineParams &p, int64_t e, int slot_lo, int slot_hi,
                                              int lane) {
  return p.expanded ? choices_agree(e, p.E, p.K, slot_lo, lane)
                    : ranks_agree(e, p.E, p.epr, p.R, slot_lo, slot_hi, lane);
}

// Warp-collective: the coefficient of destination `lane`.  A rank row: the
// fp32 sum, in k order, of the weights of the token's experts on that rank.
// An expanded row: its own gate weight.
__device__ __forceinline__ float coefficient(const CombineParams &p, int64_t e_lane, float w_lane, int lane) {
  if (p.expanded) return w_lane;
  float coef = 0.0f;
  for (int k = 0; k < p.K; ++k) {
    const int64_t e = __shfl_sync(0xffffffffu, e_lane, k);
    const float w = __shfl_sync(0xffffffffu, w_lane, k);
    if (e >= 0 && e < p.E && static_cast<int>(e) / p.epr == lane) coef = __fadd_rn(coef, w);
  }
  return coef;
}

// Warp-collective: where destination `lane` goes among the token's rows
// (bal: the lanes with a row).  Rank rows in ascending rank (lane) order;
// expanded rows in ascending row order.
__device__ __forceinline__ int row_position(const CombineParams &p, int slot, uint32_t bal, uint32_t lanes_below) {
  if (!p.expanded) return __popc(bal & lanes_below);
  int pos = 0;
  for (int j = 0; j < p.D; ++j) {
    const int s = __shfl_sync(0xffffffffu, slot, j);
    pos += (s >= 0 && s < slot) ? 1 : 0;
  }
  return pos;
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
  griddep_wait();
  griddep_launch_dependents();

  int i = 0;
  for (int t = blockIdx.x; t < p.T; t += gridDim.x, ++i) {
    const int b = i & 1;
    if (warp == 0) {
      int count = 0;
      if (p.expanded) {  // one pass: K <= 32 rows, placed in ascending row order
        int slot = lane < p.D ? __ldg(p.token_slot + (size_t)t * p.D + lane) : -1;
        const int64_t e = (WEIGHTED && lane < p.K) ? __ldg(p.topk_idx + (size_t)t * p.K + lane) : -1;
        const float w = (WEIGHTED && lane < p.K) ? __ldg(p.topk_weights + (size_t)t * p.K + lane) : 0.0f;
        if (WEIGHTED && !layout_agrees(p, e, slot, -1, lane) && lane == 0)
          set_error(p.error_word, EP_ERRBIT_STALE_LAYOUT);
        if (slot >= p.cap) {
          set_error(p.error_word, EP_ERRBIT_CAPACITY);
          slot = -1;
        }
        const uint32_t bal = __ballot_sync(0xffffffffu, slot >= 0);
        const int pos = row_position(p, slot, bal, lanes_below);
        if (slot >= 0) {
          s_slot[b][pos] = slot;
          s_coef[b][pos] = WEIGHTED ? w : 1.0f;
        }
        count = __popc(bal);
      } else {
        if (WEIGHTED) {
          const int64_t e = lane < p.K ? __ldg(p.topk_idx + (size_t)t * p.K + lane) : -1;
          const int lo = lane < p.R ? __ldg(p.token_slot + (size_t)t * p.R + lane) : -1;
          const int hi = lane + kWarpSize < p.R ? __ldg(p.token_slot + (size_t)t * p.R + lane + kWarpSize) : -1;
          if (!ranks_agree(e, p.E, p.epr, p.R, lo, hi, lane) && lane == 0)
            set_error(p.error_word, EP_ERRBIT_STALE_LAYOUT);
        }
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
      }
      if (lane == 0) s_n[b] = count;
    }
    __syncthreads();

    const int n = s_n[b];
    uint16_t *out_row = p.out + (size_t)t * p.H;
    for (int col0 = tid; col0 < ncol; col0 += kCombineThreads * kCombineCols) {
      float acc[kCombineCols][8];
#pragma unroll
      for (int c = 0; c < kCombineCols; ++c) {
        const int col = col0 + c * kCombineThreads;
        const bool in = col < ncol;
        const int4 z = make_int4(0, 0, 0, 0);
        seed(acc[c], p, (in && p.bias0) ? ld_stream_v4(p.bias0 + (size_t)t * p.H + (size_t)col * 8) : z,
             (in && p.bias1) ? ld_stream_v4(p.bias1 + (size_t)t * p.H + (size_t)col * 8) : z);
      }
      for (int j0 = 0; j0 < n; j0 += kRowsPerBatch) {
        int4 v[kCombineCols][kRowsPerBatch];
#pragma unroll
        for (int c = 0; c < kCombineCols; ++c) {
          const int col = col0 + c * kCombineThreads;
#pragma unroll
          for (int q = 0; q < kRowsPerBatch; ++q)
            if (j0 + q < n && col < ncol)
              v[c][q] = ld_stream_v4(p.y + (size_t)s_slot[b][j0 + q] * p.H + (size_t)col * 8);
        }
#pragma unroll
        for (int c = 0; c < kCombineCols; ++c)
#pragma unroll
          for (int q = 0; q < kRowsPerBatch; ++q)
            if (j0 + q < n) accumulate<WEIGHTED>(acc[c], v[c][q], s_coef[b][j0 + q]);
      }
#pragma unroll
      for (int c = 0; c < kCombineCols; ++c) {
        const int col = col0 + c * kCombineThreads;
        if (col >= ncol) continue;
        int4 o;
        o.x = (int)pack_bf16x2(acc[c][0], acc[c][1]);
        o.y = (int)pack_bf16x2(acc[c][2], acc[c][3]);
        o.z = (int)pack_bf16x2(acc[c][4], acc[c][5]);
        o.w = (int)pack_bf16x2(acc[c][6], acc[c][7]);
        st_stream_v4(out_row + (size_t)col * 8, o);
      }
    }
    // s_slot[b] is rewritten two tokens later, after the next barrier.
  }
}

// ------------------------------------------------------------------------
// Warp-specialised kernel (R <= kWsMaxRanks).  A unit is one token's
// kChunk-element slice of the row; a CTA takes tokens from its TokenSource
// (a fixed stripe, or tickets from a grid-wide counter) and all units of a
// token in a row.  Each unit's stage header carries its token and the
// CTA's next token (so the reducers can prefetch that token's bias), and a
// unit with n = -1 ends the CTA's work.
//   warp 0 (loader)   fetches a token's slots, expert ids and weights one
//                     token ahead (lanes in parallel), forms each rank's
//                     coefficient by shuffles, compacts the valid ranks in
//                     ascending order into each unit's stage header and
//                     issues one bulk (TMA 1D) load per valid row slice into
//                     the stage (one mbarrier, expected bytes = rows x slice);
//   warps 1.. (reducers) sum the stage's rows in rank order, one 16-byte
//                     column per thread (fp32, separate multiply and add),
//                     store the bf16 result and release the stage.
// The loader runs `stages` units ahead, so the memory pipe does not wait on
// the per-token metadata or on the reduction.  A stage holds ROWS rows; with
// SPLIT, a token with more rows sends each chunk as two units, the second
// header flagged, and the reducers carry the partial sum from the first in
// registers (rows stay in ascending rank order, so the sum is unchanged).

// Trace build only (warp-specialised kernel): 0 entry, 1 past the wait for
// the kernel ahead, 2 the loader's first token drawn, 3 the reducers' first
// rows in, 4 the loader draws the end, 5 the reducers done, 6 (a count) the
// loader's draws.
EP_TRACE_ARRAY(g_trace_combine);

constexpr int kWsMaxRanks = 8;
constexpr int kSmallStageRows = 6;
constexpr int kSplitMinTokens = 32768;
// L2 warm-up before the grid-dependency wait: tokens per block, leading
// chunks of each of their rows
constexpr int kWarmTokens = 2;
constexpr int kWarmChunks = 1;
constexpr int kChunk = 2048;                   // elements per unit
constexpr int kChunkBytes = kChunk * 2;
constexpr int kReducers = 8;                   // warps
constexpr int kWsCombineThreads = (1 + kReducers) * kWarpSize;
constexpr int kCombineStages = 2;
constexpr int kStageHeader = 128;              // n, token, next token, carry flag; coefficients from 16

// A plain (write-back, L2-allocating) 16-byte store.
__device__ __forceinline__ void st_v4(void *p, int4 v) {
  asm volatile("st.global.v4.s32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// One token's routing as the loader warp holds it: lane r < R has the slot
// of rank r, lane k < K the k-th expert id and gate weight.  fetch_meta reads
// them through L2 only (ld.cg; each is read once: measured against the
// read-only path, headline step -0.3 us).
struct TokenMeta {
  int slot;
  int64_t e;
  float w;
};

__device__ __forceinline__ TokenMeta fetch_meta(const CombineParams &p, int t, int lane, bool weighted) {
  TokenMeta m;
  m.slot = lane < p.D ? __ldcg(p.token_slot + (size_t)t * p.D + lane) : -1;
  m.e = (weighted && lane < p.K) ? __ldcg(p.topk_idx + (size_t)t * p.K + lane) : -1;
  m.w = (weighted && lane < p.K) ? __ldcg(p.topk_weights + (size_t)t * p.K + lane) : 0.0f;
  return m;
}

// ROWS: the rows a stage holds, the most a token can have (6 when a
// routing of at most 6 experts per token is given: smaller stages, four
// blocks per SM; else kWsMaxRanks).
// SPLIT: a token with more rows than a stage holds goes as two units per
// chunk, the first carrying its sum on to the second (else a stage holds
// every row a token can have).
template <bool WEIGHTED, int ROWS, bool SPLIT>
__global__ void __launch_bounds__(kWsCombineThreads) combine_ws_kernel(CombineParams p) {
  constexpr int kStageBytes = kStageHeader + ROWS * kChunkBytes;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // [kCombineStages]
  uint64_t *empty = full + kCombineStages;              // [kCombineStages]
  volatile int *s_abort = reinterpret_cast<volatile int *>(smem + 64);
  unsigned char *stages = smem + 128;

  const int tid = threadIdx.x;
  const int warp = tid / kWarpSize;
  const int lane = tid & (kWarpSize - 1);
  const int nchunk = (p.H + kChunk - 1) / kChunk;  // a CTA takes all chunks of a token in a row
  if (tid == 0) EP_TRACE_MARK(g_trace_combine, 0);

  if (tid == 0) {
    for (int s = 0; s < kCombineStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kReducers);
    }
    *s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (kWarmTokens > 0 && warp == 1) {
    // Before the wait for the kernel ahead, nothing is read for its value:
    // the first tokens' metadata and the first chunks of their rows are only
    // brought into L2.  Block b's first token is b (with the split units,
    // the first tickets go to tokens 0, 1, ... in some order), so block b
    // warms tokens b, b + gridDim.x, ...  The slots read
    // here may be stale; they serve as addresses only, checked against the
    // capacity.  A reducer warp does it, so that the loader, when the kernel
    // ahead has already finished, draws its first token without waiting for
    // these slot reads.
    for (int k = 0; k < kWarmTokens; ++k) {
      const int t = (int)blockIdx.x + k * (int)gridDim.x;
      if (t >= p.T) break;
      const int slot = lane < p.D ? __ldcg(p.token_slot + (size_t)t * p.D + lane) : -1;
      if (lane == 0) {
        prefetch_l2(p.token_slot + (size_t)t * p.D);
        if (p.topk_idx != nullptr) prefetch_l2(p.topk_idx + (size_t)t * p.K);
        if (p.topk_weights != nullptr) prefetch_l2(p.topk_weights + (size_t)t * p.K);
      }
      if (slot >= 0 && slot < p.cap)
        bulk_prefetch_l2(p.y + (size_t)slot * p.H, (uint32_t)min(kWarmChunks * kChunk, p.H) * 2u);
    }
  }
  griddep_wait();
  griddep_launch_dependents();
  if (tid == 0) EP_TRACE_MARK(g_trace_combine, 1);

  const uint32_t lanes_below = (1u << lane) - 1u;
  long loads_issued = 0;  // loader lane 0: units issued (loads and the end)
  if (warp == 0) {
    bool drained = false;  // lane 0: no more tokens to draw
    // Each row of y is read once, so its lines go first when L2 needs room:
    // the combine's output lines then stay in L2 longer, and their write-back
    // overlaps the next kernel's start (measured 0.3-0.9 us a step faster;
    // with the split units, at 32 768 tokens and more, the plain policy was
    // as fast, so those keep it).
    const uint64_t y_policy = SPLIT ? 0 : policy_evict_first();
    // A block's first token is its own (blockIdx.x), no ticket: the
    // blocks are resident before the wait for the kernel ahead ends, and
    // the first loads then wait for the metadata only (measured: headline
    // step -0.25 us, bf16 -0.33 us, skewed -0.24 us).  With the split
    // units every token is drawn (65 536 tokens: +0.3 us with its own).
    constexpr int kOwnFirst = SPLIT ? 0 : 1;
    auto draw = [&](int j) {
      int t = 0;
      if (lane == 0) t = draw_token(p.tokens, j, drained, kOwnFirst);
      return __shfl_sync(0xffffffffu, t, 0);
    };
    long i = 0;  // unit counter: stage i % kCombineStages
    int t = draw(0);
    if (lane == 0) EP_TRACE_MARK(g_trace_combine, 2);
    TokenMeta cur = t >= 0 ? fetch_meta(p, t, lane, WEIGHTED) : TokenMeta{-1, -1, 0.0f};
    bool ok = true;
    for (int j = 1; ok && !*s_abort; ++j) {
      if (t < 0) {  // the end: a unit with n = -1 tells the reducers
        if (lane == 0) {
          EP_TRACE_MARK(g_trace_combine, 4);
          EP_TRACE_VALUE(g_trace_combine, 6, j);
        }
        const int s = static_cast<int>(i % kCombineStages);
        if (i >= kCombineStages)
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&empty[s], (uint32_t)(i / kCombineStages - 1) & 1u));
        if (ok && lane == 0) {
          *reinterpret_cast<int *>(stages + (size_t)s * kStageBytes) = -1;
          mbar_arrive(&full[s]);
          loads_issued = i + 1;
        }
        break;
      }
      // With more than one chunk a token, the next token is drawn once this
      // token's first unit is issued, and only the token's last unit names
      // it: a block then holds less drawn work when the tickets run out
      // (measured at two chunks, against drawing before the first unit:
      // bf16 step -0.2 us, skewed -0.55 us; at more chunks it also spares a
      // block's first loads a ticket's wait).  With one chunk the single
      // unit must name the next token, so that is drawn before it.
      const bool late = nchunk > 1;
      int t_next = late ? -1 : draw(j);
      TokenMeta nxt = t_next >= 0 ? fetch_meta(p, t_next, lane, WEIGHTED) : cur;  // in flight meanwhile
      int slot = cur.slot;
      if (WEIGHTED && !layout_agrees(p, cur.e, slot, -1, lane) && lane == 0)
        set_error(p.error_word, EP_ERRBIT_STALE_LAYOUT);
      if (slot >= p.cap) {
        set_error(p.error_word, EP_ERRBIT_CAPACITY);
        slot = -1;
      }
      const float coef = WEIGHTED ? coefficient(p, cur.e, cur.w, lane) : 1.0f;
      const uint32_t bal = __ballot_sync(0xffffffffu, slot >= 0);
      int nrows = __popc(bal);
      const int pos = row_position(p, slot, bal, lanes_below);
      constexpr int kMaxRows = SPLIT ? 2 * ROWS : ROWS;
      if (nrows > kMaxRows) {  // more ranks than the routing can reach: a layout of another routing
        if (lane == 0) set_error(p.error_word, EP_ERRBIT_STALE_LAYOUT);
        if (pos >= kMaxRows) slot = -1;
        nrows = kMaxRows;
      }
      const int parts = (SPLIT && nrows > ROWS) ? 2 : 1;
      for (int c = 0; c < nchunk && ok; ++c) {
        const int elems = min(kChunk, p.H - c * kChunk);
        for (int part = 0; part < parts; ++part, ++i) {
          const int s = static_cast<int>(i % kCombineStages);
          unsigned char *stage = stages + (size_t)s * kStageBytes;
          if (i >= kCombineStages) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(&empty[s], (uint32_t)(i / kCombineStages - 1) & 1u));
            if (!ok) break;
          }
          const int r0 = part * ROWS;
          const int n = min(nrows - r0, ROWS);
          const bool mine = slot >= 0 && pos >= r0 && pos < r0 + n;
          int *hdr = reinterpret_cast<int *>(stage);
          float *hdr_coef = reinterpret_cast<float *>(stage + 16);
          if (mine) hdr_coef[pos - r0] = coef;
          if (lane == 0) {
            hdr[0] = n;
            hdr[1] = t;
            hdr[2] = t_next;
            hdr[3] = part + 1 < parts ? 1 : 0;  // the sum goes on in the next unit
          }
          __syncwarp();
          if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)n * (uint32_t)elems * 2u);
          __syncwarp();
          if (mine) {
            void *dst = stage + kStageHeader + (size_t)(pos - r0) * kChunkBytes;
            const uint16_t *src = p.y + (size_t)slot * p.H + (size_t)c * kChunk;
            if constexpr (SPLIT)
              bulk_load(dst, src, (uint32_t)elems * 2u, &full[s]);
            else
              bulk_load_hint(dst, src, (uint32_t)elems * 2u, &full[s], y_policy);
          }
          if (lane == 0) loads_issued = i + 1;
        }
        if (late && c == 0 && ok) {
          t_next = draw(j);
          if (t_next >= 0) nxt = fetch_meta(p, t_next, lane, WEIGHTED);
        }
      }
      t = t_next;
      cur = nxt;
    }
    if (!ok && lane == 0) {
      *s_abort = 1;
      set_error(p.error_word, EP_ERRBIT_TIMEOUT);
    }
    if (lane == 0) retire_tokens(p.tokens, drained);
  } else {
    const int rt = tid - kWarpSize;  // reducer thread
    long i = 0;
    int known = -1;  // the token of the next unit, when a header has named it
    bool more = true;
    while (more && !*s_abort) {
      for (int c = 0; c < nchunk; ++c, ++i) {
        int s = static_cast<int>(i % kCombineStages);
        const int cols = min(kChunk, p.H - c * kChunk) / 8;
        const unsigned char *stage = stages + (size_t)s * kStageBytes;
        // a unit has at most one column per reducer thread: its bias loads
        // are issued before the wait for the rows when the token is known
        const int4 z = make_int4(0, 0, 0, 0);
        int4 b0 = z, b1 = z;
        auto load_bias = [&](int tok) {
          const size_t bcol = (size_t)tok * p.H + (size_t)c * kChunk + (size_t)rt * 8;
          if (rt < cols && p.bias0) b0 = ld_stream_v4(p.bias0 + bcol);
          if (rt < cols && p.bias1) b1 = ld_stream_v4(p.bias1 + bcol);
        };
        if (known >= 0) load_bias(known);
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (uint32_t)(i / kCombineStages) & 1u))) {
          if (lane == 0) {
            *s_abort = 1;
            set_error(p.error_word, EP_ERRBIT_TIMEOUT);
          }
          more = false;
          break;
        }
        const int *hdr = reinterpret_cast<const int *>(stage);
        const int nrows = hdr[0];
        if (rt == 0 && i == 0) EP_TRACE_MARK(g_trace_combine, 3);
        if (nrows < 0) {  // the end
          more = false;
          break;
        }
        const int t = hdr[1];
        const int t_next = hdr[2];
        if (t < 0 || t >= p.T) {  // a hand-over that went wrong: stop, do not index with it
          if (lane == 0) {
            *s_abort = 1;
            set_error(p.error_word, EP_ERRBIT_TIMEOUT);
          }
          more = false;
          break;
        }
        if (known != t) load_bias(t);
        const float *hdr_coef = reinterpret_cast<const float *>(stage + 16);
        uint16_t *out = p.out + (size_t)t * p.H + (size_t)c * kChunk;
        static_assert(kChunk / 8 <= kReducers * kWarpSize, "one column per reducer thread");
        float acc[8];
        if (rt < cols) {
          seed(acc, p, b0, b1);
          for (int r = 0; r < nrows; ++r) {
            const int4 v =
                *reinterpret_cast<const int4 *>(stage + kStageHeader + (size_t)r * kChunkBytes + rt * 16);
            accumulate<WEIGHTED, true>(acc, v, hdr_coef[r]);
          }
        }
        // a continuation: the token's remaining rows of this chunk, summed on
        for (int carry = SPLIT ? hdr[3] : 0; carry != 0 && more;) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
          ++i;
          s = static_cast<int>(i % kCombineStages);
          stage = stages + (size_t)s * kStageBytes;
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (uint32_t)(i / kCombineStages) & 1u))) {
            if (lane == 0) {
              *s_abort = 1;
              set_error(p.error_word, EP_ERRBIT_TIMEOUT);
            }
            more = false;
            break;
          }
          const int *h2 = reinterpret_cast<const int *>(stage);
          const float *c2 = reinterpret_cast<const float *>(stage + 16);
          if (rt < cols) {
            for (int r = 0; r < h2[0]; ++r) {
              const int4 v =
                  *reinterpret_cast<const int4 *>(stage + kStageHeader + (size_t)r * kChunkBytes + rt * 16);
              accumulate<WEIGHTED, true>(acc, v, c2[r]);
            }
          }
          carry = h2[3];
        }
        if (!more) break;
        if (rt < cols) {
          int4 o;
          o.x = (int)pack_bf16x2(acc[0], acc[1]);
          o.y = (int)pack_bf16x2(acc[2], acc[3]);
          o.z = (int)pack_bf16x2(acc[4], acc[5]);
          o.w = (int)pack_bf16x2(acc[6], acc[7]);
          // rows of more than two chunks: plain stores (measured against
          // streaming ones at 7168 elements: headline step -0.6 us, the
          // combine -1.4 us; at 4096 elements, streaming stores were
          // 0.2-0.35 us faster a step and stay)
          if (!SPLIT && nchunk > 2)
            st_v4(out + (size_t)rt * 8, o);
          else
            st_stream_v4(out + (size_t)rt * 8, o);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        known = c + 1 < nchunk ? t : t_next;
      }
    }
  }

  if (tid == kWarpSize) EP_TRACE_MARK(g_trace_combine, 5);
  // After an abort, the loads of the latest units still in flight are
  // waited for (bounded) before the CTA's shared memory is released.
  __syncthreads();
  if (*s_abort && tid == 0) {
    for (long m = loads_issued > kCombineStages ? loads_issued - kCombineStages : 0; m < loads_issued; ++m)
      (void)mbar_wait_bounded(&full[m % kCombineStages], (uint32_t)(m / kCombineStages) & 1u);
  }
}

template <bool WEIGHTED, int ROWS, bool SPLIT>
ep_status_t launch_ws_rows(const CombineParams &p, const DeviceInfo &di, cudaStream_t stream) {
  static std::mutex mu;
  static bool configured[64] = {};
  const auto kernel = combine_ws_kernel<WEIGHTED, ROWS, SPLIT>;
  const size_t smem = 128 + (size_t)kCombineStages * (kStageHeader + (size_t)ROWS * kChunkBytes);
  {
    std::lock_guard<std::mutex> g(mu);
    if (di.device < 64 && !configured[di.device]) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(combine_ws_kernel)");
      configured[di.device] = true;
    }
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kWsCombineThreads, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(combine_ws)");
  if (per_sm <= 0) return fail(EP_ERR_UNSUPPORTED, "ep_combine: kernel cannot be resident");
  const int grid = std::min(p.T, per_sm * di.num_sms);
  e = launch_kernel(kernel, grid, kWsCombineThreads, smem, stream, false, p);
  if (e != cudaSuccess) return cuda_fail(e, "launch combine_ws_kernel");
  return EP_OK;
}

// A token has at most min(K, R) rank rows under a given routing.  With at
// most 6, stages of 6 rows (four blocks per SM instead of three).  With more
// and many tokens, also 6-row stages, the wider tokens split in two units:
// measured faster at 65 536 tokens (the occupancy), slower at 8192 (the
// split units), so only from kSplitMinTokens on.
template <bool WEIGHTED>
ep_status_t launch_ws(const CombineParams &p, const DeviceInfo &di, cudaStream_t stream) {
  if constexpr (WEIGHTED) {
    if (!p.expanded && std::min(p.K, p.D) <= kSmallStageRows)
      return launch_ws_rows<WEIGHTED, kSmallStageRows, false>(p, di, stream);
    if (!p.expanded && p.T >= kSplitMinTokens) return launch_ws_rows<WEIGHTED, kSmallStageRows, true>(p, di, stream);
  }
  return launch_ws_rows<WEIGHTED, kWsMaxRanks, false>(p, di, stream);
}

constexpr bool kUseWsCombine = true;

template <bool WEIGHTED>
ep_status_t launch_impl(const CombineParams &p, const DeviceInfo &di, cudaStream_t stream) {
  int per_sm = 0;
  cudaError_t e =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel<WEIGHTED>, kCombineThreads, 0);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(combine)");
  if (per_sm <= 0) return fail(EP_ERR_UNSUPPORTED, "ep_combine: kernel cannot be resident");
  const int grid = std::min(p.T, per_sm * di.num_sms);
  e = launch_kernel(combine_kernel<WEIGHTED>, grid, kCombineThreads, 0, stream, false, p);
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
  p.epr = (a.topk_weights != nullptr && !a.expanded) ? a.num_experts / a.num_ranks : 1;
  p.expanded = a.expanded;
  p.D = a.expanded ? a.num_topk : a.num_ranks;
  p.token_slot = a.token_slot;
  p.error_word = a.error_word;
  p.topk_idx = a.topk_idx;
  p.topk_weights = a.topk_weights;
  p.bias0 = a.bias0;
  p.bias1 = a.bias1;
  p.out = a.out;
  p.tokens.ticket = a.work_counters;
  p.tokens.done = a.work_counters != nullptr ? a.work_counters + 1 : nullptr;
  p.tokens.T = a.num_tokens;
  const bool weighted = a.topk_weights != nullptr;
  if (kUseWsCombine && p.D <= kWsMaxRanks)
    return weighted ? launch_ws<true>(p, *di, stream) : launch_ws<false>(p, *di, stream);
  return weighted ? launch_impl<true>(p, *di, stream) : launch_impl<false>(p, *di, stream);
}

}  // namespace ep

EP_TRACE_READER(ep_trace_read_combine, ep::g_trace_combine);
