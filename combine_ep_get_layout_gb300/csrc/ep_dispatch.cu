// Dispatch kernel: the scatter phase of TileScale PR #68 ("[Example] EP v2
// intranode dispatch/combine", PR summary: rows go straight to their final
// compact index, no copy epilogue), with the per-token, per-128-element fp8
// cast fused into the same pass (same page, commit message on packing the
// fp8 row; DeepEP's per_token_cast_to_fp8 layout).
//
// dispatch_ws_kernel (fp8 rows) and dispatch_ws_bf16_kernel (bf16 rows):
// warp-specialised, a loader warp bulk-loading rows into a ring of input
// stages, for fp8 eight caster warps, and a storer warp writing the received
// metadata and bulk-storing each row to every destination slot, handing
// buffers over through mbarriers (details above the kernel body below).
//
// dispatch_ring_kernel (bf16 rows of an expanded layout): one CTA works
// through its tokens with a ring of `stages` shared-memory row buffers;
// thread 0 draws tokens and bulk-loads their rows, warp 0 issues one bulk
// store of the stage per destination, the other warps write the metadata.
//
// Each row of x is read from HBM once and written once per destination.
#include <algorithm>
#include <climits>
#include <mutex>

#include "ep_device.cuh"
#include "ep_trace.cuh"

namespace ep {
namespace {

constexpr int kDispatchThreads = 256;
constexpr int kMaxStages = 8;
constexpr int kHeaderBytes = 1024;  // mbarriers, flags, slot buffers
constexpr size_t kSmemBudget = 80 * 1024;  // per CTA: aims at >= 2-3 CTAs per SM
constexpr int kWsStages = 2;                 // bf16 row stages of the fp8 kernel
constexpr size_t kWsSmemBudget = 64 * 1024;
constexpr bool kWsWarmL2 = true;  // fp8 kernel: L2 hints before the grid-dependency wait

struct DispatchParams {
  const uint16_t *x;
  int T, H, K, E, R, epr, groups;
  int D;          // destinations per token: R ranks, or K experts (expanded)
  bool expanded;  // token_slot is [T * K]: one row per (token, expert)
  const int32_t *xoff, *xrows;  // expanded: segment starts [E+1], rows [E]
  bool zero_padding;            // expanded: write the padding rows
  const int64_t *topk_idx;
  const float *topk_weights;
  const int32_t *token_slot;    // [T * D]
  uint32_t *error_word;
  void *recv_x;
  float *recv_x_scales;
  int32_t *recv_src_idx;
  int32_t *recv_topk_idx;
  float *recv_topk_weights;
  int cap;
  uint32_t *stats;         // [E] cumulative received (row, top-k slot) counts, or null
  int stages;
  uint32_t row_in_bytes;   // 2H
  uint32_t row_out_bytes;  // 2H (bf16), H (fp8) or the packed fp8 row
  bool packed;             // fp8 codes, scales and zero padding in one row
  uint32_t stage_stride;   // row_in_bytes rounded up to 128
  uint32_t out_stride;     // fp8 output row, H rounded up to 128
  uint32_t scale_stride;   // fp8 scales of one row, groups*4 rounded up to 16
  TokenSource tokens;      // the order in which blocks take tokens
  int early;               // rows loaded (and cast) before the wait for the previous kernel
  // warp-specialised kernels after the local layout: token_slot holds
  // block-relative slots; slot = relative + the block's base (local_base[(t /
  // 256) * R + r], or from the scanned table), written to token_slot_out
  const int32_t *local_base;
  int32_t *token_slot_out;
  int32_t *num_tokens_per_expert;
  // table mode (table_blocks = G > 0): local_base holds each 256-token
  // block's per-rank totals; the storer scans them into shared memory at
  // table_offset (bases [G*R], rank totals [R], rank offsets [R+1]) and
  // block 0 writes rank_prefix and num_tokens_per_rank
  int table_blocks;
  uint32_t table_offset;
  int32_t *rank_prefix;
  int32_t *num_tokens_per_rank;
};

// Shared-memory bytes of the table mode's scan (see DispatchParams).
inline uint32_t base_table_bytes(int table_blocks, int R) {
  return table_blocks > 0 ? ((uint32_t)(table_blocks * R + 2 * R + 1) * 4u + 15u) / 16u * 16u : 0u;
}

// Token ids travel from the loading thread to the other roles of a block
// through a ring of kTokRing shared ints: the block's idx-th token (or -1,
// the end) in entry idx % kTokRing.  A loader is at most stages + 3 tokens
// ahead of the slowest reader.
constexpr int kTokRing = 16;
constexpr int kTokPending = INT_MIN;       // entry not written yet
constexpr int kTokTimedOut = INT_MIN + 1;  // wait_token gave up

// Draws the block's idx-th token, records it in s_tok and starts the load
// of its row into stage idx % stages (mbarrier full[stage]).  Once the
// tokens are exhausted it records -1 and completes the stage's phase with a
// plain arrival instead, so every index has a phase.  Returns the token (or
// -1).  One thread.
__device__ __forceinline__ int issue_token(const DispatchParams &p, unsigned char *stages, uint64_t *full,
                                           volatile int *s_tok, int idx, bool &drained, uint64_t policy,
                                           int head = 0) {
  const int t = draw_token(p.tokens, idx, drained, head);
  const int s = idx % p.stages;
  s_tok[idx % kTokRing] = t;
  if (t < 0) {
    mbar_arrive(&full[s]);
    return t;
  }
  mbar_arrive_expect_tx(&full[s], p.row_in_bytes);
  bulk_load_hint(stages + (size_t)s * p.stage_stride, p.x + (size_t)t * p.H, p.row_in_bytes, &full[s], policy);
  return t;
}

// The token in a ring entry once the loading thread has written it
// (bounded wait: kTokTimedOut after kWaitLimitNs).
__device__ __forceinline__ int wait_token(volatile int *entry) {
  int t = *entry;
  if (t != kTokPending) return t;
  const uint64_t t0 = global_timer_ns();
  while ((t = *entry) == kTokPending) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return kTokTimedOut;
    __nanosleep(32);
  }
  return t;
}

// Warp-collective: the layout holds exactly the rows this routing needs
// (slot_lo / slot_hi: the slots of destinations lane and lane + 32; e: the
// expert of slot k = lane, -1 past K).
__device__ __forceinline__ bool layout_agrees(const DispatchParams &p, int64_t e, int slot_lo, int slot_hi,
                                              int lane) {
  return p.expanded ? choices_agree(e, p.E, p.K, slot_lo, lane)
                    : ranks_agree(e, p.E, p.epr, p.R, slot_lo, slot_hi, lane);
}

// Cumulative recv stats: lane k < K adds one to its expert's count when that
// expert's row (the rank's row, or the expanded row of slot k) was received
// (slot in [0, cap)).  Warp-collective.
__device__ __forceinline__ void count_received(const DispatchParams &p, int64_t e, int slot_lo, int slot_hi,
                                               int lane) {
  const bool valid = e >= 0 && e < p.E;
  const int r = valid ? static_cast<int>(e) / p.epr : 0;
  const int s_lo = __shfl_sync(0xffffffffu, slot_lo, r & (kWarpSize - 1));
  const int s_hi = __shfl_sync(0xffffffffu, slot_hi, r & (kWarpSize - 1));
  const int slot = p.expanded ? slot_lo : (r < kWarpSize ? s_lo : s_hi);
  if (valid && slot >= 0 && slot < p.cap) atomicAdd(p.stats + e, 1u);
}

// The destination whose received row marks top-k slot k (expert e), or -1:
// a rank row marks every expert of its rank; an expanded row marks only its
// own slot (TileScale PR #68, commit message on the expanded combine).  The
// local expert id written there is e minus the rank's first expert.
__device__ __forceinline__ int marked_dest(const DispatchParams &p, int64_t e, int k) {
  if (e < 0 || e >= p.E) return -1;
  return p.expanded ? k : static_cast<int>(e) / p.epr;
}
__device__ __forceinline__ int local_expert(const DispatchParams &p, int64_t e) {
  return static_cast<int>(e) % p.epr;
}

// Warp-collective: turns the per-block, per-rank totals the one-launch
// layout left (tot[b * R + r], G blocks of 256 tokens) into each block's
// first slot in each rank, in shared memory: base[b * R + r] (the rank's
// exclusive scan over the blocks, before its offset), rtot[r] (the rank's
// total) and roff[r] (the exclusive scan of the totals; roff[R] = N).  The
// lanes form groups of lp = 32 / (R rounded up to a power of two) lanes, at
// least one, a group per rank; a lane sums a run of ceil(G / lp) blocks of
// its rank, the runs' sums are scanned across the group by shuffles, and the
// lane rewrites its run with the running prefix.  The totals come in by one
// bulk copy (their 16-byte-aligned prefix, mbarrier `bar`, used once; the
// few left over by plain loads): one round trip to L2 for the whole table
// (measured: headline step -0.24 us against loads of four words a lane).
// False if the copy did not land within the wait limit (after a second
// bounded wait for it, so that the block does not exit with it in flight).
__device__ __forceinline__ bool scan_block_totals(const int32_t *tot, int G, int R, int32_t *base, int32_t *rtot,
                                                  int32_t *roff, int lane, uint64_t *bar) {
  const int n = G * R;
  const uint32_t bulk = ((uint32_t)n * 4u) & ~15u;
  const bool use_bulk = bulk > 0 && ((reinterpret_cast<uintptr_t>(tot) | (uintptr_t)smem_addr(base)) & 15u) == 0;
  if (use_bulk && lane == 0) {
    mbar_arrive_expect_tx(bar, bulk);
    bulk_load(base, tot, bulk, bar);
  }
  for (int q0 = use_bulk ? (int)(bulk / 4u) : 0; q0 < n; q0 += 4 * kWarpSize) {  // four loads in flight per lane
    int v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = q0 + u * kWarpSize + lane;
      v[u] = q < n ? __ldcg(tot + q) : 0;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = q0 + u * kWarpSize + lane;
      if (q < n) base[q] = v[u];
    }
  }
  const bool ok = __all_sync(0xffffffffu, !use_bulk || mbar_wait_bounded(bar, 0));
  if (!ok && lane == 0) (void)mbar_wait_bounded(bar, 0);  // the copy still in flight: once more, bounded
  __syncwarp();
  if (!ok) return false;
  int rp = 1;
  while (rp < R) rp <<= 1;
  const int lp = rp >= kWarpSize ? 1 : kWarpSize / rp;  // lanes per rank
  const int c = (G + lp - 1) / lp;                      // blocks per lane
  for (int r0 = 0; r0 < R; r0 += kWarpSize / lp) {      // two passes only when R > 32
    const int r = r0 + lane / lp, sub = lane % lp;
    const int b0 = min(sub * c, G), b1 = min(b0 + c, G);
    int sum = 0;
    if (r < R)
      for (int bb = b0; bb < b1; ++bb) sum += base[bb * R + r];
    int incl = sum;
    for (int d = 1; d < lp; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, d, lp);
      if (sub >= d) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, lp - 1, lp);
    if (r < R) {
      int run = incl - sum;
      for (int bb = b0; bb < b1; ++bb) {
        const int v = base[bb * R + r];
        base[bb * R + r] = run;
        run += v;
      }
      if (sub == 0) rtot[r] = total;
    }
  }
  __syncwarp();
  const int lo = lane < R ? rtot[lane] : 0;  // R <= 64: two ranks per lane
  const int hi = lane + kWarpSize < R ? rtot[lane + kWarpSize] : 0;
  int il = lo, ih = hi;
  for (int d = 1; d < kWarpSize; d <<= 1) {
    const int yl = __shfl_up_sync(0xffffffffu, il, d);
    const int yh = __shfl_up_sync(0xffffffffu, ih, d);
    if (lane >= d) {
      il += yl;
      ih += yh;
    }
  }
  const int sum_lo = __shfl_sync(0xffffffffu, il, kWarpSize - 1);
  const int sum_hi = __shfl_sync(0xffffffffu, ih, kWarpSize - 1);
  if (lane < R) roff[lane] = il - lo;
  if (lane + kWarpSize < R) roff[lane + kWarpSize] = sum_lo + ih - hi;
  if (lane == 0) roff[R] = sum_lo + sum_hi;
  __syncwarp();
  return true;
}

// Received metadata of token t, by threads [32, blockDim): source token,
// local expert ids and gate weights of every row the token is sent as.
__device__ __forceinline__ void write_metadata(const DispatchParams &p, int t, const int32_t *slots) {
  const int mt = threadIdx.x - kWarpSize;
  const int nt = kDispatchThreads - kWarpSize;
  if (threadIdx.x / kWarpSize == 1) {  // warp 1 checks the layout against the routing
    const int lane = threadIdx.x & (kWarpSize - 1);
    const int64_t e = lane < p.K ? __ldg(p.topk_idx + (size_t)t * p.K + lane) : -1;
    const int lo = lane < p.D ? slots[lane] : -1;
    const int hi = lane + kWarpSize < p.D ? slots[lane + kWarpSize] : -1;
    if (!layout_agrees(p, e, lo, hi, lane) && lane == 0) set_error(p.error_word, EP_ERRBIT_STALE_LAYOUT);
    if (p.stats != nullptr) count_received(p, e, lo, hi, lane);
  }
  if (p.recv_src_idx != nullptr) {
    for (int j = mt; j < p.D; j += nt) {
      const int slot = slots[j];
      if (slot >= 0 && slot < p.cap) p.recv_src_idx[slot] = t;
    }
  }
  if (p.recv_topk_idx != nullptr || p.recv_topk_weights != nullptr) {
    const int DK = p.D * p.K;
    for (int q = mt; q < DK; q += nt) {
      const int j = q / p.K;
      const int k = q - j * p.K;
      const int slot = slots[j];
      if (slot < 0 || slot >= p.cap) continue;
      const int64_t e = __ldg(p.topk_idx + (size_t)t * p.K + k);
      const bool here = marked_dest(p, e, k) == j;
      if (p.recv_topk_idx != nullptr) p.recv_topk_idx[(size_t)slot * p.K + k] = here ? local_expert(p, e) : -1;
      if (p.recv_topk_weights != nullptr)
        p.recv_topk_weights[(size_t)slot * p.K + k] = here ? __ldg(p.topk_weights + (size_t)t * p.K + k) : 0.0f;
    }
  }
}

// The fp8 cast of two 128-element groups held by a warp, one per half-warp,
// eight bf16 values per lane (`raw`, in element order): amax over the group
// by shuffles inside the half-warp, scale = amax / 448 and
// code = e4m3(x / scale) with x / scale the correctly rounded fp32 quotient,
// converted round to nearest even, saturating at +-448.  An all-zero group
// has scale 0 and keeps each zero's sign.  Returns the lane's eight codes
// (element order, low byte first); `scale` receives the group's scale in
// every lane of the half-warp.
//
// The quotient is not divided out per element.  Ziv's rounding test: with
// r = rcp_approx(scale), q = x * r lies within 2^-21 (relative) of x / scale,
// and so does the correctly rounded quotient; q * (1 -+ 2^-19) bracket both.
// The conversion is monotonic, so when the two ends of the bracket give the
// same code, that is the code of the correctly rounded quotient.  Only a
// lane with a quotient within about 2^-19 of a rounding boundary (and a
// group whose scale is too small for r to be finite) divides.
constexpr float kBracketBelow = 1.0f - 0x1p-19f;
constexpr float kBracketAbove = 1.0f + 0x1p-19f;
constexpr bool kCastPackedMul = true;  // f32x2 multiplies for the quotients and brackets

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return pack_e4m3x2(a, b) | (pack_e4m3x2(c, d) << 16);
}

__device__ __forceinline__ void mul_pair(float a, float b, float c, float &ac, float &bc) {
  if constexpr (kCastPackedMul) {
    mul2_rn(a, b, c, ac, bc);
  } else {
    ac = a * c;
    bc = b * c;
  }
}

__device__ __forceinline__ uint2 cast_pair(uint4 raw, float &scale) {
  float v[8] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y),
                bf16_lo(raw.z), bf16_hi(raw.z), bf16_lo(raw.w), bf16_hi(raw.w)};
  float a = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                  fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
  scale = __fdiv_rn(a, 448.0f);
  if (!(a > 0.0f)) return make_uint2(e4m3x4(v[0], v[1], v[2], v[3]), e4m3x4(v[4], v[5], v[6], v[7]));
  if (scale >= 0x1p-125f) {  // 1 / scale is finite
    const float r = rcp_approx(scale);
    float q[8], lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      mul_pair(v[i], v[i + 1], r, q[i], q[i + 1]);
      mul_pair(q[i], q[i + 1], kBracketBelow, lo[i], lo[i + 1]);
      mul_pair(q[i], q[i + 1], kBracketAbove, hi[i], hi[i + 1]);
    }
    const uint2 cl = make_uint2(e4m3x4(lo[0], lo[1], lo[2], lo[3]), e4m3x4(lo[4], lo[5], lo[6], lo[7]));
    const uint2 ch = make_uint2(e4m3x4(hi[0], hi[1], hi[2], hi[3]), e4m3x4(hi[4], hi[5], hi[6], hi[7]));
    if (cl.x == ch.x && cl.y == ch.y) return cl;
  }
  float u[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) u[i] = __fdiv_rn(v[i], scale);
  return make_uint2(e4m3x4(u[0], u[1], u[2], u[3]), e4m3x4(u[4], u[5], u[6], u[7]));
}

// Casts groups [g0, g0 + 2) of a staged bf16 row (`stage`, 256 bytes per
// group) into `orow` (128 codes per group) and `oscale`; a group index at or
// past `groups` is skipped.  Warp-collective.
__device__ __forceinline__ void cast_two_groups(const unsigned char *stage, unsigned char *orow, float *oscale,
                                                int g0, int groups, int lane) {
  const int g = g0 + (lane >> 4);
  const bool live = g < groups;
  const uint4 raw = live ? *reinterpret_cast<const uint4 *>(stage + (size_t)g0 * 256 + lane * 16)
                         : make_uint4(0u, 0u, 0u, 0u);
  float scale;
  const uint2 codes = cast_pair(raw, scale);
  if (live) {
    *reinterpret_cast<uint2 *>(orow + (size_t)g0 * 128 + lane * 8) = codes;
    if ((lane & 15) == 0) oscale[g] = scale;
  }
}

__global__ void __launch_bounds__(kDispatchThreads) dispatch_ring_kernel(DispatchParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);               // [kMaxStages]
  int *s_abort = reinterpret_cast<int *>(smem + 64);
  int32_t *s_slot = reinterpret_cast<int32_t *>(smem + 128);         // [2][EP_MAX_RANKS]
  volatile int *s_tok = reinterpret_cast<volatile int *>(smem + 640);  // [kTokRing]
  unsigned char *stages = smem + kHeaderBytes;

  const int tid = threadIdx.x;
  const int warp = tid / kWarpSize;
  const int lane = tid & (kWarpSize - 1);
  const int S = p.stages;

  if (tid < kTokRing) s_tok[tid] = kTokPending;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();
  const uint64_t policy = policy_evict_first();  // x is read exactly once
  bool drained = false;  // thread 0: no more tokens to draw
  int issued = 0;        // thread 0: token indices drawn (loads and the end)
  if (tid == 0)
    for (; issued < S && !drained; ++issued) issue_token(p, stages, full, s_tok, issued, drained, policy);
  __syncthreads();

  int i = 0;
  for (;; ++i) {
    // Thread 0 may have drawn token i during the previous iteration, after
    // that iteration's last barrier (bf16 with two stages): this barrier
    // makes its ring entry visible.
    if (i > 0) __syncthreads();
    const int t = s_tok[i % kTokRing];
    if (t < 0) break;  // the end (or an entry never written)
    if (t >= p.T) {    // a hand-over that went wrong: stop, do not index with it
      if (tid == 0) set_error(p.error_word, EP_ERRBIT_TIMEOUT);
      break;
    }
    const int s = i % S;
    const uint32_t parity = (uint32_t)(i / S) & 1u;
    const int b = i & 1;
    int32_t *slots = s_slot + b * EP_MAX_RANKS;
    unsigned char *stage = stages + (size_t)s * p.stage_stride;

    if (tid < p.D) slots[tid] = __ldg(p.token_slot + (size_t)t * p.D + tid);
    __syncthreads();
    if (*s_abort) break;

    {
      if (warp == 0) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], parity));
        if (!ok) {
          if (lane == 0) {
            *s_abort = 1;
            set_error(p.error_word, EP_ERRBIT_TIMEOUT);
          }
        } else {
          for (int j = lane; j < p.D; j += kWarpSize) {
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
          if (lane == 0 && i >= 1 && !drained) issue_token(p, stages, full, s_tok, issued++, drained, policy);
        }
      } else {
        write_metadata(p, t, slots);
      }
    }
  }

  // Drain: stores must finish reading shared memory before the CTA exits;
  // after an abort, loads still in flight are waited for (bounded).
  if (tid == 0) retire_tokens(p.tokens, drained);
  if (warp == 0) bulk_wait<0>();
  __syncthreads();
  if (*s_abort && tid == 0) {
    for (int m = i; m < issued; ++m) (void)mbar_wait_bounded(&full[m % S], (uint32_t)(m / S) & 1u);
  }
}



// ------------------------------------------------------------------------
// Warp-specialised kernel.  Roles inside one CTA, handing buffers over
// through mbarriers (no CTA-wide barrier in the loop):
//   warp 0 (loader)    bulk-loads token rows into a ring of `stages` bf16
//                      row buffers (full_in), reusing a buffer once every
//                      caster has released it (empty_in);
//   warp 1 (storer)    writes the received metadata, then bulk-stores each
//                      cast row and its scales to every destination slot
//                      (full_out), releasing the buffer once the stores have
//                      read it (empty_out);
//   warps 2.. (casters) cast 128-element groups of a row into one of two
//                      fp8 row buffers.
// Casting token i+1 thus overlaps the stores of token i and the loads of
// the tokens after it.  For bf16 rows (dispatch_ws_bf16_kernel) there are
// no casters: the storer stores each row from its input stage and releases
// the stage (empty_in) one token late, once those stores have read it.

// Trace build only (warp-specialised kernels): 0 entry, 3 the storer past
// its wait for the kernel ahead, 1 past the table scan too, 2 its first
// token, 4 it sees the end, 5 its stores done, 6 (a count) the tokens it
// stored, 7 the loader past its wait.
EP_TRACE_ARRAY(g_trace_dispatch);

constexpr int kWsCasters = 8;
constexpr int kWsThreads = (2 + kWsCasters) * kWarpSize;
constexpr int kWsBf16Threads = 2 * kWarpSize;  // loader and storer
constexpr int kWsBf16Stages = 8;                // bf16 row stages (fewer for wide rows)
constexpr size_t kWsBf16SmemBudget = 64 * 1024;
// Two output buffers: measured against three, the headline step -1.3 us (the
// same 4 blocks per SM, 15 KB less shared memory per SM in use).
constexpr int kWsOut = 2;
// Once a block has drawn one of the last kNearEndBlocks * gridDim.x tokens,
// its loader draws the next token only when the storer is at most one token
// behind, so the last tokens go to blocks with little left in their
// pipelines and the grid's blocks finish closer together (measured: fp8
// rows, headline step -1.2 us, 65 536 tokens -0.7 us; bf16 rows, whose
// loader otherwise runs up to seven stages ahead, bf16 step -0.45 us and
// skewed -0.3 us, two tokens ahead timing the same).
constexpr int kNearEndBlocks = 2;
// The storer releases an output buffer one token late (once the next
// token's stores are issued), so waiting for the stores to read a buffer
// overlaps the next token's metadata instead of preceding it.
constexpr bool kWsLateRelease = true;

// Storer, after committing token i's stores: hand an output buffer back to
// the casters once the bulk stores have read it -- token i's buffer, or with
// late release token i-1's (the stores of token i may still be reading).
__device__ __forceinline__ void release_out(uint64_t *empty_out, int i, int lane) {
  if constexpr (kWsLateRelease) {
    bulk_wait_read<1>();
    __syncwarp();
    if (lane == 0 && i > 0) mbar_arrive(&empty_out[(i - 1) % kWsOut]);
  } else {
    bulk_wait_read<0>();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_out[i % kWsOut]);
  }
}

// CAST: fp8 rows (casters between the loader and the storer); otherwise
// bf16 rows, which the storer bulk-stores straight from the input stage
// (two warps, no casters, no output buffers).
template <bool CAST>
__device__ __forceinline__ void dispatch_ws_body(const DispatchParams &p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int S = p.stages;
  uint64_t *full_in = reinterpret_cast<uint64_t *>(smem);  // [S]
  uint64_t *empty_in = full_in + kMaxStages;                // [S]
  uint64_t *full_out = empty_in + kMaxStages;               // [kWsOut]
  uint64_t *empty_out = full_out + kWsOut;                  // [kWsOut]
  uint64_t *table_full = empty_out + kWsOut;                // the table's bulk copy
  volatile int *s_abort = reinterpret_cast<volatile int *>(smem + 256);
  int32_t *s_slot = reinterpret_cast<int32_t *>(smem + 512);  // [EP_MAX_RANKS], storer only
  volatile int *s_tok = reinterpret_cast<volatile int *>(smem + 768);  // [kTokRing]
  volatile int *s_stored = reinterpret_cast<volatile int *>(smem + 896);  // tokens the storer is past
  unsigned char *in = smem + kHeaderBytes;
  unsigned char *out = in + (size_t)S * p.stage_stride;
  float *osc = reinterpret_cast<float *>(out + (size_t)kWsOut * p.out_stride);

  const int tid = threadIdx.x;
  const int warp = tid / kWarpSize;
  const int lane = tid & (kWarpSize - 1);

  if (tid == 0) EP_TRACE_MARK(g_trace_dispatch, 0);
  if (tid < kTokRing) s_tok[tid] = kTokPending;
  if (tid == 0) *s_stored = 0;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_in[s], 1);
      mbar_init(&empty_in[s], CAST ? kWsCasters : 1);
    }
    for (int o = 0; o < kWsOut; ++o) {
      mbar_init(&full_out[o], kWsCasters);
      mbar_init(&empty_out[o], 1);
    }
    mbar_init(table_full, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (p.packed) {  // the padding of both packed output rows stays zero
    const uint32_t used = (uint32_t)p.H + (uint32_t)p.groups * 4u;
    for (int o = 0; o < kWsOut; ++o)
      for (uint32_t b = used + tid; b < p.row_out_bytes; b += blockDim.x) out[(size_t)o * p.out_stride + b] = 0;
    fence_proxy_async_smem();
  }
  __syncthreads();
  // With p.early > 0 the previous kernel on the stream (the layout) writes
  // nothing this kernel reads before its wait: the loader brings in the rows
  // of its first p.early tokens (its own stripe) and the casters cast them
  // while the layout is still running; the loader waits before its first
  // ticket, the storer before it reads the layout.  The casters touch no
  // global memory.
  if (p.early == 0) {
    // Before the wait, only hints: the row of token blockIdx.x (the first
    // tickets go to tokens 0 .. gridDim.x - 1 in some order) and its layout
    // row are brought into L2, no value is read.
    if (kWsWarmL2 && tid == 0 && (int)blockIdx.x < p.T) {
      bulk_prefetch_l2(p.x + (size_t)blockIdx.x * p.H, p.row_in_bytes);
      prefetch_l2(p.token_slot + (size_t)blockIdx.x * p.D);
      prefetch_l2(p.topk_idx + (size_t)blockIdx.x * p.K);
    }
    griddep_wait();
  }
  griddep_launch_dependents();

  int issued = 0;        // loader lane 0: token indices drawn (loads and the end)
  bool drained = false;  // loader lane 0: no more tokens to draw
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t policy = policy_evict_first();
      bool waited = p.early == 0;
      bool near_end = false;
      for (int i = 0; !drained && !*s_abort; ++i) {
        const int s = i % S;
        if (i >= S && !mbar_wait_bounded(&empty_in[s], (uint32_t)(i / S - 1) & 1u)) {
          *s_abort = 1;
          set_error(p.error_word, EP_ERRBIT_TIMEOUT);
          break;
        }
        if (near_end && i >= 1) {  // at most one token ahead of the storer (bounded wait)
          const uint64_t t0 = global_timer_ns();
          while (*s_stored < i - 1 && !*s_abort) {
            if (global_timer_ns() - t0 > kWaitLimitNs) {
              *s_abort = 1;
              set_error(p.error_word, EP_ERRBIT_TIMEOUT);
              break;
            }
            __nanosleep(32);
          }
          if (*s_abort) break;
        }
        // the first draw that may touch the counter (a ticket, or the end)
        if (!waited && (i >= p.early || (long)blockIdx.x + (long)i * gridDim.x >= p.T)) {
          griddep_wait();
          waited = true;
          EP_TRACE_MARK(g_trace_dispatch, 7);
        }
        const int t = issue_token(p, in, full_in, s_tok, i, drained, policy, p.early);
        issued = i + 1;
        if (t >= p.T - kNearEndBlocks * (int)gridDim.x) near_end = true;
      }
      if (!waited) griddep_wait();
      retire_tokens(p.tokens, drained);
    }
  } else if (warp == 1) {
    if (p.early > 0) griddep_wait();
    if (lane == 0) EP_TRACE_MARK(g_trace_dispatch, 3);
    const bool scale_bulk = p.scale_stride == (uint32_t)p.groups * 4u &&
                            (reinterpret_cast<uintptr_t>(p.recv_x_scales) & 15u) == 0;
    // Table mode: the layout left each 256-token block's per-rank totals;
    // each rank's exclusive scan over the blocks, plus the rank's offset
    // (the exclusive scan of the rank totals), is each block's base.
    int32_t *s_base = reinterpret_cast<int32_t *>(smem + p.table_offset);  // [G * R]
    int32_t *s_rtot = s_base + p.table_blocks * p.R;                        // [R]
    int32_t *s_roff = s_rtot + p.R;                                         // [R + 1]
    if (p.table_blocks > 0) {
      const int R = p.R;
      if (!scan_block_totals(p.local_base, p.table_blocks, R, s_base, s_rtot, s_roff, lane, table_full)) {
        if (lane == 0) {
          *s_abort = 1;
          set_error(p.error_word, EP_ERRBIT_TIMEOUT);
        }
      } else if (blockIdx.x == 0) {
        for (int r = lane; r <= R; r += kWarpSize) {
          p.rank_prefix[r] = s_roff[r];
          if (r < R) p.num_tokens_per_rank[r] = s_rtot[r];
        }
      }
    }
    if (lane == 0) EP_TRACE_MARK(g_trace_dispatch, 1);
    for (int i = 0; !*s_abort; ++i) {
      if (lane == 0) *s_stored = i;  // tokens before i are stored
      const int t = wait_token(&s_tok[i % kTokRing]);
      if (t == kTokTimedOut) {
        if (lane == 0) {
          *s_abort = 1;
          set_error(p.error_word, EP_ERRBIT_TIMEOUT);
        }
        break;
      }
      if (t < 0) {
        if (lane == 0) {
          EP_TRACE_MARK(g_trace_dispatch, 4);
          EP_TRACE_VALUE(g_trace_dispatch, 6, i);
        }
        break;
      }
      if (i == 0 && lane == 0) EP_TRACE_MARK(g_trace_dispatch, 2);
      if (t >= p.T) {  // a hand-over that went wrong: stop, do not index with it
        if (lane == 0) {
          *s_abort = 1;
          set_error(p.error_word, EP_ERRBIT_TIMEOUT);
        }
        break;
      }
      const int o = i % kWsOut;
      const int32_t *srow = p.token_slot + (size_t)t * p.D;
      int slot_lo = lane < p.D ? __ldg(srow + lane) : -1;
      int slot_hi = lane + kWarpSize < p.D ? __ldg(srow + lane + kWarpSize) : -1;
      const int64_t e = lane < p.K ? __ldg(p.topk_idx + (size_t)t * p.K + lane) : -1;
      const float w = (lane < p.K && p.recv_topk_weights != nullptr)
                          ? __ldg(p.topk_weights + (size_t)t * p.K + lane) : 0.0f;
      // local layout: the block's bases, loaded alongside the slots (or
      // taken from the scanned table)
      const size_t blk = (size_t)(t / kLocalTokensPerBlock) * p.R;
      int base_lo = 0, base_hi = 0;
      if (p.table_blocks > 0) {
        if (lane < p.D) base_lo = s_base[blk + lane] + s_roff[lane];
        if (lane + kWarpSize < p.D) base_hi = s_base[blk + lane + kWarpSize] + s_roff[lane + kWarpSize];
      } else if (p.local_base != nullptr) {
        if (lane < p.D) base_lo = __ldg(p.local_base + blk + lane);
        if (lane + kWarpSize < p.D) base_hi = __ldg(p.local_base + blk + lane + kWarpSize);
      }
      if (p.local_base != nullptr) {
        // finish the layout of token t: absolute slots, written back; its
        // experts counted; ids outside [-1, E) flagged
        if (slot_lo >= 0) slot_lo += base_lo;
        if (slot_hi >= 0) slot_hi += base_hi;
        int32_t *orow = p.token_slot_out + (size_t)t * p.D;
        if (lane < p.D) orow[lane] = slot_lo;
        if (lane + kWarpSize < p.D) orow[lane + kWarpSize] = slot_hi;
        const bool valid = e >= 0 && e < p.E;
        if (valid) atomicAdd(p.num_tokens_per_expert + e, 1);
        if (__any_sync(0xffffffffu, !valid && e != -1 && lane < p.K) && lane == 0)
          set_error(p.error_word, EP_ERRBIT_BAD_INDEX);
      } else if (!layout_agrees(p, e, slot_lo, slot_hi, lane) && lane == 0) {
        set_error(p.error_word, EP_ERRBIT_STALE_LAYOUT);
      }
      if (slot_lo >= p.cap) {
        set_error(p.error_word, EP_ERRBIT_CAPACITY);
        slot_lo = -1;
      }
      if (slot_hi >= p.cap) {
        set_error(p.error_word, EP_ERRBIT_CAPACITY);
        slot_hi = -1;
      }
      if (p.stats != nullptr) count_received(p, e, slot_lo, slot_hi, lane);
      const int dest = marked_dest(p, e, lane);
      const int local = dest >= 0 ? local_expert(p, e) : -1;
      // received metadata: needs no shared memory, runs ahead of the cast
      for (int r = 0; r < p.D; ++r) {
        const int slot = __shfl_sync(0xffffffffu, r < kWarpSize ? slot_lo : slot_hi, r & (kWarpSize - 1));
        if (slot < 0) continue;
        if (lane == 0 && p.recv_src_idx != nullptr) p.recv_src_idx[slot] = t;
        if (lane < p.K) {
          const bool here = dest == r;
          if (p.recv_topk_idx != nullptr) p.recv_topk_idx[(size_t)slot * p.K + lane] = here ? local : -1;
          if (p.recv_topk_weights != nullptr) p.recv_topk_weights[(size_t)slot * p.K + lane] = here ? w : 0.0f;
        }
      }
      if constexpr (!CAST) {  // bf16: the row goes out from its input stage
        const int s = i % S;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full_in[s], (uint32_t)(i / S) & 1u))) {
          if (lane == 0) {
            *s_abort = 1;
            set_error(p.error_word, EP_ERRBIT_TIMEOUT);
          }
          break;
        }
        if (lane == 0) s_tok[i % kTokRing] = kTokPending;
        const unsigned char *stage = in + (size_t)s * p.stage_stride;
        if (slot_lo >= 0)
          bulk_store(static_cast<unsigned char *>(p.recv_x) + (size_t)slot_lo * p.row_out_bytes, stage,
                     p.row_out_bytes);
        if (slot_hi >= 0)
          bulk_store(static_cast<unsigned char *>(p.recv_x) + (size_t)slot_hi * p.row_out_bytes, stage,
                     p.row_out_bytes);
        bulk_commit();
        // the stores of token i-1 have read their stage: the loader may refill it
        bulk_wait_read<1>();
        __syncwarp();
        if (lane == 0 && i > 0) mbar_arrive(&empty_in[(i - 1) % S]);
        continue;
      }
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full_out[o], (uint32_t)(i / kWsOut) & 1u));
      if (!ok) {
        if (lane == 0) {
          *s_abort = 1;
          set_error(p.error_word, EP_ERRBIT_TIMEOUT);
        }
        break;
      }
      __syncwarp();
      if (lane == 0) s_tok[i % kTokRing] = kTokPending;  // every caster has read it
      const unsigned char *orow = out + (size_t)o * p.out_stride;
      const float *oscale = osc + (size_t)o * (p.scale_stride / 4);
      if (p.packed) {  // codes, scales and padding go out as one row
        if (slot_lo >= 0)
          bulk_store(static_cast<unsigned char *>(p.recv_x) + (size_t)slot_lo * p.row_out_bytes, orow,
                     p.row_out_bytes);
        if (slot_hi >= 0)
          bulk_store(static_cast<unsigned char *>(p.recv_x) + (size_t)slot_hi * p.row_out_bytes, orow,
                     p.row_out_bytes);
        bulk_commit();
        release_out(empty_out, i, lane);
        continue;
      }
      if (slot_lo >= 0) {
        bulk_store(static_cast<unsigned char *>(p.recv_x) + (size_t)slot_lo * p.H, orow, p.row_out_bytes);
        if (scale_bulk) bulk_store(p.recv_x_scales + (size_t)slot_lo * p.groups, oscale, p.scale_stride);
      }
      if (slot_hi >= 0) {
        bulk_store(static_cast<unsigned char *>(p.recv_x) + (size_t)slot_hi * p.H, orow, p.row_out_bytes);
        if (scale_bulk) bulk_store(p.recv_x_scales + (size_t)slot_hi * p.groups, oscale, p.scale_stride);
      }
      bulk_commit();
      if (!scale_bulk) {
        s_slot[lane] = slot_lo;
        if (p.D > kWarpSize) s_slot[lane + kWarpSize] = slot_hi;
        __syncwarp();
        const int RG = p.D * p.groups;
        for (int q = lane; q < RG; q += kWarpSize) {
          const int r = q / p.groups;
          const int g = q - r * p.groups;
          const int slot = s_slot[r];
          if (slot >= 0) p.recv_x_scales[(size_t)slot * p.groups + g] = oscale[g];
        }
      }
      release_out(empty_out, i, lane);
    }
    bulk_wait<0>();
    if (lane == 0) EP_TRACE_MARK(g_trace_dispatch, 5);
  } else if (CAST) {
    const int cw = warp - 2;
    for (int i = 0; !*s_abort; ++i) {
      const int s = i % S;
      const int o = i % kWsOut;
      bool ok = mbar_wait_bounded(&full_in[s], (uint32_t)(i / S) & 1u);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          *s_abort = 1;
          set_error(p.error_word, EP_ERRBIT_TIMEOUT);
        }
        break;
      }
      const int tc = s_tok[i % kTokRing];
      if (tc < 0 || tc >= p.T) break;  // the end (the storer flags a bad entry)
      if (i >= kWsOut) ok = mbar_wait_bounded(&empty_out[o], (uint32_t)(i / kWsOut - 1) & 1u);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          *s_abort = 1;
          set_error(p.error_word, EP_ERRBIT_TIMEOUT);
        }
        break;
      }
      const unsigned char *stage = in + (size_t)s * p.stage_stride;
      unsigned char *orow = out + (size_t)o * p.out_stride;
      float *oscale = p.packed ? reinterpret_cast<float *>(orow + p.H) : osc + (size_t)o * (p.scale_stride / 4);
      for (int g0 = 2 * cw; g0 < p.groups; g0 += 2 * kWsCasters)
        cast_two_groups(stage, orow, oscale, g0, p.groups, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&empty_in[s]);
        mbar_arrive(&full_out[o]);
      }
    }
  }

  // After an abort, loads still in flight are waited for (bounded) before
  // the CTA's shared memory is released.  Only the latest load of each stage
  // (the last S issued) can still be in flight.
  __syncthreads();
  if (*s_abort && tid == 0) {
    for (int m = max(0, issued - S); m < issued; ++m) (void)mbar_wait_bounded(&full_in[m % S], (uint32_t)(m / S) & 1u);
  }
}

__global__ void __launch_bounds__(kWsThreads) dispatch_ws_kernel(DispatchParams p) { dispatch_ws_body<true>(p); }
__global__ void __launch_bounds__(kWsBf16Threads) dispatch_ws_bf16_kernel(DispatchParams p) {
  dispatch_ws_body<false>(p);
}

size_t ws_smem_bytes(const DispatchParams &p) {
  return kHeaderBytes + (size_t)p.stages * p.stage_stride + kWsOut * ((size_t)p.out_stride + p.scale_stride);
}

ep_status_t launch_ws(DispatchParams &p, const DeviceInfo &di, cudaStream_t stream) {
  static std::mutex mu;
  static bool configured[64] = {};
  {
    std::lock_guard<std::mutex> g(mu);
    if (di.device < 64 && !configured[di.device]) {
      cudaError_t e = cudaFuncSetAttribute(dispatch_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)di.max_smem_per_block_optin);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(dispatch_ws_kernel)");
      configured[di.device] = true;
    }
  }
  p.stages = kWsStages;
  while (p.stages > 2 && ws_smem_bytes(p) > kWsSmemBudget) --p.stages;
  p.table_offset = (uint32_t)ws_smem_bytes(p);
  const size_t smem = ws_smem_bytes(p) + base_table_bytes(p.table_blocks, p.R);
  if (smem > di.max_smem_per_block_optin)
    return fail(EP_ERR_UNSUPPORTED, "ep_dispatch: hidden %d needs %zu bytes of shared memory", p.H, smem);
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_ws_kernel, kWsThreads, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(dispatch_ws)");
  if (per_sm <= 0) return fail(EP_ERR_UNSUPPORTED, "ep_dispatch: kernel cannot be resident");
  const int grid = std::min(p.T, per_sm * di.num_sms);
  e = launch_kernel(dispatch_ws_kernel, grid, kWsThreads, smem, stream, false, p);
  if (e != cudaSuccess) return cuda_fail(e, "launch dispatch_ws_kernel");
  return EP_OK;
}

// bf16 rows through the warp-specialised kernel's loader and storer.
ep_status_t launch_ws_bf16(DispatchParams &p, const DeviceInfo &di, cudaStream_t stream) {
  static std::mutex mu;
  static bool configured[64] = {};
  {
    std::lock_guard<std::mutex> g(mu);
    if (di.device < 64 && !configured[di.device]) {
      cudaError_t e = cudaFuncSetAttribute(dispatch_ws_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)di.max_smem_per_block_optin);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(dispatch_ws_bf16_kernel)");
      configured[di.device] = true;
    }
  }
  auto smem_of = [&](int stages) { return kHeaderBytes + (size_t)stages * p.stage_stride; };
  p.stages = kWsBf16Stages;
  while (p.stages > 2 && smem_of(p.stages) > kWsBf16SmemBudget) --p.stages;
  p.table_offset = (uint32_t)smem_of(p.stages);
  const size_t smem = smem_of(p.stages) + base_table_bytes(p.table_blocks, p.R);
  if (smem > di.max_smem_per_block_optin)
    return fail(EP_ERR_UNSUPPORTED, "ep_dispatch: hidden %d needs %zu bytes of shared memory", p.H, smem);
  int per_sm = 0;
  cudaError_t e =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_ws_bf16_kernel, kWsBf16Threads, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(dispatch_ws_bf16)");
  if (per_sm <= 0) return fail(EP_ERR_UNSUPPORTED, "ep_dispatch: kernel cannot be resident");
  const int grid = std::min(p.T, per_sm * di.num_sms);
  e = launch_kernel(dispatch_ws_bf16_kernel, grid, kWsBf16Threads, smem, stream, false, p);
  if (e != cudaSuccess) return cuda_fail(e, "launch dispatch_ws_bf16_kernel");
  return EP_OK;
}


// ------------------------------------------------------------------------
// Padding rows of an expanded layout (zero_padding): each expert's rows past
// its last selection, up to the aligned end of its segment, get a zero
// payload (and zero scales), source -1, all top-k slots -1 and weights 0.
// Every block scans the experts' padding counts into a prefix in shared
// memory; the padding rows are numbered 0.. across experts and row g goes to
// block g % gridDim.x, one row per thread, which finds its expert by binary
// search and zeroes the row with bulk stores from a zeroed shared buffer.

constexpr int kPadThreads = 128;
constexpr int kPadZeroBytes = 8192;

size_t pad_smem_bytes(int E) { return kPadZeroBytes + (size_t)(E + 1) * sizeof(int32_t); }

__global__ void __launch_bounds__(kPadThreads) pad_kernel(DispatchParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *zero = smem;                                   // [kPadZeroBytes]
  int *pre = reinterpret_cast<int *>(smem + kPadZeroBytes);     // [E + 1] padding rows before expert e
  const int tid = threadIdx.x;
  for (int i = tid; i < kPadZeroBytes / 16; i += kPadThreads)
    reinterpret_cast<int4 *>(zero)[i] = make_int4(0, 0, 0, 0);
  fence_proxy_async_smem();
  griddep_wait();
  griddep_launch_dependents();

  // exclusive prefix of the padding counts: a contiguous run of experts per
  // thread, then thread 0 scans the runs' sums
  const int E = p.E;
  const int per = (E + kPadThreads - 1) / kPadThreads;
  const int e0 = min(tid * per, E), e1 = min(e0 + per, E);
  int mine = 0;
  for (int e = e0; e < e1; ++e) mine += __ldg(p.xoff + e + 1) - __ldg(p.xoff + e) - __ldg(p.xrows + e);
  __shared__ int runs[kPadThreads + 1];
  runs[tid] = mine;
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int i = 0; i < kPadThreads; ++i) {
      const int v = runs[i];
      runs[i] = acc;
      acc += v;
    }
    runs[kPadThreads] = acc;
  }
  __syncthreads();
  {
    int acc = runs[tid];
    for (int e = e0; e < e1; ++e) {
      pre[e] = acc;
      acc += __ldg(p.xoff + e + 1) - __ldg(p.xoff + e) - __ldg(p.xrows + e);
    }
    if (tid == 0) pre[E] = runs[kPadThreads];
  }
  __syncthreads();

  const int total = pre[E];
  const bool scale_bulk = p.groups > 0 && !p.packed && (p.groups * 4) % 16 == 0 &&
                          (reinterpret_cast<uintptr_t>(p.recv_x_scales) & 15u) == 0;
  for (int g = blockIdx.x + tid * (int)gridDim.x; g < total; g += kPadThreads * (int)gridDim.x) {
    int lo = 0, hi = E;  // the expert e with pre[e] <= g < pre[e + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pre[mid] <= g) lo = mid;
      else hi = mid;
    }
    const int s = __ldg(p.xoff + lo) + __ldg(p.xrows + lo) + (g - pre[lo]);
    if (s < 0 || s >= p.cap) {
      set_error(p.error_word, EP_ERRBIT_CAPACITY);
      continue;
    }
    unsigned char *row = static_cast<unsigned char *>(p.recv_x) + (size_t)s * p.row_out_bytes;
    for (uint32_t off = 0; off < p.row_out_bytes; off += kPadZeroBytes)
      bulk_store(row + off, zero, min((uint32_t)kPadZeroBytes, p.row_out_bytes - off));
    if (scale_bulk) {
      bulk_store(p.recv_x_scales + (size_t)s * p.groups, zero, (uint32_t)p.groups * 4u);
    } else if (p.groups > 0 && !p.packed) {
      for (int q = 0; q < p.groups; ++q) p.recv_x_scales[(size_t)s * p.groups + q] = 0.0f;
    }
    if (p.recv_src_idx != nullptr) p.recv_src_idx[s] = -1;
    for (int k = 0; k < p.K; ++k) {
      if (p.recv_topk_idx != nullptr) p.recv_topk_idx[(size_t)s * p.K + k] = -1;
      if (p.recv_topk_weights != nullptr) p.recv_topk_weights[(size_t)s * p.K + k] = 0.0f;
    }
  }
  bulk_commit();
  bulk_wait_read<0>();  // the stores have read the zero buffer before the block exits
}

ep_status_t launch_pad(const DispatchParams &p, const DeviceInfo &di, cudaStream_t stream) {
  const size_t smem = pad_smem_bytes(p.E);  // under 48 KB for every E <= EP_MAX_EXPERTS
  static_assert(kPadZeroBytes + (EP_MAX_EXPERTS + 1) * 4 + (kPadThreads + 1) * 4 <= 48 * 1024,
                "pad_kernel fits the default shared-memory limit");
  const int grid = 2 * di.num_sms;
  // An ordinary stream-ordered launch, not a programmatic dependent of the
  // dispatch: measured on GB300, padding blocks launched early sit on the
  // SMs beside the warp-specialised dispatch and slow it (~170 against
  // ~120 us for 82 176 rows of 7168 at the 8192-token, top-8 workload).
  pad_kernel<<<grid, kPadThreads, smem, stream>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch pad_kernel");
  return EP_OK;
}

size_t dispatch_smem_bytes(const DispatchParams &p) { return kHeaderBytes + (size_t)p.stages * p.stage_stride; }

// bf16 rows of an expanded layout.
ep_status_t launch_ring(DispatchParams &p, const DeviceInfo &di, cudaStream_t stream) {
  static std::mutex mu;
  static bool configured[64] = {};
  {
    std::lock_guard<std::mutex> g(mu);
    if (di.device < 64 && !configured[di.device]) {
      cudaError_t e = cudaFuncSetAttribute(dispatch_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)di.max_smem_per_block_optin);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(dispatch_ring_kernel)");
      configured[di.device] = true;
    }
  }
  // Deepest ring that keeps the CTA within budget (at least 2 stages).
  p.stages = kMaxStages > 4 ? 4 : kMaxStages;
  while (p.stages > 2 && dispatch_smem_bytes(p) > kSmemBudget) --p.stages;
  const size_t smem = dispatch_smem_bytes(p);
  if (smem > di.max_smem_per_block_optin)
    return fail(EP_ERR_UNSUPPORTED, "ep_dispatch: hidden %d needs %zu bytes of shared memory", p.H, smem);
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_ring_kernel,
                                                                kDispatchThreads, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(dispatch)");
  if (per_sm <= 0) return fail(EP_ERR_UNSUPPORTED, "ep_dispatch: kernel cannot be resident");
  const int grid = std::min(p.T, per_sm * di.num_sms);
  e = launch_kernel(dispatch_ring_kernel, grid, kDispatchThreads, smem, stream, false, p);
  if (e != cudaSuccess) return cuda_fail(e, "launch dispatch_ring_kernel");
  return EP_OK;
}

}  // namespace

ep_status_t launch_dispatch(const DispatchArgs &a, cudaStream_t stream) {
  const bool pad = a.expanded && a.zero_padding;
  if (a.num_tokens == 0 && !pad) return EP_OK;
  const DeviceInfo *di = current_device_info();
  if (di == nullptr) return EP_ERR_CUDA;
  DispatchParams p = {};
  p.D = a.expanded ? a.num_topk : a.num_ranks;
  p.expanded = a.expanded;
  p.xoff = a.expert_offset;
  p.xrows = a.num_rows_per_expert;
  p.zero_padding = a.zero_padding;
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
  p.stats = a.recv_stats;
  p.packed = a.packed_row_bytes > 0;
  p.row_in_bytes = 2u * (uint32_t)a.hidden;
  p.row_out_bytes = p.packed ? (uint32_t)a.packed_row_bytes : a.fp8 ? (uint32_t)a.hidden : 2u * (uint32_t)a.hidden;
  p.stage_stride = (p.row_in_bytes + 127u) / 128u * 128u;
  p.out_stride = a.fp8 ? (p.row_out_bytes + 127u) / 128u * 128u : 0u;
  p.scale_stride = (a.fp8 && !p.packed) ? ((uint32_t)p.groups * 4u + 15u) / 16u * 16u : 0u;
  p.tokens.ticket = a.work_counters;
  p.tokens.done = a.work_counters != nullptr ? a.work_counters + 1 : nullptr;
  p.tokens.T = a.num_tokens;
  p.early = a.early_rows;
  p.local_base = a.local_base;
  p.token_slot_out = a.token_slot_out;
  p.num_tokens_per_expert = a.num_tokens_per_expert;
  p.table_blocks = a.local_base != nullptr ? a.local_table_blocks : 0;
  p.rank_prefix = a.rank_prefix;
  p.num_tokens_per_rank = a.num_tokens_per_rank;
  ep_status_t st = EP_OK;
  if (a.num_tokens > 0) {
    // packed rows are only built by the warp-specialised kernel
    if (a.fp8)
      st = launch_ws(p, *di, stream);
    else
      st = (kBf16WarpSpecialised && !p.expanded) || p.local_base != nullptr ? launch_ws_bf16(p, *di, stream)
                                                                            : launch_ring(p, *di, stream);
  }
  if (st == EP_OK && pad) st = launch_pad(p, *di, stream);
  return st;
}

}  // namespace ep

EP_TRACE_READER(ep_trace_read_dispatch, ep::g_trace_dispatch);
