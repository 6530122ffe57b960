/*
 * CPU oracle for MoE expert-parallel layout / dispatch / combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant generator with
 * the CUDA library; it is written directly from the definitions below, in
 * plain loops, so that a reader can check it against the sources by eye.
 *
 * Sources (pages, by title and section):
 *   [TS-PR]     TileScale PR #68 "[Example] EP v2 intranode dispatch/combine",
 *               PR summary: dispatch = count, count exchange, scatter straight
 *               to the final compact index; combine = one block per source
 *               token reducing the rows its token was sent as; payload bf16
 *               or fp8 with per-token, per-128-element scales.
 *   [TS-DESIGN] same page, README section "Design": count deduplicates each
 *               (token, destination) pair; the exchange gives every sender a
 *               base send_base[d]; the scatter adds a locally claimed slot.
 *   [TS-MASK]   same page, commit message on the masked-topk case: -1 in
 *               topk_idx is "no selection"; a token with no selection at all
 *               combines back to zero.
 *   [TS-FP8]    same page, commit message on packing the fp8 row: per-token
 *               per-128-element fp32 scales in DeepEP's per_token_cast_to_fp8
 *               layout.
 *   [TS-EXPAND] same page, commit message on do_expand: "local expert",
 *               experts_per_rank, phase 1 tallies per destination, phase 2
 *               turns tallies into a base, phase 3 adds a locally-claimed slot.
 *   [TS-STATS]  same page, commit message adding cumulative recv stats and
 *               combine bias: recv_topk_idx holds the local expert of every
 *               received (row, top-k slot).
 *   [TS-PACK]   same page, commit message on packing the fp8 row: payload,
 *               then the per-group fp32 scales, in one row padded to 16
 *               bytes always and to 512 only when that padding costs under 5%.
 *   [TS-BIAS]   same page, commit message adding combine bias and cumulative
 *               recv stats: bias_0/bias_1 seed the reduce accumulator; the
 *               stats accumulate each local expert's received count.
 *   [TS-EXPAND] (also) one received row per (token, expert) instead of per
 *               (token, rank), grouped by local expert, each segment rounded
 *               up to expert_alignment rows, zero_padding clearing the gap;
 *               an expanded row marks only the expert it belongs to; the
 *               expanded combine sums a token's rows (kDoExpandedSend).
 *   [TS-CACHE]  same page, commit messages on the cached-layout dispatch
 *               (handle=): a layout depends only on the routing; a stale one
 *               misroutes silently, so it is guarded.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - expert e lives on rank floor(e / (E/R)) (contiguous blocks).
 *   - slots inside a rank are claimed in ascending token order (stable).
 *   - received rows are rank-major: rank 0's block, then rank 1's, ...
 *   - an index outside [-1, E) is treated as -1 and flags EP_ORA_BAD_INDEX.
 *   - combine bias: acc starts at bias0 (else 0), then acc = acc + bias1.
 *   - recv stats: stats[e] += 1 for every received (row, top-k slot) whose
 *     expert is e (rank r's local expert e - r*E/R).
 *   - packed row: the 5% is the padding of the 512-byte form relative to the
 *     unpadded row (the page's +3.9% at hidden 7168, +21% at 2048, +9% at
 *     4096); padding bytes are zero.
 *   - expanded layout: rows are expert-major (rank-major, then local
 *     expert); inside an expert's segment in ascending (token, k) order;
 *     a token naming an expert a second time gets no second row (flag
 *     EP_ORA_DUP); padding rows, when zero_padding is asked for, hold zeros
 *     and are marked unoccupied (source -1, every top-k slot -1, weight 0);
 *     the expanded combine adds a token's rows in ascending row order, each
 *     times its own gate weight (or 1), in fp32 after the biases.
 *   - stale layout: dispatch and weighted combine flag EP_ORA_STALE for a
 *     token whose set of ranks under the routing they are given differs
 *     from the ranks with a slot in the layout (the slots depend on nothing
 *     else, so a routing with the same rank sets may reuse the layout).
 *   - fp8: amax = max |x| over the group, scale = amax / 448 (fp32 division,
 *     round to nearest even), q = e4m3(x / scale) rounded to nearest even
 *     with saturation at +-448; an all-zero group has scale 0 and keeps the
 *     sign of each zero.
 *   - combine: acc = 0; for ranks in ascending order acc = acc + c * y
 *     (separate fp32 multiply and add; c = 1 without weights, else the fp32
 *     sum in k order of the weights of the token's experts on that rank);
 *     out = bf16(acc) rounded to nearest even.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (the flag forbids
 * fused multiply-add so that every float operation rounds on its own).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define EP_ORA_BAD_INDEX 1
#define EP_ORA_CAPACITY 2
#define EP_ORA_STALE 8      /* routing and layout disagree on a token's ranks */
#define EP_ORA_DUP 16       /* expanded layout: a token names an expert twice */

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
float ora_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bf16, round to nearest, ties to even.  NaN stays NaN. */
uint16_t ora_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)             /* NaN: keep it quiet */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;                          /* truncated value */
    uint32_t dropped = u & 0xffffu;                   /* discarded half */
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1;                                    /* carries into exponent */
    return (uint16_t)kept;
}

/*
 * float8 e4m3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite 448.
 * Exponent field 0 holds subnormals m * 2^-9.
 */
double ora_e4m3_to_f64(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return s ? -NAN : NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Magnitudes of codes 0x00..0x7e, ascending (the format is monotone). */
static double g_e4m3_mag[127];
static int g_e4m3_ready;

static void e4m3_table(void)
{
    if (g_e4m3_ready)
        return;
    for (int c = 0; c < 127; ++c)
        g_e4m3_mag[c] = ora_e4m3_to_f64((uint8_t)c);
    g_e4m3_ready = 1;
}

/* Nearest e4m3 code, ties to the even code (even mantissa), saturating to
 * +-448.  The sign of zero is kept.  NaN maps to NaN. */
uint8_t ora_f32_to_e4m3(float x)
{
    e4m3_table();
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x))
        return (uint8_t)(sign | 0x7f);
    double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7e);
    /* largest code whose magnitude is <= a (binary search on the table) */
    int lo = 0, hi = 126;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (g_e4m3_mag[mid] <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    /* a lies in [mag[lo], mag[lo+1]); both distances are exact in double */
    double below = a - g_e4m3_mag[lo];
    double above = g_e4m3_mag[lo + 1] - a;
    int code;
    if (below < above)
        code = lo;
    else if (above < below)
        code = lo + 1;
    else
        code = (lo & 1) ? lo + 1 : lo;   /* tie: the code with even mantissa */
    return (uint8_t)(sign | code);
}

/*
 * Per-token, per-128-element fp8 cast of one bf16 row of length H
 * (H a multiple of 128).  q receives H codes, scales receives H/128 floats.
 */
void ora_quantize_row(const uint16_t *x, int H, uint8_t *q, float *scales)
{
    for (int g = 0; g < H / 128; ++g) {
        const uint16_t *xg = x + (size_t)g * 128;
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            float a = fabsf(ora_bf16_to_f32(xg[i]));
            if (a > amax)
                amax = a;
        }
        float scale = amax / 448.0f;
        scales[g] = scale;
        for (int i = 0; i < 128; ++i) {
            float v = ora_bf16_to_f32(xg[i]);
            /* an all-zero group: every element is +-0 and stays so */
            float u = (amax > 0.0f) ? v / scale : v;
            q[(size_t)g * 128 + i] = ora_f32_to_e4m3(u);
        }
    }
}

/* ------------------------------------------------------------------ */
/* Layout: dedup per (token, rank), histograms, stable slots           */
/* ------------------------------------------------------------------ */

static int valid_expert(int64_t e, int E) { return e >= 0 && e < E; }

/*
 * Outputs (all caller-allocated):
 *   num_tokens_per_expert [E], num_tokens_per_rank [R], rank_prefix [R+1],
 *   is_token_in_rank [T*R], token_slot [T*R] (-1 where absent).
 * Returns error bits (EP_ORA_BAD_INDEX).
 */
int ora_get_layout(const int64_t *topk_idx, int T, int K, int E, int R,
                   int32_t *num_tokens_per_expert, int32_t *num_tokens_per_rank,
                   int32_t *rank_prefix, uint8_t *is_token_in_rank,
                   int32_t *token_slot)
{
    int err = 0;
    int epr = E / R;
    memset(num_tokens_per_expert, 0, sizeof(int32_t) * (size_t)E);
    memset(num_tokens_per_rank, 0, sizeof(int32_t) * (size_t)R);
    memset(is_token_in_rank, 0, (size_t)T * (size_t)R);

    /* Count: every valid selection counts for its expert; a token is in a
     * rank once, however many of its experts that rank holds. */
    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[(size_t)t * K + k];
            if (e == -1)
                continue;
            if (!valid_expert(e, E)) {
                err |= EP_ORA_BAD_INDEX;
                continue;
            }
            num_tokens_per_expert[e] += 1;
            is_token_in_rank[(size_t)t * R + (size_t)(e / epr)] = 1;
        }
    }
    for (int t = 0; t < T; ++t)
        for (int r = 0; r < R; ++r)
            num_tokens_per_rank[r] += is_token_in_rank[(size_t)t * R + r];

    /* Exchange, collapsed to one sender: the base of rank r's block. */
    rank_prefix[0] = 0;
    for (int r = 0; r < R; ++r)
        rank_prefix[r + 1] = rank_prefix[r] + num_tokens_per_rank[r];

    /* Slots: base plus a running count, claimed in token order. */
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)R);
    for (int r = 0; r < R; ++r)
        next[r] = rank_prefix[r];
    for (int t = 0; t < T; ++t)
        for (int r = 0; r < R; ++r)
            token_slot[(size_t)t * R + r] =
                is_token_in_rank[(size_t)t * R + r] ? next[r]++ : -1;
    free(next);
    return err;
}

/* 1 if token t's ranks under topk_idx are exactly its ranks with a slot. */
static int ranks_agree(const int64_t *topk_idx, int t, int K, int E, int R,
                       const int32_t *token_slot)
{
    int epr = E / R;
    for (int r = 0; r < R; ++r) {
        int routed = 0;
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[(size_t)t * K + k];
            if (valid_expert(e, E) && (int)(e / epr) == r)
                routed = 1;
        }
        if (routed != (token_slot[(size_t)t * R + r] >= 0))
            return 0;
    }
    return 1;
}

/* ------------------------------------------------------------------ */
/* Dispatch: scatter (bf16 or fp8) plus received metadata               */
/* ------------------------------------------------------------------ */

/* Bytes of one packed fp8 row (payload, scales, zero padding). */
int ora_fp8_packed_row_bytes(int H)
{
    int raw = H + (H / 128) * 4;
    int pad16 = (raw + 15) / 16 * 16;
    int pad512 = (raw + 511) / 512 * 512;
    return (pad512 - raw) * 20 < raw ? pad512 : pad16;   /* under 5% */
}

/*
 * fp8 == 0: recv_x is uint16 [cap * H], a bit copy of each row.
 * fp8 == 1: recv_x is uint8 [cap * H], recv_x_scales float [cap * H/128].
 * fp8 == 2: recv_x is uint8 [cap * ora_fp8_packed_row_bytes(H)]: each row
 *   holds the H codes, then the H/128 scales, then zero padding.
 * recv_src_idx [cap], recv_topk_idx [cap*K], recv_topk_weights [cap*K] and
 * stats [E] may be NULL.  Rows with slot >= cap are skipped and flag
 * EP_ORA_CAPACITY.
 */
int ora_dispatch_ex(const uint16_t *x, int T, int H, const int64_t *topk_idx,
                    const float *topk_weights, int K, int E, int R,
                    const int32_t *token_slot, int fp8, void *recv_x,
                    float *recv_x_scales, int32_t *recv_src_idx,
                    int32_t *recv_topk_idx, float *recv_topk_weights, int cap,
                    uint32_t *stats)
{
    int err = 0;
    int epr = E / R;
    int G = H / 128;
    uint8_t *q = NULL;
    float *sc = NULL;
    if (fp8) {
        q = (uint8_t *)malloc((size_t)H);
        sc = (float *)malloc(sizeof(float) * (size_t)(G > 0 ? G : 1));
    }
    for (int t = 0; t < T; ++t) {
        const uint16_t *row = x + (size_t)t * H;
        int quantised = 0;
        if (!ranks_agree(topk_idx, t, K, E, R, token_slot))
            err |= EP_ORA_STALE;
        for (int r = 0; r < R; ++r) {
            int32_t slot = token_slot[(size_t)t * R + r];
            if (slot < 0)
                continue;
            if (slot >= cap) {
                err |= EP_ORA_CAPACITY;
                continue;
            }
            if (!fp8) {
                memcpy((uint16_t *)recv_x + (size_t)slot * H, row,
                       sizeof(uint16_t) * (size_t)H);
            } else {
                if (!quantised) {
                    ora_quantize_row(row, H, q, sc);
                    quantised = 1;
                }
                if (fp8 == 1) {
                    memcpy((uint8_t *)recv_x + (size_t)slot * H, q, (size_t)H);
                    memcpy(recv_x_scales + (size_t)slot * G, sc,
                           sizeof(float) * (size_t)G);
                } else {
                    size_t rb = (size_t)ora_fp8_packed_row_bytes(H);
                    uint8_t *dst = (uint8_t *)recv_x + (size_t)slot * rb;
                    memset(dst, 0, rb);
                    memcpy(dst, q, (size_t)H);
                    memcpy(dst + H, sc, sizeof(float) * (size_t)G);
                }
            }
            if (recv_src_idx)
                recv_src_idx[slot] = t;
            for (int k = 0; k < K; ++k) {
                int64_t e = topk_idx[(size_t)t * K + k];
                int here = valid_expert(e, E) && (int)(e / epr) == r;
                if (recv_topk_idx)
                    recv_topk_idx[(size_t)slot * K + k] =
                        here ? (int32_t)(e - (int64_t)r * epr) : -1;
                if (recv_topk_weights)
                    recv_topk_weights[(size_t)slot * K + k] =
                        here ? topk_weights[(size_t)t * K + k] : 0.0f;
                if (stats && here)
                    stats[e] += 1;
            }
        }
    }
    free(q);
    free(sc);
    return err;
}

int ora_dispatch(const uint16_t *x, int T, int H, const int64_t *topk_idx,
                 const float *topk_weights, int K, int E, int R,
                 const int32_t *token_slot, int fp8, void *recv_x,
                 float *recv_x_scales, int32_t *recv_src_idx,
                 int32_t *recv_topk_idx, float *recv_topk_weights, int cap)
{
    return ora_dispatch_ex(x, T, H, topk_idx, topk_weights, K, E, R,
                           token_slot, fp8, recv_x, recv_x_scales,
                           recv_src_idx, recv_topk_idx, recv_topk_weights,
                           cap, NULL);
}

/* ------------------------------------------------------------------ */
/* Combine: per-token gather-reduce in ascending rank order            */
/* ------------------------------------------------------------------ */

/*
 * y: uint16 bf16 [cap * H], row s is the expert-stage output for received
 * row s.  out: uint16 bf16 [T * H].  topk_weights == NULL: plain sum.
 * bias0, bias1: bf16 [T * H] or NULL; they seed the accumulator.
 */
int ora_combine_ex(const uint16_t *y, int cap, int H, const int32_t *token_slot,
                   int T, int R, const int64_t *topk_idx,
                   const float *topk_weights, int K, int E,
                   const uint16_t *bias0, const uint16_t *bias1, uint16_t *out)
{
    int err = 0;
    int epr = (R > 0) ? E / R : 0;
    float *acc = (float *)malloc(sizeof(float) * (size_t)(H > 0 ? H : 1));
    for (int t = 0; t < T; ++t) {
        if (topk_weights && !ranks_agree(topk_idx, t, K, E, R, token_slot))
            err |= EP_ORA_STALE;
        for (int h = 0; h < H; ++h) {
            acc[h] = bias0 ? ora_bf16_to_f32(bias0[(size_t)t * H + h]) : 0.0f;
            if (bias1)
                acc[h] = acc[h] + ora_bf16_to_f32(bias1[(size_t)t * H + h]);
        }
        for (int r = 0; r < R; ++r) {
            int32_t slot = token_slot[(size_t)t * R + r];
            if (slot < 0)
                continue;
            if (slot >= cap) {
                err |= EP_ORA_CAPACITY;
                continue;
            }
            const uint16_t *row = y + (size_t)slot * H;
            if (topk_weights) {
                float c = 0.0f;
                for (int k = 0; k < K; ++k) {
                    int64_t e = topk_idx[(size_t)t * K + k];
                    if (valid_expert(e, E) && (int)(e / epr) == r)
                        c = c + topk_weights[(size_t)t * K + k];
                }
                for (int h = 0; h < H; ++h) {
                    float p = c * ora_bf16_to_f32(row[h]);
                    acc[h] = acc[h] + p;
                }
            } else {
                for (int h = 0; h < H; ++h)
                    acc[h] = acc[h] + ora_bf16_to_f32(row[h]);
            }
        }
        for (int h = 0; h < H; ++h)
            out[(size_t)t * H + h] = ora_f32_to_bf16(acc[h]);
    }
    free(acc);
    return err;
}

int ora_combine(const uint16_t *y, int cap, int H, const int32_t *token_slot,
                int T, int R, const int64_t *topk_idx,
                const float *topk_weights, int K, int E, uint16_t *out)
{
    return ora_combine_ex(y, cap, H, token_slot, T, R, topk_idx, topk_weights,
                          K, E, NULL, NULL, out);
}

/* ------------------------------------------------------------------ */
/* Array forms of the format functions (used by the pin tests)         */
/* ------------------------------------------------------------------ */

void ora_f32_to_e4m3_array(const float *x, long n, uint8_t *q)
{
    for (long i = 0; i < n; ++i)
        q[i] = ora_f32_to_e4m3(x[i]);
}

void ora_f32_to_bf16_array(const float *x, long n, uint16_t *b)
{
    for (long i = 0; i < n; ++i)
        b[i] = ora_f32_to_bf16(x[i]);
}


/* ------------------------------------------------------------------ */
/* Expanded layout: one row per (token, expert), grouped by expert      */
/* ------------------------------------------------------------------ */

/* 1 if topk_idx[t][k] is a valid expert not named at an earlier k of t. */
static int first_choice(const int64_t *topk_idx, int t, int k, int K, int E)
{
    int64_t e = topk_idx[(size_t)t * K + k];
    if (!valid_expert(e, E))
        return 0;
    for (int j = 0; j < k; ++j)
        if (topk_idx[(size_t)t * K + j] == e)
            return 0;
    return 1;
}

/*
 * Outputs: num_rows_per_expert [E] (rows, one per first choice),
 * expert_offset [E+1] (aligned exclusive prefix; [E] = rows incl. padding),
 * token_slot [T*K] (row of (t, k), -1 where none).  Returns error bits.
 */
int ora_get_layout_expanded(const int64_t *topk_idx, int T, int K, int E,
                            int align, int32_t *num_rows_per_expert,
                            int32_t *expert_offset, int32_t *token_slot)
{
    int err = 0;
    memset(num_rows_per_expert, 0, sizeof(int32_t) * (size_t)E);
    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[(size_t)t * K + k];
            if (e == -1)
                continue;
            if (!valid_expert(e, E)) {
                err |= EP_ORA_BAD_INDEX;
                continue;
            }
            if (!first_choice(topk_idx, t, k, K, E)) {
                err |= EP_ORA_DUP;
                continue;
            }
            num_rows_per_expert[e] += 1;
        }
    }
    expert_offset[0] = 0;
    for (int e = 0; e < E; ++e) {
        int rows = num_rows_per_expert[e];
        int aligned = (rows + align - 1) / align * align;
        expert_offset[e + 1] = expert_offset[e] + aligned;
    }
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; ++e)
        next[e] = expert_offset[e];
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k)
            token_slot[(size_t)t * K + k] =
                first_choice(topk_idx, t, k, K, E)
                    ? next[topk_idx[(size_t)t * K + k]]++ : -1;
    free(next);
    return err;
}

/* Whether the expanded layout's slots of token t match its first choices. */
static int choices_agree(const int64_t *topk_idx, int t, int K, int E,
                         const int32_t *token_slot)
{
    for (int k = 0; k < K; ++k)
        if (first_choice(topk_idx, t, k, K, E) != (token_slot[(size_t)t * K + k] >= 0))
            return 0;
    return 1;
}

/*
 * Expanded dispatch.  fp8 as in ora_dispatch_ex (0 bf16, 1 fp8 + scales,
 * 2 packed).  Padding rows of each expert's segment are written only when
 * zero_padding != 0.  Rows with slot >= cap are skipped (EP_ORA_CAPACITY).
 */
int ora_dispatch_expanded(const uint16_t *x, int T, int H, const int64_t *topk_idx,
                          const float *topk_weights, int K, int E, int R,
                          const int32_t *token_slot, const int32_t *expert_offset,
                          const int32_t *num_rows_per_expert, int fp8,
                          int zero_padding, void *recv_x, float *recv_x_scales,
                          int32_t *recv_src_idx, int32_t *recv_topk_idx,
                          float *recv_topk_weights, int cap, uint32_t *stats)
{
    int err = 0;
    int epr = E / R;
    int G = H / 128;
    size_t width = fp8 == 2 ? (size_t)ora_fp8_packed_row_bytes(H)
                            : (size_t)H * (fp8 ? 1 : 2);
    uint8_t *q = (uint8_t *)malloc((size_t)(H > 0 ? H : 1));
    float *sc = (float *)malloc(sizeof(float) * (size_t)(G > 0 ? G : 1));
    for (int t = 0; t < T; ++t) {
        const uint16_t *row = x + (size_t)t * H;
        if (!choices_agree(topk_idx, t, K, E, token_slot))
            err |= EP_ORA_STALE;
        if (fp8)
            ora_quantize_row(row, H, q, sc);
        for (int k = 0; k < K; ++k) {
            int32_t slot = token_slot[(size_t)t * K + k];
            if (slot < 0)
                continue;
            if (slot >= cap) {
                err |= EP_ORA_CAPACITY;
                continue;
            }
            int64_t e = topk_idx[(size_t)t * K + k];
            uint8_t *dst = (uint8_t *)recv_x + (size_t)slot * width;
            if (!fp8) {
                memcpy(dst, row, sizeof(uint16_t) * (size_t)H);
            } else if (fp8 == 1) {
                memcpy(dst, q, (size_t)H);
                memcpy(recv_x_scales + (size_t)slot * G, sc, sizeof(float) * (size_t)G);
            } else {
                memset(dst, 0, width);
                memcpy(dst, q, (size_t)H);
                memcpy(dst + H, sc, sizeof(float) * (size_t)G);
            }
            if (recv_src_idx)
                recv_src_idx[slot] = t;
            for (int j = 0; j < K; ++j) {
                /* an expanded row marks only the expert it belongs to */
                int here = j == k && valid_expert(e, E);
                if (recv_topk_idx)
                    recv_topk_idx[(size_t)slot * K + j] =
                        here ? (int32_t)(e - (e / epr) * epr) : -1;
                if (recv_topk_weights)
                    recv_topk_weights[(size_t)slot * K + j] =
                        here ? topk_weights[(size_t)t * K + k] : 0.0f;
            }
            if (stats)
                stats[e] += 1;
        }
    }
    if (zero_padding) {
        for (int e = 0; e < E; ++e) {
            for (int s = expert_offset[e] + num_rows_per_expert[e];
                 s < expert_offset[e + 1]; ++s) {
                if (s >= cap) {
                    err |= EP_ORA_CAPACITY;
                    continue;
                }
                memset((uint8_t *)recv_x + (size_t)s * width, 0, width);
                if (fp8 == 1)
                    memset(recv_x_scales + (size_t)s * G, 0, sizeof(float) * (size_t)G);
                if (recv_src_idx)
                    recv_src_idx[s] = -1;
                for (int j = 0; j < K; ++j) {
                    if (recv_topk_idx)
                        recv_topk_idx[(size_t)s * K + j] = -1;
                    if (recv_topk_weights)
                        recv_topk_weights[(size_t)s * K + j] = 0.0f;
                }
            }
        }
    }
    free(q);
    free(sc);
    return err;
}

/*
 * Expanded combine: out[t] = bf16(bias0 + bias1 + sum over t's rows in
 * ascending row order of c * y[row]), c = the row's gate weight (or 1).
 */
int ora_combine_expanded(const uint16_t *y, int cap, int H, const int32_t *token_slot,
                         int T, int K, const int64_t *topk_idx,
                         const float *topk_weights, int E, const uint16_t *bias0,
                         const uint16_t *bias1, uint16_t *out)
{
    int err = 0;
    float *acc = (float *)malloc(sizeof(float) * (size_t)(H > 0 ? H : 1));
    for (int t = 0; t < T; ++t) {
        if (topk_weights && !choices_agree(topk_idx, t, K, E, token_slot))
            err |= EP_ORA_STALE;
        for (int h = 0; h < H; ++h) {
            acc[h] = bias0 ? ora_bf16_to_f32(bias0[(size_t)t * H + h]) : 0.0f;
            if (bias1)
                acc[h] = acc[h] + ora_bf16_to_f32(bias1[(size_t)t * H + h]);
        }
        /* rows in ascending order: repeatedly take the smallest unused slot */
        int32_t last = -1;
        for (;;) {
            int best = -1;
            for (int k = 0; k < K; ++k) {
                int32_t s = token_slot[(size_t)t * K + k];
                if (s > last && (best < 0 || s < token_slot[(size_t)t * K + best]))
                    best = k;
            }
            if (best < 0)
                break;
            int32_t slot = token_slot[(size_t)t * K + best];
            last = slot;
            if (slot >= cap) {
                err |= EP_ORA_CAPACITY;
                continue;
            }
            const uint16_t *row = y + (size_t)slot * H;
            float c = topk_weights ? topk_weights[(size_t)t * K + best] : 1.0f;
            for (int h = 0; h < H; ++h) {
                if (topk_weights) {
                    float p = c * ora_bf16_to_f32(row[h]);
                    acc[h] = acc[h] + p;
                } else {
                    acc[h] = acc[h] + ora_bf16_to_f32(row[h]);
                }
            }
        }
        for (int h = 0; h < H; ++h)
            out[(size_t)t * H + h] = ora_f32_to_bf16(acc[h]);
    }
    free(acc);
    return err;
}
