/*
 * Plain fp64 CPU oracle for shared-prefix (cascade) beam decode attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke() check and the
 * benchmark's CPU-baseline leg may load this library. The product path never
 * calls it and shares no code with it.
 *
 * What it computes (the plain definition, no splitting, no tiling):
 *
 *   For request b, beam w (row r = b*W + w), query head h, kv head g = h / G:
 *   the logical key list of the beam is positions 0 .. P_b + T_b - 1.
 *     - positions j < P_b (the shared prompt) are read through beam 0's prompt
 *       page table: page = prefix_pages[b][j / ps], slot = j % ps
 *       (TensorRT-LLM PR #21738, "Add opt-in cascade attention for wide beam
 *       search on KVCM V2": description, the prefix half: one pass over a
 *       request's prompt serves all of its beams; the commit for the V2 cache
 *       manager: beam 0's prompt page table is the one the manager provides).
 *     - positions j = P_b + t, t < T_b (the beam's generated tail) are gathered
 *       through cache_indirection: source beam s = ci[b][w][j], page =
 *       beam_pages[b*W + s][j / ps], slot = j % ps (same page, description,
 *       the tail half: the tokens a beam generated itself, located through
 *       cache_indirection).
 *   s_j = scale * <q, k_j>;  O = sum_j softmax(s)_j v_j;  LSE = ln sum_j exp(s_j).
 *   An empty key list gives O = 0 and LSE = -inf.
 *   The page's cascade splits this into prefix and tail and merges the two by
 *   log-sum-exp, which reaches this unsplit result exactly (description: the
 *   split into prefix and tail loses nothing once the log-sum-exp merge joins
 *   them).
 *
 *   Only valid rows are read, never the whole allocation (TensorRT-Model-Connect
 *   PR #2202, "prefill and decode over the cached prefix, not the whole KV
 *   allocation", Exit Criteria and Implementation: kv_cache.{h,cpp}).
 *
 *   The paged append writes each new token's K and V rows at its flat slot:
 *   page = loc / ps, offset = loc % ps (TensorRT-LLM PR #18614, "Fuse MiniMax-M3
 *   MSA per-layer KV-cache writes into one kernel": description: the page and
 *   in-page row of each slot come from out_cache_loc).
 *
 * Pool layout: [num_pages][Hkv][ps][D] of 16-bit floats (bf16 or fp16 bits).
 * q layout: [R][Hq][D]. cache_indirection: [B][W][max_seq] int32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BF16 0
#define ORC_FP16 1

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_INDEX 2
#define ORC_ERR_NOMEM 3

/* Exact value of a bf16 or IEEE binary16 bit pattern. bf16 is the top half of
 * an IEEE binary32; binary16 has 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double orc_half_to_double(uint16_t bits, int dtype)
{
    if (dtype == ORC_BF16) {
        uint32_t u = ((uint32_t)bits) << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1f;
    int m = bits & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);  /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Bound cache rows for a valid prefix of `valid` rows: the next multiple of
 * 256 rows, or a single row when nothing is cached, at most the allocation
 * (TensorRT-Model-Connect PR #2202, Implementation: kv_cache.{h,cpp},
 * kCacheRowBucket; Notes For Future Readers). */
int32_t orc_bucket_rows(int32_t valid, int32_t capacity)
{
    if (valid <= 0)
        return 1;
    int64_t r = (((int64_t)valid + 255) / 256) * 256;
    return r < capacity ? (int32_t)r : capacity;
}

/* One query against n explicit keys, all in fp64.
 * s_j = scale <q, k_j>, m = max s_j, Z = sum exp(s_j - m),
 * O = sum exp(s_j - m) v_j / Z, LSE = m + ln Z. n == 0: O = 0, LSE = -inf.
 * `s` is caller scratch of n doubles. */
void orc_attend(int D, int n, const double *q, const double *K, const double *V,
                double scale, double *s, double *o, double *lse)
{
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += q[d] * K[(size_t)j * D + d];
        s[j] = scale * acc;
        if (s[j] > m)
            m = s[j];
    }
    double Z = 0.0;
    for (int j = 0; j < n; ++j) {
        double p = exp(s[j] - m);
        Z += p;
        for (int d = 0; d < D; ++d)
            o[d] += p * V[(size_t)j * D + d];
    }
    for (int d = 0; d < D; ++d)
        o[d] /= Z;
    *lse = m + log(Z);
}

/* Log-sum-exp merge of k partial attention states (O_i, L_i) over disjoint key
 * sets: L = ln sum exp(L_i), O = sum exp(L_i - L) O_i. All L_i = -inf (every
 * set empty) gives O = 0, L = -inf (TensorRT-LLM PR #21738, description: the
 * prefix and tail states are joined without loss by a log-sum-exp merge). */
void orc_merge(int D, int k, const double *O, const double *L, double *o, double *lse)
{
    double m = -INFINITY;
    for (int i = 0; i < k; ++i)
        if (L[i] > m)
            m = L[i];
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double Z = 0.0;
    for (int i = 0; i < k; ++i)
        Z += exp(L[i] - m);
    double total = m + log(Z);
    for (int i = 0; i < k; ++i) {
        double wgt = exp(L[i] - total);
        for (int d = 0; d < D; ++d)
            o[d] += wgt * O[(size_t)i * D + d];
    }
    *lse = total;
}

/* Physical (page, slot) of logical position j of row r, or -1 on a bad index. */
static int64_t orc_key_row(int j, int b, int w, int W, int P, int ps, int num_pages,
                           const int32_t *prefix_pages, int maxp_prefix,
                           const int32_t *beam_pages, int maxp, const int32_t *ci, int max_seq,
                           int *bad)
{
    int page;
    if (j < P) {
        if (j / ps >= maxp_prefix) { *bad = 1; return -1; }
        page = prefix_pages[(size_t)b * maxp_prefix + j / ps];
    } else {
        if (j >= max_seq) { *bad = 1; return -1; }
        int src = ci[((size_t)b * W + w) * max_seq + j];
        if (src < 0 || src >= W) { *bad = 1; return -1; }
        if (j / ps >= maxp) { *bad = 1; return -1; }
        page = beam_pages[((size_t)b * W + src) * maxp + j / ps];
    }
    if (page < 0 || page >= num_pages) { *bad = 1; return -1; }
    return (int64_t)page * ps + (j % ps);
}

/* Unsplit decode attention for the rows listed in `rows` (all R rows when
 * rows == NULL). Outputs: O [nrows][Hq][D], LSE [nrows][Hq], fp64.
 * Returns ORC_ERR_INDEX if any page id or indirection value it would read is
 * out of range (nothing is read from a bad index). */
int orc_decode_attn(int dtype, int B, int W, int Hq, int Hkv, int D, int ps, int num_pages,
                    const int32_t *prefix_len, const int32_t *tail_len,
                    const int32_t *prefix_pages, int maxp_prefix,
                    const int32_t *beam_pages, int maxp, const int32_t *ci, int max_seq,
                    const uint16_t *q, const uint16_t *kpool, const uint16_t *vpool,
                    double scale, const int32_t *rows, int nrows, double *O, double *LSE)
{
    if (B < 0 || W <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || ps <= 0)
        return ORC_ERR_ARG;
    const int G = Hq / Hkv;
    const int R = B * W;
    if (rows == NULL)
        nrows = R;
    int err = ORC_OK;

#pragma omp parallel
    {
        int maxn = 0;
        for (int b = 0; b < B; ++b)
            if (prefix_len[b] + tail_len[b] > maxn)
                maxn = prefix_len[b] + tail_len[b];
        double *K = malloc(sizeof(double) * ((size_t)maxn * D + 1));
        double *V = malloc(sizeof(double) * ((size_t)maxn * D + 1));
        double *s = malloc(sizeof(double) * ((size_t)maxn + 1));
        double *qd = malloc(sizeof(double) * (size_t)D);
        if (!K || !V || !s || !qd) {
#pragma omp atomic write
            err = ORC_ERR_NOMEM;
        }
#pragma omp for collapse(2) schedule(dynamic, 1)
        for (int i = 0; i < nrows; ++i) {
            for (int g = 0; g < Hkv; ++g) {
                if (err != ORC_OK)
                    continue;
                int r = rows ? rows[i] : i;
                if (r < 0 || r >= R) {
#pragma omp atomic write
                    err = ORC_ERR_ARG;
                    continue;
                }
                int b = r / W, w = r % W;
                int P = prefix_len[b], T = tail_len[b], n = P + T;
                int bad = 0;
                for (int j = 0; j < n && !bad; ++j) {
                    int64_t kr = orc_key_row(j, b, w, W, P, ps, num_pages, prefix_pages, maxp_prefix,
                                             beam_pages, maxp, ci, max_seq, &bad);
                    if (bad)
                        break;
                    int64_t page = kr / ps, slot = kr % ps;
                    size_t base = (((size_t)page * Hkv + g) * ps + (size_t)slot) * D;
                    for (int d = 0; d < D; ++d) {
                        K[(size_t)j * D + d] = orc_half_to_double(kpool[base + d], dtype);
                        V[(size_t)j * D + d] = orc_half_to_double(vpool[base + d], dtype);
                    }
                }
                if (bad) {
#pragma omp atomic write
                    err = ORC_ERR_INDEX;
                    continue;
                }
                for (int hh = 0; hh < G; ++hh) {
                    int h = g * G + hh;
                    for (int d = 0; d < D; ++d)
                        qd[d] = orc_half_to_double(q[((size_t)r * Hq + h) * D + d], dtype);
                    orc_attend(D, n, qd, K, V, scale, s, O + ((size_t)i * Hq + h) * D,
                               LSE + (size_t)i * Hq + h);
                }
            }
        }
        free(K);
        free(V);
        free(s);
        free(qd);
    }
    return err;
}

/* Prefill over the cached prefix (TensorRT-Model-Connect PR #2202, "prefill and
 * decode over the cached prefix, not the whole KV allocation", Implementation:
 * the prompt rows attend the bound cache rows followed by the prompt rows, a
 * [Sq, cache_rows + Sq] mask with the prompt columns after the cache rows; only
 * the valid cached prefix is bound). Request b holds C_b valid cached rows and
 * S_b prompt tokens, whose K/V already sit at logical positions C_b .. C_b+S_b-1;
 * every position p of request b is read through its page table:
 * page = pages[b][p / ps], slot = p % ps. Query row r = off_b + i (prompt token
 * i of request b; off_b = S_0 + ... + S_{b-1}) attends positions 0 .. C_b + i
 * when `causal` (each prompt token sees the cache and the prompt up to itself),
 * else 0 .. C_b + S_b - 1. q is [R][Hq][D] with R = sum S_b; O [R][Hq][D],
 * LSE [R][Hq] (natural log). */
int orc_prefill_attn(int dtype, int B, int Hq, int Hkv, int D, int ps, int num_pages,
                     const int32_t *cached_len, const int32_t *prompt_len, const int32_t *pages, int maxp,
                     int causal, const uint16_t *q, const uint16_t *kpool, const uint16_t *vpool,
                     double scale, double *O, double *LSE)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || ps <= 0)
        return ORC_ERR_ARG;
    const int G = Hq / Hkv;
    int R = 0, maxn = 0;
    for (int b = 0; b < B; ++b) {
        if (cached_len[b] < 0 || prompt_len[b] < 0)
            return ORC_ERR_ARG;
        R += prompt_len[b];
        if (cached_len[b] + prompt_len[b] > maxn)
            maxn = cached_len[b] + prompt_len[b];
    }
    int *req_of = malloc(sizeof(int) * ((size_t)R + 1));
    int *tok_of = malloc(sizeof(int) * ((size_t)R + 1));
    if (!req_of || !tok_of) {
        free(req_of);
        free(tok_of);
        return ORC_ERR_NOMEM;
    }
    for (int b = 0, r = 0; b < B; ++b)
        for (int i = 0; i < prompt_len[b]; ++i, ++r) {
            req_of[r] = b;
            tok_of[r] = i;
        }
    int err = ORC_OK;
#pragma omp parallel
    {
        double *K = malloc(sizeof(double) * ((size_t)maxn * D + 1));
        double *V = malloc(sizeof(double) * ((size_t)maxn * D + 1));
        double *s = malloc(sizeof(double) * ((size_t)maxn + 1));
        double *qd = malloc(sizeof(double) * (size_t)D);
        if (!K || !V || !s || !qd) {
#pragma omp atomic write
            err = ORC_ERR_NOMEM;
        }
#pragma omp for collapse(2) schedule(dynamic, 1)
        for (int r = 0; r < R; ++r) {
            for (int g = 0; g < Hkv; ++g) {
                if (err != ORC_OK)
                    continue;
                const int b = req_of[r], i = tok_of[r];
                const int n = causal ? cached_len[b] + i + 1 : cached_len[b] + prompt_len[b];
                int bad = 0;
                for (int j = 0; j < n; ++j) {
                    if (j / ps >= maxp) {
                        bad = 1;
                        break;
                    }
                    const int32_t page = pages[(size_t)b * maxp + j / ps];
                    if (page < 0 || page >= num_pages) {
                        bad = 1;
                        break;
                    }
                    size_t base = (((size_t)page * Hkv + g) * ps + (size_t)(j % ps)) * D;
                    for (int d = 0; d < D; ++d) {
                        K[(size_t)j * D + d] = orc_half_to_double(kpool[base + d], dtype);
                        V[(size_t)j * D + d] = orc_half_to_double(vpool[base + d], dtype);
                    }
                }
                if (bad) {
#pragma omp atomic write
                    err = ORC_ERR_INDEX;
                    continue;
                }
                for (int hh = 0; hh < G; ++hh) {
                    int h = g * G + hh;
                    for (int d = 0; d < D; ++d)
                        qd[d] = orc_half_to_double(q[((size_t)r * Hq + h) * D + d], dtype);
                    orc_attend(D, n, qd, K, V, scale, s, O + ((size_t)r * Hq + h) * D, LSE + (size_t)r * Hq + h);
                }
            }
        }
        free(K);
        free(V);
        free(s);
        free(qd);
    }
    free(req_of);
    free(tok_of);
    return err;
}

/* Paged KV append: for each new token i and kv head h, copy the D-element K and
 * V rows to pool[loc_i / ps][h][loc_i % ps][:], as bits. All slots are checked
 * before anything is written, so a bad slot leaves both pools unchanged. */
int orc_append_kv(int Hkv, int D, int ps, int num_pages, int n, const int32_t *loc,
                  const uint16_t *knew, const uint16_t *vnew, int64_t row_stride,
                  uint16_t *kpool, uint16_t *vpool)
{
    for (int i = 0; i < n; ++i)
        if (loc[i] < 0 || (int64_t)loc[i] >= (int64_t)num_pages * ps)
            return ORC_ERR_INDEX;
    for (int i = 0; i < n; ++i) {
        int64_t page = loc[i] / ps, off = loc[i] % ps;
        for (int h = 0; h < Hkv; ++h) {
            size_t dst = (((size_t)page * Hkv + h) * ps + (size_t)off) * D;
            size_t src = (size_t)i * (size_t)row_stride + (size_t)h * D;
            memcpy(kpool + dst, knew + src, sizeof(uint16_t) * (size_t)D);
            memcpy(vpool + dst, vnew + src, sizeof(uint16_t) * (size_t)D);
        }
    }
    return ORC_OK;
}

/* Nearest bf16 or IEEE binary16 value of a double, ties to the even fraction
 * (round to nearest even, the IEEE default), as a bit pattern. Values past the
 * largest finite one by half a unit or more become infinity; NaN becomes the
 * quiet NaN with a clear sign bit. Written from the formats' definitions:
 * bf16 has 8 exponent bits (bias 127) and 7 fraction bits, binary16 has 5
 * (bias 15) and 10; below the smallest normal the spacing stays that of the
 * smallest binade (subnormals). */
uint16_t orc_round_half(double x, int dtype)
{
    const int frac_bits = dtype == ORC_BF16 ? 7 : 10;
    const int emin = dtype == ORC_BF16 ? -126 : -14;   /* exponent of the smallest normal */
    const int emax = dtype == ORC_BF16 ? 127 : 15;     /* exponent of the largest binade */
    const int bias = dtype == ORC_BF16 ? 127 : 15;
    const uint16_t exp_ones = (uint16_t)(((1u << (15 - frac_bits)) - 1u) << frac_bits);
    if (isnan(x))
        return (uint16_t)(exp_ones | (1u << (frac_bits - 1)));
    const uint16_t sign = signbit(x) ? (uint16_t)0x8000u : (uint16_t)0;
    const double a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | exp_ones);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);                       /* a in [2^(e-1), 2^e) */
    int be = e - 1;
    if (be < emin)
        be = emin;
    const double spacing = ldexp(1.0, be - frac_bits);
    const double r = nearbyint(a / spacing) * spacing;   /* default mode: ties to even */
    if (r >= ldexp(1.0, emax + 1))
        return (uint16_t)(sign | exp_ones);
    if (r == 0.0)                       /* below half the smallest subnormal */
        return sign;
    int re;
    frexp(r, &re);
    const int rbe = re - 1;
    if (rbe < emin)                     /* subnormal: exponent field 0 */
        return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, emin - frac_bits)));
    const uint32_t frac = (uint32_t)(r / ldexp(1.0, rbe - frac_bits)) - (1u << frac_bits);
    return (uint16_t)(sign | (uint16_t)((uint32_t)(rbe + bias) << frac_bits) | (uint16_t)frac);
}

/* Rotary position embedding (RoPE; Su et al., "RoFormer: Enhanced Transformer
 * with Rotary Position Embedding", the rotation matrix of its section 3.2). The
 * pages apply it to K before the paged write (TensorRT-LLM PR #21738, the review
 * of flash_attn4_kernels.py: the rope_write_kv_paged helper and its partial-RoPE
 * partner lookup; the description: the model applies RoPE itself, Qwen3 for
 * instance), but do not define it; this is the published definition.
 *
 * The first `rot` of the D dims of a head row form rot/2 pairs; pair j turns by
 * the angle pos * theta_j with theta_j = base^(-2j/rot). Pair j is (j, j + rot/2)
 * (the rotate-half layout of GPT-NeoX-style models such as Qwen3) or, with
 * `interleaved`, (2j, 2j + 1) (the paper's own layout). A pair (x, y) becomes
 * (x cos - y sin, y cos + x sin). Dims >= rot are left as they are. */
void orc_rope_cos_sin(int max_pos, int rot, double base, double *cs)
{
    const int half = rot / 2;
    for (int p = 0; p < max_pos; ++p)
        for (int j = 0; j < half; ++j) {
            const double angle = (double)p * pow(base, -2.0 * (double)j / (double)rot);
            cs[(size_t)p * rot + j] = cos(angle);
            cs[(size_t)p * rot + half + j] = sin(angle);
        }
}

void orc_rope_rotate(int D, int rot, int interleaved, double base, int pos, const double *x, double *y)
{
    const int half = rot / 2;
    for (int d = rot; d < D; ++d)
        y[d] = x[d];
    for (int j = 0; j < half; ++j) {
        const double angle = (double)pos * pow(base, -2.0 * (double)j / (double)rot);
        const double c = cos(angle), s = sin(angle);
        const int i0 = interleaved ? 2 * j : j;
        const int i1 = interleaved ? 2 * j + 1 : j + half;
        y[i0] = x[i0] * c - x[i1] * s;
        y[i1] = x[i1] * c + x[i0] * s;
    }
}

/* RoPE on the paged append: for each new token i (position pos[i], slot loc[i])
 * and kv head h, the rotated K row and the V row are written at
 * pool[loc / ps][h][loc % ps][:]; when q is non-NULL, the token's Hq query rows
 * (q + i*q_row_stride + h*D) are rotated in place by the same position. Rotated
 * values are computed in fp64 from the exact inputs and rounded once to the
 * dtype (orc_round_half). All slots and positions (0 <= pos < max_pos) are
 * checked first: a bad one leaves pools and q unchanged. */
int orc_rope_append_kv(int dtype, int Hq, int Hkv, int D, int rot, int interleaved, double base, int max_pos,
                       int ps, int num_pages, int n, const int32_t *pos, const int32_t *loc,
                       uint16_t *q, int64_t q_row_stride, const uint16_t *knew, const uint16_t *vnew,
                       int64_t row_stride, uint16_t *kpool, uint16_t *vpool)
{
    if (rot < 2 || rot > D || (rot & 1) || !(base > 0.0))
        return ORC_ERR_ARG;
    for (int i = 0; i < n; ++i) {
        if (loc[i] < 0 || (int64_t)loc[i] >= (int64_t)num_pages * ps)
            return ORC_ERR_INDEX;
        if (pos[i] < 0 || pos[i] >= max_pos)
            return ORC_ERR_INDEX;
    }
    double *x = malloc(sizeof(double) * (size_t)D), *y = malloc(sizeof(double) * (size_t)D);
    if (!x || !y) {
        free(x);
        free(y);
        return ORC_ERR_NOMEM;
    }
    for (int i = 0; i < n; ++i) {
        const int64_t page = loc[i] / ps, off = loc[i] % ps;
        for (int h = 0; h < Hkv; ++h) {
            const size_t dst = (((size_t)page * Hkv + h) * ps + (size_t)off) * D;
            const size_t src = (size_t)i * (size_t)row_stride + (size_t)h * D;
            for (int d = 0; d < D; ++d)
                x[d] = orc_half_to_double(knew[src + d], dtype);
            orc_rope_rotate(D, rot, interleaved, base, pos[i], x, y);
            for (int d = 0; d < D; ++d)
                kpool[dst + d] = orc_round_half(y[d], dtype);
            memcpy(vpool + dst, vnew + src, sizeof(uint16_t) * (size_t)D);
        }
        if (q)
            for (int h = 0; h < Hq; ++h) {
                uint16_t *row = q + (size_t)i * (size_t)q_row_stride + (size_t)h * D;
                for (int d = 0; d < D; ++d)
                    x[d] = orc_half_to_double(row[d], dtype);
                orc_rope_rotate(D, rot, interleaved, base, pos[i], x, y);
                for (int d = 0; d < D; ++d)
                    row[d] = orc_round_half(y[d], dtype);
            }
    }
    free(x);
    free(y);
    return ORC_OK;
}

/* orc_round_half over an array. */
void orc_round_half_array(int64_t n, const double *x, uint16_t *out, int dtype)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_round_half(x[i], dtype);
}

/* orc_rope_rotate over `rows` head rows of D values, row i by position pos[i]. */
void orc_rope_rotate_rows(int64_t rows, int D, int rot, int interleaved, double base, const int32_t *pos,
                          const double *x, double *y)
{
    for (int64_t i = 0; i < rows; ++i)
        orc_rope_rotate(D, rot, interleaved, base, pos[i], x + i * D, y + i * D);
}

/* FP8 E4M3 (the OCP 8-bit format, "e4m3fn"): 1 sign, 4 exponent (bias 7) and 3
 * fraction bits, no infinities, exponent 15 with fraction 7 is NaN, so the
 * largest finite value is 1.75 * 2^8 = 448; below 2^-6 the spacing stays 2^-9
 * (subnormals). Exact value of a pattern. */
double orc_e4m3_to_double(uint8_t bits)
{
    const int sign = bits >> 7, e = (bits >> 3) & 15, m = bits & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(m + 8), e - 10);   /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* Nearest E4M3 value, ties to the even fraction, saturating: a finite value past
 * 448 becomes +-448 (the satfinite conversion of CUDA's fp8 types), NaN the NaN
 * pattern 0x7F. */
uint8_t orc_round_e4m3(double x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);
    int be = e - 1;
    if (be < -6)
        be = -6;
    const double spacing = ldexp(1.0, be - 3);
    const double r = nearbyint(a / spacing) * spacing;
    if (r >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (r == 0.0)
        return sign;
    int re;
    frexp(r, &re);
    const int rbe = re - 1;
    if (rbe < -6)
        return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));
    const unsigned frac = (unsigned)(r / ldexp(1.0, rbe - 3)) - 8u;
    return (uint8_t)(sign | (uint8_t)((unsigned)(rbe + 7) << 3) | (uint8_t)frac);
}

/* Paged append into E4M3 pools ([num_pages][Hkv][ps][D] bytes). A 16-bit source
 * element x (bf16 or fp16, src_dtype) is stored as round_e4m3(fp32(x) * mul),
 * the product rounded once to fp32 (the conversion of a KV cache kept in fp8
 * with a per-tensor quantisation multiplier, k_mul for K and v_mul for V); an
 * E4M3 source (src_dtype 2) is copied bit for bit. Slots are checked first: a
 * bad one leaves both pools unchanged. */
int orc_append_kv_fp8(int src_dtype, int Hkv, int D, int ps, int num_pages, int n, const int32_t *loc,
                      const void *knew, const void *vnew, int64_t row_stride, float k_mul, float v_mul,
                      uint8_t *kpool, uint8_t *vpool)
{
    for (int i = 0; i < n; ++i)
        if (loc[i] < 0 || (int64_t)loc[i] >= (int64_t)num_pages * ps)
            return ORC_ERR_INDEX;
    for (int i = 0; i < n; ++i) {
        const int64_t page = loc[i] / ps, off = loc[i] % ps;
        for (int h = 0; h < Hkv; ++h) {
            const size_t dst = (((size_t)page * Hkv + h) * ps + (size_t)off) * D;
            const size_t src = (size_t)i * (size_t)row_stride + (size_t)h * D;
            if (src_dtype == 2) {
                memcpy(kpool + dst, (const uint8_t *)knew + src, (size_t)D);
                memcpy(vpool + dst, (const uint8_t *)vnew + src, (size_t)D);
                continue;
            }
            for (int d = 0; d < D; ++d) {
                const float kx = (float)orc_half_to_double(((const uint16_t *)knew)[src + d], src_dtype);
                const float vx = (float)orc_half_to_double(((const uint16_t *)vnew)[src + d], src_dtype);
                const float ky = kx * k_mul, vy = vx * v_mul;   /* one fp32 product each */
                kpool[dst + d] = orc_round_e4m3((double)ky);
                vpool[dst + d] = orc_round_e4m3((double)vy);
            }
        }
    }
    return ORC_OK;
}

/* RoPE on the append into E4M3 pools: the K row is rotated as in orc_rope_append_kv
 * and its exact rotated value times k_mul rounded once to E4M3 (orc_round_e4m3);
 * the V row is quantised as in orc_append_kv_fp8 (fp32 product with v_mul); the
 * query rows, when q is non-NULL, are rotated in place in their 16-bit dtype.
 * Slots and positions are checked first (nothing written on a bad one). */
int orc_rope_append_kv_fp8(int dtype, int Hq, int Hkv, int D, int rot, int interleaved, double base, int max_pos,
                           int ps, int num_pages, int n, const int32_t *pos, const int32_t *loc, uint16_t *q,
                           int64_t q_row_stride, const uint16_t *knew, const uint16_t *vnew, int64_t row_stride,
                           float k_mul, float v_mul, uint8_t *kpool, uint8_t *vpool)
{
    if (rot < 2 || rot > D || (rot & 1) || !(base > 0.0))
        return ORC_ERR_ARG;
    for (int i = 0; i < n; ++i) {
        if (loc[i] < 0 || (int64_t)loc[i] >= (int64_t)num_pages * ps)
            return ORC_ERR_INDEX;
        if (pos[i] < 0 || pos[i] >= max_pos)
            return ORC_ERR_INDEX;
    }
    double *x = malloc(sizeof(double) * (size_t)D), *y = malloc(sizeof(double) * (size_t)D);
    if (!x || !y) {
        free(x);
        free(y);
        return ORC_ERR_NOMEM;
    }
    for (int i = 0; i < n; ++i) {
        const int64_t page = loc[i] / ps, off = loc[i] % ps;
        for (int h = 0; h < Hkv; ++h) {
            const size_t dst = (((size_t)page * Hkv + h) * ps + (size_t)off) * D;
            const size_t src = (size_t)i * (size_t)row_stride + (size_t)h * D;
            for (int d = 0; d < D; ++d)
                x[d] = orc_half_to_double(knew[src + d], dtype);
            orc_rope_rotate(D, rot, interleaved, base, pos[i], x, y);
            for (int d = 0; d < D; ++d) {
                kpool[dst + d] = orc_round_e4m3(y[d] * (double)k_mul);
                const float vx = (float)orc_half_to_double(vnew[src + d], dtype);
                const float vy = vx * v_mul;
                vpool[dst + d] = orc_round_e4m3((double)vy);
            }
        }
        if (q)
            for (int h = 0; h < Hq; ++h) {
                uint16_t *row = q + (size_t)i * (size_t)q_row_stride + (size_t)h * D;
                for (int d = 0; d < D; ++d)
                    x[d] = orc_half_to_double(row[d], dtype);
                orc_rope_rotate(D, rot, interleaved, base, pos[i], x, y);
                for (int d = 0; d < D; ++d)
                    row[d] = orc_round_half(y[d], dtype);
            }
    }
    free(x);
    free(y);
    return ORC_OK;
}
