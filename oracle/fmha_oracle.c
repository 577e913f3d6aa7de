/*
 * fmha_oracle.c -- CPU oracle for the fused multi-head attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this file: only the tests, the package's smoke check and the
 * benchmark's CPU-baseline / reference arm use it.  It shares no code, header
 * or table with the CUDA library; it reads the raw bits of the stored inputs
 * and decodes them with its own decoders.
 *
 * What it computes is the plain definition, written out in double precision:
 *
 *   for every batch b (or packed sequence b), query head h, key/value head
 *   g = floor(h / (H / H_k)), and query row i of that sequence:
 *     s_j   = scale * sum_d Q[b,i,h,d] * K[b,j,g,d]          for allowed keys j
 *     m     = max_j s_j
 *     l     = sum_j exp(s_j - m)
 *     O_d   = out_scale * sum_j exp(s_j - m) * V[b,j,g,d] / l
 *     LSE   = m + ln(l)
 *
 * Sources (page title, section):
 *  - "fmha sm120 : 超越 torch.sdpa(flash-attention-2)", §1 flash attention:
 *    MHA = softmax(q @ k^T * scale) @ v, layout [batch, seq, heads, head_dim],
 *    O has Q's shape; §2 fmha 实现: GQA maps query head h to kv head
 *    h / (q_heads / kv_heads).
 *  - "CUTLASS Blackwell FMHA 示例完全解析", §融合扩展点 (fmha_fusion.hpp):
 *    masked scores become -infinity before the softmax; causal q-begin keeps
 *    key <= query, causal q-end shifts the diagonal by seqlen_k - seqlen_q;
 *    the residual mask only removes keys at or beyond seqlen_k.
 *  - same page, §变长序列 (Variable Sequence Length): packed sequences are
 *    addressed through cumulative lengths; sequence b owns rows
 *    [cum[b], cum[b+1]).
 *  - same page, §验证机制: both O and the log-sum-exp (LSE) are checked.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - a row with no allowed key (causal q-end with seqlen_q > seqlen_k, or a
 *    zero-length key sequence) yields O = 0 and LSE = -infinity;
 *  - LSE is the natural-log log-sum-exp of the scaled scores; out_scale does
 *    not enter it;
 *  - mask NONE and mask RESIDUAL define the same result.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F16 = 0, OR_BF16 = 1, OR_E4M3 = 2 };
enum { OR_MASK_NONE = 0, OR_MASK_RESIDUAL = 1, OR_MASK_CAUSAL = 2 };
enum { OR_QBEGIN = 0, OR_QEND = 1 };

/* ------------------------------------------------------------------------- */
/* Bit decoders.  Each storage format is sign | exponent | mantissa.          */
/* ------------------------------------------------------------------------- */

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
static double decode_f16(uint32_t bits) {
    int s = (bits >> 15) & 1, e = (bits >> 10) & 31, m = bits & 1023;
    double mag;
    if (e == 0)       mag = ldexp((double)m, -24);                 /* subnormal */
    else if (e == 31) mag = m ? NAN : INFINITY;
    else              mag = ldexp(1024.0 + m, e - 25);
    return s ? -mag : mag;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa bits. */
static double decode_bf16(uint32_t bits) {
    int s = (bits >> 15) & 1, e = (bits >> 7) & 255, m = bits & 127;
    double mag;
    if (e == 0)        mag = ldexp((double)m, -133);               /* 2^-126 * m/128 */
    else if (e == 255) mag = m ? NAN : INFINITY;
    else               mag = ldexp(128.0 + m, e - 134);
    return s ? -mag : mag;
}

/* OCP fp8 E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
 * no infinities, exponent 15 with mantissa 7 is NaN, largest finite 448. */
static double decode_e4m3(uint32_t bits) {
    int s = (bits >> 7) & 1, e = (bits >> 3) & 15, m = bits & 7;
    double mag;
    if (e == 0)                 mag = ldexp((double)m, -9);        /* 2^-6 * m/8 */
    else if (e == 15 && m == 7) mag = NAN;
    else                        mag = ldexp(8.0 + m, e - 10);
    return s ? -mag : mag;
}

double oracle_decode(int dtype, uint32_t bits) {
    switch (dtype) {
    case OR_F16:  return decode_f16(bits & 0xFFFF);
    case OR_BF16: return decode_bf16(bits & 0xFFFF);
    case OR_E4M3: return decode_e4m3(bits & 0xFF);
    default:      return NAN;
    }
}

/* ------------------------------------------------------------------------- */
/* Round-to-nearest-even encoders (used to report O rounded to the output     */
/* type).  e4m3 saturates to +-448 (satfinite); fp16/bf16 overflow to inf.    */
/* ------------------------------------------------------------------------- */

typedef struct { int ebits, mbits, bias, has_inf; double maxfinite; } fmt_t;

static const fmt_t FMT_F16  = {5, 10, 15, 1, 65504.0};
static const fmt_t FMT_BF16 = {8, 7, 127, 1, 3.3895313892515355e38};
static const fmt_t FMT_E4M3 = {4, 3, 7, 0, 448.0};

/* Round |x| to the format's grid, ties to even.  Returns the rounded magnitude. */
static double round_to_grid(double a, const fmt_t *f) {
    int e2;
    if (a == 0.0) return 0.0;
    frexp(a, &e2);                       /* a = frac * 2^e2, frac in [0.5, 1) */
    int E = e2 - 1;                      /* a in [2^E, 2^(E+1)) */
    int emin = 1 - f->bias;              /* smallest normal exponent */
    if (E < emin) E = emin;              /* subnormals share the smallest quantum */
    double quantum = ldexp(1.0, E - f->mbits);
    double q = a / quantum;              /* exact: power-of-two scaling */
    double n = floor(q);
    double rem = q - n;
    if (rem > 0.5 || (rem == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;
    return n * quantum;
}

static uint32_t encode_fmt(double x, const fmt_t *f) {
    uint32_t sign_bit = 1u << (f->ebits + f->mbits);
    uint32_t exp_all = (1u << f->ebits) - 1;
    if (isnan(x)) {
        /* canonical quiet NaN: all exponent bits and all mantissa bits set */
        return (exp_all << f->mbits) | ((1u << f->mbits) - 1);
    }
    uint32_t s = signbit(x) ? sign_bit : 0;
    double a = fabs(x);
    double r = isinf(a) ? a : round_to_grid(a, f);
    if (r > f->maxfinite) {
        if (f->has_inf) return s | (exp_all << f->mbits);           /* +-inf */
        r = f->maxfinite;                                            /* satfinite */
    }
    if (r == 0.0) return s;
    int e2;
    frexp(r, &e2);
    int E = e2 - 1;
    int emin = 1 - f->bias;
    if (E < emin) {                                                  /* subnormal */
        uint32_t m = (uint32_t)(r / ldexp(1.0, emin - f->mbits));
        return s | m;
    }
    uint32_t m = (uint32_t)(r / ldexp(1.0, E - f->mbits)) - (1u << f->mbits);
    return s | ((uint32_t)(E + f->bias) << f->mbits) | m;
}

uint32_t oracle_encode(int dtype, double x) {
    switch (dtype) {
    case OR_F16:  return encode_fmt(x, &FMT_F16);
    case OR_BF16: return encode_fmt(x, &FMT_BF16);
    case OR_E4M3: return encode_fmt(x, &FMT_E4M3);
    default:      return 0;
    }
}

void oracle_decode_array(int dtype, const void *bits, int64_t n, double *out) {
    for (int64_t i = 0; i < n; ++i) {
        uint32_t b = dtype == OR_E4M3 ? ((const uint8_t *)bits)[i]
                                      : ((const uint16_t *)bits)[i];
        out[i] = oracle_decode(dtype, b);
    }
}

void oracle_encode_array(int dtype, const double *x, int64_t n, void *bits) {
    for (int64_t i = 0; i < n; ++i) {
        uint32_t b = oracle_encode(dtype, x[i]);
        if (dtype == OR_E4M3) ((uint8_t *)bits)[i] = (uint8_t)b;
        else                  ((uint16_t *)bits)[i] = (uint16_t)b;
    }
}

/* ------------------------------------------------------------------------- */
/* Attention forward, one output row at a time.                               */
/* ------------------------------------------------------------------------- */

static inline uint32_t load_bits(const void *p, int dtype, int64_t idx) {
    return dtype == OR_E4M3 ? ((const uint8_t *)p)[idx] : ((const uint16_t *)p)[idx];
}

/* Is key j visible to query i of a sequence with sq query and sk key rows?
 * ("CUTLASS Blackwell FMHA 示例完全解析", §融合扩展点: CausalMask q-begin keeps
 * key <= query; q-end adds the offset seqlen_k - seqlen_q; the residual mask
 * drops keys at or past seqlen_k, which the loop bound below already does.) */
static inline int key_allowed(int mask, int causal_type, int64_t i, int64_t j,
                              int64_t sq, int64_t sk) {
    if (j >= sk) return 0;
    if (mask == OR_MASK_CAUSAL) {
        int64_t off = causal_type == OR_QEND ? sk - sq : 0;
        return j <= i + off;
    }
    return 1;
}

/*
 * Compute O and LSE for selected output rows.
 *
 * Inputs are raw storage bits (uint16 for fp16/bf16, uint8 for e4m3):
 *   fixed length: q [B, Sq, H, D], k/v [B, Sk, H_k, D]
 *   varlen (cu_q and cu_k both non-NULL, B+1 entries each):
 *                 q [total, H, D], k/v [total, H_k, D]; sequence b owns
 *                 q rows [cu_q[b], cu_q[b+1]) and k rows [cu_k[b], cu_k[b+1]).
 * A row index r follows the LSE layout:
 *   fixed length: r = (b*H + h)*Sq + i   (LSE [B, H, Sq])
 *   varlen:       r = h*total + t        (LSE [H, total]), t a packed q row.
 * rows == NULL selects every row 0..n_rows-1.
 * Outputs: o_out [n_rows, D] (before rounding to the output type) and
 * lse_out [n_rows].  A varlen row t >= cu_q[B] belongs to no sequence and is
 * reported as NaN.  Returns 0, or -1 on inconsistent arguments.
 */
int oracle_fmha_fwd(const void *q, const void *k, const void *v, int dtype,
                    int B, int H, int H_k, int Sq, int Sk, int D,
                    double scale, double out_scale, int mask, int causal_type,
                    const int *cu_q, const int *cu_k, int64_t total_length,
                    const int64_t *rows, int64_t n_rows,
                    double *o_out, double *lse_out, int n_threads) {
    int varlen = cu_q != NULL && cu_k != NULL;
    if (B < 0 || H <= 0 || H_k <= 0 || H % H_k != 0 || D <= 0) return -1;
    if ((cu_q == NULL) != (cu_k == NULL)) return -1;
    if (!varlen && (Sq < 0 || Sk < 0)) return -1;
    int64_t max_sk = varlen ? 0 : Sk;
    if (varlen) {
        for (int b = 0; b < B; ++b) {
            int64_t lk = (int64_t)cu_k[b + 1] - cu_k[b];
            if (lk < 0 || cu_q[b + 1] < cu_q[b]) return -1;
            if (lk > max_sk) max_sk = lk;
        }
        if (cu_q[B] > total_length || cu_k[B] > total_length) return -1;
    }
    const int group = H / H_k;

    double dtab[256];
    double *table = NULL;               /* lookup for 16-bit codes */
    if (dtype == OR_E4M3) {
        for (int c = 0; c < 256; ++c) dtab[c] = decode_e4m3((uint32_t)c);
    } else {
        table = (double *)malloc(65536 * sizeof(double));
        if (!table) return -1;
        for (int c = 0; c < 65536; ++c) table[c] = oracle_decode(dtype, (uint32_t)c);
    }
    const double *lut = dtype == OR_E4M3 ? dtab : table;

#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
#endif
    {
        double *s = (double *)malloc((size_t)(max_sk > 0 ? max_sk : 1) * sizeof(double));
        double *qrow = (double *)malloc((size_t)D * sizeof(double));
        double *acc = (double *)malloc((size_t)D * sizeof(double));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t n = 0; n < n_rows; ++n) {
            int64_t r = rows ? rows[n] : n;
            double *orow = o_out + n * D;
            int64_t b, h, i, sq, sk, q_base_row, k_base_row;
            if (!varlen) {
                b = r / ((int64_t)H * Sq);
                h = (r / Sq) % H;
                i = r % Sq;
                sq = Sq; sk = Sk;
                q_base_row = b * Sq;          /* row index into [B*S] */
                k_base_row = b * Sk;
            } else {
                h = r / total_length;
                int64_t t = r % total_length;
                /* find the sequence that owns packed row t */
                b = -1;
                for (int bb = 0; bb < B; ++bb)
                    if (t >= cu_q[bb] && t < cu_q[bb + 1]) { b = bb; break; }
                if (b < 0) {
                    for (int d = 0; d < D; ++d) orow[d] = NAN;
                    lse_out[n] = NAN;
                    continue;
                }
                i = t - cu_q[b];
                sq = (int64_t)cu_q[b + 1] - cu_q[b];
                sk = (int64_t)cu_k[b + 1] - cu_k[b];
                q_base_row = cu_q[b];
                k_base_row = cu_k[b];
            }
            int64_t g = h / group;
            const int64_t qoff = ((q_base_row + i) * H + h) * D;
            for (int d = 0; d < D; ++d) qrow[d] = lut[load_bits(q, dtype, qoff + d)];

            /* step 1: scaled scores of the allowed keys, and their maximum */
            double m = -INFINITY;
            int64_t n_allowed = 0;
            for (int64_t j = 0; j < sk; ++j) {
                if (!key_allowed(mask, causal_type, i, j, sq, sk)) { s[j] = -INFINITY; continue; }
                const int64_t koff = ((k_base_row + j) * H_k + g) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += qrow[d] * lut[load_bits(k, dtype, koff + d)];
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
                ++n_allowed;
            }
            if (n_allowed == 0) {             /* no visible key */
                for (int d = 0; d < D; ++d) orow[d] = 0.0;
                lse_out[n] = -INFINITY;
                continue;
            }
            /* step 2: softmax numerators, their sum, and P.V */
            double l = 0.0;
            for (int d = 0; d < D; ++d) acc[d] = 0.0;
            for (int64_t j = 0; j < sk; ++j) {
                if (s[j] == -INFINITY) continue;
                double p = exp(s[j] - m);
                l += p;
                const int64_t voff = ((k_base_row + j) * H_k + g) * D;
                for (int d = 0; d < D; ++d) acc[d] += p * lut[load_bits(v, dtype, voff + d)];
            }
            for (int d = 0; d < D; ++d) orow[d] = out_scale * acc[d] / l;
            lse_out[n] = m + log(l);
        }
        free(s); free(qrow); free(acc);
    }
    free(table);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Generation phase: one new query token per sequence against a K/V cache.    */
/* ------------------------------------------------------------------------- */

/*
 * Source: "CUTLASS Blackwell FMHA 示例完全解析", §FMHA for Blackwell 生成阶段
 * (fmha_gen): the generation-phase forward attends one new token of every
 * sequence to that sequence's entry of a K/V cache; with batch remapping the
 * entry of sequence b is batch_idx[b]; cache entries hold different numbers
 * of valid tokens; in cache-only mode the kernel neither reads nor inserts a
 * new K/V entry, otherwise the new token's K/V join the cache.  The same page
 * fixes head dim 128 and one query-head group per thread block.
 *
 * Reading used here (the page gives no formula): for sequence b, query head
 * h, kv head g = h / (H / H_k), cache entry c = batch_idx ? batch_idx[b] : b
 * and L = seqlen[b] valid cached tokens, the keys are
 *     K_cache[c, 0..L-1, g, :]                      (cache-only), or
 *     K_cache[c, 0..L-1, g, :] followed by K_new[b, g, :]   (insert mode),
 * with V alike, and the output is the plain definition of the prefill oracle
 * above with one query row and no mask:
 *     s_j = scale * q[b,h,:] . k_j ,  m = max s_j ,  l = sum exp(s_j - m)
 *     O[b,h,:] = out_scale * sum_j exp(s_j - m) v_j / l ,  LSE = m + ln l
 * (no key: O = 0, LSE = -inf).  Layouts: q, O [B, H, D]; caches
 * [B_cache, S_max, H_k, D]; new K/V [B, H_k, D]; LSE [B, H].
 * Returns 0, or -1 on inconsistent arguments (bad entry index, L outside
 * [0, S_max], or L = S_max in insert mode).
 */
int oracle_gen_fwd(const void *q, const void *k_cache, const void *v_cache,
                   const void *k_new, const void *v_new, int dtype,
                   int B, int H, int H_k, int D, int B_cache, int S_max,
                   const int *seqlen, const int *batch_idx,
                   double scale, double out_scale,
                   double *o_out, double *lse_out, int n_threads) {
    if (B < 0 || H <= 0 || H_k <= 0 || H % H_k != 0 || D <= 0 || S_max < 0 || B_cache < 0) return -1;
    if ((k_new == NULL) != (v_new == NULL)) return -1;
    const int insert = k_new != NULL;
    for (int b = 0; b < B; ++b) {
        int c = batch_idx ? batch_idx[b] : b;
        if (c < 0 || c >= B_cache) return -1;
        if (seqlen[b] < 0 || seqlen[b] > S_max || (insert && seqlen[b] == S_max)) return -1;
    }
    const int group = H / H_k;
    double dtab[256];
    double *table = NULL;
    if (dtype == OR_E4M3) {
        for (int c = 0; c < 256; ++c) dtab[c] = decode_e4m3((uint32_t)c);
    } else {
        table = (double *)malloc(65536 * sizeof(double));
        if (!table) return -1;
        for (int c = 0; c < 65536; ++c) table[c] = oracle_decode(dtype, (uint32_t)c);
    }
    const double *lut = dtype == OR_E4M3 ? dtab : table;
    const int64_t n_rows = (int64_t)B * H;

#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
#endif
    {
        double *s = (double *)malloc((size_t)(S_max + 1) * sizeof(double));
        double *qrow = (double *)malloc((size_t)D * sizeof(double));
        double *acc = (double *)malloc((size_t)D * sizeof(double));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t r = 0; r < n_rows; ++r) {
            const int64_t b = r / H, h = r % H, g = h / group;
            const int64_t c = batch_idx ? batch_idx[b] : b;
            const int64_t L = seqlen[b], n_keys = L + insert;
            for (int d = 0; d < D; ++d) qrow[d] = lut[load_bits(q, dtype, (b * H + h) * D + d)];
            /* key j < L lives in the cache entry; key L (insert mode) is the new token */
            double m = -INFINITY;
            for (int64_t j = 0; j < n_keys; ++j) {
                const void *src = j < L ? k_cache : k_new;
                const int64_t off = j < L ? ((c * S_max + j) * H_k + g) * D : (b * H_k + g) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += qrow[d] * lut[load_bits(src, dtype, off + d)];
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
            }
            double *orow = o_out + r * D;
            if (n_keys == 0) {
                for (int d = 0; d < D; ++d) orow[d] = 0.0;
                lse_out[r] = -INFINITY;
                continue;
            }
            double l = 0.0;
            for (int d = 0; d < D; ++d) acc[d] = 0.0;
            for (int64_t j = 0; j < n_keys; ++j) {
                const double p = exp(s[j] - m);
                const void *src = j < L ? v_cache : v_new;
                const int64_t off = j < L ? ((c * S_max + j) * H_k + g) * D : (b * H_k + g) * D;
                l += p;
                for (int d = 0; d < D; ++d) acc[d] += p * lut[load_bits(src, dtype, off + d)];
            }
            for (int d = 0; d < D; ++d) orow[d] = out_scale * acc[d] / l;
            lse_out[r] = m + log(l);
        }
        free(s);
        free(qrow);
        free(acc);
    }
    free(table);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Backward pass, on real (already decoded) values.                           */
/* ------------------------------------------------------------------------- */

/*
 * Source: "CUTLASS Blackwell FMHA 示例完全解析", §FMHA for Blackwell 反向
 * (Backward): the backward pass produces dQ, dK and dV from dO, uses the row
 * sums of O * dO, supports causal masking (a key past the query's position
 * plus the q-end offset, or outside the problem, is masked to -infinity) and
 * no GQA.  What it differentiates is the forward definition above:
 *     P = softmax_j(scale * Q K^T + mask),  O = P V.
 * For a loss with gradient dO the chain rule gives, per (b, h):
 *     dV_j  = sum_i P_ij dO_i
 *     dP_ij = dO_i . V_j
 *     D_i   = sum_j P_ij dP_ij            (= dO_i . O_i)
 *     dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i  = scale * sum_j dS_ij K_j ,   dK_j = scale * sum_i dS_ij Q_i
 * Layouts as the forward (fixed length): q, dq, do [B, Sq, H, D];
 * k, v, dk, dv [B, Sk, H, D] (H_k = H).  All arrays are double.  Rows without
 * a visible key contribute nothing.  Returns 0, or -1 on bad arguments.
 *
 * oracle_attn_bwd_o_f64 takes O as an input and forms D_i = dO_i . O_i from
 * it, the page's first step (row sums of O * dO): with the exact O the two
 * agree; with a stored O (rounded to the input type) this is what a backward
 * pass that reads that O computes.
 */
int oracle_attn_fwd_f64(const double *q, const double *k, const double *v, int B, int H, int Sq, int Sk,
                        int D, double scale, int mask, int causal_type, double *o, double *lse) {
    if (B < 0 || H <= 0 || Sq < 0 || Sk < 0 || D <= 0) return -1;
    double *s = (double *)malloc((size_t)(Sk > 0 ? Sk : 1) * sizeof(double));
    if (!s) return -1;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t i = 0; i < Sq; ++i) {
                const double *qi = q + ((b * Sq + i) * H + h) * D;
                double m = -INFINITY;
                for (int64_t j = 0; j < Sk; ++j) {
                    if (!key_allowed(mask, causal_type, i, j, Sq, Sk)) { s[j] = -INFINITY; continue; }
                    const double *kj = k + ((b * Sk + j) * H + h) * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += qi[d] * kj[d];
                    s[j] = scale * dot;
                    if (s[j] > m) m = s[j];
                }
                double *oi = o + ((b * Sq + i) * H + h) * D;
                for (int d = 0; d < D; ++d) oi[d] = 0.0;
                if (m == -INFINITY) { lse[(b * H + h) * Sq + i] = -INFINITY; continue; }
                double l = 0.0;
                for (int64_t j = 0; j < Sk; ++j) {
                    if (s[j] == -INFINITY) continue;
                    const double p = exp(s[j] - m);
                    const double *vj = v + ((b * Sk + j) * H + h) * D;
                    l += p;
                    for (int d = 0; d < D; ++d) oi[d] += p * vj[d];
                }
                for (int d = 0; d < D; ++d) oi[d] /= l;
                lse[(b * H + h) * Sq + i] = m + log(l);
            }
    free(s);
    return 0;
}

static int attn_bwd(const double *q, const double *k, const double *v, const double *o, const double *dout,
                    int B, int H, int Sq, int Sk, int D, double scale, int mask, int causal_type, double *dq,
                    double *dk, double *dv, int n_threads) {
    if (B < 0 || H <= 0 || Sq < 0 || Sk < 0 || D <= 0) return -1;
    const int64_t nq = (int64_t)B * Sq * H * D, nk = (int64_t)B * Sk * H * D;
    for (int64_t x = 0; x < nq; ++x) dq[x] = 0.0;
    for (int64_t x = 0; x < nk; ++x) { dk[x] = 0.0; dv[x] = 0.0; }
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
#endif
    {
        double *p = (double *)malloc((size_t)(Sk > 0 ? Sk : 1) * sizeof(double));
        double *dp = (double *)malloc((size_t)(Sk > 0 ? Sk : 1) * sizeof(double));
        /* one (b, h) per task: dK and dV rows of (b, h) are written by that task only */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
            const int64_t b = bh / H, h = bh % H;
            for (int64_t i = 0; i < Sq; ++i) {
                const double *qi = q + ((b * Sq + i) * H + h) * D;
                const double *gi = dout + ((b * Sq + i) * H + h) * D;
                /* P row: softmax of the visible scaled scores */
                double m = -INFINITY;
                for (int64_t j = 0; j < Sk; ++j) {
                    if (!key_allowed(mask, causal_type, i, j, Sq, Sk)) { p[j] = -INFINITY; continue; }
                    const double *kj = k + ((b * Sk + j) * H + h) * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += qi[d] * kj[d];
                    p[j] = scale * dot;
                    if (p[j] > m) m = p[j];
                }
                if (m == -INFINITY) continue;
                double l = 0.0;
                for (int64_t j = 0; j < Sk; ++j) {
                    p[j] = p[j] == -INFINITY ? 0.0 : exp(p[j] - m);
                    l += p[j];
                }
                /* dP = dO_i . V_j, and D_i = sum_j P_ij dP_ij (or dO_i . O_i from a given O) */
                double Di = 0.0;
                for (int64_t j = 0; j < Sk; ++j) {
                    p[j] /= l;
                    if (p[j] == 0.0) { dp[j] = 0.0; continue; }
                    const double *vj = v + ((b * Sk + j) * H + h) * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += gi[d] * vj[d];
                    dp[j] = dot;
                    Di += p[j] * dot;
                }
                if (o) {
                    const double *oi = o + ((b * Sq + i) * H + h) * D;
                    Di = 0.0;
                    for (int d = 0; d < D; ++d) Di += gi[d] * oi[d];
                }
                double *dqi = dq + ((b * Sq + i) * H + h) * D;
                for (int64_t j = 0; j < Sk; ++j) {
                    if (p[j] == 0.0) continue;
                    const double ds = p[j] * (dp[j] - Di);
                    const double *kj = k + ((b * Sk + j) * H + h) * D;
                    double *dkj = dk + ((b * Sk + j) * H + h) * D;
                    double *dvj = dv + ((b * Sk + j) * H + h) * D;
                    for (int d = 0; d < D; ++d) {
                        dqi[d] += scale * ds * kj[d];
                        dkj[d] += scale * ds * qi[d];
                        dvj[d] += p[j] * gi[d];
                    }
                }
            }
        }
        free(p);
        free(dp);
    }
    return 0;
}

int oracle_attn_bwd_f64(const double *q, const double *k, const double *v, const double *dout, int B, int H,
                        int Sq, int Sk, int D, double scale, int mask, int causal_type, double *dq, double *dk,
                        double *dv, int n_threads) {
    return attn_bwd(q, k, v, NULL, dout, B, H, Sq, Sk, D, scale, mask, causal_type, dq, dk, dv, n_threads);
}

int oracle_attn_bwd_o_f64(const double *q, const double *k, const double *v, const double *o, const double *dout,
                          int B, int H, int Sq, int Sk, int D, double scale, int mask, int causal_type, double *dq,
                          double *dk, double *dv, int n_threads) {
    if (!o) return -1;
    return attn_bwd(q, k, v, o, dout, B, H, Sq, Sk, D, scale, mask, causal_type, dq, dk, dv, n_threads);
}
