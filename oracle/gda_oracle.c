/*
 * gda_oracle.c -- plain FP64 CPU oracle for gated split-KV GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load or run this code.  The CUDA library
 * never links, includes or calls it, and it shares no code, header or table
 * with the CUDA path.
 *
 * What it computes (one decode token per sequence b, query head h):
 *
 *   kvh      = h / (Hq / Hkv)                        consecutive GQA grouping
 *   rows     = kv_indices[kv_indptr[b] .. kv_indptr[b+1])
 *   s_j      = scale * sum_d q[b,h,d] * K[rows_j, kvh, d]
 *   p        = softmax(s)                             (natural exp, max-shifted)
 *   O        = sum_j p_j * V[rows_j, kvh, :]
 *   o_b      = RNE_bf16(O)                            (double rounded directly)
 *   s_b      = RNE_bf16(1 / (1 + exp(-gate)))         (gate widened to double)
 *   out      = RNE_bf16(o_b * s_b)                    (product exact in double)
 *
 * Sources:
 *  - FreeToken PR #781 "Fuse the BF16 attention output sigmoid gate into the
 *    existing Triton decode stage2", Summary: stage1 + stage2 FP32 reduction are
 *    kept, the output is rounded to BF16, the sigmoid of the gate is taken in
 *    BF16 (a per-device table of BF16 sigmoid values) and the product is rounded
 *    to nearest even; Correctness: the fused output equals the unfused
 *    Torch sigmoid followed by Torch multiply element by element.
 *  - FreeToken PR #781, Automatic dispatch: query [1,16,256], two KV heads, a
 *    CSR slot index, default full attention (no window, sinks or custom scale).
 *  - cuDNN FE-OSS "Gated Attention Block (SM107)", Overview, stages (4) and (5):
 *    O = softmax(Q K^T * scale) V with GQA H_q / H_kv, then O * sigmoid(GATE);
 *    Forward / fp4 notes: a dead (zero-length) row produces zeros.
 *
 * Variants FreeToken PR #781 lists among the cases its fused path leaves to the
 * fallback (Automatic dispatch: "no window, sinks, custom scale"; Correctness:
 * "sinks/window and non-power GQA groups"):
 *   window W > 0   only the last W positions of each sequence are attended
 *                  (rows kv_indices[kv_indptr[b] + max(0, L - W) .. kv_indptr[b+1]))
 *   sinks[h]       a per-head logit that joins the softmax denominator with a
 *                  zero value row: O = sum_j e^{s_j} V_j / (e^{sink_h} + sum_j e^{s_j}),
 *                  lse = log(e^{sink_h} + sum_j e^{s_j})
 *   any G = Hq / Hkv (including non-powers of two), any scale.
 *
 * FP8 KV cache (cuDNN FE-OSS "Gated Attention Block (SM107)", API, QuantSpec:
 * static per-tensor scales with dtype torch.float8_e4m3fn): the K and V pools may
 * hold e4m3 codes; the value of a code c is descale * e4m3(c), with one descale
 * for K and one for V, and everything above runs on those values unchanged.
 *
 * Readings where the pages are silent: the sigmoid is the correctly rounded
 * BF16 value of the real sigmoid (no page fixes a device's sigmoid), the KV
 * head of query head h is h / G, a zero-length sequence gives O = 0 and
 * lse = -inf, and rounding to BF16 is round-to-nearest-even straight from the
 * double (never through an intermediate float, which would round twice).
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (no fast-math, no
 * FMA contraction), so the arithmetic is the plain IEEE double arithmetic the
 * formulas above describe, on x86-64 and on aarch64 alike.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_SHAPE (-1)
#define ORACLE_ERR_INDEX (-2)
#define ORACLE_ERR_NOMEM (-3)

/* ---- BF16 <-> double ------------------------------------------------------ */

/* Widen a BF16 bit pattern: BF16 is the upper half of an IEEE binary32. */
double oracle_double_from_bf16(uint16_t b) {
    uint32_t bits = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round a double to the nearest BF16 value, ties to even, in one step.
 * BF16: 1 sign, 8 exponent, 7 fraction bits; normal quantum 2^(E-7) for values
 * in [2^E, 2^(E+1)), subnormal quantum 2^-133, overflow to infinity from
 * (2 - 2^-8) * 2^127 upward.  NaN maps to the canonical quiet NaN. */
uint16_t oracle_bf16_from_double(double x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    int e;
    (void)frexp(a, &e);            /* a in [2^(e-1), 2^e) */
    int qexp = e - 8;              /* quantum of that binade: 8 significant bits */
    if (qexp < -133) qexp = -133;  /* subnormal grid */
    double r = nearbyint(ldexp(a, -qexp)); /* exact scaling, then RNE to integer */
    double v = ldexp(r, qexp);
    if (v >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
    float f = (float)v;            /* exact: v has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

/* ---- e4m3 -> double ---------------------------------------------------------
 * The e4m3 ("fn") 8-bit float that torch.float8_e4m3fn stores: 1 sign bit, 4
 * exponent bits with bias 7, 3 fraction bits; exponent field 0 holds the
 * subnormals m * 2^-9; exponent field 15 with fraction 7 is NaN; there are no
 * infinities, so the largest finite value is 1.75 * 2^8 = 448. */
double oracle_double_from_e4m3(uint8_t c) {
    int e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);          /* 0.m * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10); /* 1.m * 2^(e-7) */
    return (c & 0x80) ? -v : v;
}

/* A K or V pool: BF16 bit patterns, or e4m3 codes scaled by a per-tensor descale. */
typedef struct {
    const void* data;
    int fp8;
    double descale;
} kv_pool;

static double kv_value(const kv_pool* p, int64_t off) {
    if (p->fp8) return p->descale * oracle_double_from_e4m3(((const uint8_t*)p->data)[off]);
    return oracle_double_from_bf16(((const uint16_t*)p->data)[off]);
}

/* ---- the output gate ------------------------------------------------------ */

/* RNE_bf16(sigmoid(g)) for a BF16 gate value g, sigmoid taken in double. */
uint16_t oracle_sigmoid_bf16(uint16_t g) {
    double x = oracle_double_from_bf16(g);
    double s = 1.0 / (1.0 + exp(-x));
    return oracle_bf16_from_double(s);
}

/* out = RNE_bf16(o * RNE_bf16(sigmoid(gate))), element by element.
 * The product of two BF16 values is exact in double. */
void oracle_gate(const uint16_t* o, const uint16_t* gate, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        double ov = oracle_double_from_bf16(o[i]);
        double sv = oracle_double_from_bf16(oracle_sigmoid_bf16(gate[i]));
        out[i] = oracle_bf16_from_double(ov * sv);
    }
}

/* ---- attention for one (b, h) ---------------------------------------------- */

/* Softmax-weighted sum over the positions [p0, p1) of sequence b for query
 * head h.  Writes the normalised O (length D) and returns lse = m + ln(sum)
 * over those positions; an empty range gives O = 0 and lse = -inf. */
static double attend_range(const uint16_t* q, const kv_pool* kp, const kv_pool* vp,
                           const int32_t* idx, int64_t p0, int64_t p1,
                           int Hkv, int kvh, int D, double scale, double* s_buf, double* O) {
    for (int d = 0; d < D; ++d) O[d] = 0.0;
    if (p1 <= p0) return -INFINITY;
    double m = -INFINITY;
    for (int64_t j = p0; j < p1; ++j) {
        int64_t krow = ((int64_t)idx[j] * Hkv + kvh) * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += oracle_double_from_bf16(q[d]) * kv_value(kp, krow + d);
        double s = scale * acc;
        s_buf[j - p0] = s;
        if (s > m) m = s;
    }
    double z = 0.0;
    for (int64_t j = p0; j < p1; ++j) {
        double p = exp(s_buf[j - p0] - m);
        z += p;
        int64_t vrow = ((int64_t)idx[j] * Hkv + kvh) * D;
        for (int d = 0; d < D; ++d) O[d] += p * kv_value(vp, vrow + d);
    }
    for (int d = 0; d < D; ++d) O[d] /= z;
    return m + log(z);
}

static int check_inputs(const int32_t* indptr, const int32_t* indices, int64_t num_slots,
                        int B, int Hq, int Hkv, int D) {
    if (B < 0 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv != 0) return ORACLE_ERR_SHAPE;
    if (B > 0 && indptr[0] != 0) return ORACLE_ERR_SHAPE;
    for (int b = 0; b < B; ++b)
        if (indptr[b + 1] < indptr[b]) return ORACLE_ERR_SHAPE;
    int64_t nnz = B > 0 ? indptr[B] : 0;
    for (int64_t j = 0; j < nnz; ++j)
        if (indices[j] < 0 || indices[j] >= num_slots) return ORACLE_ERR_INDEX;
    return ORACLE_OK;
}

/* Full path for the (b, h) pairs listed in `pairs` (2*n_pairs ints: b, h), or
 * (window > 0: only the last `window` positions of each sequence; sinks != NULL:
 * the per-head sink logits sinks[h] join every softmax denominator)
 * for every pair in row-major order when pairs == NULL.  Outputs are indexed
 * like the inputs ([B, Hq, D] and [B, Hq]); any output pointer may be NULL.
 *   o_f64  : O in double, before any rounding
 *   o_bf16 : RNE_bf16(O)
 *   out    : the gated output RNE_bf16(o_bf16 * RNE_bf16(sigmoid(gate)))
 *   lse    : natural-log log-sum-exp of the scaled scores
 * num_splits > 0 evaluates O through the split-merge formulation instead:
 * split s covers positions [s*c, min(L, (s+1)*c)) with c = ceil(L / S); each
 * split gives a normalised partial O_s and lse_s; the merge weights them by
 * exp(lse_s - max lse) (empty splits weigh 0).  Mathematically it is the same O.
 * kv_fp8 != 0: k_pool and v_pool hold e4m3 codes (one byte per element) whose
 * values are k_descale * e4m3(c) and v_descale * e4m3(c); otherwise they hold
 * BF16 bit patterns and the descales are not used.
 */
int oracle_decode(const uint16_t* q, const uint16_t* gate,
                  const void* k_pool, const void* v_pool, int kv_fp8, double k_descale, double v_descale,
                  const int32_t* kv_indptr, const int32_t* kv_indices, int64_t num_slots,
                  int B, int Hq, int Hkv, int D, double scale, int num_splits,
                  int window, const double* sinks,
                  const int32_t* pairs, int64_t n_pairs,
                  double* o_f64, uint16_t* o_bf16, uint16_t* out, double* lse, int nthreads) {
    int rc = check_inputs(kv_indptr, kv_indices, num_slots, B, Hq, Hkv, D);
    if (rc != ORACLE_OK) return rc;
    if (num_splits < 0 || window < 0) return ORACLE_ERR_SHAPE;
    int G = Hq / Hkv;
    int64_t total = pairs ? n_pairs : (int64_t)B * Hq;
    int64_t max_len = 0;
    for (int b = 0; b < B; ++b) {
        int64_t L = kv_indptr[b + 1] - kv_indptr[b];
        if (L > max_len) max_len = L;
    }
    for (int64_t t = 0; t < total; ++t) {
        int b = pairs ? pairs[2 * t] : (int)(t / Hq);
        int h = pairs ? pairs[2 * t + 1] : (int)(t % Hq);
        if (b < 0 || b >= B || h < 0 || h >= Hq) return ORACLE_ERR_SHAPE;
    }
    int err = ORACLE_OK;
    const kv_pool kp = {k_pool, kv_fp8 != 0, k_descale};
    const kv_pool vp = {v_pool, kv_fp8 != 0, v_descale};
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double* s_buf = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        double* O = (double*)malloc(sizeof(double) * (size_t)D);
        int ns = num_splits > 0 ? num_splits : 1;
        double* Os = (double*)malloc(sizeof(double) * (size_t)D * (size_t)ns);
        double* lse_s = (double*)malloc(sizeof(double) * (size_t)ns);
        if (!s_buf || !O || !Os || !lse_s) {
#pragma omp atomic write
            err = ORACLE_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < total; ++t) {
                int b = pairs ? pairs[2 * t] : (int)(t / Hq);
                int h = pairs ? pairs[2 * t + 1] : (int)(t % Hq);
                int kvh = h / G;
                const uint16_t* qrow = q + ((int64_t)b * Hq + h) * D;
                int64_t L = kv_indptr[b + 1] - kv_indptr[b];
                int64_t first = (window > 0 && L > window) ? L - window : 0;  /* window: last positions */
                const int32_t* idx = kv_indices + kv_indptr[b] + first;
                L -= first;
                double l_out;
                if (num_splits == 0) {
                    l_out = attend_range(qrow, &kp, &vp, idx, 0, L, Hkv, kvh, D, scale, s_buf, O);
                } else {
                    /* split-merge: every split's (O_s, lse_s), then the LSE merge */
                    int64_t c = (L + num_splits - 1) / num_splits;
                    double M = -INFINITY;
                    for (int s = 0; s < num_splits; ++s) {
                        int64_t p0 = (int64_t)s * c, p1 = p0 + c < L ? p0 + c : L;
                        lse_s[s] = attend_range(qrow, &kp, &vp, idx, p0, p1, Hkv, kvh, D, scale,
                                                s_buf, Os + (int64_t)s * D);
                        if (lse_s[s] > M) M = lse_s[s];
                    }
                    double W = 0.0;
                    for (int d = 0; d < D; ++d) O[d] = 0.0;
                    if (M > -INFINITY) {
                        for (int s = 0; s < num_splits; ++s) {
                            if (lse_s[s] == -INFINITY) continue;
                            double w = exp(lse_s[s] - M);
                            W += w;
                            for (int d = 0; d < D; ++d) O[d] += w * Os[(int64_t)s * D + d];
                        }
                        for (int d = 0; d < D; ++d) O[d] /= W;
                        l_out = M + log(W);
                    } else {
                        l_out = -INFINITY;
                    }
                }
                if (sinks) {
                    /* the sink joins the denominator: O_total = O * Z / (Z + e^sink),
                     * written with the max shift of both terms */
                    double sk = sinks[h];
                    double M = l_out > sk ? l_out : sk;
                    if (M > -INFINITY) {
                        double wo = (l_out == -INFINITY) ? 0.0 : exp(l_out - M);
                        double ws = (sk == -INFINITY) ? 0.0 : exp(sk - M);
                        for (int d = 0; d < D; ++d) O[d] = O[d] * wo / (wo + ws);
                        l_out = M + log(wo + ws);
                    }
                }
                int64_t base = ((int64_t)b * Hq + h) * D;
                const uint16_t* grow = gate ? gate + base : NULL;
                for (int d = 0; d < D; ++d) {
                    uint16_t ob = oracle_bf16_from_double(O[d]);
                    if (o_f64) o_f64[base + d] = O[d];
                    if (o_bf16) o_bf16[base + d] = ob;
                    if (out && grow) {
                        double sv = oracle_double_from_bf16(oracle_sigmoid_bf16(grow[d]));
                        out[base + d] = oracle_bf16_from_double(oracle_double_from_bf16(ob) * sv);
                    }
                }
                if (lse) lse[(int64_t)b * Hq + h] = l_out;
            }
        }
        free(s_buf);
        free(O);
        free(Os);
        free(lse_s);
    }
    return err;
}

/* ---- the step before attention: Q/K RMSNorm, partial RoPE, KV write ------------
 *
 * cuDNN FE-OSS "Gated Attention Block (SM107)", Overview stages (2)+(3): per head,
 * an optional RMSNorm of Q and K (weights w_q_norm, w_k_norm [D]) and a rotary
 * embedding of the first rope_dim dims in the rotate-half convention (Weights and
 * tables: cos, sin [B, rope_dim]); V passes through.  The projection output of
 * one token is the flat row [q (Hq*D) | gate (Hq*D) | k (Hkv*D) | v (Hkv*D)]
 * (W_qkvg column blocks Q | GATE | K | V).  For each token b:
 *   y   = x / sqrt(mean(x^2) + eps) * w           (RMSNorm, when w != NULL)
 *   for i < rope_dim/2, j = i + rope_dim/2:
 *     out_i = y_i cos_i - y_j sin_i,   out_j = y_j cos_j + y_i sin_j
 *   out_i = y_i for i >= rope_dim
 * all in double, rounded once to BF16.  Outputs: q_out [B,Hq,D], gate_out [B,Hq,D]
 * (a copy), and the token's K and V rows written to k_pool / v_pool at slots[b].
 */
static void norm_rope_row(const uint16_t* x, const uint16_t* w, double eps, const uint16_t* cs,
                          const uint16_t* sn, int rope_dim, int D, uint16_t* out) {
    double y[1024];
    double ss = 0.0;
    for (int d = 0; d < D; ++d) {
        y[d] = oracle_double_from_bf16(x[d]);
        ss += y[d] * y[d];
    }
    if (w) {
        double r = 1.0 / sqrt(ss / D + eps);
        for (int d = 0; d < D; ++d) y[d] = y[d] * r * oracle_double_from_bf16(w[d]);
    }
    int half = rope_dim / 2;
    for (int d = 0; d < D; ++d) {
        double v = y[d];
        if (d < half) {
            v = y[d] * oracle_double_from_bf16(cs[d]) - y[d + half] * oracle_double_from_bf16(sn[d]);
        } else if (d < rope_dim) {
            v = y[d] * oracle_double_from_bf16(cs[d]) + y[d - half] * oracle_double_from_bf16(sn[d]);
        }
        out[d] = oracle_bf16_from_double(v);
    }
}

int oracle_qk_norm_rope_kv_write(const uint16_t* qgkv, int64_t row_stride, const uint16_t* w_q,
                                 const uint16_t* w_k, double eps, const uint16_t* cos_t,
                                 const uint16_t* sin_t, int rope_dim, const int32_t* slots,
                                 uint16_t* q_out, uint16_t* gate_out, uint16_t* k_pool,
                                 uint16_t* v_pool, int64_t num_slots, int B, int Hq, int Hkv, int D) {
    if (B < 0 || Hq < 1 || Hkv < 1 || D < 1 || D > 1024 || rope_dim < 0 || rope_dim > D || rope_dim % 2)
        return ORACLE_ERR_SHAPE;
    if (row_stride < (int64_t)(2 * Hq + 2 * Hkv) * D) return ORACLE_ERR_SHAPE;
    for (int b = 0; b < B; ++b)
        if (slots[b] < 0 || slots[b] >= num_slots) return ORACLE_ERR_INDEX;
    for (int b = 0; b < B; ++b) {
        const uint16_t* row = qgkv + (int64_t)b * row_stride;
        const uint16_t* cs = cos_t + (int64_t)b * rope_dim;
        const uint16_t* sn = sin_t + (int64_t)b * rope_dim;
        for (int h = 0; h < Hq; ++h) {
            norm_rope_row(row + (int64_t)h * D, w_q, eps, cs, sn, rope_dim, D,
                          q_out + ((int64_t)b * Hq + h) * D);
            memcpy(gate_out + ((int64_t)b * Hq + h) * D, row + (int64_t)(Hq + h) * D, sizeof(uint16_t) * D);
        }
        for (int h = 0; h < Hkv; ++h) {
            norm_rope_row(row + (int64_t)(2 * Hq + h) * D, w_k, eps, cs, sn, rope_dim, D,
                          k_pool + ((int64_t)slots[b] * Hkv + h) * D);
            memcpy(v_pool + ((int64_t)slots[b] * Hkv + h) * D, row + (int64_t)(2 * Hq + Hkv + h) * D,
                   sizeof(uint16_t) * D);
        }
    }
    return ORACLE_OK;
}

/* ---- prefill / extend: gated SDPA over per-sequence K and V -------------------
 *
 * cuDNN FE-OSS "Gated Attention Block (SM107)", Overview stage (4) SDPA
 * O = softmax(Q K^T * scale + mask) V with GQA H_q / H_kv, and stage (5) with the
 * Fusion knob fuse_gate: O *= sigmoid(GATE) in the SDPA epilogue, after the dead-row
 * select; Forward: return_lse writes the softmax statistics [B, H_q, S] in fp32,
 * seq_lens gives per-batch KV lengths (padding).  Layout: q, gate [B, Sq, Hq, D];
 * k, v [B, Skv, Hkv, D] (BF16 bits).  For sequence b with L = kv_lens[b] (Skv when
 * kv_lens is NULL) key j is visible to query i when j < L and, with the causal mask,
 * j <= i + (L - Sq): the Sq queries are the last Sq positions of the L keys (a
 * plain prefill has Sq == L).  A query with no visible key is a dead row: O = 0 and
 * lse = -inf.  Then, per element, out = RNE(RNE(O) * RNE(sigmoid(gate))) as in the
 * decode path.  Every sum runs over j in increasing order, in double.
 *   rows / n_rows: optional (b, i, h) triples to evaluate (NULL: all), outputs indexed
 *   like the inputs ([B, Sq, Hq, D]; lse [B, Hq, Sq]); any output may be NULL.
 */
int oracle_prefill(const uint16_t* q, const uint16_t* gate, const uint16_t* k, const uint16_t* v,
                   const int32_t* kv_lens, int B, int Sq, int Skv, int Hq, int Hkv, int D, double scale,
                   int causal, const int32_t* rows, int64_t n_rows, double* o_f64, uint16_t* o_bf16,
                   uint16_t* out, double* lse, int nthreads) {
    if (B < 0 || Sq < 0 || Skv < 0 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv != 0) return ORACLE_ERR_SHAPE;
    if (kv_lens)
        for (int b = 0; b < B; ++b)
            if (kv_lens[b] < 0 || kv_lens[b] > Skv) return ORACLE_ERR_SHAPE;
    int64_t total = rows ? n_rows : (int64_t)B * Sq * Hq;
    for (int64_t t = 0; rows && t < total; ++t)
        if (rows[3 * t] < 0 || rows[3 * t] >= B || rows[3 * t + 1] < 0 || rows[3 * t + 1] >= Sq ||
            rows[3 * t + 2] < 0 || rows[3 * t + 2] >= Hq)
            return ORACLE_ERR_SHAPE;
    int G = Hq / Hkv;
    int err = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double* sc = (double*)malloc(sizeof(double) * (size_t)(Skv > 0 ? Skv : 1));
        double* O = (double*)malloc(sizeof(double) * (size_t)D);
        if (!sc || !O) {
#pragma omp atomic write
            err = ORACLE_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < total; ++t) {
                int b, i, h;
                if (rows) {
                    b = rows[3 * t];
                    i = rows[3 * t + 1];
                    h = rows[3 * t + 2];
                } else {
                    b = (int)(t / ((int64_t)Sq * Hq));
                    i = (int)((t / Hq) % Sq);
                    h = (int)(t % Hq);
                }
                int L = kv_lens ? kv_lens[b] : Skv;
                int64_t last = causal ? (int64_t)i + (L - Sq) : (int64_t)L - 1;  /* last visible key */
                if (last > L - 1) last = L - 1;
                const uint16_t* qi = q + (((int64_t)b * Sq + i) * Hq + h) * D;
                int kvh = h / G;
                for (int d = 0; d < D; ++d) O[d] = 0.0;
                double l_out = -INFINITY;
                if (last >= 0) {
                    double m = -INFINITY;
                    for (int64_t j = 0; j <= last; ++j) {
                        const uint16_t* kj = k + (((int64_t)b * Skv + j) * Hkv + kvh) * D;
                        double acc = 0.0;
                        for (int d = 0; d < D; ++d)
                            acc += oracle_double_from_bf16(qi[d]) * oracle_double_from_bf16(kj[d]);
                        sc[j] = scale * acc;
                        if (sc[j] > m) m = sc[j];
                    }
                    double z = 0.0;
                    for (int64_t j = 0; j <= last; ++j) {
                        double p = exp(sc[j] - m);
                        z += p;
                        const uint16_t* vj = v + (((int64_t)b * Skv + j) * Hkv + kvh) * D;
                        for (int d = 0; d < D; ++d) O[d] += p * oracle_double_from_bf16(vj[d]);
                    }
                    for (int d = 0; d < D; ++d) O[d] /= z;
                    l_out = m + log(z);
                }
                int64_t base = (((int64_t)b * Sq + i) * Hq + h) * D;
                for (int d = 0; d < D; ++d) {
                    uint16_t ob = oracle_bf16_from_double(O[d]);
                    if (o_f64) o_f64[base + d] = O[d];
                    if (o_bf16) o_bf16[base + d] = ob;
                    if (out && gate) {
                        double sv = oracle_double_from_bf16(oracle_sigmoid_bf16(gate[base + d]));
                        out[base + d] = oracle_bf16_from_double(oracle_double_from_bf16(ob) * sv);
                    }
                }
                if (lse) lse[((int64_t)b * Hq + h) * Sq + i] = l_out;
            }
        }
        free(sc);
        free(O);
    }
    return err;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
