/*
 * mc_oracle.c -- plain, slow, fp64 CPU oracle for the MuonClip optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA
 * library.
 *
 * Every routine restates the pages' definitions with plain loops in double
 * precision, in the order the pages give them:
 *
 *   [K2-review]   "Kimi K2: 1T MoE, MuonClip and Agentic training system"
 *                 (wineandchord.com), section "Muon 为何在规模扩大后撞上
 *                 attention logit" (S_max, gamma, MHA clip, semantic
 *                 reference) and section "MLA 为什么要非对称缩放" (MLA table).
 *   [K2-digest]   "Kimi K2: Open Agentic Intelligence" (hugoean.github.io),
 *                 paragraph "Taming Muon with QK-Clip".
 *   [K2-zh 2.1]   Kimi K2 Chinese translation, section 2.1 "MuonClip".
 *   [Moonlight]   "Notes on Moonlight", sections "Background" (Muon
 *                 momentum / Newton-Schulz equations) and "Scaling up Muon"
 *                 (weight decay, RMS lemma, RMS-matched update).
 *   [Muon-blog]   "Notes on Muon blog", sections "Newton-Schulz" and
 *                 "Algorithm" (quintic iteration, coefficients, transpose
 *                 rule, normalisation eps).
 *
 * Readings where the pages are silent (the library takes the same ones):
 *   - d in 1/sqrt(d) is the per-head q.k dimension (head_dim for MHA,
 *     nope + rope for MLA).
 *   - i == j pairs are included; a causal mask keeps j <= i.
 *   - MLA: c_Q = x W_qa; per head [q^C | q^R] = c_Q W_qb[:, head block];
 *     [c_KV | k^R] = x W_kva; k^C per head = c_KV W_kb[:, head block];
 *     RoPE (rotate-half pairs (f, f + rope/2), theta_f = base^(-2f/rope),
 *     position = token index within its sequence) on q^R and k^R.  No
 *     latent normalisation.
 *   - Muon: M_t = mu M_{t-1} + G_t; O_t = NS5(M_t) (Nesterov variant:
 *     NS5(G_t + mu M_t)); W_t = W_{t-1} - lr (rms * sqrt(max(A,B)) O_t
 *     + wd W_{t-1}).
 *   - Newton-Schulz: X0 = U / (||U||_F + eps); transpose when rows > cols;
 *     X <- aX + (b A + c A A) X with A = X X^T.
 *
 *   - Attention forward (the row that takes the max logit inside the forward
 *     pass): O_i = sum_j softmax_j(s_ij / sqrt(dh)) v_j with s_ij = q_i . k_j
 *     over the keys j the mask allows ([K2-zh 2.1] calls S the largest
 *     softmax input: the logits are the inputs of this softmax).  MLA:
 *     s_ij = q^C_i . k^C_j + q^R_i . k^R_j with the shared k^R, d = nope +
 *     rope, and a value head dimension of its own.
 *
 * Parity status: every function here is pinned by the CPU tests against
 * closed forms, special cases, library routines or brute force (see
 * tests/test_oracle_pins.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_MEM 2

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* bf16 bit pattern -> double (exact: a bf16 is the top half of a float). */
double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* double -> bf16 with ONE round-to-nearest-even step (no pass through
 * float, which would round twice).  bf16 keeps 8 significant bits and
 * float's exponent range (normal down to 2^-126, subnormal step 2^-133). */
uint16_t oracle_f64_to_bf16(double x) {
    if (isnan(x)) return (uint16_t)0x7FC0;
    if (x == 0.0) return signbit(x) ? (uint16_t)0x8000 : (uint16_t)0x0000;
    if (isinf(x)) return x > 0 ? (uint16_t)0x7F80 : (uint16_t)0xFF80;
    int e;
    (void)frexp(x, &e);                 /* x = m * 2^e, 0.5 <= |m| < 1 */
    int q = e - 8;                      /* unit in the last of 8 bits  */
    if (q < -133) q = -133;             /* subnormal spacing           */
    double scaled = ldexp(x, -q);       /* exact (power-of-two scale)  */
    double r = nearbyint(scaled);       /* ties to even (default mode) */
    double y = ldexp(r, q);
    const double max_bf16 = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (fabs(y) > max_bf16) return x > 0 ? (uint16_t)0x7F80 : (uint16_t)0xFF80;
    float f = (float)y;                 /* exact: y has <= 8 bits      */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

void oracle_bf16_array_to_f64(const uint16_t* in, double* out, long n) {
    for (long i = 0; i < n; ++i) out[i] = oracle_bf16_to_f64(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Plain helpers                                                            */
/* ------------------------------------------------------------------------ */

/* out[r][c] = sum_k a[r*lda + k] * w[k*ldw + c]   for r < rows, c < cols.
 * The columns of w start at w (the caller offsets the pointer). */
static void matmul_rows(const double* a, long lda, const double* w, long ldw,
                        double* out, long ldo, long rows, long inner, long cols) {
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        double* o = out + r * ldo;
        for (long c = 0; c < cols; ++c) o[c] = 0.0;
        for (long k = 0; k < inner; ++k) {
            double av = a[r * lda + k];
            const double* wr = w + k * ldw;
            for (long c = 0; c < cols; ++c) o[c] += av * wr[c];
        }
    }
}

/* RoPE on one token's rope part v[0..rope) at position pos:
 * out[f]          = v[f] cos(pos th_f) - v[f+h] sin(pos th_f)
 * out[f+h]        = v[f+h] cos(pos th_f) + v[f] sin(pos th_f)
 * with h = rope/2 and th_f = base^(-2f/rope). */
static void rope_apply(double* v, int rope, long pos, double base) {
    int half = rope / 2;
    for (int f = 0; f < half; ++f) {
        double theta = pow(base, -2.0 * (double)f / (double)rope);
        double ang = (double)pos * theta;
        double cs = cos(ang), sn = sin(ang);
        double lo = v[f], hi = v[f + half];
        v[f] = lo * cs - hi * sn;
        v[f + half] = hi * cs + lo * sn;
    }
}

/* max over i, j (j <= i when causal) of q_i . k_j, with q, k [T][dim]
 * given as up to two (pointer, leading dim, width) parts that are summed:
 * dot = sum_f qa_i[f] ka_j[f] + sum_f qb_i[f] kb_j[f]. */
static double max_pair_dot(long T, int causal,
                           const double* qa, long ldqa, const double* ka, long ldka, int wa,
                           const double* qb, long ldqb, const double* kb, long ldkb, int wb) {
    double best = -INFINITY;
    int saw_nan = 0;
#pragma omp parallel for schedule(dynamic, 8) reduction(max : best) reduction(| : saw_nan)
    for (long i = 0; i < T; ++i) {
        long jend = causal ? i + 1 : T;
        for (long j = 0; j < jend; ++j) {
            double s = 0.0;
            for (int f = 0; f < wa; ++f) s += qa[i * ldqa + f] * ka[j * ldka + f];
            for (int f = 0; f < wb; ++f) s += qb[i * ldqb + f] * kb[j * ldkb + f];
            if (isnan(s)) saw_nan = 1;
            else if (s > best) best = s;
        }
    }
    /* like a max-reduction over tensors, a NaN logit makes the maximum NaN */
    return saw_nan ? NAN : best;
}

/* ------------------------------------------------------------------------ */
/* (1) Per-head max logit                                                   */
/* ------------------------------------------------------------------------ */

/*
 * MHA: S^h = (1/sqrt(dh)) max_{X in batch} max_{i,j} Q_i^h . K_j^h,
 * Q^h = X W_q^h, K^h = X W_k^h   ([K2-review] S_max equation;
 * [K2-zh 2.1] eq. for S_max^h; [K2-digest] QK-Clip paragraph).
 *
 * x [B][T][D]; wq, wk [D][H*dh] (x @ W convention, head h = columns
 * [h*dh, (h+1)*dh)).  For each listed batch b (batches[ib]) and head h
 * (heads[ih]) writes s_bh[ib*nheads + ih] = max_{i,j} q.k / sqrt(dh)
 * over that one sequence.  heads/batches may be NULL (= all).
 */
int oracle_max_logits_mha(const double* x, int B, int T, int D,
                          const double* wq, const double* wk, int H, int dh, int causal,
                          const int* heads, int nheads, const int* batches, int nbatches,
                          double* s_bh) {
    if (B <= 0 || T <= 0 || D <= 0 || H <= 0 || dh <= 0) return ORACLE_ERR_ARG;
    if (!heads) nheads = H;
    if (!batches) nbatches = B;
    long ld = (long)H * dh;
    double* q = (double*)malloc(sizeof(double) * (size_t)T * dh);
    double* k = (double*)malloc(sizeof(double) * (size_t)T * dh);
    if (!q || !k) { free(q); free(k); return ORACLE_ERR_MEM; }
    for (int ib = 0; ib < nbatches; ++ib) {
        int b = batches ? batches[ib] : ib;
        const double* xb = x + (long)b * T * D;
        for (int ih = 0; ih < nheads; ++ih) {
            int h = heads ? heads[ih] : ih;
            matmul_rows(xb, D, wq + (long)h * dh, ld, q, dh, T, D, dh);
            matmul_rows(xb, D, wk + (long)h * dh, ld, k, dh, T, D, dh);
            double m = max_pair_dot(T, causal, q, dh, k, dh, dh, NULL, 0, NULL, 0, 0);
            s_bh[(long)ib * nheads + ih] = m / sqrt((double)dh);
        }
    }
    free(q);
    free(k);
    return ORACLE_OK;
}

/*
 * MLA: per head the logit is q^C_i . k^C_j + q^R_i . k^R_j, divided by
 * sqrt(nope + rope) ([K2-review] MLA table lists the four components;
 * [K2-zh 2.1] names q^C, k^C, q^R and the shared k^R).
 *   c_Q = x W_qa                          [T][q_lora]
 *   [q^C | q^R]_h = c_Q W_qb[:, h block]  block = h*(nope+rope) .. +nope+rope
 *   [c_KV | k^R] = x W_kva                [T][kv_lora + rope], k^R shared
 *   k^C_h = c_KV W_kb[:, h*nope .. +nope]
 *   RoPE on q^R and k^R at the token's position.
 */
int oracle_max_logits_mla(const double* x, int B, int T, int D,
                          const double* w_qa, int q_lora, const double* w_qb,
                          const double* w_kva, int kv_lora, const double* w_kb,
                          int H, int nope, int rope, double rope_base, int causal,
                          const int* heads, int nheads, const int* batches, int nbatches,
                          double* s_bh) {
    if (B <= 0 || T <= 0 || D <= 0 || H <= 0 || nope < 0 || rope < 0 || (rope & 1))
        return ORACLE_ERR_ARG;
    if (!heads) nheads = H;
    if (!batches) nbatches = B;
    int qk = nope + rope;
    long ld_qb = (long)H * qk, ld_kva = (long)kv_lora + rope, ld_kb = (long)H * nope;
    double* cq = (double*)malloc(sizeof(double) * (size_t)T * q_lora);
    double* ckv = (double*)malloc(sizeof(double) * (size_t)T * ld_kva);
    double* qh = (double*)malloc(sizeof(double) * (size_t)T * (qk > 0 ? qk : 1));
    double* kc = (double*)malloc(sizeof(double) * (size_t)T * (nope > 0 ? nope : 1));
    if (!cq || !ckv || !qh || !kc) {
        free(cq); free(ckv); free(qh); free(kc);
        return ORACLE_ERR_MEM;
    }
    for (int ib = 0; ib < nbatches; ++ib) {
        int b = batches ? batches[ib] : ib;
        const double* xb = x + (long)b * T * D;
        matmul_rows(xb, D, w_qa, q_lora, cq, q_lora, T, D, q_lora);
        matmul_rows(xb, D, w_kva, ld_kva, ckv, ld_kva, T, D, ld_kva);
        for (long t = 0; t < T; ++t) rope_apply(ckv + t * ld_kva + kv_lora, rope, t, rope_base);
        for (int ih = 0; ih < nheads; ++ih) {
            int h = heads ? heads[ih] : ih;
            matmul_rows(cq, q_lora, w_qb + (long)h * qk, ld_qb, qh, qk, T, q_lora, qk);
            for (long t = 0; t < T; ++t) rope_apply(qh + t * qk + nope, rope, t, rope_base);
            matmul_rows(ckv, ld_kva, w_kb + (long)h * nope, ld_kb, kc, nope, T, kv_lora, nope);
            double m = max_pair_dot(T, causal, qh, qk, kc, nope, nope,
                                    qh + nope, qk, ckv + kv_lora, ld_kva, rope);
            s_bh[(long)ib * nheads + ih] = m / sqrt((double)qk);
        }
    }
    free(cq); free(ckv); free(qh); free(kc);
    return ORACLE_OK;
}

/*
 * Softmax attention forward of an MHA layer, with the max logit taken on
 * the way.  For each sequence b, head h and query i:
 *   s_ij = q_i . k_j for the keys j the mask allows (j <= i when causal),
 *   O_i  = sum_j exp(s_ij / sqrt(dh) - m_i) v_j / sum_j exp(s_ij / sqrt(dh) - m_i),
 *          m_i = max_j s_ij / sqrt(dh) (the usual shift; the ratio is the softmax),
 *   S_bh = max_{i,j} s_ij / sqrt(dh): the same max logit as
 *          oracle_max_logits_mha, taken here from the given q and k.
 * q, k, v, o [B][T][H*dh] (head h = columns [h*dh, (h+1)*dh)); s_bh [B][H].
 * A NaN logit makes S_bh NaN (like a tensor max) and the row's output NaN.
 */
int oracle_attention_mha(const double* q, const double* k, const double* v, int B, int T, int H,
                         int dh, int causal, double* o, double* s_bh) {
    if (B <= 0 || T <= 0 || H <= 0 || dh <= 0) return ORACLE_ERR_ARG;
    const long ld = (long)H * dh;
    const double scale = 1.0 / sqrt((double)dh);
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double best = -INFINITY;
            int saw_nan = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(max : best) reduction(| : saw_nan)
            for (long i = 0; i < T; ++i) {
                const double* qi = q + ((long)b * T + i) * ld + (long)h * dh;
                const long jend = causal ? i + 1 : T;
                double* s = (double*)malloc(sizeof(double) * (size_t)jend);
                double m = -INFINITY;
                int row_nan = 0;
                for (long j = 0; j < jend; ++j) {
                    const double* kj = k + ((long)b * T + j) * ld + (long)h * dh;
                    double d = 0.0;
                    for (int f = 0; f < dh; ++f) d += qi[f] * kj[f];
                    s[j] = d * scale;
                    if (isnan(d)) row_nan = 1;
                    else if (s[j] > m) m = s[j];
                }
                double* oi = o + ((long)b * T + i) * ld + (long)h * dh;
                if (row_nan) {
                    saw_nan = 1;
                    for (int f = 0; f < dh; ++f) oi[f] = NAN;
                } else {
                    if (m > best) best = m;
                    double l = 0.0;
                    for (int f = 0; f < dh; ++f) oi[f] = 0.0;
                    for (long j = 0; j < jend; ++j) {
                        const double p = exp(s[j] - m);
                        const double* vj = v + ((long)b * T + j) * ld + (long)h * dh;
                        l += p;
                        for (int f = 0; f < dh; ++f) oi[f] += p * vj[f];
                    }
                    for (int f = 0; f < dh; ++f) oi[f] /= l;
                }
                free(s);
            }
            s_bh[(long)b * H + h] = saw_nan ? NAN : best;
        }
    }
    return ORACLE_OK;
}

/*
 * MLA attention forward with the max logit taken along.  Per head h the
 * logit is the content dot product plus the rope dot product against the
 * key rope part that every head shares ([K2-review] MLA table: q^C, k^C per
 * head, q^R per head, k^R shared), over the q.k dimension d = nope + rope:
 *   s_ij = (q^C_i . k^C_j + q^R_i . k^R_j) / sqrt(nope + rope)
 *   O_i  = sum_j softmax_j(s_ij) v_j          (j <= i when causal)
 * q [B][T][H][nope + rope] (q^C then q^R of each head, RoPE applied),
 * kc [B][T][H][nope], kr [B][T][rope], v [B][T][H][dv] -> o [B][T][H][dv];
 * s_bh[b][h] = max_{i,j} s_ij (NaN if any logit of (b, h) is NaN).
 */
int oracle_attention_mla(const double* q, const double* kc, const double* kr, const double* v, int B, int T,
                         int H, int nope, int rope, int dv, int causal, double* o, double* s_bh) {
    if (B <= 0 || T <= 0 || H <= 0 || nope < 0 || rope < 0 || nope + rope <= 0 || dv <= 0) return ORACLE_ERR_ARG;
    const int dq = nope + rope;
    const double scale = 1.0 / sqrt((double)dq);
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double best = -INFINITY;
            int saw_nan = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(max : best) reduction(| : saw_nan)
            for (long i = 0; i < T; ++i) {
                const double* qi = q + (((long)b * T + i) * H + h) * dq;
                const long jend = causal ? i + 1 : T;
                double* s = (double*)malloc(sizeof(double) * (size_t)jend);
                double m = -INFINITY;
                int row_nan = 0;
                for (long j = 0; j < jend; ++j) {
                    const double* kcj = kc + (((long)b * T + j) * H + h) * nope;
                    const double* krj = kr + ((long)b * T + j) * rope;
                    double d = 0.0;
                    for (int f = 0; f < nope; ++f) d += qi[f] * kcj[f];
                    for (int f = 0; f < rope; ++f) d += qi[nope + f] * krj[f];
                    s[j] = d * scale;
                    if (isnan(d)) row_nan = 1;
                    else if (s[j] > m) m = s[j];
                }
                double* oi = o + (((long)b * T + i) * H + h) * dv;
                if (row_nan) {
                    saw_nan = 1;
                    for (int f = 0; f < dv; ++f) oi[f] = NAN;
                } else {
                    if (m > best) best = m;
                    double l = 0.0;
                    for (int f = 0; f < dv; ++f) oi[f] = 0.0;
                    for (long j = 0; j < jend; ++j) {
                        const double p = exp(s[j] - m);
                        const double* vj = v + (((long)b * T + j) * H + h) * dv;
                        l += p;
                        for (int f = 0; f < dv; ++f) oi[f] += p * vj[f];
                    }
                    for (int f = 0; f < dv; ++f) oi[f] /= l;
                }
                free(s);
            }
            s_bh[(long)b * H + h] = saw_nan ? NAN : best;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* (2) Clip factor and QK-Clip                                              */
/* ------------------------------------------------------------------------ */

/*
 * gamma_h = min(1, tau / S^h), and 1 when S^h is not positive
 * ([K2-review] gamma equation and the reference's
 * where(before > 0, tau / before, 1).clamp(max=1)).  Computed from an
 * fp32 S: the quotient is formed in double and rounded once to float,
 * which equals IEEE float division (double rounding through a 53-bit
 * format is innocuous for 24-bit operands).  sqrt_gamma likewise.
 */
void oracle_gamma(const float* s, int H, float tau, float* gamma, float* sqrt_gamma) {
    for (int h = 0; h < H; ++h) {
        float g;
        if (!(s[h] > 0.0f)) {
            g = 1.0f;
        } else {
            float r = (float)((double)tau / (double)s[h]);
            g = r < 1.0f ? r : 1.0f;
        }
        gamma[h] = g;
        if (sqrt_gamma) sqrt_gamma[h] = (float)sqrt((double)g);
    }
}

/* Scale columns [c0, c1) of a row-major matrix by `factor` with a single
 * rounding of the exact product to the storage format (bf16 x float and
 * float x float products are exact in double). */
void oracle_scale_cols_bf16(uint16_t* w, long rows, long ld, long c0, long c1, float factor) {
    for (long r = 0; r < rows; ++r)
        for (long c = c0; c < c1; ++c) {
            double v = oracle_bf16_to_f64(w[r * ld + c]) * (double)factor;
            w[r * ld + c] = oracle_f64_to_bf16(v);
        }
}

void oracle_scale_cols_f32(float* w, long rows, long ld, long c0, long c1, float factor) {
    for (long r = 0; r < rows; ++r)
        for (long c = c0; c < c1; ++c) w[r * ld + c] = (float)((double)w[r * ld + c] * (double)factor);
}

static void scale_cols(void* w, int is_bf16, long rows, long ld, long c0, long c1, float f) {
    if (is_bf16) oracle_scale_cols_bf16((uint16_t*)w, rows, ld, c0, c1, f);
    else oracle_scale_cols_f32((float*)w, rows, ld, c0, c1, f);
}

/*
 * MHA QK-Clip: W_q^h <- sqrt(gamma_h) W_q^h, W_k^h <- sqrt(gamma_h) W_k^h
 * ([K2-review] MHA clip equations).  wq, wk [D][H*dh].  Heads with
 * gamma == 1 are left untouched.  gamma_out may be NULL.
 */
void oracle_qk_clip_mha(void* wq, void* wk, int is_bf16, int D, int H, int dh,
                        const float* s_max, float tau, float* gamma_out) {
    float* g = (float*)malloc(sizeof(float) * H);
    float* sg = (float*)malloc(sizeof(float) * H);
    oracle_gamma(s_max, H, tau, g, sg);
    long ld = (long)H * dh;
    for (int h = 0; h < H; ++h) {
        if (g[h] == 1.0f) continue;
        scale_cols(wq, is_bf16, D, ld, (long)h * dh, (long)(h + 1) * dh, sg[h]);
        scale_cols(wk, is_bf16, D, ld, (long)h * dh, (long)(h + 1) * dh, sg[h]);
    }
    if (gamma_out) memcpy(gamma_out, g, sizeof(float) * H);
    free(g);
    free(sg);
}

/*
 * MLA QK-Clip ([K2-review] MLA table; [K2-zh 2.1] bullet list):
 *   q^C columns of W_qb (head block, first nope) x sqrt(gamma_h)
 *   q^R columns of W_qb (head block, last rope)  x gamma_h
 *   k^C columns of W_kb (head block)             x sqrt(gamma_h)
 *   k^R (shared, inside W_kva) and W_qa are never written.
 */
void oracle_qk_clip_mla(void* w_qb, void* w_kb, int is_bf16, int q_lora, int kv_lora,
                        int H, int nope, int rope, const float* s_max, float tau,
                        float* gamma_out) {
    float* g = (float*)malloc(sizeof(float) * H);
    float* sg = (float*)malloc(sizeof(float) * H);
    oracle_gamma(s_max, H, tau, g, sg);
    long qk = nope + rope;
    long ld_qb = (long)H * qk, ld_kb = (long)H * nope;
    for (int h = 0; h < H; ++h) {
        if (g[h] == 1.0f) continue;
        scale_cols(w_qb, is_bf16, q_lora, ld_qb, h * qk, h * qk + nope, sg[h]);
        scale_cols(w_qb, is_bf16, q_lora, ld_qb, h * qk + nope, (h + 1) * qk, g[h]);
        scale_cols(w_kb, is_bf16, kv_lora, ld_kb, (long)h * nope, (long)(h + 1) * nope, sg[h]);
    }
    if (gamma_out) memcpy(gamma_out, g, sizeof(float) * H);
    free(g);
    free(sg);
}

/* Naive global clip ([K2-zh 2.1], the all-heads variant):
 * gamma = min(1, tau / max_h S^h); W_q <- gamma^alpha W_q,
 * W_k <- gamma^(1-alpha) W_k (every head).  Factors are formed in double
 * and rounded once to float. */
void oracle_qk_clip_global(void* wq, void* wk, int is_bf16, int D, int ncols,
                           const float* s_max, int H, float tau, float alpha,
                           float* gamma_out) {
    float smax = s_max[0];
    for (int h = 1; h < H; ++h)
        if (s_max[h] > smax || isnan(s_max[h])) smax = s_max[h];
    float g, sg;
    oracle_gamma(&smax, 1, tau, &g, &sg);
    if (gamma_out) *gamma_out = g;
    if (g == 1.0f) return;
    float fq = (float)pow((double)g, (double)alpha);
    float fk = (float)pow((double)g, 1.0 - (double)alpha);
    scale_cols(wq, is_bf16, D, ncols, 0, ncols, fq);
    scale_cols(wk, is_bf16, D, ncols, 0, ncols, fk);
}

/* ------------------------------------------------------------------------ */
/* (3) Muon: Newton-Schulz and the update                                   */
/* ------------------------------------------------------------------------ */

/*
 * Quintic Newton-Schulz ([Muon-blog] "Newton-Schulz" and "Algorithm";
 * [Moonlight] NS equation):
 *   X0 = G / (||G||_F + eps), transposed when rows > cols (X is m x n,
 *   m <= n);  repeat `steps` times:  A = X X^T;  B = b A + c A A;
 *   X = a X + B X;  transpose back.
 * g and out are [rows][cols]; out may alias g.
 */
int oracle_newton_schulz(const double* g, int rows, int cols, int steps,
                         double a, double b, double c, double eps, double* out) {
    if (rows <= 0 || cols <= 0 || steps < 0) return ORACLE_ERR_ARG;
    int tr = rows > cols;
    long m = tr ? cols : rows, n = tr ? rows : cols;
    double* X = (double*)malloc(sizeof(double) * (size_t)(m * n));
    double* Xn = (double*)malloc(sizeof(double) * (size_t)(m * n));
    double* A = (double*)malloc(sizeof(double) * (size_t)(m * m));
    double* Bm = (double*)malloc(sizeof(double) * (size_t)(m * m));
    if (!X || !Xn || !A || !Bm) {
        free(X); free(Xn); free(A); free(Bm);
        return ORACLE_ERR_MEM;
    }
    for (long i = 0; i < m; ++i)
        for (long j = 0; j < n; ++j) X[i * n + j] = tr ? g[j * cols + i] : g[i * cols + j];
    double ss = 0.0;
    for (long i = 0; i < m * n; ++i) ss += X[i] * X[i];
    double inv = 1.0 / (sqrt(ss) + eps);
    for (long i = 0; i < m * n; ++i) X[i] *= inv;
    for (int it = 0; it < steps; ++it) {
        /* A = X X^T */
#pragma omp parallel for schedule(dynamic, 4)
        for (long i = 0; i < m; ++i)
            for (long j = 0; j < m; ++j) {
                double s = 0.0;
                for (long k = 0; k < n; ++k) s += X[i * n + k] * X[j * n + k];
                A[i * m + j] = s;
            }
        /* B = b A + c A A */
#pragma omp parallel for schedule(dynamic, 4)
        for (long i = 0; i < m; ++i)
            for (long j = 0; j < m; ++j) {
                double s = 0.0;
                for (long k = 0; k < m; ++k) s += A[i * m + k] * A[k * m + j];
                Bm[i * m + j] = b * A[i * m + j] + c * s;
            }
        /* X = a X + B X */
#pragma omp parallel for schedule(dynamic, 4)
        for (long i = 0; i < m; ++i) {
            double* o = Xn + i * n;
            for (long j = 0; j < n; ++j) o[j] = a * X[i * n + j];
            for (long k = 0; k < m; ++k) {
                double bv = Bm[i * m + k];
                const double* xr = X + k * n;
                for (long j = 0; j < n; ++j) o[j] += bv * xr[j];
            }
        }
        double* t = X; X = Xn; Xn = t;
    }
    for (long i = 0; i < m; ++i)
        for (long j = 0; j < n; ++j) {
            if (tr) out[j * cols + i] = X[i * n + j];
            else out[i * cols + j] = X[i * n + j];
        }
    free(X); free(Xn); free(A); free(Bm);
    return ORACLE_OK;
}

/*
 * One Muon step with decoupled weight decay and RMS matching
 * ([Moonlight] "Background": M_t = mu M_{t-1} + G_t, O_t = NS(M_t);
 * "Scaling up Muon": W_t = W_{t-1} - lr (0.2 sqrt(max(A,B)) O_t
 * + wd W_{t-1}); the 0.2 is `rms`).  Nesterov variant feeds
 * G_t + mu M_t to Newton-Schulz ([Muon-blog] remark on Nesterov).
 * w, m updated in place; o_out (may be NULL) receives O_t.
 */
int oracle_muon_step(double* w, const double* g, double* m, int rows, int cols,
                     double lr, double mu, double wd, double rms, int steps,
                     double a, double b, double c, double eps, int nesterov,
                     double* o_out) {
    long n = (long)rows * cols;
    double* u = (double*)malloc(sizeof(double) * (size_t)n);
    double* o = (double*)malloc(sizeof(double) * (size_t)n);
    if (!u || !o) { free(u); free(o); return ORACLE_ERR_MEM; }
    for (long i = 0; i < n; ++i) {
        m[i] = mu * m[i] + g[i];
        u[i] = nesterov ? g[i] + mu * m[i] : m[i];
    }
    int rc = oracle_newton_schulz(u, rows, cols, steps, a, b, c, eps, o);
    if (rc != ORACLE_OK) { free(u); free(o); return rc; }
    double scale = rms * sqrt((double)(rows > cols ? rows : cols));
    for (long i = 0; i < n; ++i) w[i] = w[i] - lr * (scale * o[i] + wd * w[i]);
    if (o_out) memcpy(o_out, o, sizeof(double) * (size_t)n);
    free(u);
    free(o);
    return ORACLE_OK;
}
