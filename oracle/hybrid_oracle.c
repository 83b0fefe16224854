/*
 * hybrid_oracle.c -- CPU oracle, in double precision, of the two per-layer steps that come before
 * the MoE FFN in the 80B hybrid stack: the Gated DeltaNet decode step (36 of the 48 layers) and the
 * gated grouped-query attention decode step over a K/V cache (the other 12).
 *
 * TEST INFRASTRUCTURE: only the tests, the smoke entry point and the benchmark's CPU-baseline leg
 * call this file. It shares no code with the CUDA library.
 *
 * Sources:
 *  - alphalab.site, "Swiftlet 實測資料解讀", section "Swiftlet 是什麼？MoE expert streaming 白話解釋":
 *    the 80B model has 48 layers, 36 with a fixed-size DeltaNet recurrent state (about 72 MiB in
 *    all) and 12 with full attention whose K/V cache is kept in 32-bit floats (at least 48 KiB per
 *    token; about 384 MiB at an 8K context).
 *  - paotong.dev commentary on Swiftlet, paragraph on the hybrid layers: 75% of the layers are
 *    Gated DeltaNet linear attention with a fixed-size recurrent state.
 *  - cheshm.ai item on Swiftlet, architecture paragraph: Gated DeltaNet linear attention, gated
 *    GQA and a high-sparsity MoE with shared experts.
 * The pages name the layer types but not their equations. The equations below are the published
 * definitions of those layer types, restated:
 *  - Gated DeltaNet (Yang, Kautz and Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with
 *    Delta Rule", ICLR 2025), the gated delta rule: the state S (d_v x d_k) maps keys to values;
 *    S_t = S_{t-1} * alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T and o_t = S_t q_t, with
 *    L2-normalised q and k, a per-head decay alpha_t in (0, 1] and a write strength beta_t in
 *    (0, 1). The decay takes the Mamba2 form alpha = exp(-exp(A_log) softplus(a + dt_bias)), and
 *    beta = sigmoid(b); a and b are per-head scalars from the input projection. The head output is
 *    RMS-normalised, scaled by a learned weight and gated by silu(z).
 *  - Grouped-query attention with an output gate: the new token's key and value are appended to the
 *    cache; query head h attends, with softmax(scale q_h . K_t) over every cached position t
 *    including the new one, to the K/V head h / (Hq / Hkv); the result is gated element-wise by
 *    sigmoid(gate).
 * Projections (x -> q, k, v, z, a, b, gate and the output projection), the short convolution,
 * rotary position encoding and q/k normalisation before rotation belong to the dense projection
 * step and are not part of these two steps: they receive q, k, v, z, a, b and gate as inputs.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

static double softplus(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Per-head decay alpha and write strength beta of the gated delta rule (Mamba2-form decay). */
void orc_gdn_gates(int Hv, const double* a, const double* b, const double* A_log, const double* dt_bias,
                   double* alpha, double* beta)
{
    for (int h = 0; h < Hv; ++h) {
        alpha[h] = exp(-exp(A_log[h]) * softplus(a[h] + dt_bias[h]));
        beta[h] = sigmoid(b[h]);
    }
}

/* x / sqrt(sum x^2 + eps_l2) * mul, over n values. */
static void l2_normalise(const double* x, int n, double eps_l2, double mul, double* out)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i)
        ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss + eps_l2);
    for (int i = 0; i < n; ++i)
        out[i] = x[i] * r * mul;
}

/*
 * One decode step of one sequence.
 *   S       [Hv][dv][dk]  recurrent state, updated in place (row r of head h: value index r)
 *   q, k    [Hk][dk]      query and key of each key head; value head h uses key head h / (Hv / Hk)
 *   v, z    [Hv][dv]      value and output-gate input of each value head
 *   a, b    [Hv]          decay and write-strength inputs; A_log, dt_bias [Hv] learned per head
 *   norm_w  [dv]          RMS-norm weight shared by the heads
 *   o       [Hv][dv]      head outputs S_t q_t (before the norm); y [Hv][dv] gated normalised outputs
 */
void orc_gdn_step(int Hk, int Hv, int dk, int dv, double* S, const double* q, const double* k, const double* v,
                  const double* z, const double* a, const double* b, const double* A_log, const double* dt_bias,
                  const double* norm_w, double scale, double eps_l2, double eps, double* o, double* y)
{
    const int rep = Hv / Hk;
    double* alpha = malloc(sizeof(double) * Hv);
    double* beta = malloc(sizeof(double) * Hv);
    double* kn = malloc(sizeof(double) * dk);
    double* qn = malloc(sizeof(double) * dk);
    double* M = malloc(sizeof(double) * (size_t)dk * dk);
    double* Sn = malloc(sizeof(double) * (size_t)dv * dk);
    orc_gdn_gates(Hv, a, b, A_log, dt_bias, alpha, beta);
    for (int h = 0; h < Hv; ++h) {
        const int g = h / rep;
        l2_normalise(k + (size_t)g * dk, dk, eps_l2, 1.0, kn);
        l2_normalise(q + (size_t)g * dk, dk, eps_l2, scale, qn);
        /* transition of the gated delta rule: M = alpha (I - beta kn kn^T) */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dk; ++j)
                M[(size_t)i * dk + j] = alpha[h] * ((i == j ? 1.0 : 0.0) - beta[h] * kn[i] * kn[j]);
        /* S_t = S_{t-1} M + beta v kn^T */
        double* Sh = S + (size_t)h * dv * dk;
        const double* vh = v + (size_t)h * dv;
        for (int r = 0; r < dv; ++r)
            for (int c = 0; c < dk; ++c) {
                double acc = 0.0;
                for (int j = 0; j < dk; ++j)
                    acc += Sh[(size_t)r * dk + j] * M[(size_t)j * dk + c];
                Sn[(size_t)r * dk + c] = acc + beta[h] * vh[r] * kn[c];
            }
        memcpy(Sh, Sn, sizeof(double) * (size_t)dv * dk);
        /* o_t = S_t q_t, then y = RMSNorm(o) * norm_w * silu(z) over the head's dv values */
        double* oh = o + (size_t)h * dv;
        double ss = 0.0;
        for (int r = 0; r < dv; ++r) {
            double acc = 0.0;
            for (int c = 0; c < dk; ++c)
                acc += Sh[(size_t)r * dk + c] * qn[c];
            oh[r] = acc;
            ss += acc * acc;
        }
        const double rinv = 1.0 / sqrt(ss / dv + eps);
        for (int r = 0; r < dv; ++r) {
            const double zz = z[(size_t)h * dv + r];
            y[(size_t)h * dv + r] = oh[r] * rinv * norm_w[r] * (zz * sigmoid(zz));
        }
    }
    free(alpha);
    free(beta);
    free(kn);
    free(qn);
    free(M);
    free(Sn);
}

/*
 * One decode step of gated grouped-query attention for one sequence.
 *   Kc, Vc  [Hkv][Lmax][D]  caches; the new token's k and v are written at position pos
 *   q, gate [Hq][D]; k, v [Hkv][D]
 *   o       [Hq][D] attention outputs; y [Hq][D] = o * sigmoid(gate)
 * Query head h reads K/V head h / (Hq / Hkv) over positions 0..pos (pos + 1 positions).
 */
void orc_gqa_step(int Hq, int Hkv, int D, int Lmax, int pos, double* Kc, double* Vc, const double* q, const double* k,
                  const double* v, const double* gate, double scale, double* o, double* y)
{
    const int rep = Hq / Hkv;
    const int n = pos + 1;
    for (int g = 0; g < Hkv; ++g) {
        memcpy(Kc + ((size_t)g * Lmax + pos) * D, k + (size_t)g * D, sizeof(double) * D);
        memcpy(Vc + ((size_t)g * Lmax + pos) * D, v + (size_t)g * D, sizeof(double) * D);
    }
    double* s = malloc(sizeof(double) * n);
    for (int h = 0; h < Hq; ++h) {
        const int g = h / rep;
        const double* qh = q + (size_t)h * D;
        double m = -INFINITY;
        for (int t = 0; t < n; ++t) {
            const double* kt = Kc + ((size_t)g * Lmax + t) * D;
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += qh[d] * kt[d];
            s[t] = scale * acc;
            if (s[t] > m)
                m = s[t];
        }
        /* softmax with the maximum taken out first (the same quotient, without overflow) */
        double Z = 0.0;
        for (int t = 0; t < n; ++t) {
            s[t] = exp(s[t] - m);
            Z += s[t];
        }
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int t = 0; t < n; ++t)
                acc += s[t] / Z * Vc[((size_t)g * Lmax + t) * D + d];
            o[(size_t)h * D + d] = acc;
            y[(size_t)h * D + d] = acc * sigmoid(gate[(size_t)h * D + d]);
        }
    }
    free(s);
}
