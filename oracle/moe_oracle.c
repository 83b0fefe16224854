/*
 * moe_oracle.c -- plain, slow CPU reference of the routed-expert MoE FFN layer.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg load this file (through oracle/__init__.py). The product library never links, loads or
 * calls it, and it shares no code, header or table with the CUDA path.
 *
 * Everything is evaluated in double from the stored bytes: bf16 router rows, bf16 shared-gate
 * vector, blob codes and bf16 scale/bias. There is no blocking, fusion or reordering beyond what
 * the definitions below state. Sources (web pages about the Swiftlet runtime):
 *   [qpack]  paotong.dev commentary on Swiftlet (paotong.dev/a/b3a48bd74abb1ebf): experts are
 *            repacked into one fixed-stride blob each, fetched at base + index * stride.
 *   [route]  cheshm.ai news item "Swiftlet fits an 80B-level Qwen giant into Mac", paragraph on
 *            scheduling: each layer routes a token to 10 of 512 (80B) or 8 of 256 (35B) experts;
 *            dense weights (router, shared experts) stay resident.
 *   [quant]  the same cheshm.ai item, closing paragraph: MLX-style int4/int8 group quantisation,
 *            byte-addressed kernels with 64-bit offsets, MoE with shared experts.
 *   [renorm] alphalab.site "Swiftlet 實測資料解讀", section on the 35B correctness fix: the top-k
 *            routing weights are renormalised (norm_topk_prob); the 80B config sets it true.
 *   [size]   the same alphalab.site page, section on SSD reads: with no cache hits the 80B model
 *            requests at most 480 experts, about 810 MiB, per token.
 * Where the pages are silent the reading taken is stated at the function (readings R1..R13).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Threads of the row loops (the oracle's timing on all host cores). Default 1: serial. Rows are
 * independent and each row's sums keep their order, so the results do not depend on the count. */
static int orc_threads = 1;
void orc_set_threads(int n) { orc_threads = n < 1 ? 1 : n; }
int orc_get_threads(void) { return orc_threads; }

/* ------------------------------------------------------------------------------------------ */
/* bf16 values                                                                                 */
/* ------------------------------------------------------------------------------------------ */

/* Value of a bf16 bit pattern: the upper 16 bits of an IEEE binary32. Exact. */
double orc_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits), ties to even, by the IEEE rule.
 * Written for zero and normal-range magnitudes (2^-126 <= |v| < 2^128), which is all the
 * layer produces; smaller magnitudes are flushed to signed zero. */
uint16_t orc_round_bf16(double v)
{
    if (v == 0.0 || fabs(v) < ldexp(1.0, -126))
        return signbit(v) ? 0x8000u : 0x0000u;
    int e;
    double m = frexp(fabs(v), &e);            /* |v| = m * 2^e, m in [0.5, 1) */
    double scaled = ldexp(m, 8);              /* 8 significant bits -> [128, 256) */
    double r = floor(scaled);
    double frac = scaled - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    double q = ldexp(r, e - 8);               /* exactly representable in bf16 */
    float f = (float)(signbit(v) ? -q : q);   /* exact conversion */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------------------------ */
/* Blob format: one expert = one contiguous blob ([qpack]); layout is reading R2               */
/* ------------------------------------------------------------------------------------------ */
/*
 * R2 (the pages only say "fixed stride"): the nine sections follow one another with no gaps,
 *   gate.q | up.q | down.q | gate.s | gate.b | up.s | up.b | down.s | down.b
 * gate and up are [I][H] (out x in), down is [H][I]. Codes are row-major, packed along the input
 * dimension: int4 element c of a row sits in byte c/2 of that row, in the low nibble when c is
 * even and the high nibble when c is odd; int8 codes take one byte each. Scale and bias are bf16,
 * row-major [out][in/group]. The stride between blobs is the blob size rounded up to 4096 bytes.
 */

static size_t q_bytes(int rows, int cols, int bits) { return (size_t)rows * cols * bits / 8; }
static size_t sb_bytes(int rows, int cols, int group) { return (size_t)rows * (cols / group) * 2; }

/* Byte offsets of the nine sections and the total blob size. */
static void blob_sections(int H, int I, int bits, int group, size_t off[9], size_t* total)
{
    size_t sz[9];
    sz[0] = q_bytes(I, H, bits);          /* gate.q */
    sz[1] = q_bytes(I, H, bits);          /* up.q   */
    sz[2] = q_bytes(H, I, bits);          /* down.q */
    sz[3] = sb_bytes(I, H, group);        /* gate.s */
    sz[4] = sb_bytes(I, H, group);        /* gate.b */
    sz[5] = sb_bytes(I, H, group);        /* up.s   */
    sz[6] = sb_bytes(I, H, group);        /* up.b   */
    sz[7] = sb_bytes(H, I, group);        /* down.s */
    sz[8] = sb_bytes(H, I, group);        /* down.b */
    size_t o = 0;
    for (int i = 0; i < 9; ++i) {
        off[i] = o;
        o += sz[i];
    }
    *total = o;
}

size_t orc_blob_bytes(int H, int I, int bits, int group)
{
    size_t off[9], total;
    blob_sections(H, I, bits, group, off, &total);
    return total;
}

size_t orc_blob_stride(int H, int I, int bits, int group)
{
    size_t b = orc_blob_bytes(H, I, bits, group);
    return (b + 4095) / 4096 * 4096;
}

/* Code of element (r, c) of a [rows][cols] code section. */
static int code_at(const uint8_t* sec, int cols, int bits, int r, int c)
{
    if (bits == 8)
        return sec[(size_t)r * cols + c];
    uint8_t byte = sec[(size_t)r * (cols / 2) + c / 2];
    return (c % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
}

static void put_code(uint8_t* sec, int cols, int bits, int r, int c, int q)
{
    if (bits == 8) {
        sec[(size_t)r * cols + c] = (uint8_t)q;
        return;
    }
    uint8_t* byte = &sec[(size_t)r * (cols / 2) + c / 2];
    if (c % 2 == 0)
        *byte = (uint8_t)((*byte & 0xF0) | (q & 0x0F));
    else
        *byte = (uint8_t)((*byte & 0x0F) | ((q & 0x0F) << 4));
}

static uint16_t get_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void put_u16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xFF); p[1] = (uint8_t)(v >> 8); }

/* Write one blob (blob_bytes long; the caller zeroes any padding up to the stride).
 * codes[m]: uint8 [out][in] of matrix m (0 gate, 1 up, 2 down); scale[m], bias[m]: bf16 bits
 * [out][in/group]. */
void orc_blob_pack(int H, int I, int bits, int group, const uint8_t* const codes[3],
                   const uint16_t* const scale[3], const uint16_t* const bias[3], uint8_t* blob)
{
    size_t off[9], total;
    blob_sections(H, I, bits, group, off, &total);
    memset(blob, 0, total);
    for (int m = 0; m < 3; ++m) {
        int rows = (m == 2) ? H : I, cols = (m == 2) ? I : H;
        for (int r = 0; r < rows; ++r)
            for (int c = 0; c < cols; ++c)
                put_code(blob + off[m], cols, bits, r, c, codes[m][(size_t)r * cols + c]);
        int ng = cols / group;
        for (int r = 0; r < rows; ++r)
            for (int gi = 0; gi < ng; ++gi) {
                put_u16(blob + off[3 + 2 * m] + 2 * ((size_t)r * ng + gi), scale[m][(size_t)r * ng + gi]);
                put_u16(blob + off[4 + 2 * m] + 2 * ((size_t)r * ng + gi), bias[m][(size_t)r * ng + gi]);
            }
    }
}

/* Read one blob back into codes and scale/bias bit patterns (the inverse of orc_blob_pack). */
void orc_blob_unpack(int H, int I, int bits, int group, const uint8_t* blob, uint8_t* const codes[3],
                     uint16_t* const scale[3], uint16_t* const bias[3])
{
    size_t off[9], total;
    blob_sections(H, I, bits, group, off, &total);
    for (int m = 0; m < 3; ++m) {
        int rows = (m == 2) ? H : I, cols = (m == 2) ? I : H;
        for (int r = 0; r < rows; ++r)
            for (int c = 0; c < cols; ++c)
                codes[m][(size_t)r * cols + c] = (uint8_t)code_at(blob + off[m], cols, bits, r, c);
        int ng = cols / group;
        for (int r = 0; r < rows; ++r)
            for (int gi = 0; gi < ng; ++gi) {
                scale[m][(size_t)r * ng + gi] = get_u16(blob + off[3 + 2 * m] + 2 * ((size_t)r * ng + gi));
                bias[m][(size_t)r * ng + gi] = get_u16(blob + off[4 + 2 * m] + 2 * ((size_t)r * ng + gi));
            }
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Dequantisation ([quant]); reading R1                                                        */
/* ------------------------------------------------------------------------------------------ */
/*
 * R1: MLX-style affine group quantisation, w = s * q + b, q the unsigned code (int4 0..15,
 * int8 0..255), s and b the bf16 scale and bias of the group of `group` consecutive input
 * columns that holds the element.
 * Writes matrix `which` (0 gate [I][H], 1 up [I][H], 2 down [H][I]) of the blob as doubles.
 */
void orc_dequant(const uint8_t* blob, int H, int I, int bits, int group, int which, double* W)
{
    size_t off[9], total;
    blob_sections(H, I, bits, group, off, &total);
    int rows = (which == 2) ? H : I, cols = (which == 2) ? I : H;
    int ng = cols / group;
    const uint8_t* q = blob + off[which];
    const uint8_t* s = blob + off[3 + 2 * which];
    const uint8_t* b = blob + off[4 + 2 * which];
#pragma omp parallel for num_threads(orc_threads) if (orc_threads > 1)
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c) {
            size_t gi = (size_t)r * ng + c / group;
            double sc = orc_bf16(get_u16(s + 2 * gi));
            double bi = orc_bf16(get_u16(b + 2 * gi));
            W[(size_t)r * cols + c] = sc * (double)code_at(q, cols, bits, r, c) + bi;
        }
}

/* ------------------------------------------------------------------------------------------ */
/* Router, softmax, top-k, renormalisation ([route], [renorm])                                 */
/* ------------------------------------------------------------------------------------------ */

/* logits[e] = sum_h Wr[e][h] * u[h] (+ bias[e]) in double.
 * bound[e] (if not NULL) is gamma_{H+1} * (sum_h |Wr[e][h] u[h]| + |bias[e]|), gamma_n =
 * n*2^-24 / (1 - n*2^-24): the classical bound on the error of any binary32 summation order of
 * exactly representable products (Higham, "Accuracy and Stability of Numerical Algorithms",
 * section 4.2). bf16 x bf16 products are exact in binary32, so it bounds a binary32 GPU logit. */
void orc_router_logits(const uint16_t* Wr, const uint16_t* u, const float* bias, int E, int H,
                       double* logits, double* bound)
{
    double unit = ldexp(1.0, -24);
    double gam = (H + 1) * unit / (1.0 - (H + 1) * unit);
#pragma omp parallel for num_threads(orc_threads) if (orc_threads > 1)
    for (int e = 0; e < E; ++e) {
        double acc = 0.0, mag = 0.0;
        for (int h = 0; h < H; ++h) {
            double p = orc_bf16(Wr[(size_t)e * H + h]) * orc_bf16(u[h]);
            acc += p;
            mag += fabs(p);
        }
        if (bias) {
            acc += (double)bias[e];
            mag += fabs((double)bias[e]);
        }
        logits[e] = acc;
        if (bound)
            bound[e] = gam * mag;
    }
}

/* R4/R5: the routing weights of a selection idx[k] (rank order): the softmax of the logits over
 * all E experts at the selected ones, renormalised over the k selected when renorm. */
void orc_route_weights(const double* logits, int E, int k, int renorm, const int32_t* idx, double* w)
{
    double mx = logits[0];
    for (int e = 1; e < E; ++e)
        if (logits[e] > mx)
            mx = logits[e];
    double all = 0.0;
    for (int e = 0; e < E; ++e)
        all += exp(logits[e] - mx);
    double sel = 0.0;
    for (int j = 0; j < k; ++j)
        sel += exp(logits[idx[j]] - mx);
    for (int j = 0; j < k; ++j) {
        double p = exp(logits[idx[j]] - mx) / all;
        w[j] = renorm ? p / (sel / all) : p;
    }
}

/*
 * Top-k selection and routing weights.
 * Selection (R4, R5): the decision is taken in the precision the GPU path takes it, binary32:
 * each logit is rounded to the nearest float, the k largest floats are chosen, and equal floats go
 * to the lower expert index. idx[] lists the chosen experts from the largest logit down.
 * Weights: p = softmax over all E logits (max subtracted); with renorm (R3, [renorm])
 * w_j = p[idx_j] / sum_m p[idx_m], without it w_j = p[idx_j].
 */
void orc_topk(const double* logits, int E, int k, int renorm, int32_t* idx, double* w)
{
    char* taken = (char*)calloc((size_t)E, 1);
    for (int j = 0; j < k; ++j) {
        int best = -1;
        float bestv = 0.0f;
        for (int e = 0; e < E; ++e) {
            if (taken[e])
                continue;
            float v = (float)logits[e];
            if (best < 0 || v > bestv) {   /* strict: an equal later index never replaces */
                best = e;
                bestv = v;
            }
        }
        taken[best] = 1;
        idx[j] = best;
    }
    free(taken);
    orc_route_weights(logits, E, k, renorm, idx, w);
}

/* ------------------------------------------------------------------------------------------ */
/* Expert MLP (SwiGLU), shared-expert gate, combine                                            */
/* ------------------------------------------------------------------------------------------ */

/* y = Wd * (silu(Wg*u) .* (Wu*u)), silu(z) = z / (1 + exp(-z)), all in double (reading R6: no
 * intermediate rounding). h_out (if not NULL) receives the I intermediate values. */
void orc_expert_ffn(const uint8_t* blob, int H, int I, int bits, int group, const uint16_t* u,
                    double* y, double* h_out)
{
    double* Wg = (double*)malloc(sizeof(double) * (size_t)I * H);
    double* Wu = (double*)malloc(sizeof(double) * (size_t)I * H);
    double* Wd = (double*)malloc(sizeof(double) * (size_t)H * I);
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    orc_dequant(blob, H, I, bits, group, 0, Wg);
    orc_dequant(blob, H, I, bits, group, 1, Wu);
    orc_dequant(blob, H, I, bits, group, 2, Wd);
#pragma omp parallel for num_threads(orc_threads) if (orc_threads > 1)
    for (int r = 0; r < I; ++r) {
        double g = 0.0, v = 0.0;
        for (int c = 0; c < H; ++c) {
            double x = orc_bf16(u[c]);
            g += Wg[(size_t)r * H + c] * x;
            v += Wu[(size_t)r * H + c] * x;
        }
        h[r] = g / (1.0 + exp(-g)) * v;
        if (h_out)
            h_out[r] = h[r];
    }
#pragma omp parallel for num_threads(orc_threads) if (orc_threads > 1)
    for (int o = 0; o < H; ++o) {
        double acc = 0.0;
        for (int r = 0; r < I; ++r)
            acc += Wd[(size_t)o * I + r] * h[r];
        y[o] = acc;
    }
    free(Wg);
    free(Wu);
    free(Wd);
    free(h);
}

/* R7: the always-on shared expert is scaled by sigmoid(w_sg . u), w_sg a bf16 vector [H]. */
double orc_shared_gate(const uint16_t* w_sg, const uint16_t* u, int H)
{
    double z = 0.0;
    for (int h = 0; h < H; ++h)
        z += orc_bf16(w_sg[h]) * orc_bf16(u[h]);
    return 1.0 / (1.0 + exp(-z));
}

/*
 * One MoE FFN layer for one token u (bf16 [H]):
 *   logits = Wr u (+ bias); (idx, w) = top-k of the logits with routing weights;
 *   y = sum_{j=0}^{k-1} w_j * E_{idx_j}(u) + sigmoid(w_sg . u) * S(u)
 * with E_e the SwiGLU expert stored in expert_blobs[e] and S the shared expert (shared_blob,
 * intermediate Is). The sum runs over j in rank order, then the shared term.
 * Outputs: idx[k], w[k], y[H]; logits[E], bound[E] and gamma[1] when not NULL.
 */
void orc_moe_layer_sel(int H, int E, int k, int I, int Is, int bits, int group, int renorm,
                       const uint16_t* u, const uint16_t* Wr, const float* bias, const uint16_t* w_sg,
                       const uint8_t* const* expert_blobs, const uint8_t* shared_blob, int forced,
                       int32_t* idx, double* w, double* y, double* logits, double* bound, double* gamma);

void orc_moe_layer(int H, int E, int k, int I, int Is, int bits, int group, int renorm,
                   const uint16_t* u, const uint16_t* Wr, const float* bias, const uint16_t* w_sg,
                   const uint8_t* const* expert_blobs, const uint8_t* shared_blob,
                   int32_t* idx, double* w, double* y, double* logits, double* bound, double* gamma)
{
    orc_moe_layer_sel(H, E, k, I, Is, bits, group, renorm, u, Wr, bias, w_sg, expert_blobs, shared_blob, 0, idx, w,
                      y, logits, bound, gamma);
}

/*
 * The same layer with the selection either chosen by the top-k (forced = 0: idx is an output) or
 * given (forced = 1: idx[k] is an input, in rank order, and only the routing weights and y are
 * computed for it). A caller that meets a near tie (two logits closer than their binary32 error
 * bound) evaluates the layer for the other valid selection this way.
 */
void orc_moe_layer_sel(int H, int E, int k, int I, int Is, int bits, int group, int renorm,
                       const uint16_t* u, const uint16_t* Wr, const float* bias, const uint16_t* w_sg,
                       const uint8_t* const* expert_blobs, const uint8_t* shared_blob, int forced,
                       int32_t* idx, double* w, double* y, double* logits, double* bound, double* gamma)
{
    double* lg = logits ? logits : (double*)malloc(sizeof(double) * (size_t)E);
    orc_router_logits(Wr, u, bias, E, H, lg, bound);
    if (forced)
        orc_route_weights(lg, E, k, renorm, idx, w);
    else
        orc_topk(lg, E, k, renorm, idx, w);

    double* ye = (double*)malloc(sizeof(double) * (size_t)H);
    for (int o = 0; o < H; ++o)
        y[o] = 0.0;
    for (int j = 0; j < k; ++j) {
        orc_expert_ffn(expert_blobs[idx[j]], H, I, bits, group, u, ye, NULL);
        for (int o = 0; o < H; ++o)
            y[o] += w[j] * ye[o];
    }
    double gs = orc_shared_gate(w_sg, u, H);
    orc_expert_ffn(shared_blob, H, Is, bits, group, u, ye, NULL);
    for (int o = 0; o < H; ++o)
        y[o] += gs * ye[o];
    if (gamma)
        *gamma = gs;
    free(ye);
    if (!logits)
        free(lg);
}

/* ------------------------------------------------------------------------------------------ */
/* Stack pre-norm (reading R9)                                                                 */
/* ------------------------------------------------------------------------------------------ */
/*
 * R9: a stack with only a residual add between layers diverges (SwiGLU is quadratic in its
 * input), so each layer sees an unweighted RMSNorm of the residual stream:
 *   u = bf16( x / sqrt(mean(x^2) + eps) ),   x <- x + MoE(u).
 */
void orc_rmsnorm_bf16(const double* x, int H, double eps, uint16_t* u)
{
    double ss = 0.0;
    for (int h = 0; h < H; ++h)
        ss += x[h] * x[h];
    double r = sqrt(ss / H + eps);
    for (int h = 0; h < H; ++h)
        u[h] = orc_round_bf16(x[h] / r);
}
