/*
 * hybrid.h -- C ABI of the two per-layer decode steps that precede the MoE FFN in the 80B hybrid
 * stack, built into libmoe next to the entry points of moe.h:
 *   moe_gdn_step    Gated DeltaNet decode step (36 of the 48 layers): a fixed-size recurrent state
 *                   per value head, updated in place by the gated delta rule, read out with q and
 *                   passed through a gated RMS norm.
 *   moe_gqa_decode  gated grouped-query attention decode step (the other 12 layers): the new
 *                   token's key and value are appended to a K/V cache kept in 32-bit floats, every
 *                   query head attends over all cached positions of its K/V head, and the result is
 *                   gated by sigmoid(gate).
 *
 * Sources:
 *  [mix]   alphalab.site, "Swiftlet 實測資料解讀", section explaining the 80B layer mix: 48 layers,
 *          36 with a fixed DeltaNet recurrent state (about 72 MiB in all), 12 with full attention
 *          whose K/V cache is held in 32-bit floats (at least 48 KiB per token, about 384 MiB at
 *          an 8K context).
 *  [gdn]   paotong.dev commentary on Swiftlet, paragraph on the hybrid layers (75% of the layers
 *          are Gated DeltaNet linear attention with a fixed-size state); cheshm.ai item on
 *          Swiftlet, architecture paragraph (Gated DeltaNet, gated GQA, sparse MoE).
 * The pages name the layer types without their equations; the equations are the published ones:
 * the gated delta rule of Gated DeltaNet (Yang, Kautz and Hatamizadeh, ICLR 2025) with a
 * Mamba2-form decay, and softmax attention with grouped K/V heads and an element-wise output gate.
 *
 * Conventions are those of moe.h: d_* pointers are caller-owned device memory, streams are
 * cudaStream_t values passed as void* (NULL = legacy default stream), work is enqueued and the call
 * returns without waiting, nothing is allocated, and errors come back as moe_status with a message
 * in moe_last_error(). bf16 values are passed as their 16-bit patterns (uint16_t).
 */
#ifndef MOE_HYBRID_H
#define MOE_HYBRID_H

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- Gated DeltaNet decode step */

/* Hk key heads and Hv value heads (Hv a multiple of Hk; value head h reads key head h / (Hv / Hk)),
 * key_dim dk and value_dim dv. Supported: dk == 128, dv in {32, 64, 128, 256}, 1 <= Hk <= Hv. */
typedef struct {
    int32_t n_key_heads;
    int32_t n_value_heads;
    int32_t key_dim;
    int32_t value_dim;
} moe_gdn_shape;

#define MOE_GDN_L2_EPS   1e-6f /* q^ = scale q / sqrt(|q|^2 + eps), k^ = k / sqrt(|k|^2 + eps) */
#define MOE_GDN_NORM_EPS 1e-6f /* head norm: o / sqrt(mean(o^2) + eps) */

/* One decode step of `batch` independent sequences ([gdn], [mix]). Per sequence and value head h
 * (g = h / (Hv / Hk)):
 *     alpha = exp(-exp(A_log[h]) * softplus(a[h] + dt_bias[h])),   beta = sigmoid(b[h])
 *     S <- alpha S + beta (v_h - alpha S k^_g) k^_g^T        (the gated delta rule)
 *     o_h = S q^_g;   y_h = o_h / sqrt(mean(o_h^2) + eps) * norm_w * silu(z_h)
 * Layouts (row-major, fp32 unless noted):
 *   d_state   [batch][Hv][dv][dk]   the recurrent state, read and written in place (dv rows of dk)
 *   d_q, d_k  [batch][Hk][dk] bf16;  d_v, d_z [batch][Hv][dv] bf16
 *   d_a, d_b  [batch][Hv];  d_A_log, d_dt_bias [Hv];  d_norm_w [dv]
 *   d_o       [batch][Hv][dv] head outputs before the norm (may be NULL);  d_y [batch][Hv][dv]
 * All pointers 16-byte aligned. The state must not overlap any other argument.
 * Errors: MOE_E_INVALID (null or misaligned pointer, batch < 1), MOE_E_SHAPE (unsupported shape),
 * MOE_E_CUDA (launch failure). The kernel has no waits and no device status. */
moe_status moe_gdn_step(const moe_gdn_shape* shape, int32_t batch, float* d_state, const uint16_t* d_q,
                        const uint16_t* d_k, const uint16_t* d_v, const uint16_t* d_z, const float* d_a,
                        const float* d_b, const float* d_A_log, const float* d_dt_bias, const float* d_norm_w,
                        float scale, float* d_o, float* d_y, void* stream);

/* ---------------------------------------------------------------- gated GQA decode attention */

/* Hq query heads over Hkv K/V heads (query head h reads K/V head h / (Hq / Hkv)), head_dim D, and
 * a cache capacity of max_len positions per sequence. Supported: D == 256 with Hq / Hkv in
 * {1, 2, 4, 8}; D == 128 with Hq / Hkv in {1, 2, 4, 8, 16}; max_len >= 1. */
typedef struct {
    int32_t n_q_heads;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t max_len;
} moe_gqa_shape;

/* Workspace bytes moe_gqa_decode needs for `batch` sequences when no sequence holds more than
 * max_pos positions after the step (1 <= max_pos <= max_len); 0 for an unsupported shape. */
size_t moe_gqa_workspace_bytes(const moe_gqa_shape* shape, int32_t batch, int32_t max_pos);

/* One decode step of `batch` sequences ([mix]). Sequence b holds d_pos[b] cached positions; its
 * new key and value are written at position d_pos[b], and query head h attends over positions
 * 0 .. d_pos[b] of its K/V head:
 *     o_h = sum_t softmax_t(scale q_h . K_t) V_t,    y_h = o_h * sigmoid(gate_h)
 * Layouts (row-major):
 *   d_k_cache, d_v_cache  [batch][Hkv][max_len][D] fp32, row d_pos[b] of each written in place
 *   d_pos     [batch] int32, read only (the caller advances it after the step)
 *   d_q, d_gate [batch][Hq][D] bf16;  d_k, d_v [batch][Hkv][D] bf16
 *   d_o       [batch][Hq][D] fp32 attention output before the gate (may be NULL);  d_y likewise
 *   d_work    at least moe_gqa_workspace_bytes(shape, batch, max_pos) bytes, 16-byte aligned
 *   d_status  one int32 the caller clears to 0 before the call (required)
 * max_pos bounds the step's positions: every d_pos[b] + 1 <= max_pos <= max_len; it sets how the
 * positions are split across thread blocks (the split depends on it alone, so results are the same
 * bit for bit for equal max_pos). The partial results are combined in a fixed order: the call is
 * deterministic.
 * Errors returned: MOE_E_INVALID (null or misaligned pointer, batch < 1, max_pos out of range),
 * MOE_E_SHAPE, MOE_E_NOMEM (work_bytes too small), MOE_E_CUDA. Found on the device and written to
 * *d_status (first problem wins): MOE_E_RANGE when some d_pos[b] is outside 0 .. max_pos - 1
 * (that sequence's cache rows and outputs are left untouched), MOE_E_TIMEOUT when a copy into shared
 * memory did not arrive within about a second (outputs then unspecified). */
moe_status moe_gqa_decode(const moe_gqa_shape* shape, int32_t batch, int32_t max_pos, float* d_k_cache,
                          float* d_v_cache, const int32_t* d_pos, const uint16_t* d_q, const uint16_t* d_k,
                          const uint16_t* d_v, const uint16_t* d_gate, float scale, void* d_work, size_t work_bytes,
                          float* d_o, float* d_y, int32_t* d_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_HYBRID_H */
