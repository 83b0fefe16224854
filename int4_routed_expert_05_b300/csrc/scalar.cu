// scalar.cu -- plain reference kernels of one MoE FFN layer for one token.
//
// One thread per router logit, one thread for the top-k selection, one thread per gate/up row
// and one thread per output row; every sum runs in index order in fp32 with the weight
// dequantised as s * q + b first. These kernels exist to cross-check the fused decode kernel on
// the GPU (the pages' practice of keeping a "fast" and a "scalar" kernel of the same layer;
// paotong.dev commentary on Swiftlet, paragraph on correctness).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "layout.h"

namespace moe {
namespace {

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ int code_at(const uint8_t* row, int bits, int c)
{
    if (bits == 8)
        return row[c];
    const uint8_t b = row[c >> 1];
    return (c & 1) ? (b >> 4) : (b & 15);
}

// w[r][c] of matrix m of a blob
__device__ __forceinline__ float weight(const uint8_t* blob, const BlobGeo& g, int bits, int group, int m, int r, int c)
{
    const uint8_t* row = blob + g.q_off[m] + (uint64_t)r * g.row_bytes[m];
    const uint64_t gi = (uint64_t)r * g.groups[m] + c / group;
    const float s = bf(*reinterpret_cast<const uint16_t*>(blob + g.s_off[m] + 2 * gi));
    const float b = bf(*reinterpret_cast<const uint16_t*>(blob + g.b_off[m] + 2 * gi));
    return s * (float)code_at(row, bits, c) + b;
}

}  // namespace

__global__ void scalar_router(const StepParams P)
{
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= P.E)
        return;
    const LayerDesc L = P.layers[P.layer0];
    const uint16_t* u = (const uint16_t*)P.x_in;
    float acc = 0.f;
    for (int h = 0; h < P.H; ++h)
        acc = fmaf(bf(L.router[(size_t)e * P.H + h]), bf(u[h]), acc);
    if (L.logit_bias)
        acc += L.logit_bias[e];
    P.logits[e] = acc;
}

// sel: int32 [kMaxK] indices, then float [kMaxK] weights, then int32 [kMaxK] slots
__global__ void scalar_topk(const StepParams P, int32_t* sel)
{
    if (threadIdx.x != 0 || blockIdx.x != 0)
        return;
    int32_t* idx = sel;
    float* w = reinterpret_cast<float*>(sel + kMaxK);
    int32_t* slot = sel + 2 * kMaxK;
    for (int j = 0; j < P.k; ++j) {
        int best = -1;
        float bv = 0.f;
        for (int e = 0; e < P.E; ++e) {
            bool taken = false;
            for (int q = 0; q < j; ++q)
                taken |= idx[q] == e;
            if (taken)
                continue;
            const float v = P.logits[e];
            if (best < 0 || v > bv) {
                best = e;
                bv = v;
            }
        }
        idx[j] = best;
    }
    const float mx = P.logits[idx[0]];
    float denom = 0.f;
    if (P.flags & kRenorm) {
        for (int j = 0; j < P.k; ++j)
            denom += expf(P.logits[idx[j]] - mx);
    } else {
        for (int e = 0; e < P.E; ++e)
            denom += expf(P.logits[e] - mx);
    }
    for (int j = 0; j < P.k; ++j) {
        w[j] = expf(P.logits[idx[j]] - mx) / denom;
        slot[j] = P.table[(size_t)P.layer0 * P.E + idx[j]];
        if (P.topk_idx)
            P.topk_idx[j] = idx[j];
        if (P.topk_w)
            P.topk_w[j] = w[j];
    }
}

// thread (j, r): h_j[r] = silu(Wg_j[r] . u) * (Wu_j[r] . u); j == k is the shared expert
__global__ void scalar_gateup(const StepParams P, const int32_t* sel)
{
    const int Imax = P.I > P.Is ? P.I : P.Is;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const int j = t / Imax, r = t % Imax;
    if (j > P.k)
        return;
    const int Ij = j < P.k ? P.I : P.Is;
    if (r >= Ij)
        return;
    const LayerDesc L = P.layers[P.layer0];
    const uint8_t* blob;
    if (j < P.k) {
        const int s = sel[2 * kMaxK + j];
        if (s < 0)
            return;
        blob = P.arena + (uint64_t)s * P.stride;
    } else {
        blob = L.shared_blob;
    }
    const BlobGeo& g = j < P.k ? P.geo : P.geo_s;
    const uint16_t* u = (const uint16_t*)P.x_in;
    float gs = 0.f, vs = 0.f;
    for (int c = 0; c < P.H; ++c) {
        gs = fmaf(weight(blob, g, P.bits, P.group, 0, r, c), bf(u[c]), gs);
        vs = fmaf(weight(blob, g, P.bits, P.group, 1, r, c), bf(u[c]), vs);
    }
    P.hbuf[(size_t)j * Imax + r] = gs / (1.f + expf(-gs)) * vs;
}

// thread o: y[o] = sum_j w_j (Wd_j[o] . h_j) + sigmoid(w_sg . u) (Wd_s[o] . h_s)
__global__ void scalar_down(const StepParams P, const int32_t* sel)
{
    const int o = blockIdx.x * blockDim.x + threadIdx.x;
    if (o >= P.H)
        return;
    const int Imax = P.I > P.Is ? P.I : P.Is;
    const LayerDesc L = P.layers[P.layer0];
    const uint16_t* u = (const uint16_t*)P.x_in;
    const float* w = reinterpret_cast<const float*>(sel + kMaxK);
    float y = 0.f;
    for (int j = 0; j <= P.k; ++j) {
        const uint8_t* blob;
        float wj;
        if (j < P.k) {
            const int s = sel[2 * kMaxK + j];
            if (s < 0)
                continue;
            blob = P.arena + (uint64_t)s * P.stride;
            wj = w[j];
        } else {
            blob = L.shared_blob;
            float z = 0.f;
            for (int h = 0; h < P.H; ++h)
                z = fmaf(bf(L.shared_gate[h]), bf(u[h]), z);
            wj = 1.f / (1.f + expf(-z));
        }
        const BlobGeo& g = j < P.k ? P.geo : P.geo_s;
        const int Ij = j < P.k ? P.I : P.Is;
        float acc = 0.f;
        for (int r = 0; r < Ij; ++r)
            acc = fmaf(weight(blob, g, P.bits, P.group, 2, o, r), P.hbuf[(size_t)j * Imax + r], acc);
        y = fmaf(wj, acc, y);
    }
    P.y_out[o] = y;
}

}  // namespace moe
