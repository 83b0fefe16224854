// batched.cu -- the MoE FFN layer for a batch of tokens (prefill or batched decode), sm_103a.
//
// Same layer as the decode kernel (cheshm.ai item "Swiftlet fits an 80B-level Qwen giant into
// Mac": k of E routed experts plus always-on shared experts, MLX-style int4/int8 group
// quantisation; alphalab.site "Swiftlet 實測資料解讀", the 35B router-normalisation fix), organised
// for many tokens at once, where the expert matrices are real GEMMs:
//   1. router GEMM  logits[T][E] = U[T][H] Wr^T (bf16 x bf16, fp32 accumulate, exact products);
//   2. per token: top-k (equal logits to the lower index), renormalised weights, shared gate;
//   3. counting sort of the T*k assignments by expert (the shared expert takes all T tokens as
//      "expert" E), so each expert's tokens are contiguous;
//   4. grouped gate/up GEMM per expert with SwiGLU in the epilogue -> h[assignment][I] (fp16);
//   5. grouped down GEMM per expert, scaled by the assignment's weight, added into y by fp32
//      reductions in tile completion order (the sum of a token's k + 1 contributions is then not
//      bit reproducible), or, with MOE_DETERMINISTIC, stored per assignment;
//   6. (MOE_DETERMINISTIC) per token: y = its k routed contributions in rank order, then the
//      shared expert's (a fixed order, bit reproducible).
// Range: the expert GEMMs take fp16 operands. Input elements above 65504 in magnitude, scales
// below fp16's normal range (their relative precision would be lost on every code of the group) or
// above it, biases above it, and weights s q + b or SwiGLU outputs that would overflow fp16 set
// MOE_E_RANGE in the status word. (Elements in fp16's subnormal range lose at most 2^-25 absolute,
// which no output notices: they are not reported.)
// This file holds everything around the GEMMs (grouped.cu): top-k, the device-side plan (offsets
// per expert, GEMM task lists), the placement of assignments and the input rows in assignment order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "grouped.h"
#include "layout.h"

namespace moe {
namespace bat {

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// The expert GEMMs' input operand: row p = the fp16 copy of the input row of assignment p's token,
// K-permuted within 8-element blocks in the order the dequantiser emits weight pairs (tc::kperm).
// One warp per row, one 8-element block per lane and step. bf16 -> fp16 is exact for |x| in
// [2^-14, 65504] (bf16's 8-bit significand fits in fp16's 11 bits).
__global__ void gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ list, int A, int H,
                                   int bits, __half* __restrict__ us, int* status)
{
    bool inexact = false;  // an element fp16 cannot hold
    const int lane = threadIdx.x & 31;
    for (int p = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < A; p += (gridDim.x * blockDim.x) >> 5) {
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)list[p] * H);
        uint4* dst = reinterpret_cast<uint4*>(us + (size_t)p * H);
        for (int c = lane; c < H / 8; c += 32) {
            const uint4 v = __ldg(src + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            __half h[8], o[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float f = bf((uint16_t)(w[j >> 1] >> (16 * (j & 1))));
                h[j] = __float2half_rn(f);
                inexact |= !(fabsf(f) <= 65504.f);  // beyond fp16's range
            }
            if (bits == 4) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    o[tc::kperm(j, 4)] = h[j];
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    o[tc::kperm(j, 8)] = h[j];
            }
            dst[c] = *reinterpret_cast<const uint4*>(o);
        }
    }
    if (inexact)
        atomicCAS(status, 0, kStatusRange);
}

__device__ __forceinline__ uint32_t ord_key(float f)
{
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp per token: top-k of the E logits (ties -> lower index), weights, shared gate, counts.
__global__ void topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E, int k,
                            int renorm, const uint16_t* __restrict__ u, const uint16_t* __restrict__ wsg, int H,
                            int32_t* __restrict__ idx, float* __restrict__ w, float* __restrict__ gamma,
                            int32_t* __restrict__ counts)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= T)
        return;
    const float* lg = logits + (size_t)warp * E;
    // each lane keeps its keys in registers (E <= 512 -> 16 per lane)
    uint32_t keys[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int e = lane + 32 * i;
        keys[i] = e < E ? ord_key(lg[e] + (bias ? bias[e] : 0.f)) : 0u;
    }
    int sel[kMaxK];
    for (int j = 0; j < k; ++j) {
        uint32_t bk = 0u;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int e = lane + 32 * i;
            if (keys[i] > bk || (keys[i] == bk && e < bi)) {
                bk = keys[i];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const uint32_t ok = __shfl_xor_sync(0xffffffffu, bk, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ok > bk || (ok == bk && oi < bi)) {
                bk = ok;
                bi = oi;
            }
        }
        sel[j] = bi;
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (lane + 32 * i == bi)
                keys[i] = 0u;
    }
    // weights: softmax (max subtracted) renormalised over the k selected, or over all E
    const float lmax = lg[sel[0]] + (bias ? bias[sel[0]] : 0.f);
    float denom = 0.f;
    if (renorm) {
        for (int j = 0; j < k; ++j)
            denom += expf(lg[sel[j]] + (bias ? bias[sel[j]] : 0.f) - lmax);
    } else {
        float s = 0.f;
        for (int e = lane; e < E; e += 32)
            s += expf(lg[e] + (bias ? bias[e] : 0.f) - lmax);
#pragma unroll
        for (int o = 16; o; o >>= 1)
            s += __shfl_xor_sync(0xffffffffu, s, o);
        denom = s;
    }
    if (lane < k) {
        int mine = sel[0];
        for (int j = 0; j < k; ++j)
            if (j == lane)
                mine = sel[j];
        idx[(size_t)warp * k + lane] = mine;
        w[(size_t)warp * k + lane] = expf(lg[mine] + (bias ? bias[mine] : 0.f) - lmax) / denom;
        atomicAdd(&counts[mine], 1);
    }
    // shared gate sigmoid(w_sg . u)
    float z = 0.f;
    for (int i = lane; i < H; i += 32)
        z = fmaf(bf(wsg[i]), bf(u[(size_t)warp * H + i]), z);
#pragma unroll
    for (int o = 16; o; o >>= 1)
        z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane == 0)
        gamma[warp] = 1.f / (1.f + expf(-z));
}

// Block-wide exclusive scan (blockDim.x == 1024); returns the total in *total.
__device__ int block_scan(int v, int* total)
{
    __shared__ int warp_sum[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        warp_sum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        warp_sum[lane] = w;
    }
    __syncthreads();
    const int excl = x - v + (warp ? warp_sum[warp - 1] : 0);
    *total = warp_sum[31];
    __syncthreads();
    return excl;
}

// The plan, on the device (one block of 1024 threads): assignment offsets per expert (the shared
// expert, index E, takes all T tokens last) and the GEMM task lists. A task is one 128-token chunk
// of one expert's assignments against one M tile: 64 rows of gate and of up, or 128 rows of down.
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ counts, int E, int T, int I, int Is,
                                                    int H, int32_t* __restrict__ offs, int32_t* __restrict__ cursor,
                                                    int4* __restrict__ tasks_gu, int4* __restrict__ tasks_dn,
                                                    int32_t* __restrict__ n_tasks)
{
    const int e = threadIdx.x;
    const bool on = e <= E;
    const int cnt = on ? (e < E ? counts[e] : T) : 0;
    int total;
    const int off = block_scan(cnt, &total);
    if (on) {
        offs[e] = off;
        cursor[e] = off;
    }
    if (e == 0)
        offs[E + 1] = total;
    const int chunks = (cnt + tc::kNT - 1) / tc::kNT;
    const int mgu = (e < E ? I : Is) / 64, mdn = (H + 127) / 128;
    int ngu, ndn;
    const int bgu = block_scan(chunks * mgu, &ngu);
    const int bdn = block_scan(chunks * mdn, &ndn);
    for (int c = 0; c < chunks; ++c) {
        const int n0 = off + c * tc::kNT, nn = min(tc::kNT, cnt - c * tc::kNT);
        for (int m = 0; m < mgu; ++m)
            tasks_gu[bgu + c * mgu + m] = make_int4(e, m * 64, n0, nn);
        for (int m = 0; m < mdn; ++m)
            tasks_dn[bdn + c * mdn + m] = make_int4(e, m * 128, n0, nn);
    }
    if (e == 0) {
        n_tasks[0] = ngu;
        n_tasks[1] = ndn;
    }
}

// Assignments grouped by expert: assignment (t, j) takes the next free position of expert idx[t][j]
// (the shared expert, E, takes every token). The order inside an expert does not change the
// result: every column of the expert GEMMs is computed on its own.
__global__ void place_kernel(const int32_t* __restrict__ idx, const float* __restrict__ w, const float* __restrict__ gamma,
                             int T, int E, int k, int32_t* __restrict__ cursor, int32_t* __restrict__ list,
                             float* __restrict__ aw, int32_t* __restrict__ apos)
{
    const int n = T * (k + 1);
    for (int a = blockIdx.x * blockDim.x + threadIdx.x; a < n; a += gridDim.x * blockDim.x) {
        const int t = a / (k + 1), j = a - t * (k + 1);
        const int e = j < k ? idx[(size_t)t * k + j] : E;
        const int p = atomicAdd(&cursor[e], 1);
        list[p] = t;
        aw[p] = j < k ? w[(size_t)t * k + j] : gamma[t];
        apos[a] = p;
    }
}

// Deterministic combine: y[t] = sum over j = 0..k (rank order, the shared expert last) of the
// weighted down rows of assignment (t, j).
__global__ void combine_kernel(const float* __restrict__ ypart, const int32_t* __restrict__ apos, int T, int k, int H,
                               float* __restrict__ y)
{
    const int n4 = H / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)T * n4; i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / n4), c = (int)(i - (size_t)t * n4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j <= k; ++j) {
            const float4 v = reinterpret_cast<const float4*>(ypart + (size_t)apos[(size_t)t * (k + 1) + j] * H)[c];
            acc = make_float4(acc.x + v.x, acc.y + v.y, acc.z + v.z, acc.w + v.w);
        }
        reinterpret_cast<float4*>(y + (size_t)t * H)[c] = acc;
    }
}

void launch_gather_rows(const uint16_t* x, const int32_t* list, int A, int H, int bits, __half* us, int* status,
                        cudaStream_t st)
{
    gather_rows_kernel<<<(A + 7) / 8 < 2368 ? (A + 7) / 8 : 2368, 256, 0, st>>>(x, list, A, H, bits, us, status);
}

void launch_combine(const float* ypart, const int32_t* apos, int T, int k, int H, float* y, cudaStream_t st)
{
    const size_t n = (size_t)T * (H / 4);
    const size_t blocks = (n + 255) / 256;
    combine_kernel<<<blocks < 2368 ? (int)blocks : 2368, 256, 0, st>>>(ypart, apos, T, k, H, y);
}

void launch_topk(const float* logits, const float* bias, int T, int E, int k, int renorm, const uint16_t* u,
                 const uint16_t* wsg, int H, int32_t* idx, float* w, float* gamma, int32_t* counts, cudaStream_t st)
{
    topk_kernel<<<(T * 32 + 255) / 256, 256, 0, st>>>(logits, bias, T, E, k, renorm, u, wsg, H, idx, w, gamma, counts);
}

void launch_plan(const int32_t* counts, int E, int T, int I, int Is, int H, int32_t* offs, int32_t* cursor,
                 int4* tasks_gu, int4* tasks_dn, int32_t* n_tasks, cudaStream_t st)
{
    plan_kernel<<<1, 1024, 0, st>>>(counts, E, T, I, Is, H, offs, cursor, tasks_gu, tasks_dn, n_tasks);
}

void launch_place(const int32_t* idx, const float* w, const float* gamma, int T, int E, int k, int32_t* cursor,
                  int32_t* list, float* aw, int32_t* apos, cudaStream_t st)
{
    const int n = T * (k + 1);
    place_kernel<<<(n + 255) / 256, 256, 0, st>>>(idx, w, gamma, T, E, k, cursor, list, aw, apos);
}

}  // namespace bat
}  // namespace moe
