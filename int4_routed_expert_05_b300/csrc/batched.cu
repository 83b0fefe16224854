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
//   5. grouped down GEMM per expert, scaled by the assignment's weight -> partial y rows (fp32);
//   6. per token: y = sum of its partials in rank order, then the shared expert's (fixed order).
// The GEMMs run on the tensor cores (mma.m16n8k16, fp32 accumulate); a producer dequantises the
// int4/int8 codes of each K-slice into fp16 weights w = s * q + b in shared memory (rounding to
// fp16 costs at most 2^-11 relative per weight).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "layout.h"

namespace moe {
namespace bat {

constexpr int kBM = 128, kBN = 64, kBK = 32;  // CTA tile (weights rows x tokens x K-slice)
constexpr int kThreadsG = 256;                // 8 warps: 4 along M x 2 along N
constexpr int kLdA = kBK + 8, kLdB = kBK + 8;  // padded smem rows (halves): conflict-free ldmatrix

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"((uint32_t)__cvta_generic_to_shared(p)));
}

__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const void* p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"((uint32_t)__cvta_generic_to_shared(p)));
}

template <bool kBf16>
__device__ __forceinline__ void mma(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2])
{
    if (kBf16)
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                     "{%0,%1,%2,%3};"
                     : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
    else
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                     "{%0,%1,%2,%3};"
                     : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// One GEMM task: rows [m0, m0 + kBM) of a weight matrix (row-major [M][K], K = inputs) against
// the activation rows of tokens listed in [n0, n0 + nn) of an assignment range.
struct GemmArgs {
    int kind;                  // 0: router (bf16 weights), 1: gate/up (quantised), 2: down (quantised)
    int T, H, E, k, I, Is, bits, n_exp;
    BlobGeo geo, geo_s;
    const uint8_t* arena;
    uint64_t stride;
    const int32_t* table;      // [E] slot of each expert of this layer
    const uint16_t* router;    // bf16 [E][H]
    const uint8_t* shared_blob;
    const uint16_t* u_bf16;    // [T][H] bf16 layer input (router)
    const __half* u_h;         // [T][H] fp16 copy of the input (expert B operand)
    const int32_t* list;       // [T*(k+1)] assignment -> token, sorted by expert
    const int32_t* offs;       // [E+2] assignment offsets per expert (E = shared)
    const float* aw;           // [T*(k+1)] weight of each sorted assignment
    __half* hbuf;              // [T*(k+1)][Imax] SwiGLU output per assignment
    float* ypart;              // [T*(k+1)][H] weighted down output per assignment
    float* logits;             // [T][E]
    int* status;
};

// Task decoding: tiles over (expert, M-tile, N-tile).
struct Task {
    int e, m0, n0, nn, M, K, rows_in;  // rows_in: rows of the matrix (for gate/up: I per matrix)
};

__device__ __forceinline__ const uint8_t* expert_blob(const GemmArgs& A, int e)
{
    if (e == A.E)
        return A.shared_blob;
    const int s = A.table[e];
    return s >= 0 ? A.arena + (uint64_t)s * A.stride : nullptr;
}

// Producer, first half: the thread's share of a K-slice, global -> registers. The thread owns one
// tile row and 16 consecutive K-elements of it (256 threads x 16 = 128 rows x 32).
// Gate/up tiles interleave gate and up rows: tile rows [0, 64) are gate rows m0 .. m0+63 and rows
// [64, 128) the same up rows, so the epilogue finds both halves of a SwiGLU pair in one tile.
struct AFrag {
    uint4 q;      // 16 codes (int4: .x/.y used) or 16 bf16 router values (with q2)
    uint4 q2;
    float s, b;   // scale and bias of the group (quantised matrices)
    bool on;
};

template <int kKind>
__device__ __forceinline__ AFrag fetch_a(const GemmArgs& A, const Task& t, const uint8_t* blob, const BlobGeo& g, int k0)
{
    AFrag f;
    f.q = f.q2 = make_uint4(0, 0, 0, 0);
    f.s = f.b = 0.f;
    const int r = threadIdx.x >> 1;
    const int kk = (threadIdx.x & 1) * 16;
    if (kKind == 0) {
        const int row = t.m0 + r;
        f.on = row < t.M;
        if (f.on) {
            const uint4* src = reinterpret_cast<const uint4*>(A.router + (size_t)row * A.H + k0 + kk);
            f.q = __ldg(src);
            f.q2 = __ldg(src + 1);
        }
        return f;
    }
    const int m = kKind == 1 ? (r < 64 ? 0 : 1) : 2;
    const int row = kKind == 1 ? t.m0 + (r & 63) : t.m0 + r;
    f.on = blob != nullptr && row < g.rows[m];
    if (f.on) {
        const int gidx = (k0 + kk) >> 6;
        f.s = bf(__ldg(reinterpret_cast<const uint16_t*>(blob + g.s_off[m]) + (size_t)row * g.groups[m] + gidx));
        f.b = bf(__ldg(reinterpret_cast<const uint16_t*>(blob + g.b_off[m]) + (size_t)row * g.groups[m] + gidx));
        const uint8_t* qrow = blob + g.q_off[m] + (size_t)row * g.row_bytes[m];
        if (A.bits == 4) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(qrow + (k0 + kk) / 2));
            f.q = make_uint4(v.x, v.y, 0, 0);
        } else {
            f.q = __ldg(reinterpret_cast<const uint4*>(qrow + k0 + kk));
        }
    }
    return f;
}

// Producer, second half: dequantise (w = s * q + b, rounded to fp16) and store into As.
template <int kKind>
__device__ __forceinline__ void store_a(const GemmArgs& A, const AFrag& f, uint16_t* As)
{
    const int r = threadIdx.x >> 1;
    const int kk = (threadIdx.x & 1) * 16;
    uint16_t* dst = As + r * kLdA + kk;
    if (kKind == 0) {
        *reinterpret_cast<uint4*>(dst) = f.q;
        *reinterpret_cast<uint4*>(dst + 8) = f.q2;
        return;
    }
    uint32_t out[8];
    if (!f.on) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            out[i] = 0u;
    } else if (A.bits == 4) {
        const uint32_t w[2] = {f.q.x, f.q.y};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t byte = (w[i >> 2] >> (8 * (i & 3))) & 0xFFu;
            const __half2 h = __floats2half2_rn(fmaf(f.s, (float)(byte & 15u), f.b), fmaf(f.s, (float)(byte >> 4), f.b));
            out[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
    } else {
        const uint32_t w[4] = {f.q.x, f.q.y, f.q.z, f.q.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t pair = (w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
            const __half2 h = __floats2half2_rn(fmaf(f.s, (float)(pair & 0xFFu), f.b), fmaf(f.s, (float)(pair >> 8), f.b));
            out[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
    }
    *reinterpret_cast<uint4*>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
    *reinterpret_cast<uint4*>(dst + 8) = make_uint4(out[4], out[5], out[6], out[7]);
}

// The activation rows of the task's tokens: 64 rows x 32 K-elements, 8 per thread.
template <int kKind>
__device__ __forceinline__ uint4 fetch_b(const GemmArgs& A, const Task& t, int k0)
{
    const int n = threadIdx.x >> 2;
    const int kk = (threadIdx.x & 3) * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < t.nn) {
        if (kKind == 0) {
            v = __ldg(reinterpret_cast<const uint4*>(A.u_bf16 + (size_t)(t.n0 + n) * A.H + k0 + kk));
        } else if (kKind == 1) {
            const int tok = A.list[t.n0 + n];
            v = __ldg(reinterpret_cast<const uint4*>(A.u_h + (size_t)tok * A.H + k0 + kk));
        } else {
            const int Imax = A.I > A.Is ? A.I : A.Is;
            v = *reinterpret_cast<const uint4*>(A.hbuf + (size_t)(t.n0 + n) * Imax + k0 + kk);
        }
    }
    return v;
}

__device__ __forceinline__ void store_b(uint4 v, uint16_t* Bs)
{
    const int n = threadIdx.x >> 2;
    const int kk = (threadIdx.x & 3) * 8;
    *reinterpret_cast<uint4*>(Bs + n * kLdB + kk) = v;
}

template <int kKind>
__global__ void __launch_bounds__(kThreadsG) gemm_kernel(const __grid_constant__ GemmArgs A, const int4* __restrict__ tasks,
                                                         int n_tasks)
{
    __shared__ __align__(16) uint16_t As[2][kBM * kLdA];
    __shared__ __align__(16) uint16_t Bs[2][kBN * kLdB];
    __shared__ float sc_w[kBN];
    constexpr bool kBf = kKind == 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wm = warp & 3, wn = warp >> 2;  // warp tile 32 x 32
    for (int ti = blockIdx.x; ti < n_tasks; ti += gridDim.x) {
        const int4 tv = tasks[ti];
        Task t;
        t.e = tv.x;
        t.m0 = tv.y;
        t.n0 = tv.z;
        t.nn = tv.w;
        const bool shared = t.e == A.E;
        const BlobGeo& g = shared ? A.geo_s : A.geo;
        const uint8_t* blob = kKind == 0 ? nullptr : expert_blob(A, t.e);
        if (kKind == 0) {
            t.M = A.E;
            t.K = A.H;
        } else if (kKind == 1) {
            t.M = g.rows[0];
            t.K = A.H;
        } else {
            t.M = A.H;
            t.K = g.cols[2];
        }
        float acc[2][4][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    acc[i][j][q] = 0.f;
        const int nk = t.K / kBK;
        store_a<kKind>(A, fetch_a<kKind>(A, t, blob, g, 0), As[0]);
        store_b(fetch_b<kKind>(A, t, 0), Bs[0]);
        __syncthreads();
        for (int ks = 0; ks < nk; ++ks) {
            const int cur = ks & 1;
            AFrag fa;
            uint4 fb = make_uint4(0, 0, 0, 0);
            const bool more = ks + 1 < nk;
            if (more) {  // next slice's loads in flight while this slice's MMAs run
                fa = fetch_a<kKind>(A, t, blob, g, (ks + 1) * kBK);
                fb = fetch_b<kKind>(A, t, (ks + 1) * kBK);
            }
#pragma unroll
            for (int kk = 0; kk < kBK; kk += 16) {
                uint32_t af[2][4], bfr[4][2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int row = wm * 32 + i * 16 + (lane & 15);
                    const int col = kk + (lane >> 4) * 8;
                    ldsm_x4(af[i], &As[cur][row * kLdA + col]);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int row = wn * 32 + j * 8 + (lane & 7);
                    const int col = kk + ((lane >> 3) & 1) * 8;
                    ldsm_x2(bfr[j], &Bs[cur][row * kLdB + col]);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        mma<kBf>(acc[i][j], af[i], bfr[j]);
            }
            if (more) {
                store_a<kKind>(A, fa, As[cur ^ 1]);
                store_b(fb, Bs[cur ^ 1]);
            }
            __syncthreads();
        }
        // ---- epilogue ----
        // acc[i][j][q]: row = wm*32 + i*16 + (lane>>2) + (q>=2 ? 8 : 0), col = wn*32 + j*8 + (lane&3)*2 + (q&1)
        if (kKind == 0) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int r = t.m0 + wm * 32 + i * 16 + (lane >> 2) + (q >= 2 ? 8 : 0);
                        const int n = wn * 32 + j * 8 + (lane & 3) * 2 + (q & 1);
                        if (r < t.M && n < t.nn)
                            A.logits[(size_t)(t.n0 + n) * A.E + r] = acc[i][j][q];
                    }
        } else if (kKind == 1) {
            // tile rows [0, 64): gate rows, [64, 128): up rows of the same matrix rows; the warp
            // pairs wm (gate) and wm + 2 (up) hold matching rows: exchange through shared memory
            float* ex = reinterpret_cast<float*>(As);  // reuse: 64 x 64 fp32 = 16 KB < sizeof As
            if (wm >= 2) {
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int rr = (wm - 2) * 32 + i * 16 + (lane >> 2) + (q >= 2 ? 8 : 0);
                            const int n = wn * 32 + j * 8 + (lane & 3) * 2 + (q & 1);
                            ex[rr * kBN + n] = acc[i][j][q];
                        }
            }
            __syncthreads();
            if (wm < 2) {
                const int Imax = A.I > A.Is ? A.I : A.Is;
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int rr = wm * 32 + i * 16 + (lane >> 2) + (q >= 2 ? 8 : 0);
                            const int n = wn * 32 + j * 8 + (lane & 3) * 2 + (q & 1);
                            const int row = t.m0 + rr;
                            if (row < t.M && n < t.nn) {
                                const float gg = acc[i][j][q], vv = ex[rr * kBN + n];
                                const float h = gg / (1.f + expf(-gg)) * vv;
                                A.hbuf[(size_t)(t.n0 + n) * Imax + row] = __float2half_rn(h);
                            }
                        }
            }
            __syncthreads();
        } else {
            if (threadIdx.x < kBN)
                sc_w[threadIdx.x] = threadIdx.x < t.nn ? A.aw[t.n0 + threadIdx.x] : 0.f;
            __syncthreads();
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int r = t.m0 + wm * 32 + i * 16 + (lane >> 2) + (q >= 2 ? 8 : 0);
                        const int n = wn * 32 + j * 8 + (lane & 3) * 2 + (q & 1);
                        if (r < t.M && n < t.nn)
                            A.ypart[(size_t)(t.n0 + n) * A.H + r] = sc_w[n] * acc[i][j][q];
                    }
            __syncthreads();
        }
    }
}

// bf16 input -> fp16 copy (B operand of the expert GEMMs)
__global__ void to_half_kernel(const uint16_t* __restrict__ x, __half* __restrict__ y, size_t n)
{
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        y[i] = __float2half_rn(bf(x[i]));
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

// Exclusive scan of the E counts (one block), the shared expert's T assignments last.
__global__ void scan_kernel(const int32_t* __restrict__ counts, int E, int T, int32_t* __restrict__ offs,
                            int32_t* __restrict__ cursor)
{
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int e = 0; e < E; ++e) {
            offs[e] = acc;
            cursor[e] = acc;
            acc += counts[e];
        }
        offs[E] = acc;
        cursor[E] = acc;
        offs[E + 1] = acc + T;
    }
}

// Assignments grouped by expert: assignment (t, j) takes the next free position of expert idx[t][j]
// (the shared expert, E, takes every token). The order inside an expert does not change any result:
// every column of the expert GEMMs is computed on its own.
__global__ void place_kernel(const int32_t* __restrict__ idx, const float* __restrict__ w, const float* __restrict__ gamma,
                             int T, int E, int k, int32_t* __restrict__ cursor, int32_t* __restrict__ list,
                             float* __restrict__ aw, int32_t* __restrict__ pos)
{
    const int n = T * (k + 1);
    for (int a = blockIdx.x * blockDim.x + threadIdx.x; a < n; a += gridDim.x * blockDim.x) {
        const int t = a / (k + 1), j = a - t * (k + 1);
        const int e = j < k ? idx[(size_t)t * k + j] : E;
        const int p = atomicAdd(&cursor[e], 1);
        list[p] = t;
        aw[p] = j < k ? w[(size_t)t * k + j] : gamma[t];
        pos[a] = p;
    }
}

// y[t][o] = sum_j ypart[pos(t, j)][o] in rank order, then the shared expert's partial.
__global__ void combine_kernel(const float* __restrict__ ypart, const int32_t* __restrict__ pos, int T, int H, int k,
                               float* __restrict__ y)
{
    const size_t n = (size_t)T * H;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / H), o = (int)(i - (size_t)t * H);
        float acc = 0.f;
        for (int j = 0; j <= k; ++j)
            acc += ypart[(size_t)pos[(size_t)t * (k + 1) + j] * H + o];
        y[i] = acc;
    }
}

void launch_to_half(const uint16_t* x, __half* y, size_t n, cudaStream_t st)
{
    to_half_kernel<<<1184, 256, 0, st>>>(x, y, n);
}

void launch_gemm(int kind, const GemmArgs& A, const int4* tasks, int n_tasks, int grid, cudaStream_t st)
{
    if (n_tasks <= 0)
        return;
    const int g = n_tasks < grid ? n_tasks : grid;
    if (kind == 0)
        gemm_kernel<0><<<g, kThreadsG, 0, st>>>(A, tasks, n_tasks);
    else if (kind == 1)
        gemm_kernel<1><<<g, kThreadsG, 0, st>>>(A, tasks, n_tasks);
    else
        gemm_kernel<2><<<g, kThreadsG, 0, st>>>(A, tasks, n_tasks);
}

void launch_topk(const float* logits, const float* bias, int T, int E, int k, int renorm, const uint16_t* u,
                 const uint16_t* wsg, int H, int32_t* idx, float* w, float* gamma, int32_t* counts, cudaStream_t st)
{
    topk_kernel<<<(T * 32 + 255) / 256, 256, 0, st>>>(logits, bias, T, E, k, renorm, u, wsg, H, idx, w, gamma, counts);
}

void launch_scan(const int32_t* counts, int E, int T, int32_t* offs, int32_t* cursor, cudaStream_t st)
{
    scan_kernel<<<1, 32, 0, st>>>(counts, E, T, offs, cursor);
}

void launch_place(const int32_t* idx, const float* w, const float* gamma, int T, int E, int k, int32_t* cursor,
                  int32_t* list, float* aw, int32_t* pos, cudaStream_t st)
{
    const int n = T * (k + 1);
    place_kernel<<<(n + 255) / 256, 256, 0, st>>>(idx, w, gamma, T, E, k, cursor, list, aw, pos);
}

void launch_combine(const float* ypart, const int32_t* pos, int T, int H, int k, float* y, cudaStream_t st)
{
    combine_kernel<<<1184, 256, 0, st>>>(ypart, pos, T, H, k, y);
}

}  // namespace bat
}  // namespace moe
