// gemv.cu -- the batched layer's expert products for small token counts (T <= kGemvMaxTokens).
//
// With few tokens per expert the expert matrices are matrix-vector products: each touched expert's
// weights are read once and used for its one or few assignments, so the work is bound by the bytes
// of the weights, not by tensor-core rate. These kernels replace the two tcgen05 GEMM launches of
// the batched path for such T and keep everything around them: the same task lists (from the plan
// kernel), the same fp16 operand rows in assignment order (K-permuted within 8-element blocks in
// the order the dequantiser emits code pairs), the same SwiGLU and down epilogues. The weights
// enter exactly: a code q goes into the MMA as the fp16 value 1024 + q (one lop3 per code pair),
// a second MMA with A = 1 gives each column's sum of x over the 64-element group, and the affine
// dequantisation is applied per group in fp32, s (sum (1024 + q) x - 1024 sum x) + b sum x (the
// GEMM path instead rounds s q + b to fp16 and reports scales fp16 cannot hold; here any bf16 scale
// is exact).
//
// Work: a gate/up task (64 rows of gate and of up) runs as 4 rounds of 16 gate + 16 up rows; a down
// task (128 rows) as one round. A round's rows arrive as one 1D bulk copy per row (plus
// the rows' scale and bias spans) into shared-memory rows padded by 16 bytes, so that the 8 rows a
// warp's fragment load touches fall in distinct banks; two rounds are in flight. The 8 warps split
// K into 64-element groups of four 16-element slices; per slice each warp feeds its rows' codes
// straight into the A fragments of mma.sync m16n8k16 (rows = weight rows, K = 16, N = 8
// assignments) with the activations as B, fp32 accumulation; a warp takes whole quantisation groups
// (w, w + 8, ...), so each row's scale and bias are read once per group, and fetches the next
// group's activation fragments while it works on the current one. The warps' partial sums are added in
// warp order through shared memory, so the result does not depend on timing.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attr.h"
#include "grouped.h"
#include "layout.h"

namespace moe {
namespace gv {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 2;
constexpr int kPad = 16;  // bytes added to every staged row

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ void mbar_init(uint64_t* m, int n)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(m)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_expect(uint64_t* m, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(m)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* m, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(su32(m)), "r"(parity)
                 : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* m, uint32_t parity, long long limit)
{
    const long long t0 = clock64();
    while (!mbar_try(m, parity))
        if (clock64() - t0 > limit)
            return false;
    return true;
}
// 1D bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* m)
{
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(su32(dst)),
                 "l"(src), "r"(bytes), "r"(su32(m))
                 : "memory");
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Code pair p (0..3) of an 8-element K block as fp16 (1024 + q_i, 1024 + q_j), in the K-permuted
// storage order: int4, one 32-bit word per block, pair p = nibbles (p, p + 4); int8, two words per
// block, pair p = bytes (0, 2) or (1, 3) of word p / 2.
template <int BITS>
__device__ __forceinline__ uint32_t code_pair(const uint32_t* w, int p)
{
    if (BITS == 4) {
        uint32_t x;
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(x) : "r"(w[0] >> (4 * p)), "r"(0x000F000Fu), "r"(0x64006400u));
        return x;
    }
    return __byte_perm((p >> 1) ? w[1] : w[0], 0x64646464u, (p & 1) ? 0x4341u : 0x4240u);
}

struct Round {
    int task, rr;      // task index, round within the task
    int e, m0, n0, nn; // expert (E = the shared one), first row of the round, assignments
    bool live;         // false: no task, or rows past the matrix (nothing staged, nothing computed)
};

// Geometry of one kind: KIND 1 = gate/up (16 rows of each, K = H), KIND 2 = down (64 rows, K = I).
template <int KIND>
struct Kind {
    static constexpr int kRounds = KIND == 1 ? 4 : 1;   // rounds per task
    static constexpr int kRows = KIND == 1 ? 16 : 128;  // rows per matrix per round
    static constexpr int kMats = KIND == 1 ? 2 : 1;     // matrices per round
    static constexpr int kUnits = kMats * kRows / 16;   // 16-row MMA tiles per round
};

struct Smem {
    uint32_t row_stride, code, sc, stage, red, bar, total;
};

template <int KIND>
__host__ __device__ inline Smem smem_plan(int H, int Imax, int bits)
{
    using K = Kind<KIND>;
    const int kdim = KIND == 1 ? H : Imax;
    const int G = kdim / 64;
    Smem s{};
    s.row_stride = (uint32_t)(kdim * bits / 8 + kPad);
    s.code = 0;
    s.sc = s.row_stride * K::kMats * K::kRows;                      // [mat][s | b][row][G] bf16
    s.stage = (s.sc + (uint32_t)(K::kMats * 2 * K::kRows * G * 2) + 127) & ~127u;
    s.red = kStages * s.stage;                                      // [warp][unit][16][8] fp32
    s.bar = s.red + (uint32_t)(kWarps * K::kUnits * 16 * 8 * 4);
    s.total = s.bar + kStages * 8;
    return s;
}

template <int KIND, int BITS>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const tc::GroupedArgs P, const int4* __restrict__ tasks,
                                                         const int32_t* __restrict__ n_tasks_p, const __half* __restrict__ bop)
{
    using K = Kind<KIND>;
    extern __shared__ __align__(128) uint8_t sm[];
    const Smem pl = smem_plan<KIND>(P.H, P.Imax, BITS);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + pl.bar);
    float* red = reinterpret_cast<float*>(sm + pl.red);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    const int n_tasks = *n_tasks_p;
    const int my_tasks = blockIdx.x < n_tasks ? (n_tasks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int n_rounds = my_tasks * K::kRounds;
    const long long lim = P.timeout_cycles;

    auto round_of = [&](int j) {
        Round r{};
        r.task = blockIdx.x + (j / K::kRounds) * gridDim.x;
        r.rr = j % K::kRounds;
        const int4 t = tasks[r.task];
        r.e = t.x;
        r.n0 = t.z;
        r.nn = t.w;
        r.m0 = t.y + r.rr * K::kRows;
        const int rows = KIND == 1 ? (r.e < P.E ? P.I : P.Is) : P.H;
        r.live = r.m0 < rows;
        return r;
    };
    // the blob of expert e (the shared one for e == E); null when a routed expert has no slot
    auto blob_of = [&](int e) -> const uint8_t* {
        if (e >= P.E)
            return P.shared_blob;
        const int slot = P.table[e];
        return slot < 0 ? nullptr : P.arena + (uint64_t)slot * P.stride;
    };

    // warp 0 stages round j into stage j % kStages: every row of the round by its own bulk copy
    auto issue = [&](int j) {
        const Round r = round_of(j);
        uint64_t* b = bar + (j % kStages);
        uint8_t* st = sm + (j % kStages) * pl.stage;
        const uint8_t* blob = r.live ? blob_of(r.e) : nullptr;
        if (r.live && !blob && lane == 0)
            atomicCAS(P.status, 0, kStatusNotResident);
        const BlobGeo& geo = r.e < P.E ? P.geo : P.geo_s;
        const int kd = KIND == 1 ? P.H : geo.cols[2];
        const int G = kd / 64;
        const uint32_t rb = (uint32_t)(kd * BITS / 8);          // code bytes of a row
        // rows of the round inside the matrix: a down round may pass its end (H a multiple of 64,
        // rounds of 128); rows past it are neither copied nor used
        const int rows_total = KIND == 1 ? (r.e < P.E ? P.I : P.Is) : P.H;
        const int nr = r.live ? min(K::kRows, rows_total - r.m0) : 0;
        const uint32_t sstride = (uint32_t)(K::kRows * G * 2);  // shared-memory span of scales (or biases)
        const uint32_t sb = (uint32_t)(nr * G * 2);             // bytes of it copied
        const uint32_t total = blob ? K::kMats * (nr * rb + 2 * sb) : 0;
        if (lane == 0)
            mbar_expect(b, total);
        __syncwarp();
        if (!blob)
            return;
        for (int i = lane; i < K::kMats * (K::kRows + 2); i += 32) {
            const int mat = i / (K::kRows + 2), q = i % (K::kRows + 2);
            const int m = KIND == 1 ? mat : 2;                   // gate, up / down
            if (q < nr) {
                bulk_g2s(st + pl.code + (uint32_t)(mat * K::kRows + q) * pl.row_stride,
                         blob + geo.q_off[m] + (uint64_t)(r.m0 + q) * rb, rb, b);
            } else if (q >= K::kRows) {
                const uint64_t off = (q == K::kRows ? geo.s_off[m] : geo.b_off[m]) + (uint64_t)r.m0 * G * 2;
                bulk_g2s(st + pl.sc + (uint32_t)(mat * 2 + (q - K::kRows)) * sstride, blob + off, sb, b);
            }
        }
    };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s)
            mbar_init(bar + s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp == 0)
        for (int j = 0; j < n_rounds && j < kStages; ++j)
            issue(j);

    for (int j = 0; j < n_rounds; ++j) {
        const Round r = round_of(j);
        const bool ok = mbar_wait(bar + (j % kStages), (uint32_t)(j / kStages) & 1u, lim);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicCAS(P.status, 0, kStatusTimeout);
                for (int jj = j; jj < n_rounds && jj < j + kStages; ++jj)  // copies in flight land first
                    mbar_wait(bar + (jj % kStages), (uint32_t)(jj / kStages) & 1u, lim);
            }
            return;
        }
        const uint8_t* blob = r.live ? blob_of(r.e) : nullptr;
        if (blob) {
            const BlobGeo& geo = r.e < P.E ? P.geo : P.geo_s;
            const int kd = KIND == 1 ? P.H : geo.cols[2];
            const int G = kd / 64;
            const int ldb = KIND == 1 ? P.H : P.Imax;  // row length of the B operand rows
            const uint8_t* st = sm + (j % kStages) * pl.stage;
            const uint16_t* ssc = reinterpret_cast<const uint16_t*>(st + pl.sc);
            // passes of 8 assignments (the MMA's N); this thread feeds column g and holds rows g, g + 8
            for (int cg0 = 0; cg0 < r.nn; cg0 += 8) {
                float acc[K::kUnits][4];
#pragma unroll
                for (int u = 0; u < K::kUnits; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        acc[u][i] = 0.0f;
                const bool colv = cg0 + g < r.nn;
                const __half* brow = bop + (size_t)(r.n0 + (colv ? cg0 + g : 0)) * ldb + 2 * c;
                // B fragments of one quantisation group (its 4 slices), fetched one group ahead so
                // that their latency overlaps the current group's work
                uint32_t bc[8], bn[8];
                auto load_b = [&](int grp, uint32_t (&x)[8]) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const bool v = colv && grp < G;
                        const __half* q = brow + (4 * grp + i) * 16;
                        x[2 * i] = v ? *reinterpret_cast<const uint32_t*>(q) : 0u;
                        x[2 * i + 1] = v ? *reinterpret_cast<const uint32_t*>(q + 8) : 0u;
                    }
                };
                load_b(warp, bn);
                // warp w takes the quantisation groups w, w + 8, ...: one scale and bias per row and
                // group, four 16-element slices each
                for (int grp = warp; grp < G; grp += kWarps) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        bc[i] = bn[i];
                    load_b(grp + kWarps, bn);
                    // sum of the group's activations per column (an MMA with A = 1), the same in
                    // every row of the fragment: accx[i] belongs to column 2c + (i & 1)
                    float accx[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        mma16816(accx, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, bc[2 * i], bc[2 * i + 1]);
#pragma unroll
                    for (int u = 0; u < K::kUnits; ++u) {
                        const int mat = u / (K::kRows / 16), rt = u % (K::kRows / 16);
                        const int ra = rt * 16 + g, rb2 = ra + 8;  // rows within the matrix's round
                        const uint8_t* ca = st + pl.code + (uint32_t)(mat * K::kRows + ra) * pl.row_stride;
                        const uint8_t* cb = st + pl.code + (uint32_t)(mat * K::kRows + rb2) * pl.row_stride;
                        const uint16_t* sp = ssc + (size_t)(mat * 2) * K::kRows * G;
                        const uint16_t* bp = sp + (size_t)K::kRows * G;
                        const float sa = bf2f(sp[ra * G + grp]), ba = bf2f(bp[ra * G + grp]);
                        const float sb2 = bf2f(sp[rb2 * G + grp]), bb = bf2f(bp[rb2 * G + grp]);
                        float accq[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // sum of (1024 + q) x over the group
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int sl = 4 * grp + i;
                            uint32_t wa[4], wb[4];
                            if (BITS == 4) {
                                const uint2 va = *reinterpret_cast<const uint2*>(ca + sl * 8);
                                const uint2 vb = *reinterpret_cast<const uint2*>(cb + sl * 8);
                                wa[0] = va.x; wa[1] = va.y; wb[0] = vb.x; wb[1] = vb.y;
                            } else {
                                const uint4 va = *reinterpret_cast<const uint4*>(ca + sl * 16);
                                const uint4 vb = *reinterpret_cast<const uint4*>(cb + sl * 16);
                                wa[0] = va.x; wa[1] = va.y; wa[2] = va.z; wa[3] = va.w;
                                wb[0] = vb.x; wb[1] = vb.y; wb[2] = vb.z; wb[3] = vb.w;
                            }
                            // K block 0 of the slice = word 0 (int4) / words 0-1 (int8), block 1 the next;
                            // the codes enter as the exact fp16 values 1024 + q
                            const uint32_t a0 = code_pair<BITS>(wa, c);
                            const uint32_t a1 = code_pair<BITS>(wb, c);
                            const uint32_t a2 = code_pair<BITS>(wa + (BITS == 4 ? 1 : 2), c);
                            const uint32_t a3 = code_pair<BITS>(wb + (BITS == 4 ? 1 : 2), c);
                            mma16816(accq, a0, a1, a2, a3, bc[2 * i], bc[2 * i + 1]);
                        }
                        // w = s q + b over the group: s (sum (1024 + q) x - 1024 sum x) + b sum x
                        acc[u][0] += sa * (accq[0] - 1024.0f * accx[0]) + ba * accx[0];
                        acc[u][1] += sa * (accq[1] - 1024.0f * accx[1]) + ba * accx[1];
                        acc[u][2] += sb2 * (accq[2] - 1024.0f * accx[2]) + bb * accx[2];
                        acc[u][3] += sb2 * (accq[3] - 1024.0f * accx[3]) + bb * accx[3];
                    }
                }
                // the warps' partial sums -> shared memory [warp][unit][row 16][col 8]
#pragma unroll
                for (int u = 0; u < K::kUnits; ++u) {
                    float* rp = red + ((size_t)(warp * K::kUnits + u) * 16) * 8 + 2 * c;
                    rp[g * 8] = acc[u][0];
                    rp[g * 8 + 1] = acc[u][1];
                    rp[(g + 8) * 8] = acc[u][2];
                    rp[(g + 8) * 8 + 1] = acc[u][3];
                }
                __syncthreads();
                auto sum_warps = [&](int u, int row, int col) {
                    float v = 0.0f;
#pragma unroll
                    for (int w = 0; w < kWarps; ++w)
                        v += red[((size_t)(w * K::kUnits + u) * 16 + row) * 8 + col];
                    return v;
                };
                if (KIND == 1) {
                    // h = silu(gate) * up for the round's 16 rows and the pass's assignments
                    for (int i = tid; i < 16 * 8; i += kThreads) {
                        const int row = i / 8, col = i % 8;
                        if (cg0 + col < r.nn) {
                            const float gt = sum_warps(0, row, col), up = sum_warps(1, row, col);
                            const float h = __fdividef(gt, 1.f + __expf(-gt)) * up;
                            if (!(fabsf(h) <= 65504.f))
                                atomicCAS(P.status, 0, kStatusRange);
                            const int rowi = r.m0 + row;
                            const int pos = (rowi & ~7) | tc::kperm(rowi & 7, BITS);
                            P.hbuf[(size_t)(r.n0 + cg0 + col) * P.Imax + pos] = __float2half_rn(h);
                        }
                    }
                } else {
                    for (int i = tid; i < K::kRows * 8; i += kThreads) {
                        const int row = i / 8, col = i % 8;
                        const int o = r.m0 + row;
                        if (cg0 + col < r.nn && o < P.H) {
                            const int a = r.n0 + cg0 + col;
                            const float v = sum_warps(row >> 4, row & 15, col);
                            if (P.ypart)
                                P.ypart[(size_t)a * P.H + o] = P.aw[a] * v;
                            else
                                atomicAdd(P.y + (size_t)P.list[a] * P.H + o, P.aw[a] * v);
                        }
                    }
                }
                __syncthreads();  // the reduction buffer is free again
            }
        }
        __syncthreads();  // every warp is done with the stage
        if (warp == 0 && j + kStages < n_rounds)
            issue(j + kStages);
    }
}

template <int KIND, int BITS>
void launch_one(const tc::GroupedArgs& A, const int4* tasks, const int32_t* n_tasks, int grid, cudaStream_t st)
{
    const Smem pl = smem_plan<KIND>(A.H, A.Imax, BITS);
    static std::atomic<int> done[kMaxDevices];
    raise_smem_limit(gemv_kernel<KIND, BITS>, (int)pl.total, done);
    const __half* bop = KIND == 1 ? A.us : A.hbuf;
    gemv_kernel<KIND, BITS><<<grid, kThreads, pl.total, st>>>(A, tasks, n_tasks, bop);
}

}  // namespace

size_t smem_bytes(int H, int Imax, int bits)
{
    const size_t a = smem_plan<1>(H, Imax, bits).total, b = smem_plan<2>(H, Imax, bits).total;
    return a > b ? a : b;
}

bool geometry_ok(const BlobGeo& g)
{
    for (int m = 0; m < 3; ++m)
        if ((g.q_off[m] | g.s_off[m] | g.b_off[m] | (uint64_t)g.row_bytes[m]) & 15u)
            return false;
    return true;
}

void launch(int kind, const tc::GroupedArgs& A, const int4* tasks, const int32_t* n_tasks, int grid, cudaStream_t st)
{
    if (kind == 1)
        A.bits == 4 ? launch_one<1, 4>(A, tasks, n_tasks, grid, st) : launch_one<1, 8>(A, tasks, n_tasks, grid, st);
    else
        A.bits == 4 ? launch_one<2, 4>(A, tasks, n_tasks, grid, st) : launch_one<2, 8>(A, tasks, n_tasks, grid, st);
}

}  // namespace gv
}  // namespace moe
