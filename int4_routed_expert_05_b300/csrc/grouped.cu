// grouped.cu -- the GEMMs of the batched MoE layer on the fifth-generation tensor cores (sm_103a).
//
// The layer is the one of the decode kernel (cheshm.ai item "Swiftlet fits an 80B-level Qwen giant
// into Mac": router, top-k of E experts, SwiGLU experts with MLX-style group-64 int4/int8 codes and
// per-group scale and bias, weighted combine, sigmoid-gated shared expert), here for T tokens at
// once, where the expert matrices are real GEMMs over the tokens routed to each expert.
//
// Both kernels are persistent (one CTA per SM) and warp-specialised around one MMA-issuing thread;
// tcgen05.mma (M = 128, N = tokens rounded up to 16, K = 16, fp32 accumulate) accumulates in tensor
// memory (two accumulators, so the epilogue of one task overlaps the main loop of the next):
//   * router GEMM: A = router rows (bf16) and B = token rows (bf16), both brought in by TMA with
//     the 128-byte swizzle as K-major shared-memory tiles, so a slice goes global -> shared ->
//     tensor core untouched;
//   * expert GEMMs: TMA stages the packed codes (64 bytes per row and slice, 64-byte swizzled);
//     eight dequantising warps turn them into fp16 weights w = s * q + b (one rounding; s is
//     checked to be a normal fp16 value and w to stay finite, else MOE_E_RANGE) and write them straight into tensor memory
//     (tcgen05.st; the MMA reads A from there); TMA brings the expert's token rows (input rows in
//     assignment order, or h rows) into 128-byte swizzled B tiles in shared memory; four epilogue
//     warps read the accumulators with tcgen05.ld and apply SwiGLU (gate/up: h to a per-assignment
//     buffer) or the combine weight (down: fp32 reductions into y, or per-assignment rows that a
//     fixed-order combine sums).
//   Operand tiles the MMA reads come from TMA or from tcgen05.st (rows written by cp.async and
//   released after cp.async.wait_group + fence.proxy.async were measured to reach tcgen05.mma stale
//   at times, and are not used).
// Every wait is bounded: on expiry the kernel records MOE timeout status, drains its own copies and
// frees its tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attr.h"
#include "grouped.h"
#include "layout.h"

namespace moe {
namespace tc {

namespace {

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ---- mbarriers ----
__device__ __forceinline__ void bar_init(uint64_t* m, int n)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(m)), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* m)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(m)) : "memory");
}
// One arrival per warp: the warp's lanes are ordered before lane 0's release by __syncwarp.
__device__ __forceinline__ void bar_arrive_warp(uint64_t* m)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        bar_arrive(m);
}
__device__ __forceinline__ void bar_expect(uint64_t* m, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(m)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool bar_try(uint64_t* m, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(su32(m)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Shared block state: the abort flag every wait checks, the tensor-memory base address.
struct Ctl {
    volatile int abort;
    uint32_t tmem;
};

// Bounded wait on phase `parity` of m. False on timeout or when another role gave up. The test of
// an already completed phase stays inline; only the polling loop is a call.
__device__ __noinline__ bool bar_wait_slow(uint64_t* m, uint32_t parity, Ctl* ctl, int* status, long long limit)
{
    const long long t0 = clock64();
    for (int it = 1;; ++it) {
        if (bar_try(m, parity))
            return true;
        if ((it & 255) == 0) {
            if (ctl->abort)
                return false;
            if (clock64() - t0 > limit) {
                ctl->abort = 1;
                atomicOr(status, kStatusTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool bar_wait(uint64_t* m, uint32_t parity, Ctl* ctl, int* status, long long limit)
{
    return bar_try(m, parity) || bar_wait_slow(m, parity, ctl, status, limit);
}

// ---- copies ----
__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* m)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            su32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(su32(m))
        : "memory");
}
__device__ __forceinline__ void tma3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* m)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(su32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(su32(m))
        : "memory");
}
__device__ __forceinline__ void bulk(void* dst, const void* src, uint32_t bytes, uint64_t* m)
{
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(su32(dst)),
                 "l"(src), "r"(bytes), "r"(su32(m))
                 : "memory");
}

// ---- tcgen05 ----
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand tile, 128-byte swizzle, 8-row groups 1024 bytes
// apart (start address and offsets in 16-byte units; bits 46-48 hold the fixed value 1).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc(int n, bool bf16)
{
    const uint32_t f = bf16 ? 1u : 0u;
    return (1u << 4) | (f << 7) | (f << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc)
{
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}
// A operand from tensor memory (lane = row, 32-bit columns holding fp16 pairs along K)
__device__ __forceinline__ void mma_ta(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc)
{
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(id), "r"(acc)
        : "memory");
}

// 16 / 32 consecutive 32-bit columns of this thread's TMEM lane from registers
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mma_commit(uint64_t* m)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(m))
                 : "memory");
}

// 16 consecutive fp32 columns of this thread's accumulator row (lane = row)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

// 4 consecutive fp32 columns of this thread's accumulator row
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4])
{
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 4; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols = kTmemCols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(slot)), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_free(uint32_t base, uint32_t cols = kTmemCols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// 8 int4 codes of one 32-bit word -> 4 fp16 pairs w = s * q + b, pair j = (code j, code j + 4):
// (word >> 4j) & 0x000F000F | 0x6400_6400 is the fp16 pair (1024 + q_j, 1024 + q_{j+4}); taking
// 1024 back off is exact, and the fma rounds s * q + b once.
__device__ __forceinline__ uint4 deq_int4(uint32_t w, __half2 s, __half2 b)
{
    const __half2 k1024 = u2h(0x64006400u);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t x;
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(x) : "r"(w >> (4 * j)), "r"(0x000F000Fu), "r"(0x64006400u));
        o[j] = h2u(__hfma2(__hsub2(u2h(x), k1024), s, b));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// 8 int8 codes of two 32-bit words -> 4 fp16 pairs, pair order (0,2), (1,3) within each word.
__device__ __forceinline__ uint4 deq_int8(uint32_t w0, uint32_t w1, __half2 s, __half2 b)
{
    const __half2 k1024 = u2h(0x64006400u);
    uint32_t o[4];
    const uint32_t w[2] = {w0, w1};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t x = __byte_perm(w[j >> 1], 0x64646464u, (j & 1) ? 0x4341u : 0x4240u);
        o[j] = h2u(__hfma2(__hsub2(u2h(x), k1024), s, b));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint16_t pick16(const uint4& v, int i)
{
    const uint32_t w = (i & 4) ? ((i & 2) ? v.w : v.z) : ((i & 2) ? v.y : v.x);
    return (uint16_t)((i & 1) ? (w >> 16) : (w & 0xFFFFu));
}

struct TaskX {
    int e, m0, n0, nn, nk, nh, shared, slot;  // nk slices of 128 K; nh = 64-element halves in all
    const uint8_t* blob;
};

__device__ __forceinline__ TaskX decode_task(const GroupedArgs& P, int kind, int4 t, int sub = 1)
{
    TaskX x;
    x.e = t.x;
    x.m0 = t.y;
    x.n0 = t.z;
    x.nn = t.w;
    x.shared = x.e == P.E;
    x.slot = 0;
    if (x.shared) {
        x.blob = P.shared_blob;
    } else {
        int s = P.table[x.e];
        if (s < 0) {
            atomicOr(P.status, kStatusNotResident);
            s = 0;
        }
        x.slot = s;
        x.blob = P.arena + (uint64_t)s * P.stride;
    }
    const BlobGeo& g = x.shared ? P.geo_s : P.geo;
    x.nh = (kind == 1 ? P.H : g.cols[2]) / kKS;
    x.nk = (x.nh + sub - 1) / sub;
    return x;
}

__device__ __forceinline__ int n_mma(int nn) { return (nn + 15) & ~15; }

}  // namespace

// ------------------------------------------------------------------------------------------------
// Router GEMM: logits[t][e] = sum_h Wr[e][h] u[t][h], tiles of 128 experts x 128 tokens.
// ------------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreadsR, 1) router_kernel(const __grid_constant__ GroupedArgs P)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sa = sm;                                   // kStagesR A tiles
    uint8_t* sbuf = sm + kStagesR * kTileBytes;         // kStagesR B tiles
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + 2 * kStagesR * kTileBytes);
    uint64_t* full = bars;                 // [kStagesR]
    uint64_t* empty = bars + kStagesR;     // [kStagesR]
    uint64_t* acc_full = bars + 2 * kStagesR;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* fin = acc_empty + 2;
    Ctl* ctl = reinterpret_cast<Ctl*>(fin + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = (P.E + 127) / 128, n_tasks = mt * ((P.T + kNT - 1) / kNT);
    const int nk = P.H / kKS;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStagesR; ++i) {
            bar_init(full + i, 1);
            bar_init(empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            bar_init(acc_full + i, 1);
            bar_init(acc_empty + i, 4);
        }
        bar_init(fin, 1);
        ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 5)
        tmem_alloc(&ctl->tmem);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;
    const long long lim = P.timeout_cycles;

    if (warp == 4) {
        if (lane == 0) {  // TMA producer
            asm volatile("prefetch.tensormap [%0];" ::"l"(&P.map_wr) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&P.map_u) : "memory");
            uint32_t it = 0;
            for (int ti = blockIdx.x; ti < n_tasks; ti += gridDim.x) {
                const int m0 = (ti % mt) * 128, n0 = (ti / mt) * kNT;
                for (int g = 0; g < nk; ++g, ++it) {
                    const int s = it % kStagesR;
                    if (!bar_wait(empty + s, ((it / kStagesR) & 1) ^ 1, ctl, P.status, lim))
                        goto tma_done;
                    bar_expect(full + s, 2 * kTileBytes);
                    tma2d(sa + s * kTileBytes, &P.map_wr, g * kKS, m0, full + s);
                    tma2d(sbuf + s * kTileBytes, &P.map_u, g * kKS, n0, full + s);
                }
            }
        tma_done:
            // every issued copy has landed before the block can exit
            for (uint32_t i = it > (uint32_t)kStagesR ? it - kStagesR : 0; i < it; ++i)
                bar_wait(full + i % kStagesR, (i / kStagesR) & 1, ctl, P.status, lim);
        }
    } else if (warp == 5) {
        if (lane == 0) {  // MMA issuer
            uint32_t it = 0, j = 0;
            for (int ti = blockIdx.x; ti < n_tasks; ti += gridDim.x, ++j) {
                const int n0 = (ti / mt) * kNT;
                const int nn = min(kNT, P.T - n0);
                const uint32_t id = idesc(n_mma(nn), true);
                const int ab = j & 1;
                if (!bar_wait(acc_empty + ab, ((j >> 1) & 1) ^ 1, ctl, P.status, lim))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + ab * kNT;
                bool ok = true;
                for (int g = 0; g < nk; ++g, ++it) {
                    const int s = it % kStagesR;
                    if (!bar_wait(full + s, (it / kStagesR) & 1, ctl, P.status, lim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a = sdesc(su32(sa + s * kTileBytes)), b = sdesc(su32(sbuf + s * kTileBytes));
#pragma unroll
                    for (int kk = 0; kk < kKS / 16; ++kk)
                        mma(d, a + 2 * kk, b + 2 * kk, id, (g | kk) != 0);
                    mma_commit(empty + s);
                }
                if (!ok)
                    break;
                mma_commit(acc_full + ab);
            }
            mma_commit(fin);
            bar_wait(fin, 0, ctl, P.status, lim);
        }
    } else {  // epilogue warps 0-3: TMEM lanes 32 * warp ..
        const int r = warp * 32 + lane;
        uint32_t j = 0;
        for (int ti = blockIdx.x; ti < n_tasks; ti += gridDim.x, ++j) {
            const int m0 = (ti % mt) * 128, n0 = (ti / mt) * kNT;
            const int nn = min(kNT, P.T - n0);
            const int ab = j & 1;
            bar_wait(acc_full + ab, (j >> 1) & 1, ctl, P.status, lim);  // no early exit (warp-collective loads)
            tc_fence_after();
            const int row = m0 + r;
            for (int c0 = 0; c0 < n_mma(nn); c0 += 16) {
                float v[16];
                tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + ab * kNT + c0, v);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (row < P.E && c0 + i < nn)
                        P.logits[(size_t)(n0 + c0 + i) * P.E + row] = v[i];
            }
            tc_fence_before();
            bar_arrive_warp(acc_empty + ab);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_free(tmem);
    }
}

// ------------------------------------------------------------------------------------------------
// Expert GEMMs. kind 1: gate/up tiles (64 gate rows + the same 64 up rows) against the expert's
// tokens, SwiGLU epilogue -> hbuf. kind 2: down tiles (128 rows) against the expert's h rows,
// epilogue y[token] += weight * acc.
// ------------------------------------------------------------------------------------------------
template <int kKind, int kBits>
__global__ void __launch_bounds__(kThreadsX, 1) expert_kernel(const __grid_constant__ GroupedArgs P)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const XPlan pl = xplan(P.H, P.Imax, kBits);
    uint8_t* sbt = sm + pl.b;
    uint8_t* scode = sm + pl.code;
    uint8_t* ssc = sm + pl.sc;
    float* xch = reinterpret_cast<float*>(sm + pl.xch);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + pl.bar);
    const int NC = (int)pl.n_code;
    uint64_t* full_a = bars;
    uint64_t* full_b = full_a;  // the B-operand TMA's arrive.expect_tx joins the producers' arrivals
    uint64_t* empty = bars + kTiles;
    uint64_t* code_full = bars + 2 * kTiles;
    uint64_t* code_empty = code_full + 8;
    uint64_t* sc_full = code_empty + 8;
    uint64_t* sc_empty = sc_full + 2;
    uint64_t* acc_full = sc_empty + 2;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* fin = acc_empty + 2;
    Ctl* ctl = reinterpret_cast<Ctl*>(bars + 64);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tasks = *P.n_tasks;
    const long long lim = P.timeout_cycles;
    constexpr int kSub = slice_sub(kBits);         // sub-tiles per slice
    constexpr int kStages = kTiles / kSub;         // slices in flight
    // tensor memory: two accumulators (columns 0..255), then the A stages (kSub x 32 columns each)
    constexpr uint32_t kAccCols = 2 * kNT, kAStageCols = kSub * (kKS / 2), kTmemColsX = 512;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            bar_init(full_a + i, 9);  // 8 dequantising warps + the B-operand TMA
            bar_init(empty + i, 1);
        }
        for (int i = 0; i < NC; ++i) {
            bar_init(code_full + i, 1);
            bar_init(code_empty + i, 8);
        }
        for (int i = 0; i < 2; ++i) {
            bar_init(sc_full + i, 1);
            bar_init(sc_empty + i, 8);
            bar_init(acc_full + i, 1);
            bar_init(acc_empty + i, 4);
        }
        bar_init(fin, 1);
        ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 13)
        tmem_alloc(&ctl->tmem, kTmemColsX);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem;

    if (warp < 8) {
        // ---- dequantising producers: thread (hk, r) owns 32 code bytes of row r in each slice
        // (int4: group hk of two; int8: half hk of one): two warps per SMSP share each slice ----
        const int r = threadIdx.x & 127, hk = threadIdx.x >> 7;
        uint32_t it = 0, j = 0;
        for (int ti = blockIdx.x; ti < n_tasks; ti += gridDim.x, ++j) {
            const TaskX t = decode_task(P, kKind, P.tasks[ti], kSub);
            const BlobGeo& geo = t.shared ? P.geo_s : P.geo;
            const int G = kKind == 1 ? geo.groups[0] : geo.groups[2];
            const int sb = j & 1;
            // waits of the warp-collective roles never leave the loop early: after a timeout they
            // return at once, so every lane still reaches every __syncwarp and named barrier
            bar_wait(sc_full + sb, (j >> 1) & 1, ctl, P.status, lim);
            // row r's scales and biases in the staged block: gate/up [gs 64][gb 64][us 64][ub 64] x G,
            // down [s 128][b 128] x G
            const uint16_t* scb = reinterpret_cast<const uint16_t*>(ssc + sb * pl.sc_bytes);
            const uint16_t* srow;
            const uint16_t* brow;
            if (kKind == 1) {
                const int half = r >> 6, rr = r & 63;
                srow = scb + (size_t)(2 * half) * 64 * G + rr * G;
                brow = srow + 64 * G;
            } else {
                srow = scb + (size_t)r * G;
                brow = scb + (size_t)128 * G + r * G;
            }
            const bool vec = (G & 7) == 0;
            uint4 sv = make_uint4(0, 0, 0, 0), bv = sv;
            int blk = -1;
            for (int g = 0; g < t.nk; ++g, ++it) {
                const int c = it % NC;
                // int4: this thread's quantisation group gg of the slice's two (128 elements); int8:
                // half hk of the slice's one group
                const int gg = kSub == 2 ? 2 * g + hk : g;
                const bool live = gg < t.nh;   // the last int4 slice may hold one group only
                bar_wait(code_full + c, (it / NC) & 1, ctl, P.status, lim);
                // the stage holds 64-byte rows, 64-byte swizzled: chunk cc of row r at cc ^ ((r >> 1) & 3)
                const uint8_t* crow = scode + c * pl.code_stage + r * kCodeRow;
                const int xr = (r >> 1) & 3;
                const uint4 q0 = *reinterpret_cast<const uint4*>(crow + (((2 * hk) ^ xr) << 4));
                const uint4 q1 = *reinterpret_cast<const uint4*>(crow + (((2 * hk + 1) ^ xr) << 4));
                bar_arrive_warp(code_empty + c);
                uint16_t s16 = 0, b16 = 0;
                if (live) {
                    if (vec) {
                        if ((gg >> 3) != blk) {
                            blk = gg >> 3;
                            sv = *reinterpret_cast<const uint4*>(srow + (gg & ~7));
                            bv = *reinterpret_cast<const uint4*>(brow + (gg & ~7));
                        }
                        s16 = pick16(sv, gg & 7);
                        b16 = pick16(bv, gg & 7);
                    } else {
                        s16 = srow[gg];
                        b16 = brow[gg];
                    }
                }
                const float sf = bf2f(s16), bf = bf2f(b16);
                const __half2 s2 = __half2half2(__float2half_rn(sf));
                const __half2 b2 = __half2half2(__float2half_rn(bf));
                // the fp16 dequantisation keeps s's relative precision and stays finite only when s
                // is zero or a normal fp16 value and |s| qmax + |b| is within fp16's range (b in
                // fp16's subnormal range is off by at most 2^-25, unnoticeable in a weight)
                if (live && ((sf != 0.f && !(fabsf(sf) >= 6.103515625e-05f)) ||
                             !(fabsf(sf) * (kBits == 4 ? 15.f : 255.f) + fabsf(bf) <= 65504.f)))
                    atomicCAS(P.status, 0, kStatusRange);
                const int st = it % kStages;
                bar_wait(empty + st, ((it / kStages) & 1) ^ 1, ctl, P.status, lim);
                // A row segment -> tensor memory (lane r): 32-bit columns of fp16 pairs in K order
                tc_fence_after();
                const uint32_t acol = tmem + ((uint32_t)((r >> 5) * 32) << 16) + kAccCols + st * kAStageCols;
                const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                if (kBits == 4) {  // 64 codes -> 32 columns of sub-tile hk
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t v[16];
#pragma unroll
                        for (int ch = 0; ch < 4; ++ch) {
                            const uint4 o = deq_int4(w[4 * half + ch], s2, b2);
                            v[4 * ch] = o.x;
                            v[4 * ch + 1] = o.y;
                            v[4 * ch + 2] = o.z;
                            v[4 * ch + 3] = o.w;
                        }
                        if (live)
                            tmem_st16(acol + hk * 32 + half * 16, v);
                    }
                } else {           // 32 codes -> columns 16 hk .. 16 hk + 15 of the slice
                    uint32_t v[16];
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        const uint4 o = deq_int8(w[2 * ch], w[2 * ch + 1], s2, b2);
                        v[4 * ch] = o.x;
                        v[4 * ch + 1] = o.y;
                        v[4 * ch + 2] = o.z;
                        v[4 * ch + 3] = o.w;
                    }
                    tmem_st16(acol + hk * 16, v);
                }
                tmem_st_wait();
                tc_fence_before();
                bar_arrive_warp(full_a + st);
            }
            bar_arrive_warp(sc_empty + sb);
        }
    } else if (warp < 12) {
        // ---- epilogue: warp 8 + q reads TMEM lanes 32q .. 32q + 31 (tile row = lane) ----
        const int q = warp - 8, r = q * 32 + lane;
        uint32_t j = 0;
        for (int ti = blockIdx.x; ti < n_tasks; ti += gridDim.x, ++j) {
            const TaskX t = decode_task(P, kKind, P.tasks[ti], kSub);
            const int ab = j & 1;
            bar_wait(acc_full + ab, (j >> 1) & 1, ctl, P.status, lim);  // no early exit (named barriers below)
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + ab * kNT;
            const int N = n_mma(t.nn);
            if (kKind == 1) {
                // rows 64..127 hold the up projections of rows 0..63: handed over in shared memory,
                // 16 columns at a time
                const int row = t.m0 + (r & 63);
                const int pos = (row & ~7) | kperm(row & 7, kBits);
                for (int c0 = 0; c0 < N; c0 += 16) {
                    if (q >= 2) {
#pragma unroll 1
                        for (int c = 0; c < 16; c += 4) {
                            float v[4];
                            tmem_ld4(tbase + c0 + c, v);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                xch[(r - 64) * 17 + c + i] = v[i];
                        }
                    }
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    if (q < 2) {
#pragma unroll 1
                        for (int c = 0; c < 16; c += 4) {
                            float v[4];
                            tmem_ld4(tbase + c0 + c, v);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int n = c0 + c + i;
                                if (n < t.nn) {
                                    const float gt = v[i], up = xch[r * 17 + c + i];
                                    const float h = __fdividef(gt, 1.f + __expf(-gt)) * up;
                                    if (!(fabsf(h) <= 65504.f))
                                        atomicCAS(P.status, 0, kStatusRange);
                                    P.hbuf[(size_t)(t.n0 + n) * P.Imax + pos] = __float2half_rn(h);
                                }
                            }
                        }
                    }
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                }
            } else {
                const int o = t.m0 + r;
#pragma unroll 1
                for (int c0 = 0; c0 < N; c0 += 4) {
                    float v[4];
                    tmem_ld4(tbase + c0, v);
                    if (o < P.H) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int a = t.n0 + c0 + i;
                            if (c0 + i < t.nn) {
                                if (P.ypart)
                                    P.ypart[(size_t)a * P.H + o] = P.aw[a] * v[i];
                                else
                                    atomicAdd(P.y + (size_t)P.list[a] * P.H + o, P.aw[a] * v[i]);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            bar_arrive_warp(acc_empty + ab);
        }
    } else if (warp == 12) {
        if (lane == 0) {
            // ---- TMA producer: per task the scale/bias block, per slice the code tile ----
            for (int m = 0; m < 3; ++m) {
                asm volatile("prefetch.tensormap [%0];" ::"l"(&P.map_q[0][m]) : "memory");
                asm volatile("prefetch.tensormap [%0];" ::"l"(&P.map_q[1][m]) : "memory");
            }
            uint32_t it = 0, j = 0;
            for (int ti = blockIdx.x; ti < n_tasks; ti += gridDim.x, ++j) {
                const TaskX t = decode_task(P, kKind, P.tasks[ti], kSub);
                const BlobGeo& geo = t.shared ? P.geo_s : P.geo;
                const int sb = j & 1;
                if (!bar_wait(sc_empty + sb, ((j >> 1) & 1) ^ 1, ctl, P.status, lim))
                    goto tma_done;
                {
                    uint8_t* dst = ssc + sb * pl.sc_bytes;
                    if (kKind == 1) {
                        const int G = geo.groups[0];
                        const uint32_t nb = 64u * G * 2;
                        bar_expect(sc_full + sb, 4 * nb);
                        bulk(dst, t.blob + geo.s_off[0] + (size_t)t.m0 * G * 2, nb, sc_full + sb);
                        bulk(dst + nb, t.blob + geo.b_off[0] + (size_t)t.m0 * G * 2, nb, sc_full + sb);
                        bulk(dst + 2 * nb, t.blob + geo.s_off[1] + (size_t)t.m0 * G * 2, nb, sc_full + sb);
                        bulk(dst + 3 * nb, t.blob + geo.b_off[1] + (size_t)t.m0 * G * 2, nb, sc_full + sb);
                    } else {
                        const int G = geo.groups[2];
                        const int rows = min(128, P.H - t.m0);
                        const uint32_t nb = (uint32_t)rows * G * 2;
                        bar_expect(sc_full + sb, 2 * nb);
                        bulk(dst, t.blob + geo.s_off[2] + (size_t)t.m0 * G * 2, nb, sc_full + sb);
                        bulk(dst + 128u * G * 2, t.blob + geo.b_off[2] + (size_t)t.m0 * G * 2, nb, sc_full + sb);
                    }
                }
                for (int g = 0; g < t.nk; ++g, ++it) {
                    const int c = it % NC;
                    if (!bar_wait(code_empty + c, ((it / NC) & 1) ^ 1, ctl, P.status, lim))
                        goto tma_done;
                    uint8_t* dst = scode + c * pl.code_stage;
                    bar_expect(code_full + c, pl.code_stage);
                    const int x = g * kCodeRow;
                    if (kKind == 1) {
                        tma3d(dst, &P.map_q[t.shared][0], x, t.m0, t.slot, code_full + c);
                        tma3d(dst + 64 * kCodeRow, &P.map_q[t.shared][1], x, t.m0, t.slot, code_full + c);
                    } else {
                        tma3d(dst, &P.map_q[t.shared][2], x, t.m0, t.slot, code_full + c);
                    }
                }
            }
        tma_done:
            for (uint32_t i = it > (uint32_t)NC ? it - NC : 0; i < it; ++i)
                bar_wait(code_full + i % NC, (i / NC) & 1, ctl, P.status, lim);
            for (uint32_t i = j > 2 ? j - 2 : 0; i < j; ++i)
                bar_wait(sc_full + (i & 1), (i >> 1) & 1, ctl, P.status, lim);
        }
    } else if (warp == 14) {
        if (lane == 0) {
            // ---- B operand: the task's token rows of this K slice, boxes of 16 rows ----
            const CUtensorMap* mb = &P.map_b[kKind - 1];
            asm volatile("prefetch.tensormap [%0];" ::"l"(mb) : "memory");
            uint32_t it = 0;
            for (int ti = blockIdx.x; ti < n_tasks; ti += gridDim.x) {
                const TaskX t = decode_task(P, kKind, P.tasks[ti], kSub);
                const int nb = n_mma(t.nn) / kBRows;
                bool ok = true;
                for (int g = 0; g < t.nk; ++g, ++it) {
                    const int st = it % kStages;
                    if (!bar_wait(empty + st, ((it / kStages) & 1) ^ 1, ctl, P.status, lim)) {
                        ok = false;
                        break;
                    }
                    const int halves = min(kSub, t.nh - kSub * g);
                    bar_expect(full_b + st, (uint32_t)(halves * nb) * kBRows * 128);
                    for (int h = 0; h < halves; ++h)
                        for (int q = 0; q < nb; ++q)
                            tma2d(sbt + (st * kSub + h) * kTileBytes + q * kBRows * 128, mb, (kSub * g + h) * kKS,
                                  t.n0 + q * kBRows, full_b + st);
                }
                if (!ok)
                    break;
            }
            // every issued copy has landed before the block can exit
            for (uint32_t i = it > (uint32_t)kStages ? it - kStages : 0; i < it; ++i)
                bar_wait(full_b + i % kStages, (i / kStages) & 1, ctl, P.status, lim);
        }
    } else {
        // ---- MMA issuer (warp 13): the whole warp walks the loop (converged); lane 0 issues ----
        const bool issuer = lane == 0;
        uint32_t it = 0, j = 0;
        bool ok = true;
        for (int ti = blockIdx.x; ti < n_tasks && ok; ti += gridDim.x, ++j) {
            const TaskX t = decode_task(P, kKind, P.tasks[ti], kSub);
            const uint32_t id = idesc(n_mma(t.nn), false);
            const int ab = j & 1;
            ok = __all_sync(0xffffffffu, bar_wait(acc_empty + ab, ((j >> 1) & 1) ^ 1, ctl, P.status, lim));
            if (!ok)
                break;
            tc_fence_after();
            const uint32_t d = tmem + ab * kNT;
            for (int g = 0; g < t.nk; ++g, ++it) {
                const int st = it % kStages;
                ok = __all_sync(0xffffffffu, bar_wait(full_a + st, (it / kStages) & 1, ctl, P.status, lim));
                if (!ok)
                    break;
                tc_fence_after();
                if (issuer) {
                    const int halves = min(kSub, t.nh - kSub * g);
                    for (int h = 0; h < halves; ++h) {
                        const uint32_t a = tmem + kAccCols + st * kAStageCols + h * (kKS / 2);
                        const uint64_t b = sdesc(su32(sbt + (st * kSub + h) * kTileBytes));
#pragma unroll
                        for (int kk = 0; kk < kKS / 16; ++kk)
                            mma_ta(d, a + kk * 8, b + 2 * kk, id, (g | h | kk) != 0);
                    }
                    mma_commit(empty + st);
                }
                __syncwarp();
            }
            if (ok && issuer)
                mma_commit(acc_full + ab);
            __syncwarp();
        }
        if (issuer) {
            mma_commit(fin);
            bar_wait(fin, 0, ctl, P.status, lim);
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        tc_fence_after();
        tmem_free(tmem, kTmemColsX);
    }
}

size_t router_smem_bytes() { return 2 * kStagesR * kTileBytes + 64 * 8 + 1024; }

size_t expert_smem_bytes(int H, int Imax, int bits) { return xplan(H, Imax, bits).total + 1024; }

void launch_router_gemm(const GroupedArgs& A, int grid, cudaStream_t st)
{
    static std::atomic<int> done[kMaxDevices];
    const size_t smem = router_smem_bytes();
    raise_smem_limit(router_kernel, (int)smem, done);
    router_kernel<<<grid, kThreadsR, smem, st>>>(A);
}

void launch_expert_gemm(int kind, const GroupedArgs& A, const int4* tasks, const int32_t* n_tasks, int grid,
                        cudaStream_t st)
{
    static std::atomic<int> done[4][kMaxDevices];
    GroupedArgs P = A;
    P.tasks = tasks;
    P.n_tasks = n_tasks;
    const size_t smem = expert_smem_bytes(A.H, A.Imax, A.bits);
    void (*k)(const GroupedArgs) = kind == 1 ? (A.bits == 4 ? expert_kernel<1, 4> : expert_kernel<1, 8>)
                                             : (A.bits == 4 ? expert_kernel<2, 4> : expert_kernel<2, 8>);
    const int ki = (kind - 1) * 2 + (A.bits == 4 ? 0 : 1);
    raise_smem_limit(k, 227 * 1024, done[ki]);
    k<<<grid, kThreadsX, smem, st>>>(P);
}

}  // namespace tc
}  // namespace moe
