// decode.cu -- fused batch-1 decode kernel of the routed-expert MoE FFN layer (sm_103a).
//
// What it computes (per token and layer; cheshm.ai item "Swiftlet fits an 80B-level Qwen giant
// into Mac", scheduling and closing paragraphs; alphalab.site "Swiftlet 實測資料解讀", section on
// the 35B router-normalisation fix):
//   u = input (or bf16(x / rms(x)) in a pre-norm stack)
//   logits = Wr u (+ bias);  idx = top-k (ties -> lower index);  w = softmax renormalised over idx
//   y = sum_j w_j Wd_j (silu(Wg_j u) .* (Wu_j u)) + sigmoid(w_sg . u) * S(u)
// with expert idx_j's blob at arena + slot * stride (paotong.dev commentary on Swiftlet: one
// fixed-stride blob per expert, one read per expert).
//
// Design: one cooperative launch covers every layer and token of a call, one 512-thread block per
// SM. Every step executes the whole body, so the body has to stay small enough for the SM's
// instruction caches: only the inner chunk loops of the MMA blocks are unrolled. Per step (token, layer) a block
//   1. holds the layer input x in shared memory and forms u;
//   2. computes its rows of the router (rows prefetched during the previous step) and publishes
//      them as epoch-tagged (epoch, value) pairs; computes its rows of the shared expert's gate/up
//      and publishes h_shared the same way; queues the next step's router and shared rows;
//   3. polls the logits until every pair carries this step's epoch, takes the top-k itself;
//   4. joins the group of blocks that serves one routed expert (rank j): fetches its share of the
//      expert's gate/up rows and down rows as TMA boxes into a ring of 16 slots (one per warp; a
//      warp refills its slot with its next box as soon as it has consumed it), and in the meantime
//      finishes the shared expert's down rows;
//   5. turns its gate/up rows into h_j, publishes them to its group, collects the group's h_j
//      while the down boxes land, and computes its down rows of y_j;
//   6. adds w_j y_j (and gamma y_shared) into a fixed-point accumulator with integer atomics, so
//      the sum is exact and independent of the order in which blocks arrive;
//   7. waits at one grid barrier and reads the complete layer output back.
// int4 codes become exact bf16 integers in registers (mask + bf16x2 FMA) and meet the activations
// on the tensor cores (mma.m16n8k16, fp32 accumulate), one 64-element quantisation group per chunk;
// the affine dequantisation is applied per chunk as s * (sum q u) + b * (sum u). Every sum runs in
// a fixed order, so the result depends neither on the grid size nor on pool placement.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "layout.h"

namespace moe {
namespace {

// ------------------------------------------------------------------------------------------
// small device helpers
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint16_t f2bf(float v)
{
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t*>(&h);
}

// Order-preserving map of a float onto uint32 (larger float -> larger key; finite keys > 0).
__device__ __forceinline__ uint32_t ord_key(float f)
{
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Position of element n of an expanded activation vector inside its permuted 16-element block
// (register order 0,4,1,5,2,6,3,7, 8,12,9,13,10,14,11,15 of the B fragments).
__device__ __forceinline__ int pslot(int n)
{
    const int e = n & 15;
    return (n & ~15) | (e & 8) | ((e & 3) << 1) | ((e >> 2) & 1);
}

// SM cycle counter: cheap to read, so waits check their limit on it. A limit of t ns is taken as
// 2 t cycles (about t ns at the 2.03 GHz maximum SM clock, longer at lower clocks).
__device__ __forceinline__ long long cycles() { return clock64(); }
__device__ __forceinline__ long long limit_cycles(const StepParams& P) { return (long long)(2 * P.timeout_ns); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// thread / block coordinates (kept out of the block context, which lives in shared memory)
#define TID ((int)threadIdx.x)
#define WARP ((int)threadIdx.x >> 5)
#define LANE ((int)threadIdx.x & 31)
#define CTA ((int)blockIdx.x)
#define GRID ((int)gridDim.x)

__device__ __forceinline__ uint16_t f2h(float v)
{
    __half h = __float2half_rn(v);
    return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(*reinterpret_cast<const __half*>(&b)); }

// (a & b) | c in one instruction
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Eight 4-bit fields of a word (field i = bits 4i..4i+3) as four fp16x2 registers, exactly:
// r0 = 1024 + {f0, f4}, r1 = 1024 + 16 {f1, f5}, r2 = 1024 + {f2, f6}, r3 = 1024 + 16 {f3, f7}.
// Placing a field inside the mantissa of 1024.0 (0x6400) costs one lop3 per pair and no shift for
// the odd fields; the 1024 offset and the factor 16 are taken out by the B operand and a
// per-chunk correction.
__device__ __forceinline__ void deq8(uint32_t w, uint32_t (&r)[4])
{
    const uint32_t w8 = w >> 8;
    r[0] = and_or(w, 0x000F000Fu, 0x64006400u);
    r[1] = and_or(w, 0x00F000F0u, 0x64006400u);
    r[2] = and_or(w8, 0x000F000Fu, 0x64006400u);
    r[3] = and_or(w8, 0x00F000F0u, 0x64006400u);
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 64-field chunk of a 16-row tile: thread (g, tq) holds fields [16 tq, 16 tq + 16) of row g
// (ra) and of row g + 8 (rb); b0/b1 hold the matching 16 B values in permuted register order.
// c[0] = C[g][2tq], c[1] = C[g][2tq+1], c[2] = C[g+8][2tq], c[3] = C[g+8][2tq+1].
__device__ __forceinline__ void chunk_mma(float (&c)[4], uint2 ra, uint2 rb, uint4 b0, uint4 b1)
{
    uint32_t a[4], b[4];
    c[0] = c[1] = c[2] = c[3] = 0.f;
    deq8(ra.x, a);
    deq8(rb.x, b);
    mma_f16(c, a[0], b[0], a[1], b[1], b0.x, b0.y);
    mma_f16(c, a[2], b[2], a[3], b[3], b0.z, b0.w);
    deq8(ra.y, a);
    deq8(rb.y, b);
    mma_f16(c, a[0], b[0], a[1], b[1], b1.x, b1.y);
    mma_f16(c, a[2], b[2], a[3], b[3], b1.z, b1.w);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float dot8_bf16(uint4 w, uint4 x, float acc)
{
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    const uint32_t xx[4] = {x.x, x.y, x.z, x.w};
#pragma unroll 1
    for (int i = 0; i < 4; ++i) {
        acc = fmaf(__uint_as_float(ww[i] << 16), __uint_as_float(xx[i] << 16), acc);
        acc = fmaf(__uint_as_float(ww[i] & 0xFFFF0000u), __uint_as_float(xx[i] & 0xFFFF0000u), acc);
    }
    return acc;
}

__device__ __forceinline__ void set_status(int* status, int code) { atomicCAS(status, 0, code); }

// ---- memory-model helpers ----
__device__ __forceinline__ void st_pair(unsigned long long* p, uint32_t epoch, float v)
{
    const unsigned long long x = ((unsigned long long)epoch << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(x) : "memory");
}

__device__ __forceinline__ void ld_pair2(const unsigned long long* p, unsigned long long& a, unsigned long long& b)
{
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ void red_add_s64(long long* p, long long v)
{
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void st_s64(long long* p, long long v)
{
    asm volatile("st.relaxed.gpu.global.s64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void ld_s64x2(const long long* p, long long& a, long long& b)
{
    asm volatile("ld.relaxed.gpu.global.v2.s64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}


// ---- mbarrier / TMA ----
__device__ __forceinline__ void mbar_init(uint64_t* m, int n)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(m)), "r"(n) : "memory");
}

__device__ __forceinline__ void mbar_expect(uint64_t* m, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(m)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t* m, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(smem_u32(m)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// 1D bulk copy global -> shared; dst, src 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* m)
{
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(m))
                 : "memory");
}

// 3D tiled TMA load (x in bytes: a multiple of 16)
__device__ __forceinline__ void tma3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* m)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(m))
        : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ------------------------------------------------------------------------------------------
// per-block context
// ------------------------------------------------------------------------------------------

// Block-uniform context: shape, staging geometry and shared-memory carve-up. One copy per block
// in shared memory (written by thread 0 at start), so it takes no registers.
struct Ctx {
    int H, E, k, I, Is, xp, KU, NCu, KD, NCd, KDs, NCds, ngu, ngd, ngds, rb_gu, rb_d, rb_ds;
    float invH;
    BlobGeo geo, geo_s;   // routed / shared blob geometry
    // (Ctx must fit in kCtxBytes; checked below)
    StageGeo sg;
    uint64_t* mbar;        // [kNumMbar]: ring slots, routed scales, dense, shared down
    int* sel_idx;          // [kMaxK]
    float* sel_w;          // [kMaxK]
    int* sel_slot;         // [kMaxK]
    float* red;            // [64]
    float* misc;           // [16]: [0] gamma
    int* imisc;            // [16]: staged-span offsets ([0..3] shared gate/up, [4..5] shared down,
                           //       [8..13] routed gate/up and down)
    float* sx;             // [H] layer input x (fp32)
    uint16_t* su;          // [H] u (bf16)
    uint16_t* sup;         // [KU] B operand of u (fp16, permuted blocks)
    float2* scs;           // [NCu] per chunk: sum of u, 1024 * sum of B
    float* slg;            // [E] logits
    uint32_t* lkey;        // [kWarps][kMaxK]
    int* lidx;             // [kWarps][kMaxK]
    uint16_t* srt;         // [Rr][H] router rows
    uint16_t* swsg;        // [H] shared gate vector
    uint8_t* sgq;          // [2][Rs][rb_gu] shared gate/up codes
    uint8_t* ssb;          // 4 spans: shared gate.s, gate.b, up.s, up.b rows
    uint8_t* sdq;          // [Rsd][rb_ds] shared down codes
    uint8_t* sdsb;         // 2 spans: shared down.s, down.b rows
    uint8_t* ring;         // [kWarps][slot_bytes]
    uint8_t* rsb;          // 4 spans: routed gate.s, gate.b, up.s, up.b rows
    uint8_t* rdsb;         // 2 spans: routed down.s, down.b rows
    uint16_t* shs;         // [2][KDs] B operand of h_shared (fp16 hi/lo, permuted blocks)
    float2* chs;           // [NCds] per chunk: sum of h, 1024 * sum of B
    uint16_t* shj;         // [2][KD] B operand of h_j
    float2* chj;           // [NCd]
    float* hv;             // [max(I, Is)] polled h values
    float* sp;             // gate/up partials [rows][2][ncb_gu]
    float* spd;            // down partials [rows][NCd or NCds]
    uint32_t span_gu, span_d, span_sgu, span_sd;  // bytes per staged scale span
};

static_assert(sizeof(Ctx) <= kCtxBytes, "the block context outgrew its shared-memory slot");

__device__ void make_ctx(const StepParams& P, Ctx& C, uint8_t* base)
{
    C.H = P.H;
    C.E = P.E;
    C.k = P.k;
    C.I = P.I;
    C.Is = P.Is;
    C.xp = P.bits == 8 ? 2 : 1;
    C.KU = P.H * C.xp;
    C.NCu = C.KU / kChunk;
    C.KD = P.I * C.xp;
    C.NCd = C.KD / kChunk;
    C.KDs = P.Is * C.xp;
    C.NCds = C.KDs / kChunk;
    C.ngu = P.H / 64;
    C.ngd = P.I / 64;
    C.ngds = P.Is / 64;
    C.rb_gu = P.H * P.bits / 8;
    C.rb_d = P.I * P.bits / 8;
    C.rb_ds = P.Is * P.bits / 8;
    C.sg = P.sg;
    C.invH = 1.f / (float)P.H;
    C.geo = P.geo;
    C.geo_s = P.geo_s;
    const SmemPlan s = smem_plan(P.H, P.E, P.k, P.I, P.Is, P.bits, GRID);
    C.mbar = (uint64_t*)(base + s.mbar);
    int* ctl = (int*)(base + s.ctl);
    C.sel_idx = ctl;
    C.sel_w = (float*)(ctl + kMaxK);
    C.sel_slot = ctl + 2 * kMaxK;
    C.red = (float*)(ctl + 3 * kMaxK);
    C.misc = (float*)(ctl + 3 * kMaxK + 64);
    C.imisc = ctl + 3 * kMaxK + 64 + 16;
    C.sx = (float*)(base + s.x);
    C.su = (uint16_t*)(base + s.u);
    C.sup = (uint16_t*)(base + s.up);
    C.scs = (float2*)(base + s.uc);
    C.slg = (float*)(base + s.lg);
    C.lkey = (uint32_t*)(base + s.lkey);
    C.lidx = (int*)(base + s.lidx);
    C.srt = (uint16_t*)(base + s.rt);
    C.swsg = (uint16_t*)(base + s.wsg);
    C.sgq = base + s.sgq;
    C.ssb = base + s.ssb;
    C.sdq = base + s.sdq;
    C.sdsb = base + s.sdsb;
    C.ring = base + s.ring;
    C.rsb = base + s.rsb;
    C.rdsb = base + s.rdsb;
    C.shs = (uint16_t*)(base + s.hs);
    C.chs = (float2*)(base + s.uhs);
    C.shj = (uint16_t*)(base + s.hj);
    C.chj = (float2*)(base + s.uhj);
    C.hv = (float*)(base + s.hv);
    C.sp = (float*)(base + s.sp);
    C.spd = (float*)(base + s.spd);
    C.span_gu = sb_span_max(C.sg.Rgu, 2 * C.ngu);
    C.span_d = sb_span_max(C.sg.Rd, 2 * C.ngd);
    C.span_sgu = sb_span_max(C.sg.Rs, 2 * C.ngu);
    C.span_sd = sb_span_max(C.sg.Rsd, 2 * C.ngds);
}


// Block-uniform time limit check: true once the wait that started at t0 ran past the limit.
__device__ __forceinline__ bool timed_out(const StepParams& P, long long t0)
{
    return __syncthreads_or(threadIdx.x == 0 && cycles() - t0 > limit_cycles(P)) != 0;
}

// Issue a 1D copy of rows [r0, r1) of a section whose rows hold row_b bytes (16-byte aligned
// superset); returns the bytes issued and, in *off, the offset of row r0 inside the copy.
__device__ __forceinline__ uint32_t copy_rows(void* dst, const uint8_t* sec, int r0, int r1, int row_b, uint64_t* m,
                                              uint32_t* off)
{
    if (r1 <= r0) {
        *off = 0;
        return 0;
    }
    const uintptr_t a = (uintptr_t)(sec + (size_t)r0 * row_b);
    const uintptr_t e = (uintptr_t)(sec + (size_t)r1 * row_b);
    const uintptr_t a16 = a & ~(uintptr_t)15, e16 = (e + 15) & ~(uintptr_t)15;
    *off = (uint32_t)(a - a16);
    bulk_g2s(dst, (const void*)a16, (uint32_t)(e16 - a16), m);
    return (uint32_t)(e16 - a16);
}

// ------------------------------------------------------------------------------------------
// dense (resident) rows of a step: router rows, shared gate vector, shared gate/up rows, and
// separately the shared down rows
// ------------------------------------------------------------------------------------------

struct DenseRows {
    int e0, e1;    // router rows
    int s0, s1;    // shared gate/up rows
    int o0, o1;    // shared down rows (= this block's slice of the output)
};

__device__ __forceinline__ DenseRows dense_rows(const Ctx& C)
{
    DenseRows d;
    d.e0 = part(C.E, GRID, CTA);
    d.e1 = part(C.E, GRID, CTA + 1);
    d.s0 = part(C.Is, GRID, CTA);
    d.s1 = part(C.Is, GRID, CTA + 1);
    d.o0 = part(C.H, GRID, CTA);
    d.o1 = part(C.H, GRID, CTA + 1);
    return d;
}

// Bytes copy_rows() issues for rows [r0, r1) of a section whose rows hold row_b bytes.
__device__ __forceinline__ uint32_t span_bytes(const uint8_t* sec, int r0, int r1, int row_b)
{
    if (r1 <= r0)
        return 0;
    const uintptr_t a = (uintptr_t)(sec + (size_t)r0 * row_b);
    const uintptr_t e = (uintptr_t)(sec + (size_t)r1 * row_b);
    return (uint32_t)(((e + 15) & ~(uintptr_t)15) - (a & ~(uintptr_t)15));
}

// Issued by thread 0: the router rows, the shared gate vector and the shared expert's gate/up
// rows of layer L. Offsets of the staged scale spans go to imisc[0..3].
__device__ __noinline__ void issue_dense(const StepParams& P, const Ctx& C, const LayerDesc L, bool with_router, bool with_shared)
{
    const DenseRows d = dense_rows(C);
    uint64_t* m = C.mbar + kWarps + 1;
    const BlobGeo& gs = C.geo_s;
    const bool rt = with_router && d.e1 > d.e0;
    const bool sh = with_shared && d.s1 > d.s0;
    // the expected bytes go first: the arrive must not complete the phase before the copies count
    uint32_t bytes = (uint32_t)C.H * 2;
    if (rt)
        bytes += (uint32_t)(d.e1 - d.e0) * C.H * 2;
    if (sh) {
        bytes += 2u * (uint32_t)(d.s1 - d.s0) * C.rb_gu;
        #pragma unroll 1
        for (int i = 0; i < 4; ++i)
            bytes += span_bytes(L.shared_blob + ((i & 1) ? gs.b_off[i >> 1] : gs.s_off[i >> 1]), d.s0, d.s1, C.ngu * 2);
    }
    mbar_expect(m, bytes);
    if (rt)
        bulk_g2s(C.srt, L.router + (size_t)d.e0 * C.H, (uint32_t)(d.e1 - d.e0) * C.H * 2, m);
    bulk_g2s(C.swsg, L.shared_gate, (uint32_t)C.H * 2, m);
    if (sh) {
        const uint32_t nq = (uint32_t)(d.s1 - d.s0) * C.rb_gu;
        bulk_g2s(C.sgq, L.shared_blob + gs.q_off[0] + (size_t)d.s0 * C.rb_gu, nq, m);
        bulk_g2s(C.sgq + (size_t)C.sg.Rs * C.rb_gu, L.shared_blob + gs.q_off[1] + (size_t)d.s0 * C.rb_gu, nq, m);
        #pragma unroll 1
        for (int i = 0; i < 4; ++i) {
            uint32_t off;
            copy_rows(C.ssb + i * C.span_sgu, L.shared_blob + ((i & 1) ? gs.b_off[i >> 1] : gs.s_off[i >> 1]), d.s0, d.s1,
                      C.ngu * 2, m, &off);
            C.imisc[i] = (int)off;
        }
    }
}

__device__ __noinline__ void issue_shared_down(const StepParams& P, const Ctx& C, const LayerDesc L)
{
    const DenseRows d = dense_rows(C);
    uint64_t* m = C.mbar + kWarps + 2;
    const BlobGeo& gs = C.geo_s;
    const int rowb = C.ngds * 2;
    uint32_t bytes = 0;
    if (d.o1 > d.o0)
        bytes = (uint32_t)(d.o1 - d.o0) * C.rb_ds + span_bytes(L.shared_blob + gs.s_off[2], d.o0, d.o1, rowb) +
                span_bytes(L.shared_blob + gs.b_off[2], d.o0, d.o1, rowb);
    mbar_expect(m, bytes);
    if (d.o1 > d.o0) {
        uint32_t off;
        bulk_g2s(C.sdq, L.shared_blob + gs.q_off[2] + (size_t)d.o0 * C.rb_ds, (uint32_t)(d.o1 - d.o0) * C.rb_ds, m);
        copy_rows(C.sdsb, L.shared_blob + gs.s_off[2], d.o0, d.o1, rowb, m, &off);
        C.imisc[4] = (int)off;
        copy_rows(C.sdsb + C.span_sd, L.shared_blob + gs.b_off[2], d.o0, d.o1, rowb, m, &off);
        C.imisc[5] = (int)off;
    }
}

// ------------------------------------------------------------------------------------------
// A-fragment loads from staged rows
// ------------------------------------------------------------------------------------------

// Rows staged in shared memory. Swizzled (TMA boxes of 128-byte rows, slots 1024-byte aligned):
// the 16-byte chunk j of row R sits at chunk j ^ (R & 7); linear: rows of `width` bytes one after
// another. swzmask is 7 for swizzled rows (width 128) and 0 for linear ones, so both layouts share
// one branch-free address computation.
__device__ __forceinline__ uint2 lds_a(const uint8_t* base, uint32_t swzmask, int width, int R, int byte)
{
    const uint32_t off = (uint32_t)R * (uint32_t)width + ((((uint32_t)byte >> 4) ^ ((uint32_t)R & swzmask)) << 4) +
                         ((uint32_t)byte & 15u);
    return *reinterpret_cast<const uint2*>(base + off);
}

// ------------------------------------------------------------------------------------------
// input, u, expanded u
// ------------------------------------------------------------------------------------------

// The B operand of one chunk: fp16 activations in the MMA's register order (pslot). For int4 the
// odd fields of a word enter A multiplied by 16, so their activations are divided by 16; an int8
// code is read as two fields (low, 16 x high), both paired with the code's activation.

// x (in sx) or the bf16 input u_bits -> su (bf16 u), sup (B operand), scs (per chunk sums)
__device__ void make_u(const StepParams& P, const Ctx& C, bool prenorm, const uint16_t* u_bits)
{
    const int H = C.H;
    float rinv = 1.f;
    if (prenorm) {
        float ss = 0.f;
        #pragma unroll 1
        for (int i = TID; i < H; i += kThreads)
            ss = fmaf(C.sx[i], C.sx[i], ss);
        ss = warp_sum(ss);
        if (LANE == 0)
            C.red[WARP] = ss;
        __syncthreads();
        float tot = 0.f;
        #pragma unroll 1
        for (int w = 0; w < kWarps; ++w)
            tot += C.red[w];
        rinv = rsqrtf(tot * C.invH + 1e-6f);
    }
    const int cpc = kChunk / C.xp;  // codes per chunk
    const int lpc = cpc / 4;        // threads per chunk (4 codes each)
    #pragma unroll 1
    for (int q0 = 0; q0 < H / 4; q0 += kThreads) {
        const int q = q0 + TID;
        float us = 0.f, bs = 0.f;
        if (q < H / 4) {
            #pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                const int i = 4 * q + j;
                const uint16_t ub = prenorm ? f2bf(C.sx[i] * rinv) : u_bits[i];
                const float uv = bf16f(ub);
                C.su[i] = ub;
                us += uv;
                if (C.xp == 1) {
                    const uint16_t bh = f2h((i & 1) ? uv * 0.0625f : uv);
                    C.sup[pslot(i)] = bh;
                    bs += h2f(bh);
                } else {
                    const uint16_t bh = f2h(uv);
                    C.sup[pslot(2 * i)] = bh;
                    C.sup[pslot(2 * i + 1)] = bh;
                    bs += 2.f * h2f(bh);
                }
            }
        }
        #pragma unroll 1
        for (int o = lpc / 2; o; o >>= 1) {
            us += __shfl_xor_sync(0xffffffffu, us, o);
            bs += __shfl_xor_sync(0xffffffffu, bs, o);
        }
        if (q < H / 4 && (LANE % lpc) == 0)
            C.scs[4 * q / cpc] = make_float2(us, 1024.f * bs);
    }
    __syncthreads();
}

// h values hv[0, n) -> B operand hi/lo parts (sh: [2][n * xp]) and per chunk {sum of h, 1024 *
// sum of (hi + lo)}; hi + lo carries h to about 22 bits.
__device__ __noinline__ void stage_h(int xp, const float* hv, int n, uint16_t* sh, float2* chs)
{
    const int tid = threadIdx.x, lane = tid & 31;
    const int KD = n * xp;
    uint16_t* hi = sh;
    uint16_t* lo = sh + KD;
    const int cpc = kChunk / xp;
    const int lpc = cpc / 4;
    #pragma unroll 1
    for (int q0 = 0; q0 < n / 4; q0 += kThreads) {
        const int q = q0 + tid;
        float hs = 0.f, bs = 0.f;
        if (q < n / 4) {
            #pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                const int i = 4 * q + j;
                const float v = hv[i];
                hs += v;
                if (xp == 1) {
                    const float e = (i & 1) ? v * 0.0625f : v;
                    const uint16_t hb = f2h(e);
                    const uint16_t lb = f2h(e - h2f(hb));
                    hi[pslot(i)] = hb;
                    lo[pslot(i)] = lb;
                    bs += h2f(hb) + h2f(lb);
                } else {
                    const uint16_t hb = f2h(v);
                    const uint16_t lb = f2h(v - h2f(hb));
                    hi[pslot(2 * i)] = hb;
                    hi[pslot(2 * i + 1)] = hb;
                    lo[pslot(2 * i)] = lb;
                    lo[pslot(2 * i + 1)] = lb;
                    bs += 2.f * (h2f(hb) + h2f(lb));
                }
            }
        }
        #pragma unroll 1
        for (int o = lpc / 2; o; o >>= 1) {
            hs += __shfl_xor_sync(0xffffffffu, hs, o);
            bs += __shfl_xor_sync(0xffffffffu, bs, o);
        }
        if (q < n / 4 && (lane % lpc) == 0)
            chs[4 * q / cpc] = make_float2(hs, 1024.f * bs);
    }
    __syncthreads();
}

// Poll n epoch-tagged pairs until all carry `epoch`; values -> dst (fp32). Block-uniform.
__device__ __noinline__ bool poll_pairs(long long limit, int* status, const unsigned long long* src, int n,
                                        uint32_t epoch, float* dst)
{
    const long long t0 = cycles();
    while (true) {
        int bad = 0;
        #pragma unroll 1
        for (int e = 2 * (int)threadIdx.x; e < n; e += 2 * kThreads) {
            unsigned long long a, b;
            ld_pair2(src + e, a, b);
            bad |= (uint32_t)(a >> 32) != epoch;
            dst[e] = __uint_as_float((uint32_t)a);
            if (e + 1 < n) {
                bad |= (uint32_t)(b >> 32) != epoch;
                dst[e + 1] = __uint_as_float((uint32_t)b);
            }
        }
        if (!__syncthreads_or(bad))
            return true;
        if (__syncthreads_or(threadIdx.x == 0 && cycles() - t0 > limit)) {
            if (threadIdx.x == 0)
                set_status(status, kStatusTimeout);
            return false;
        }
    }
}

// Grid barrier on a monotonically increasing counter (a multiple of the grid between launches).
__device__ __noinline__ bool grid_barrier(const StepParams& P, const Ctx& C)
{
    __syncthreads();
    int ok = 1;
    if (TID == 0) {
        const unsigned long long G = gridDim.x;
        unsigned long long ticket;
        asm volatile("atom.add.release.gpu.global.u64 %0, [%1], 1;" : "=l"(ticket) : "l"(P.bar) : "memory");
        const unsigned long long target = (ticket / G + 1) * G;
        const long long t0 = cycles();
        while (true) {
            unsigned long long v;
            asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(P.bar) : "memory");
            if (v >= target)
                break;
            if (cycles() - t0 > limit_cycles(P)) {
                ok = 0;
                set_status(P.status, kStatusTimeout);
                break;
            }
        }
    }
    return __syncthreads_or(!ok) == 0;
}

// ------------------------------------------------------------------------------------------
// the chunk work items
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ float bf16_at(const uint8_t* p) { return bf16f(*reinterpret_cast<const uint16_t*>(p)); }

// One block of up to four chunks (one 128-byte column block) of staged rows. Rows [0, nstaged) of
// the staged set are local rows rloc0 + R; chunk c0 + i starts at byte cbyte0 + 32 i of a staged
// row. For every local row r < nrows it writes s * (sum q v) + b * (sum v), summed over the
// chunks, to out[r * ostride], where v is u (gate/up rows) or h (down rows; kDown: B holds h's hi
// parts in the even columns and lo parts in the odd ones). The B operands and chunk sums are
// loaded once for all row tiles, and the four chunks of a tile run as independent MMA chains.
template <bool kDown>
__device__ __noinline__ void mma_block(const uint8_t* base, uint32_t swzmask, int width, int nstaged, int rloc0,
                                          int nrows, int c0, int nch, int cbyte0, const uint16_t* bsrc, int KD,
                                          const float2* csum, const uint8_t* sc, const uint8_t* bi, int sbrow,
                                          float* out, int ostride, int gsh)
{
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    const uint16_t* bb = kDown ? bsrc + (size_t)(g & 1) * KD : bsrc;
    const int ntile = (nstaged + 15) >> 4;
#pragma unroll 1
    for (int tile = 0; tile < ntile; ++tile) {
        const int Ra = tile * 16 + g, Rb = Ra + 8;
        const int R = tq == 0 ? Ra : Rb;
        const int r = rloc0 + R;
        const bool mine = tq < 2 && R < nstaged && r < nrows;
        float part = 0.f;
#pragma unroll 1
        for (int cp = 0; cp < 4; cp += 2) {  // two chunks at a time: two independent MMA chains
            uint2 ra[2], rb[2];
            uint4 B0[2], B1[2];
            float sv[2], bv[2];
            float2 cs[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int cl = cp + h;
                const bool on = cl < nch;
                const int c = c0 + (on ? cl : 0);
                const int byte = cbyte0 + 32 * cl + 8 * tq;
                ra[h] = (on && Ra < nstaged) ? lds_a(base, swzmask, width, Ra, byte) : make_uint2(0, 0);
                rb[h] = (on && Rb < nstaged) ? lds_a(base, swzmask, width, Rb, byte) : make_uint2(0, 0);
                const uint4* bp = reinterpret_cast<const uint4*>(bb + kChunk * c + 16 * tq);
                B0[h] = bp[0];
                B1[h] = bp[1];
                cs[h] = csum[c];
                const int gi = c >> gsh;
                sv[h] = (mine && on) ? bf16_at(sc + r * sbrow + 2 * gi) : 0.f;
                bv[h] = (mine && on) ? bf16_at(bi + r * sbrow + 2 * gi) : 0.f;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float acc[4];
                chunk_mma(acc, ra[h], rb[h], B0[h], B1[h]);
                const float a = kDown ? (tq == 0 ? acc[0] + acc[1] : acc[2] + acc[3]) : (tq == 0 ? acc[0] : acc[2]);
                part = fmaf(sv[h], a - cs[h].y, fmaf(bv[h], cs[h].x, part));
            }
        }
        if (mine)
            out[r * ostride] = part;
    }
}

// ------------------------------------------------------------------------------------------
// routing
// ------------------------------------------------------------------------------------------

// slg (logits) -> sel_idx / sel_w (rank order: larger fp32 logit first, ties -> lower index).
// Each warp ranks its 32 logits; the largest of the warps' k-th best values is a lower bound of
// the overall k-th best, so only logits at or above it (usually little more than k) take part in
// the final ranking.
__device__ void topk_select(const StepParams& P, const Ctx& C, int my_slot)
{
    const int E = C.E, k = C.k;
    const int nl = (E + 31) / 32;
    uint32_t* wkth = C.lkey;                 // [kWarps] k-th best key of each warp
    uint32_t* skey = C.lkey + kWarps;        // [E] survivors
    int* sidx = C.lidx;                      // [E]
    int* wcnt = C.lidx + kMaxE + 8;          // [kWarps] survivors per warp
    const int e = 32 * WARP + LANE;
    const uint32_t key = (WARP < nl && e < E) ? ord_key(C.slg[e]) : 0u;
    if (WARP < nl) {
        int rank = 0;
#pragma unroll
        for (int d = 1; d < 32; ++d) {
            const int src = (LANE + d) & 31;
            const uint32_t o = __shfl_sync(0xffffffffu, key, src);
            rank += (o > key) || (o == key && src < LANE);
        }
        const unsigned kth = __ballot_sync(0xffffffffu, rank == k - 1);
        const uint32_t kv = __shfl_sync(0xffffffffu, key, kth ? __ffs(kth) - 1 : 0);
        if (LANE == 0)
            wkth[WARP] = kth ? kv : 0u;
    }
    __syncthreads();
    uint32_t t0 = 0;
#pragma unroll 1
    for (int w = 0; w < nl; ++w)
        t0 = max(t0, wkth[w]);
    const bool surv = WARP < nl && e < E && key >= t0;
    const unsigned bal = __ballot_sync(0xffffffffu, surv);
    if (LANE == 0)
        wcnt[WARP] = __popc(bal);
    __syncthreads();
    int pos = 0, ns = 0;
#pragma unroll 1
    for (int w = 0; w < kWarps; ++w) {
        const int c = wcnt[w];
        pos += w < WARP ? c : 0;
        ns += c;
    }
    if (surv) {
        const int p = pos + __popc(bal & ((1u << LANE) - 1u));
        skey[p] = key;
        sidx[p] = e;
    }
    __syncthreads();
    if (TID >= ns && TID < ((ns + 3) & ~3)) {  // pad the survivor list to a multiple of 4
        skey[TID] = 0u;
        sidx[TID] = 0x7fffffff;
    }
    __syncthreads();
    if (surv) {
        int rank = 0;
        const uint4* k4 = reinterpret_cast<const uint4*>(skey);
        const int4* i4 = reinterpret_cast<const int4*>(sidx);
#pragma unroll 4
        for (int i = 0; i < (ns + 3) >> 2; ++i) {
            const uint4 kk = k4[i];
            const int4 ii = i4[i];
            rank += (kk.x > key || (kk.x == key && ii.x < e)) + (kk.y > key || (kk.y == key && ii.y < e)) +
                    (kk.z > key || (kk.z == key && ii.z < e)) + (kk.w > key || (kk.w == key && ii.w < e));
        }
        if (rank < k) {
            C.sel_idx[rank] = e;
            C.sel_slot[rank] = my_slot;
        }
    }
    __syncthreads();
    if (WARP == 0) {
        const float lmax = C.slg[C.sel_idx[0]];
        const float p = LANE < k ? __expf(C.slg[C.sel_idx[LANE]] - lmax) : 0.f;
        float denom = 0.f;
        if (P.flags & kRenorm) {
            #pragma unroll 1
            for (int j = 0; j < k; ++j)
                denom += __shfl_sync(0xffffffffu, p, j);
        } else {
            float s = 0.f;
            #pragma unroll 1
            for (int e = LANE; e < E; e += 32)
                s += __expf(C.slg[e] - lmax);
            denom = __shfl_sync(0xffffffffu, warp_sum(s), 0);
        }
        if (LANE < k)
            C.sel_w[LANE] = __fdividef(p, denom);
    }
    __syncthreads();
}

// ------------------------------------------------------------------------------------------
// routed stages
// ------------------------------------------------------------------------------------------

struct Routed {
    int j;                 // expert rank served by this block
    const uint8_t* blob;   // its blob (null: not resident)
    int slot;
    int r0, r1;            // own gate/up rows
    int d0, d1;            // own down rows
    uint32_t off[6];       // offsets of the staged scale spans: gate.s, gate.b, up.s, up.b, down.s, down.b
};

// Stage s of the block's routed work -> TMA box into ring slot (s % kWarps).
__device__ __noinline__ void issue_stage(const StepParams& P, const Ctx& C, int wslot, int r0, int d0, int s)
{
    const StageGeo& sg = C.sg;
    uint8_t* dst = C.ring + (size_t)(s % kWarps) * sg.slot_bytes;
    uint64_t* m = C.mbar + (s % kWarps);
    if (s < sg.n_gu) {
        const int rc = s % sg.nrc_gu, q = s / sg.nrc_gu, mat = q & 1, cb = q >> 1;
        mbar_expect(m, (uint32_t)sg.SR * sg.cbw_gu);
        tma3d(dst, &P.tmap[mat], cb * sg.cbw_gu, r0 + rc * sg.SR, wslot, m);
    } else {
        const int sd = s - sg.n_gu, rc = sd % sg.nrc_d, cb = sd / sg.nrc_d;
        mbar_expect(m, (uint32_t)sg.SR * sg.cbw_d);
        tma3d(dst, &P.tmap[2], cb * sg.cbw_d, d0 + rc * sg.SR, wslot, m);
    }
}

// Wait for ring slot `slot` to complete phase `parity` (warp-uniform; false after the limit).
__device__ __noinline__ bool wait_slot(const StepParams& P, const Ctx& C, int slot, uint32_t parity)
{
    const long long t0 = cycles();
    while (true) {
        if (__all_sync(0xffffffffu, mbar_try(C.mbar + slot, parity)))
            return true;
        if (__any_sync(0xffffffffu, cycles() - t0 > limit_cycles(P)))
            return false;
    }
}

// Block-uniform wait for a block-level mbarrier (all threads).
__device__ __noinline__ bool wait_block(const StepParams& P, const Ctx& C, uint64_t* m, uint32_t parity)
{
    const long long t0 = cycles();
    while (true) {
        const int ok = mbar_try(m, parity);
        if (__syncthreads_and(ok))
            return true;
        if (timed_out(P, t0))
            return false;
    }
}

}  // namespace

// Dynamic shared memory of the fused kernel: the plan plus 1024 bytes to align the ring.
__host__ __device__ uint32_t decode_smem_bytes(const StepParams& P, int grid)
{
    return smem_plan(P.H, P.E, P.k, P.I, P.Is, P.bits, grid).total + 1024;
}

__global__ void __launch_bounds__(kThreads, 1) moe_decode_kernel(const __grid_constant__ StepParams P)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const SmemPlan plan0 = smem_plan(P.H, P.E, P.k, P.I, P.Is, P.bits, GRID);
    Ctx& C = *reinterpret_cast<Ctx*>(base + plan0.ctx);
    if (TID == 0)
        make_ctx(P, C, base);
    __syncthreads();
    const StageGeo& sg = C.sg;
    const bool route = P.mode != kModeExperts;
    const bool experts = P.mode != kModeRoute;
    const int n_steps = P.n_tokens * P.n_layers;

    if (TID == 0) {
        #pragma unroll
        for (int i = 0; i < kNumMbar; ++i)
            mbar_init(C.mbar + i, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (experts)
            #pragma unroll
            for (int i = 0; i < 3; ++i)
                prefetch_map(&P.tmap[i]);
    }
    __syncthreads();

    // phase counters of the mbarriers (uniform in the block / warp)
    uint32_t ph_dense = 0, ph_sdown = 0, ph_rsc = 0, ph_slot = 0;
    bool dense_pending = false, sdown_pending = false, rsc_pending = false;
    int slot_pending = 0;  // this warp's issued-but-unconsumed stages (at most one per slot)

    if (TID == 0) {
        const LayerDesc L0 = P.layers[P.layer0];
        issue_dense(P, C, L0, route, experts);
        if (experts)
            issue_shared_down(P, C, L0);
    }
    dense_pending = true;
    sdown_pending = experts;

    const DenseRows drow = dense_rows(C);
    bool ok = true;

    // X init for token 0: this block's slice of the accumulator holds the residual base
    if (experts) {
        const bool residual = (P.flags & kResidual) != 0;
        #pragma unroll 1
        for (int o = drow.o0 + TID; o < drow.o1; o += kThreads) {
            float x0 = 0.f;
            if (residual)
                x0 = (P.flags & kPrenorm) ? ((const float*)P.x_in)[o] : bf16f(((const uint16_t*)P.x_in)[o]);
            st_s64(P.xacc + o, (long long)__float2ll_rn(x0 * kFix));
        }
        ok = grid_barrier(P, C);
    }

    #pragma unroll 1
    for (int step = 0; ok && step < n_steps; ++step) {
        const int t = step / P.n_layers, li = step - t * P.n_layers;
        const int l = P.layer0 + li;
        const LayerDesc L = P.layers[l];
        // this thread's expert's slot, loaded now so that it is in a register by the time top-k
        // names the experts (the thread of logit e is thread e)
        const int my_slot = (route && TID < C.E) ? P.table[(size_t)l * C.E + TID] : -1;
        const uint32_t epoch = P.epoch0 + (uint32_t)step;
        long long* X = P.xacc + (size_t)(step & 1) * C.H;
        const bool prenorm = (P.flags & kPrenorm) != 0;

        // ---------------- 1. layer input ----------------
        if (li == 0) {
            if (prenorm) {
                const float* src = (const float*)P.x_in + (size_t)t * C.H;
                #pragma unroll 1
                for (int i = TID; i < C.H; i += kThreads)
                    C.sx[i] = src[i];
            } else {
                const uint16_t* src = (const uint16_t*)P.x_in + (size_t)t * C.H;
                #pragma unroll 1
                for (int i = TID; i < C.H; i += kThreads)
                    C.sx[i] = bf16f(src[i]);
            }
            __syncthreads();
        }
        if (P.trace && CTA == 0)
            #pragma unroll 1
            for (int i = TID; i < C.H; i += kThreads)
                P.trace[((size_t)t * (P.n_layers + 1) + li) * C.H + i] = C.sx[i];
        make_u(P, C, prenorm, (const uint16_t*)P.x_in + (size_t)t * C.H);

        // ---------------- 2. router rows, gamma, shared gate/up ----------------
        if (!wait_block(P, C, C.mbar + kWarps + 1, ph_dense & 1)) {
            ok = false;
            break;
        }
        ++ph_dense;
        dense_pending = false;
        if (route) {
            const int nr = drow.e1 - drow.e0;
            #pragma unroll 1
            for (int r = WARP; r < nr; r += kWarps) {
                const uint16_t* row = C.srt + (size_t)r * C.H;
                float acc = 0.f;
                #pragma unroll 1
                for (int i = 0; i < C.H / 256; ++i) {
                    const uint4 w = *reinterpret_cast<const uint4*>(row + 256 * i + 8 * LANE);
                    const uint4 x = *reinterpret_cast<const uint4*>(C.su + 256 * i + 8 * LANE);
                    acc = dot8_bf16(w, x, acc);
                }
                acc = warp_sum(acc);
                if (LANE == 0) {
                    const int e = drow.e0 + r;
                    if (L.logit_bias)
                        acc += __ldg(L.logit_bias + e);
                    st_pair(P.xlog + e, epoch, acc);
                }
            }
        }
        if (experts) {
            if (WARP == kWarps - 1) {
                float z = 0.f;
                #pragma unroll 1
                for (int i = 0; i < C.H / 256; ++i) {
                    const uint4 w = *reinterpret_cast<const uint4*>(C.swsg + 256 * i + 8 * LANE);
                    const uint4 x = *reinterpret_cast<const uint4*>(C.su + 256 * i + 8 * LANE);
                    z = dot8_bf16(w, x, z);
                }
                z = warp_sum(z);
                if (LANE == 0)
                    C.misc[0] = __fdividef(1.f, 1.f + __expf(-z));
            }
            // shared gate/up rows [s0, s1): one item per (matrix, 128-byte column block)
            const int ns = drow.s1 - drow.s0;
            const int ncb = sg.ncb_gu;
            if (ns > 0) {
                #pragma unroll 1
                for (int it = WARP; it < 2 * ncb; it += kWarps) {
                    const int m = it / ncb, cb = it - m * ncb;
                    const uint8_t* q = C.sgq + (size_t)m * sg.Rs * C.rb_gu;
                    const uint8_t* sc = C.ssb + (2 * m) * C.span_sgu + C.imisc[2 * m];
                    const uint8_t* bi = C.ssb + (2 * m + 1) * C.span_sgu + C.imisc[2 * m + 1];
                    const int c0 = cb * 4;
                    mma_block<false>(q, 0u, C.rb_gu, ns, 0, ns, c0, min(4, C.NCu - c0), cb * kCb, C.sup, 0, C.scs, sc,
                                     bi, C.ngu * 2, C.sp + m * ncb + cb, 2 * ncb, C.xp - 1);
                }
            }
            __syncthreads();
            if (TID < ns) {
                const float* pg = C.sp + TID * 2 * ncb;
                float gg = 0.f, vv = 0.f;
                #pragma unroll 1
                for (int cb = 0; cb < ncb; ++cb) {
                    gg += pg[cb];
                    vv += pg[ncb + cb];
                }
                const float h = __fdividef(gg, 1.f + __expf(-gg)) * vv;
                st_pair(P.xh + (size_t)C.k * xh_stride(C.I, C.Is) + drow.s0 + TID, epoch, h);
            }
        }
        __syncthreads();
        if (experts && TID == 0) {
            // this block's step flag, after a gpu-scope fence: every store of the block so far,
            // the accumulator base included, is visible to whoever sees the flag
            fence_gpu();
            st_pair(P.xh + (size_t)C.k * xh_stride(C.I, C.Is) + C.Is + CTA, epoch, 0.f);
        }
        // next step's router rows, shared gate vector and shared gate/up rows
        if (step + 1 < n_steps) {
            if (TID == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                const int ln = P.layer0 + (step + 1) % P.n_layers;
                issue_dense(P, C, P.layers[ln], route, experts);
            }
            dense_pending = true;
        }

        // ---------------- 3. routing ----------------
        if (route) {
            if (!poll_pairs(limit_cycles(P), P.status, P.xlog, C.E, epoch, C.slg)) {
                ok = false;
                break;
            }
            topk_select(P, C, my_slot);
            if (CTA == 0 && TID < C.k) {
                const size_t o = ((size_t)t * P.n_layers + li) * C.k + TID;
                if (P.topk_idx)
                    P.topk_idx[o] = C.sel_idx[TID];
                if (P.topk_w)
                    P.topk_w[o] = C.sel_w[TID];
            }
            if (!experts)
                break;  // a route-only launch has one step
            if (TID < C.k && C.sel_slot[TID] < 0)
                set_status(P.status, kStatusNotResident);
        } else if (TID < C.k) {
            C.sel_w[TID] = P.topk_w[TID];
            C.sel_slot[TID] = P.slots[TID];
            C.sel_idx[TID] = -1;
        }
        __syncthreads();

        // ---------------- 4. routed work of this block: issue its boxes ----------------
        Routed W;
        {
            W.j = grp_of(CTA, GRID, C.k);
            const int gs0 = grp_start(W.j, GRID, C.k), gs1 = grp_start(W.j + 1, GRID, C.k);
            const int n = gs1 - gs0, mi = CTA - gs0;
            W.slot = C.sel_slot[W.j];
            W.blob = W.slot >= 0 ? P.arena + (uint64_t)W.slot * P.stride : nullptr;
            W.r0 = part(C.I, n, mi);
            W.r1 = part(C.I, n, mi + 1);
            W.d0 = part(C.H, n, mi);
            W.d1 = part(C.H, n, mi + 1);
        }
        if (W.blob) {
            if (WARP == 0 && LANE == 0) {
                // scale / bias rows of the block's gate/up rows and down rows
                uint64_t* m = C.mbar + kWarps;
                const BlobGeo& geo = C.geo;
                uint32_t bytes = 0;
                #pragma unroll 1
                for (int i = 0; i < 6; ++i) {
                    const bool dn = i >= 4;
                    const uint64_t sec = (i & 1) ? geo.b_off[i >> 1] : geo.s_off[i >> 1];
                    bytes += span_bytes(W.blob + sec, dn ? W.d0 : W.r0, dn ? W.d1 : W.r1, dn ? C.ngd * 2 : C.ngu * 2);
                }
                mbar_expect(m, bytes);
                #pragma unroll 1
                for (int i = 0; i < 6; ++i) {
                    const bool dn = i >= 4;
                    uint8_t* dst = dn ? C.rdsb + (i - 4) * C.span_d : C.rsb + i * C.span_gu;
                    uint32_t off;
                    const uint64_t sec = (i & 1) ? geo.b_off[i >> 1] : geo.s_off[i >> 1];
                    copy_rows(dst, W.blob + sec, dn ? W.d0 : W.r0, dn ? W.d1 : W.r1, dn ? C.ngd * 2 : C.ngu * 2, m, &off);
                    C.imisc[8 + i] = (int)off;
                }
            }
            rsc_pending = true;
            if (LANE == 0 && WARP < sg.n_stages) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue_stage(P, C, W.slot, W.r0, W.d0, WARP);
            }
            if (WARP < sg.n_stages)
                slot_pending = 1;
        }

        // ---------------- 5. shared expert down rows ----------------
        float* hval = C.hv;
        // the shared h values and every block's step flag: past this point the accumulator bases of all
        // blocks (stored at the end of the previous step, before their flag's fence) are visible
        if (!poll_pairs(limit_cycles(P), P.status, P.xh + (size_t)C.k * xh_stride(C.I, C.Is), C.Is + GRID, epoch, hval)) {
            ok = false;
            break;
        }
        stage_h(C.xp, hval, C.Is, C.shs, C.chs);
        if (!wait_block(P, C, C.mbar + kWarps + 2, ph_sdown & 1)) {
            ok = false;
            break;
        }
        ++ph_sdown;
        sdown_pending = false;
        {
            const int nd = drow.o1 - drow.o0;
            const int ncb = (C.NCds + 3) / 4;
            const uint8_t* sc = C.sdsb + C.imisc[4];
            const uint8_t* bi = C.sdsb + C.span_sd + C.imisc[5];
            if (nd > 0)
                #pragma unroll 1
                for (int cb = WARP; cb < ncb; cb += kWarps)
                    mma_block<true>(C.sdq, 0u, C.rb_ds, nd, 0, nd, 4 * cb, min(4, C.NCds - 4 * cb), cb * kCb, C.shs,
                                    C.KDs, C.chs, sc, bi, C.ngds * 2, C.spd + cb, ncb, C.xp - 1);
            __syncthreads();
            if (TID < nd) {
                float ys = 0.f;
                #pragma unroll 1
                for (int cb = 0; cb < ncb; ++cb)
                    ys += C.spd[TID * ncb + cb];
                const float v = C.misc[0] * ys;
                fence_gpu();  // after the shared h pairs: every block's accumulator base is in place
                if (!(fabsf(v) < kFixMax))
                    set_status(P.status, kStatusInvalid);
                else
                    red_add_s64(X + drow.o0 + TID, (long long)__float2ll_rn(v * kFix));
            }
            __syncthreads();
        }
        if (step + 1 < n_steps) {
            if (TID == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue_shared_down(P, C, P.layers[P.layer0 + (step + 1) % P.n_layers]);
            }
            sdown_pending = true;
        }

        // ---------------- 6. routed gate/up -> h_j ----------------
        const int own = W.r1 - W.r0, own_d = W.d1 - W.d0;
        if (W.blob) {
            if (!wait_block(P, C, C.mbar + kWarps, ph_rsc & 1)) {
                ok = false;
                break;
            }
            ++ph_rsc;
            rsc_pending = false;
            bool wok = true;
            // every warp works through its gate/up stages (s = warp, warp + 16, ...)
            #pragma unroll 1
            for (int s = WARP; s < sg.n_gu; s += kWarps) {
                if (!wait_slot(P, C, WARP, ph_slot & 1)) {
                    wok = false;
                    break;
                }
                ++ph_slot;
                slot_pending = 0;
                const uint8_t* slotp = C.ring + (size_t)WARP * sg.slot_bytes;
                const int rc = s % sg.nrc_gu, q = s / sg.nrc_gu, m = q & 1, cb = q >> 1;
                const int rloc0 = rc * sg.SR;
                const int nstaged = min(sg.SR, own - rloc0);
                const uint8_t* sc = C.rsb + (2 * m) * C.span_gu + C.imisc[8 + 2 * m];
                const uint8_t* bi = C.rsb + (2 * m + 1) * C.span_gu + C.imisc[8 + 2 * m + 1];
                const int cpb = sg.cbw_gu / 32;  // chunks per column block
                const int c0 = cb * cpb;
                if (nstaged > 0 && c0 < C.NCu)
                    mma_block<false>(slotp, sg.swz_gu ? 7u : 0u, sg.cbw_gu, nstaged, rloc0, own, c0, min(cpb, C.NCu - c0), 0,
                                     C.sup, 0, C.scs, sc, bi, C.ngu * 2, C.sp + m * sg.ncb_gu + cb, 2 * sg.ncb_gu, C.xp - 1);
                __syncwarp();
                const int s2 = s + kWarps;
                if (s2 < sg.n_stages) {
                    if (LANE == 0) {
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        issue_stage(P, C, W.slot, W.r0, W.d0, s2);
                    }
                    slot_pending = 1;
                }
            }
            if (__syncthreads_or(!wok)) {
                set_status(P.status, kStatusTimeout);
                ok = false;
                break;
            }
        }
        __syncthreads();
        {
            const int hdim = xh_stride(C.I, C.Is);
            unsigned long long* xh = P.xh + (size_t)W.j * hdim;
            if (TID < own) {
                float h = 0.f;
                if (W.blob) {
                    const int ncb = sg.ncb_gu;
                    const float* pg = C.sp + TID * 2 * ncb;
                    float gg = 0.f, vv = 0.f;
                    #pragma unroll 1
                    for (int cb = 0; cb < ncb; ++cb) {
                        gg += pg[cb];
                        vv += pg[ncb + cb];
                    }
                    h = __fdividef(gg, 1.f + __expf(-gg)) * vv;
                }
                st_pair(xh + W.r0 + TID, epoch, h);
            }
            __syncthreads();
            // ---------------- 7. the group's h_j, down rows ----------------
            if (!poll_pairs(limit_cycles(P), P.status, xh, C.I, epoch, hval)) {
                ok = false;
                break;
            }
        }
        if (W.blob) {
            stage_h(C.xp, hval, C.I, C.shj, C.chj);
            bool wok = true;
            const int s_first = sg.n_gu + ((WARP - sg.n_gu % kWarps + kWarps) % kWarps);
            #pragma unroll 1
            for (int s = s_first; s < sg.n_stages; s += kWarps) {
                if (!wait_slot(P, C, WARP, ph_slot & 1)) {
                    wok = false;
                    break;
                }
                ++ph_slot;
                slot_pending = 0;
                const uint8_t* slotp = C.ring + (size_t)WARP * sg.slot_bytes;
                const int sd = s - sg.n_gu, rc = sd % sg.nrc_d, cb = sd / sg.nrc_d;
                const int rloc0 = rc * sg.SR;
                const int nstaged = min(sg.SR, own_d - rloc0);
                const uint8_t* sc = C.rdsb + C.imisc[12];
                const uint8_t* bi = C.rdsb + C.span_d + C.imisc[13];
                const int cpb = sg.cbw_d / 32;
                const int c0 = cb * cpb;
                if (nstaged > 0 && c0 < C.NCd)
                    mma_block<true>(slotp, sg.swz_d ? 7u : 0u, sg.cbw_d, nstaged, rloc0, own_d, c0, min(cpb, C.NCd - c0), 0,
                                    C.shj, C.KD, C.chj, sc, bi, C.ngd * 2, C.spd + cb, sg.ncb_d, C.xp - 1);
                __syncwarp();
                const int s2 = s + kWarps;
                if (s2 < sg.n_stages) {
                    if (LANE == 0) {
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        issue_stage(P, C, W.slot, W.r0, W.d0, s2);
                    }
                    slot_pending = 1;
                }
            }
            if (__syncthreads_or(!wok)) {
                set_status(P.status, kStatusTimeout);
                ok = false;
                break;
            }
            // ---------------- 8. weighted contributions ----------------
            if (TID < own_d) {
                float yj = 0.f;
                #pragma unroll 1
                for (int cb = 0; cb < sg.ncb_d; ++cb)
                    yj += C.spd[TID * sg.ncb_d + cb];
                const float v = C.sel_w[W.j] * yj;
                fence_gpu();
                if (!(fabsf(v) < kFixMax))
                    set_status(P.status, kStatusInvalid);
                else
                    red_add_s64(X + W.d0 + TID, (long long)__float2ll_rn(v * kFix));
            }
        }

        const bool last_of_token = li == P.n_layers - 1;

        // ---------------- 9. layer output ----------------
        if (!grid_barrier(P, C)) {
            ok = false;
            break;
        }
        #pragma unroll 1
        for (int o = 2 * TID; o < C.H; o += 2 * kThreads) {
            long long a, b;
            ld_s64x2(X + o, a, b);
            C.sx[o] = __ll2float_rn(a) * kFixInv;
            C.sx[o + 1] = __ll2float_rn(b) * kFixInv;
        }
        __syncthreads();
        // The next step's accumulator starts from this block's slice of its fp32 input: this
        // layer's output (same token) or the next token's input. These stores reach the other
        // blocks before any of their atomic adds of the next step: the shared-expert h pairs that
        // every block waits for are written after a gpu-scope fence (step 2).
        if (step + 1 < n_steps) {
            long long* Xn = P.xacc + (size_t)((step + 1) & 1) * C.H;
            const bool residual = (P.flags & kResidual) != 0;
            #pragma unroll 1
            for (int o = drow.o0 + TID; o < drow.o1; o += kThreads) {
                float x0 = 0.f;
                if (!last_of_token)
                    x0 = C.sx[o];
                else if (residual)
                    x0 = prenorm ? ((const float*)P.x_in)[(size_t)(t + 1) * C.H + o]
                                 : bf16f(((const uint16_t*)P.x_in)[(size_t)(t + 1) * C.H + o]);
                st_s64(Xn + o, (long long)__float2ll_rn(x0 * kFix));
            }
        }
        if (last_of_token) {
            #pragma unroll 1
            for (int o = drow.o0 + TID; o < drow.o1; o += kThreads)
                P.y_out[(size_t)t * C.H + o] = C.sx[o];
            if (P.trace)
                #pragma unroll 1
                for (int o = drow.o0 + TID; o < drow.o1; o += kThreads)
                    P.trace[((size_t)t * (P.n_layers + 1) + P.n_layers) * C.H + o] = C.sx[o];
        }
    }

    // drain: copies still in flight into this block's shared memory finish before it exits
    {
        const long long t0 = cycles();
        auto drain = [&](uint64_t* m, uint32_t parity) {
            while (!mbar_try(m, parity) && cycles() - t0 < 4 * limit_cycles(P)) {
            }
        };
        if (LANE == 0 && slot_pending)
            drain(C.mbar + WARP, ph_slot & 1);
        if (TID == 0) {
            if (dense_pending)
                drain(C.mbar + kWarps + 1, ph_dense & 1);
            if (sdown_pending)
                drain(C.mbar + kWarps + 2, ph_sdown & 1);
            if (rsc_pending)
                drain(C.mbar + kWarps, ph_rsc & 1);
        }
    }
}

}  // namespace moe
