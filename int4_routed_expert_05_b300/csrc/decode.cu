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
// SM. Per step (token, layer) a block
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

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// int4 pair -> exact bf16 pair: nibbles at bit `sh` and `sh + 16` become 128 + q, then - 128.
__device__ __forceinline__ uint32_t nib2(uint32_t w, int sh)
{
    const uint32_t x = ((w >> sh) & 0x000F000Fu) | 0x43004300u;
    uint32_t r;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(0x3F803F80u), "r"(0xC300C300u));
    return r;
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 64-nibble chunk of a 16-row tile: thread (g, tq) holds 16 nibbles of row g (ra) and of row
// g + 8 (rb); b0/b1 hold the matching 16 activation values in permuted register order.
// c[0] = C[g][2tq], c[1] = C[g][2tq+1], c[2] = C[g+8][2tq], c[3] = C[g+8][2tq+1].
__device__ __forceinline__ void chunk_mma(float (&c)[4], uint2 ra, uint2 rb, uint4 b0, uint4 b1)
{
    c[0] = c[1] = c[2] = c[3] = 0.f;
    mma16816(c, nib2(ra.x, 0), nib2(rb.x, 0), nib2(ra.x, 4), nib2(rb.x, 4), b0.x, b0.y);
    mma16816(c, nib2(ra.x, 8), nib2(rb.x, 8), nib2(ra.x, 12), nib2(rb.x, 12), b0.z, b0.w);
    mma16816(c, nib2(ra.y, 0), nib2(rb.y, 0), nib2(ra.y, 4), nib2(rb.y, 4), b1.x, b1.y);
    mma16816(c, nib2(ra.y, 8), nib2(rb.y, 8), nib2(ra.y, 12), nib2(rb.y, 12), b1.z, b1.w);
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
#pragma unroll
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

struct Ctx {
    int H, E, k, I, Is, xp, KU, NCu, KD, NCd, KDs, NCds, ngu, ngd, ngds, rb_gu, rb_d, rb_ds;
    int G, cta, tid, warp, lane, g, tq;
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
    uint16_t* sup;         // [KU] expanded u, permuted blocks
    float* suc;            // [NCu] chunk sums of u
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
    uint16_t* shs;         // [2][KDs] shared h hi/lo, permuted blocks
    float* suhs;           // [NCds] chunk sums of h_shared
    uint16_t* shj;         // [2][KD] routed h hi/lo, permuted blocks
    float* suhj;           // [NCd]
    float* hv;             // [max(I, Is)] polled h values
    float* sp;             // gate/up partials [rows][2][NCu]
    float* spd;            // down partials [rows][NCd or NCds]
    uint32_t span_gu, span_d, span_sgu, span_sd;  // bytes per staged scale span
};

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
    C.G = gridDim.x;
    C.cta = blockIdx.x;
    C.tid = threadIdx.x;
    C.warp = C.tid >> 5;
    C.lane = C.tid & 31;
    C.g = C.lane >> 2;
    C.tq = C.lane & 3;
    C.sg = P.sg;
    const SmemPlan s = smem_plan(P.H, P.E, P.k, P.I, P.Is, P.bits, C.G);
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
    C.suc = (float*)(base + s.uc);
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
    C.suhs = (float*)(base + s.uhs);
    C.shj = (uint16_t*)(base + s.hj);
    C.suhj = (float*)(base + s.uhj);
    C.hv = (float*)(base + s.hv);
    C.sp = (float*)(base + s.sp);
    C.spd = (float*)(base + s.spd);
    C.span_gu = sb_span_max(C.sg.Rgu, 2 * C.ngu);
    C.span_d = sb_span_max(C.sg.Rd, 2 * C.ngd);
    C.span_sgu = sb_span_max(C.sg.Rs, 2 * C.ngu);
    C.span_sd = sb_span_max(C.sg.Rsd, 2 * C.ngds);
}

__device__ float block_sum(const Ctx& C, float v)
{
    v = warp_sum(v);
    __syncthreads();
    if (C.lane == 0)
        C.red[C.warp] = v;
    __syncthreads();
    if (C.warp == 0) {
        float s = C.lane < kWarps ? C.red[C.lane] : 0.f;
        s = warp_sum(s);
        if (C.lane == 0)
            C.red[32] = s;
    }
    __syncthreads();
    return C.red[32];
}

// Block-uniform time limit check: true once the wait that started at t0 ran past the limit.
__device__ __forceinline__ bool timed_out(const StepParams& P, uint64_t t0)
{
    return __syncthreads_or(threadIdx.x == 0 && globaltimer() - t0 > P.timeout_ns) != 0;
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
    d.e0 = part(C.E, C.G, C.cta);
    d.e1 = part(C.E, C.G, C.cta + 1);
    d.s0 = part(C.Is, C.G, C.cta);
    d.s1 = part(C.Is, C.G, C.cta + 1);
    d.o0 = part(C.H, C.G, C.cta);
    d.o1 = part(C.H, C.G, C.cta + 1);
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
__device__ void issue_dense(const StepParams& P, const Ctx& C, const LayerDesc& L, bool with_router, bool with_shared)
{
    const DenseRows d = dense_rows(C);
    uint64_t* m = C.mbar + kWarps + 1;
    const BlobGeo& gs = P.geo_s;
    const uint64_t secs[4] = {gs.s_off[0], gs.b_off[0], gs.s_off[1], gs.b_off[1]};
    const bool rt = with_router && d.e1 > d.e0;
    const bool sh = with_shared && d.s1 > d.s0;
    // the expected bytes go first: the arrive must not complete the phase before the copies count
    uint32_t bytes = (uint32_t)C.H * 2;
    if (rt)
        bytes += (uint32_t)(d.e1 - d.e0) * C.H * 2;
    if (sh) {
        bytes += 2u * (uint32_t)(d.s1 - d.s0) * C.rb_gu;
        for (int i = 0; i < 4; ++i)
            bytes += span_bytes(L.shared_blob + secs[i], d.s0, d.s1, C.ngu * 2);
    }
    mbar_expect(m, bytes);
    if (rt)
        bulk_g2s(C.srt, L.router + (size_t)d.e0 * C.H, (uint32_t)(d.e1 - d.e0) * C.H * 2, m);
    bulk_g2s(C.swsg, L.shared_gate, (uint32_t)C.H * 2, m);
    if (sh) {
        const uint32_t nq = (uint32_t)(d.s1 - d.s0) * C.rb_gu;
        bulk_g2s(C.sgq, L.shared_blob + gs.q_off[0] + (size_t)d.s0 * C.rb_gu, nq, m);
        bulk_g2s(C.sgq + (size_t)C.sg.Rs * C.rb_gu, L.shared_blob + gs.q_off[1] + (size_t)d.s0 * C.rb_gu, nq, m);
        for (int i = 0; i < 4; ++i) {
            uint32_t off;
            copy_rows(C.ssb + i * C.span_sgu, L.shared_blob + secs[i], d.s0, d.s1, C.ngu * 2, m, &off);
            C.imisc[i] = (int)off;
        }
    }
}

__device__ void issue_shared_down(const StepParams& P, const Ctx& C, const LayerDesc& L)
{
    const DenseRows d = dense_rows(C);
    uint64_t* m = C.mbar + kWarps + 2;
    const BlobGeo& gs = P.geo_s;
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

// Rows staged by TMA in one ring slot. Swizzled: 128-byte rows whose 16-byte chunks are permuted
// by (row & 7) (the 128B swizzle of the tensor map; slots are 1024-byte aligned). Linear: rows of
// `width` bytes one after another.
__device__ __forceinline__ uint2 lds_a(const uint8_t* base, int swz, int width, int R, int byte)
{
    uint32_t off;
    if (swz)
        off = (uint32_t)R * kCb + ((((uint32_t)byte >> 4) ^ ((uint32_t)R & 7u)) << 4) + ((uint32_t)byte & 15u);
    else
        off = (uint32_t)R * width + (uint32_t)byte;
    return *reinterpret_cast<const uint2*>(base + off);
}

// ------------------------------------------------------------------------------------------
// input, u, expanded u
// ------------------------------------------------------------------------------------------

// x (already in sx) -> su (bf16 u), sup (expanded, permuted), suc (chunk sums of u)
__device__ void make_u(const StepParams& P, const Ctx& C, bool prenorm, const uint16_t* u_bits)
{
    const int H = C.H;
    if (prenorm) {
        float ss = 0.f;
        for (int i = C.tid; i < H; i += kThreads)
            ss = fmaf(C.sx[i], C.sx[i], ss);
        ss = block_sum(C, ss);
        const float r = sqrtf(ss / (float)H + 1e-6f);
        for (int i = C.tid; i < H; i += kThreads)
            C.su[i] = f2bf(C.sx[i] / r);
    } else {
        for (int i = C.tid; i < H; i += kThreads)
            C.su[i] = u_bits[i];
    }
    __syncthreads();
    for (int n = C.tid; n < C.KU; n += kThreads) {
        float v = bf16f(C.su[C.xp == 1 ? n : (n >> 1)]);
        if (C.xp == 2 && (n & 1))
            v *= 16.f;
        C.sup[pslot(n)] = f2bf(v);
    }
    const int cpc = kChunk / C.xp;  // codes per chunk
    for (int c = C.warp; c < C.NCu; c += kWarps) {
        float s = 0.f;
        for (int i = C.lane; i < cpc; i += 32)
            s += bf16f(C.su[c * cpc + i]);
        s = warp_sum(s);
        if (C.lane == 0)
            C.suc[c] = s;
    }
    __syncthreads();
}

// h values (fp32, smem or registers already gathered into hv[0..n)) -> hi/lo bf16 permuted + sums
__device__ void stage_h(const Ctx& C, const float* hv, int n, uint16_t* sh, float* suh)
{
    const int KD = n * C.xp;
    uint16_t* hi = sh;
    uint16_t* lo = sh + KD;
    for (int i = C.tid; i < KD; i += kThreads) {
        float v = hv[C.xp == 1 ? i : (i >> 1)];
        if (C.xp == 2 && (i & 1))
            v *= 16.f;
        const uint16_t h = f2bf(v);
        hi[pslot(i)] = h;
        lo[pslot(i)] = f2bf(v - bf16f(h));
    }
    const int cpc = kChunk / C.xp;
    const int nch = KD / kChunk;
    for (int c = C.warp; c < nch; c += kWarps) {
        float s = 0.f;
        for (int i = C.lane; i < cpc; i += 32)
            s += hv[c * cpc + i];
        s = warp_sum(s);
        if (C.lane == 0)
            suh[c] = s;
    }
    __syncthreads();
}

// Poll n epoch-tagged pairs until all carry `epoch`; values -> dst (fp32). Block-uniform.
__device__ bool poll_pairs(const StepParams& P, const Ctx& C, const unsigned long long* src, int n, uint32_t epoch,
                           float* dst)
{
    const uint64_t t0 = globaltimer();
    while (true) {
        int bad = 0;
        for (int e = 2 * C.tid; e < n; e += 2 * kThreads) {
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
        if (timed_out(P, t0)) {
            if (C.tid == 0)
                set_status(P.status, kStatusTimeout);
            return false;
        }
    }
}

// Grid barrier on a monotonically increasing counter (a multiple of the grid between launches).
__device__ bool grid_barrier(const StepParams& P, const Ctx& C)
{
    __syncthreads();
    int ok = 1;
    if (C.tid == 0) {
        const unsigned long long G = gridDim.x;
        unsigned long long ticket;
        asm volatile("atom.add.release.gpu.global.u64 %0, [%1], 1;" : "=l"(ticket) : "l"(P.bar) : "memory");
        const unsigned long long target = (ticket / G + 1) * G;
        const uint64_t t0 = globaltimer();
        uint32_t spins = 0;
        while (true) {
            unsigned long long v;
            asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(P.bar) : "memory");
            if (v >= target)
                break;
            if ((++spins & 31u) == 0 && globaltimer() - t0 > P.timeout_ns) {
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

// Gate/up item of a 16-row tile: rows [R0, R0 + 16) of a staged row set, chunk c (global chunk
// index along the row), matrix m; staged bytes of the chunk start at byte `cbyte` of the staged
// row. Writes sp[(row*2 + m)*NCu + c] for rows r (local index rloc0 + R) < nrows.
__device__ __forceinline__ void gu_item(const Ctx& C, const uint8_t* base, int swz, int width, int R0, int nstaged,
                                        int c, int cbyte, int m, int rloc0, int nrows, const uint8_t* sc,
                                        const uint8_t* bi, int sb_row_b)
{
    const int Ra = R0 + C.g, Rb = Ra + 8;
    const uint2 ra = Ra < nstaged ? lds_a(base, swz, width, Ra, cbyte + 8 * C.tq) : make_uint2(0, 0);
    const uint2 rb = Rb < nstaged ? lds_a(base, swz, width, Rb, cbyte + 8 * C.tq) : make_uint2(0, 0);
    const uint4* bp = reinterpret_cast<const uint4*>(C.sup + kChunk * c + 16 * C.tq);
    float acc[4];
    chunk_mma(acc, ra, rb, bp[0], bp[1]);
    const int gi = c / C.xp;
    if (C.tq < 2) {
        const int R = C.tq == 0 ? Ra : Rb;
        const int r = rloc0 + R;
        if (R < nstaged && r < nrows) {
            const float s = bf16f(*reinterpret_cast<const uint16_t*>(sc + (size_t)r * sb_row_b + 2 * gi));
            const float b = bf16f(*reinterpret_cast<const uint16_t*>(bi + (size_t)r * sb_row_b + 2 * gi));
            C.sp[(r * 2 + m) * C.NCu + c] = fmaf(s, C.tq == 0 ? acc[0] : acc[2], b * C.suc[c]);
        }
    }
}

// Down item: like gu_item, with the h hi/lo pair in the B columns (even columns hi, odd lo).
__device__ __forceinline__ void dn_item(const Ctx& C, const uint8_t* base, int swz, int width, int R0, int nstaged,
                                        int c, int cbyte, int rloc0, int nrows, const uint16_t* sh, const float* suh,
                                        int KD, int NC, const uint8_t* sc, const uint8_t* bi, int sb_row_b)
{
    const int Ra = R0 + C.g, Rb = Ra + 8;
    const uint2 ra = Ra < nstaged ? lds_a(base, swz, width, Ra, cbyte + 8 * C.tq) : make_uint2(0, 0);
    const uint2 rb = Rb < nstaged ? lds_a(base, swz, width, Rb, cbyte + 8 * C.tq) : make_uint2(0, 0);
    const uint4* bp = reinterpret_cast<const uint4*>(sh + (size_t)(C.g & 1) * KD + kChunk * c + 16 * C.tq);
    float acc[4];
    chunk_mma(acc, ra, rb, bp[0], bp[1]);
    const int gi = c / C.xp;
    if (C.tq < 2) {
        const int R = C.tq == 0 ? Ra : Rb;
        const int r = rloc0 + R;
        if (R < nstaged && r < nrows) {
            const float s = bf16f(*reinterpret_cast<const uint16_t*>(sc + (size_t)r * sb_row_b + 2 * gi));
            const float b = bf16f(*reinterpret_cast<const uint16_t*>(bi + (size_t)r * sb_row_b + 2 * gi));
            const float a = C.tq == 0 ? acc[0] + acc[1] : acc[2] + acc[3];
            C.spd[r * NC + c] = fmaf(s, a, b * suh[c]);
        }
    }
}

// ------------------------------------------------------------------------------------------
// routing
// ------------------------------------------------------------------------------------------

// slg (logits) -> sel_idx / sel_w (rank order: larger fp32 logit first, ties -> lower index).
__device__ void topk_select(const StepParams& P, const Ctx& C)
{
    const int E = C.E, k = C.k;
    const int nl = (E + 31) / 32;
    if (C.warp < nl) {
        const int e = 32 * C.warp + C.lane;
        const uint32_t key = e < E ? ord_key(C.slg[e]) : 0u;
        int rank = 0;
        for (int d = 1; d < 32; ++d) {
            const int src = (C.lane + d) & 31;
            const uint32_t o = __shfl_sync(0xffffffffu, key, src);
            rank += (o > key) || (o == key && src < C.lane);
        }
        if (C.lane < k) {
            C.lkey[C.warp * kMaxK + C.lane] = 0u;
            C.lidx[C.warp * kMaxK + C.lane] = 0x7fffffff;
        }
        __syncwarp();
        if (e < E && rank < k) {
            C.lkey[C.warp * kMaxK + rank] = key;
            C.lidx[C.warp * kMaxK + rank] = e;
        }
    }
    __syncthreads();
    if (C.tid < nl * k) {
        const int w = C.tid / k, r = C.tid - (C.tid / k) * k;
        const uint32_t key = C.lkey[w * kMaxK + r];
        const int idx = C.lidx[w * kMaxK + r];
        if (idx != 0x7fffffff) {
            int grank = r;
            for (int w2 = 0; w2 < nl && grank < k; ++w2) {
                if (w2 == w)
                    continue;
                for (int r2 = 0; r2 < k; ++r2) {
                    const uint32_t k2 = C.lkey[w2 * kMaxK + r2];
                    const int i2 = C.lidx[w2 * kMaxK + r2];
                    if (k2 > key || (k2 == key && i2 < idx))
                        ++grank;
                    else
                        break;
                }
            }
            if (grank < k)
                C.sel_idx[grank] = idx;
        }
    }
    __syncthreads();
    if (C.warp == 0) {
        const float lmax = C.slg[C.sel_idx[0]];
        const float p = C.lane < k ? expf(C.slg[C.sel_idx[C.lane]] - lmax) : 0.f;
        float denom = 0.f;
        if (P.flags & kRenorm) {
            for (int j = 0; j < k; ++j)
                denom += __shfl_sync(0xffffffffu, p, j);
        } else {
            float s = 0.f;
            for (int e = C.lane; e < E; e += 32)
                s += expf(C.slg[e] - lmax);
            denom = __shfl_sync(0xffffffffu, warp_sum(s), 0);
        }
        if (C.lane < k)
            C.sel_w[C.lane] = p / denom;
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
__device__ __forceinline__ void issue_stage(const StepParams& P, const Ctx& C, const Routed& W, int s)
{
    const StageGeo& sg = C.sg;
    uint8_t* dst = C.ring + (size_t)(s % kWarps) * sg.slot_bytes;
    uint64_t* m = C.mbar + (s % kWarps);
    if (s < sg.n_gu) {
        const int rc = s % sg.nrc_gu, q = s / sg.nrc_gu, mat = q & 1, cb = q >> 1;
        mbar_expect(m, (uint32_t)sg.SR * sg.cbw_gu);
        tma3d(dst, &P.tmap[mat], cb * sg.cbw_gu, W.r0 + rc * sg.SR, W.slot, m);
    } else {
        const int sd = s - sg.n_gu, rc = sd % sg.nrc_d, cb = sd / sg.nrc_d;
        mbar_expect(m, (uint32_t)sg.SR * sg.cbw_d);
        tma3d(dst, &P.tmap[2], cb * sg.cbw_d, W.d0 + rc * sg.SR, W.slot, m);
    }
}

// Wait for ring slot `slot` to complete phase `parity` (warp-uniform; false after the limit).
__device__ bool wait_slot(const StepParams& P, const Ctx& C, int slot, uint32_t parity)
{
    const uint64_t t0 = globaltimer();
    uint32_t spins = 0;
    while (true) {
        if (__all_sync(0xffffffffu, mbar_try(C.mbar + slot, parity)))
            return true;
        if ((++spins & 15u) == 0 && __any_sync(0xffffffffu, globaltimer() - t0 > P.timeout_ns))
            return false;
    }
}

// Block-uniform wait for a block-level mbarrier (all threads).
__device__ bool wait_block(const StepParams& P, const Ctx& C, uint64_t* m, uint32_t parity)
{
    const uint64_t t0 = globaltimer();
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
    Ctx C;
    make_ctx(P, C, base);
    const StageGeo& sg = C.sg;
    const bool route = P.mode != kModeExperts;
    const bool experts = P.mode != kModeRoute;
    const int n_steps = P.n_tokens * P.n_layers;

    if (C.tid == 0) {
        for (int i = 0; i < kNumMbar; ++i)
            mbar_init(C.mbar + i, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (experts)
            for (int i = 0; i < 3; ++i)
                prefetch_map(&P.tmap[i]);
    }
    __syncthreads();

    // phase counters of the mbarriers (uniform in the block / warp)
    uint32_t ph_dense = 0, ph_sdown = 0, ph_rsc = 0, ph_slot = 0;
    bool dense_pending = false, sdown_pending = false, rsc_pending = false;
    int slot_pending = 0;  // this warp's issued-but-unconsumed stages (at most one per slot)

    if (C.tid == 0) {
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
        for (int o = drow.o0 + C.tid; o < drow.o1; o += kThreads) {
            float x0 = 0.f;
            if (residual)
                x0 = (P.flags & kPrenorm) ? ((const float*)P.x_in)[o] : bf16f(((const uint16_t*)P.x_in)[o]);
            st_s64(P.xacc + o, (long long)__float2ll_rn(x0 * kFix));
        }
        ok = grid_barrier(P, C);
    }

    for (int step = 0; ok && step < n_steps; ++step) {
        const int t = step / P.n_layers, li = step - t * P.n_layers;
        const int l = P.layer0 + li;
        const LayerDesc L = P.layers[l];
        const uint32_t epoch = P.epoch0 + (uint32_t)step;
        long long* X = P.xacc + (size_t)(t & 1) * C.H;
        const bool prenorm = (P.flags & kPrenorm) != 0;

        // ---------------- 1. layer input ----------------
        if (li == 0) {
            if (prenorm) {
                const float* src = (const float*)P.x_in + (size_t)t * C.H;
                for (int i = C.tid; i < C.H; i += kThreads)
                    C.sx[i] = src[i];
            } else {
                const uint16_t* src = (const uint16_t*)P.x_in + (size_t)t * C.H;
                for (int i = C.tid; i < C.H; i += kThreads)
                    C.sx[i] = bf16f(src[i]);
            }
            __syncthreads();
        }
        if (P.trace && C.cta == 0)
            for (int i = C.tid; i < C.H; i += kThreads)
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
            for (int r = C.warp; r < nr; r += kWarps) {
                const uint16_t* row = C.srt + (size_t)r * C.H;
                float acc = 0.f;
                for (int i = 0; i < C.H / 256; ++i) {
                    const uint4 w = *reinterpret_cast<const uint4*>(row + 256 * i + 8 * C.lane);
                    const uint4 x = *reinterpret_cast<const uint4*>(C.su + 256 * i + 8 * C.lane);
                    acc = dot8_bf16(w, x, acc);
                }
                acc = warp_sum(acc);
                if (C.lane == 0) {
                    const int e = drow.e0 + r;
                    if (L.logit_bias)
                        acc += __ldg(L.logit_bias + e);
                    st_pair(P.xlog + e, epoch, acc);
                }
            }
        }
        if (experts) {
            if (C.warp == kWarps - 1) {
                float z = 0.f;
                for (int i = 0; i < C.H / 256; ++i) {
                    const uint4 w = *reinterpret_cast<const uint4*>(C.swsg + 256 * i + 8 * C.lane);
                    const uint4 x = *reinterpret_cast<const uint4*>(C.su + 256 * i + 8 * C.lane);
                    z = dot8_bf16(w, x, z);
                }
                z = warp_sum(z);
                if (C.lane == 0)
                    C.misc[0] = 1.f / (1.f + expf(-z));
            }
            // shared gate/up rows [s0, s1): items (matrix, chunk) over one 16-row tile
            const int ns = drow.s1 - drow.s0;
            if (ns > 0) {
                const int nit = 2 * C.NCu;
                for (int it = C.warp; it < nit; it += kWarps) {
                    const int m = it / C.NCu, c = it - m * C.NCu;
                    const uint8_t* q = C.sgq + (size_t)m * sg.Rs * C.rb_gu;
                    const uint8_t* sc = C.ssb + (2 * m) * C.span_sgu + C.imisc[2 * m];
                    const uint8_t* bi = C.ssb + (2 * m + 1) * C.span_sgu + C.imisc[2 * m + 1];
                    gu_item(C, q, 0, C.rb_gu, 0, ns, c, 32 * c, m, 0, ns, sc, bi, C.ngu * 2);
                }
            }
            __syncthreads();
            if (C.tid < ns) {
                const float* pg = C.sp + (C.tid * 2 + 0) * C.NCu;
                const float* pv = C.sp + (C.tid * 2 + 1) * C.NCu;
                float gg = 0.f, vv = 0.f;
                for (int c = 0; c < C.NCu; ++c) {
                    gg += pg[c];
                    vv += pv[c];
                }
                const float h = gg / (1.f + expf(-gg)) * vv;
                st_pair(P.xh + (size_t)C.k * (C.I > C.Is ? C.I : C.Is) + drow.s0 + C.tid, epoch, h);
            }
        }
        __syncthreads();
        // next step's router rows, shared gate vector and shared gate/up rows
        if (step + 1 < n_steps) {
            if (C.tid == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                const int ln = P.layer0 + (step + 1) % P.n_layers;
                issue_dense(P, C, P.layers[ln], route, experts);
            }
            dense_pending = true;
        }

        // ---------------- 3. routing ----------------
        if (route) {
            if (!poll_pairs(P, C, P.xlog, C.E, epoch, C.slg)) {
                ok = false;
                break;
            }
            topk_select(P, C);
            if (C.cta == 0 && C.tid < C.k) {
                const size_t o = ((size_t)t * P.n_layers + li) * C.k + C.tid;
                if (P.topk_idx)
                    P.topk_idx[o] = C.sel_idx[C.tid];
                if (P.topk_w)
                    P.topk_w[o] = C.sel_w[C.tid];
            }
            if (!experts)
                break;  // a route-only launch has one step
            if (C.tid < C.k) {
                const int s = P.table[(size_t)l * C.E + C.sel_idx[C.tid]];
                C.sel_slot[C.tid] = s;
                if (s < 0)
                    set_status(P.status, kStatusNotResident);
            }
        } else if (C.tid < C.k) {
            C.sel_w[C.tid] = P.topk_w[C.tid];
            C.sel_slot[C.tid] = P.slots[C.tid];
            C.sel_idx[C.tid] = -1;
        }
        __syncthreads();

        // ---------------- 4. routed work of this block: issue its boxes ----------------
        Routed W;
        {
            W.j = grp_of(C.cta, C.G, C.k);
            const int gs0 = grp_start(W.j, C.G, C.k), gs1 = grp_start(W.j + 1, C.G, C.k);
            const int n = gs1 - gs0, mi = C.cta - gs0;
            W.slot = C.sel_slot[W.j];
            W.blob = W.slot >= 0 ? P.arena + (uint64_t)W.slot * P.stride : nullptr;
            W.r0 = part(C.I, n, mi);
            W.r1 = part(C.I, n, mi + 1);
            W.d0 = part(C.H, n, mi);
            W.d1 = part(C.H, n, mi + 1);
        }
        if (W.blob) {
            if (C.warp == 0 && C.lane == 0) {
                // scale / bias rows of the block's gate/up rows and down rows
                uint64_t* m = C.mbar + kWarps;
                const BlobGeo& geo = P.geo;
                const uint64_t secs[6] = {geo.s_off[0], geo.b_off[0], geo.s_off[1], geo.b_off[1], geo.s_off[2], geo.b_off[2]};
                uint32_t bytes = 0;
                for (int i = 0; i < 6; ++i) {
                    const bool dn = i >= 4;
                    bytes += span_bytes(W.blob + secs[i], dn ? W.d0 : W.r0, dn ? W.d1 : W.r1, dn ? C.ngd * 2 : C.ngu * 2);
                }
                mbar_expect(m, bytes);
                for (int i = 0; i < 6; ++i) {
                    const bool dn = i >= 4;
                    uint8_t* dst = dn ? C.rdsb + (i - 4) * C.span_d : C.rsb + i * C.span_gu;
                    uint32_t off;
                    copy_rows(dst, W.blob + secs[i], dn ? W.d0 : W.r0, dn ? W.d1 : W.r1, dn ? C.ngd * 2 : C.ngu * 2, m, &off);
                    C.imisc[8 + i] = (int)off;
                }
            }
            rsc_pending = true;
            if (C.lane == 0 && C.warp < sg.n_stages) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue_stage(P, C, W, C.warp);
            }
            if (C.warp < sg.n_stages)
                slot_pending = 1;
        }

        // ---------------- 5. shared expert down rows ----------------
        float* hval = C.hv;
        if (!poll_pairs(P, C, P.xh + (size_t)C.k * (C.I > C.Is ? C.I : C.Is), C.Is, epoch, hval)) {
            ok = false;
            break;
        }
        stage_h(C, hval, C.Is, C.shs, C.suhs);
        if (!wait_block(P, C, C.mbar + kWarps + 2, ph_sdown & 1)) {
            ok = false;
            break;
        }
        ++ph_sdown;
        sdown_pending = false;
        {
            const int nd = drow.o1 - drow.o0;
            const int ntile = (nd + 15) / 16;
            const int nit = ntile * C.NCds;
            const uint8_t* sc = C.sdsb + C.imisc[4];
            const uint8_t* bi = C.sdsb + C.span_sd + C.imisc[5];
            for (int it = C.warp; it < nit; it += kWarps) {
                const int tile = it / C.NCds, c = it - tile * C.NCds;
                dn_item(C, C.sdq, 0, C.rb_ds, tile * 16, nd, c, 32 * c, 0, nd, C.shs, C.suhs, C.KDs, C.NCds, sc, bi,
                        C.ngds * 2);
            }
            __syncthreads();
            if (C.tid < nd) {
                float ys = 0.f;
                for (int c = 0; c < C.NCds; ++c)
                    ys += C.spd[C.tid * C.NCds + c];
                const float v = C.misc[0] * ys;
                if (!(fabsf(v) < kFixMax))
                    set_status(P.status, kStatusInvalid);
                else
                    red_add_s64(X + drow.o0 + C.tid, (long long)__float2ll_rn(v * kFix));
            }
            __syncthreads();
        }
        if (step + 1 < n_steps) {
            if (C.tid == 0) {
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
            for (int s = C.warp; s < sg.n_gu; s += kWarps) {
                if (!wait_slot(P, C, C.warp, ph_slot & 1)) {
                    wok = false;
                    break;
                }
                ++ph_slot;
                slot_pending = 0;
                const uint8_t* slotp = C.ring + (size_t)C.warp * sg.slot_bytes;
                const int rc = s % sg.nrc_gu, q = s / sg.nrc_gu, m = q & 1, cb = q >> 1;
                const int rloc0 = rc * sg.SR;
                const int nstaged = min(sg.SR, own - rloc0);
                const uint8_t* sc = C.rsb + (2 * m) * C.span_gu + C.imisc[8 + 2 * m];
                const uint8_t* bi = C.rsb + (2 * m + 1) * C.span_gu + C.imisc[8 + 2 * m + 1];
                const int cpb = sg.cbw_gu / 32;  // chunks per column block
                const int ntile = (nstaged + 15) / 16;
                for (int it = 0; it < ntile * cpb; ++it) {
                    const int tile = it / cpb, cl = it - tile * cpb;
                    const int c = cb * cpb + cl;
                    if (c < C.NCu && nstaged > 0)
                        gu_item(C, slotp, sg.swz_gu, sg.cbw_gu, tile * 16, nstaged, c, 32 * cl, m, rloc0, own, sc, bi,
                                C.ngu * 2);
                }
                __syncwarp();
                const int s2 = s + kWarps;
                if (s2 < sg.n_stages) {
                    if (C.lane == 0) {
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        issue_stage(P, C, W, s2);
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
            const int hdim = C.I > C.Is ? C.I : C.Is;
            unsigned long long* xh = P.xh + (size_t)W.j * hdim;
            if (C.tid < own) {
                float h = 0.f;
                if (W.blob) {
                    const float* pg = C.sp + (C.tid * 2 + 0) * C.NCu;
                    const float* pv = C.sp + (C.tid * 2 + 1) * C.NCu;
                    float gg = 0.f, vv = 0.f;
                    for (int c = 0; c < C.NCu; ++c) {
                        gg += pg[c];
                        vv += pv[c];
                    }
                    h = gg / (1.f + expf(-gg)) * vv;
                }
                st_pair(xh + W.r0 + C.tid, epoch, h);
            }
            __syncthreads();
            // ---------------- 7. the group's h_j, down rows ----------------
            if (!poll_pairs(P, C, xh, C.I, epoch, hval)) {
                ok = false;
                break;
            }
        }
        if (W.blob) {
            stage_h(C, hval, C.I, C.shj, C.suhj);
            bool wok = true;
            const int s_first = sg.n_gu + ((C.warp - sg.n_gu % kWarps + kWarps) % kWarps);
            for (int s = s_first; s < sg.n_stages; s += kWarps) {
                if (!wait_slot(P, C, C.warp, ph_slot & 1)) {
                    wok = false;
                    break;
                }
                ++ph_slot;
                slot_pending = 0;
                const uint8_t* slotp = C.ring + (size_t)C.warp * sg.slot_bytes;
                const int sd = s - sg.n_gu, rc = sd % sg.nrc_d, cb = sd / sg.nrc_d;
                const int rloc0 = rc * sg.SR;
                const int nstaged = min(sg.SR, own_d - rloc0);
                const uint8_t* sc = C.rdsb + C.imisc[12];
                const uint8_t* bi = C.rdsb + C.span_d + C.imisc[13];
                const int cpb = sg.cbw_d / 32;
                const int ntile = (nstaged + 15) / 16;
                for (int it = 0; it < ntile * cpb; ++it) {
                    const int tile = it / cpb, cl = it - tile * cpb;
                    const int c = cb * cpb + cl;
                    if (c < C.NCd && nstaged > 0)
                        dn_item(C, slotp, sg.swz_d, sg.cbw_d, tile * 16, nstaged, c, 32 * cl, rloc0, own_d, C.shj,
                                C.suhj, C.KD, C.NCd, sc, bi, C.ngd * 2);
                }
                __syncwarp();
                const int s2 = s + kWarps;
                if (s2 < sg.n_stages) {
                    if (C.lane == 0) {
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        issue_stage(P, C, W, s2);
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
            if (C.tid < own_d) {
                float yj = 0.f;
                for (int c = 0; c < C.NCd; ++c)
                    yj += C.spd[C.tid * C.NCd + c];
                const float v = C.sel_w[W.j] * yj;
                if (!(fabsf(v) < kFixMax))
                    set_status(P.status, kStatusInvalid);
                else
                    red_add_s64(X + W.d0 + C.tid, (long long)__float2ll_rn(v * kFix));
            }
        }

        // next token's accumulator base (ordered before its use by the barrier below)
        const bool last_of_token = li == P.n_layers - 1;
        if (last_of_token && t + 1 < P.n_tokens) {
            long long* Xn = P.xacc + (size_t)((t + 1) & 1) * C.H;
            const bool residual = (P.flags & kResidual) != 0;
            for (int o = drow.o0 + C.tid; o < drow.o1; o += kThreads) {
                float x0 = 0.f;
                if (residual)
                    x0 = prenorm ? ((const float*)P.x_in)[(size_t)(t + 1) * C.H + o]
                                 : bf16f(((const uint16_t*)P.x_in)[(size_t)(t + 1) * C.H + o]);
                st_s64(Xn + o, (long long)__float2ll_rn(x0 * kFix));
            }
        }

        // ---------------- 9. layer output ----------------
        if (!grid_barrier(P, C)) {
            ok = false;
            break;
        }
        for (int o = 2 * C.tid; o < C.H; o += 2 * kThreads) {
            long long a, b;
            ld_s64x2(X + o, a, b);
            C.sx[o] = __ll2float_rn(a) * kFixInv;
            C.sx[o + 1] = __ll2float_rn(b) * kFixInv;
        }
        __syncthreads();
        if (last_of_token) {
            for (int o = drow.o0 + C.tid; o < drow.o1; o += kThreads)
                P.y_out[(size_t)t * C.H + o] = C.sx[o];
            if (P.trace)
                for (int o = drow.o0 + C.tid; o < drow.o1; o += kThreads)
                    P.trace[((size_t)t * (P.n_layers + 1) + P.n_layers) * C.H + o] = C.sx[o];
        }
    }

    // drain: copies still in flight into this block's shared memory finish before it exits
    {
        const uint64_t t0 = globaltimer();
        auto drain = [&](uint64_t* m, uint32_t parity) {
            while (!mbar_try(m, parity) && globaltimer() - t0 < 4 * P.timeout_ns) {
            }
        };
        if (C.lane == 0 && slot_pending)
            drain(C.mbar + C.warp, ph_slot & 1);
        if (C.tid == 0) {
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
