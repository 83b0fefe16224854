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
// SM. A layer at batch 1 moves about 20 MB, a few microseconds of HBM time, so the kernel is built
// around the latency of the layer's all-to-all dependencies (logits -> top-k, h -> down rows,
// output -> next layer) and around what the copy engine charges per copy. The blocks form k + 1
// groups: group j < k serves the routed expert of rank j, group k the shared expert; a block owns
// a slice of its expert's gate/up rows and a slice of its down rows. Per step (token, layer) a block
//   1. waits until the step counter says every block has added its share of the previous step's
//      output (one release add per block and step, one acquire poll per block), reads the output
//      words (coalesced) and forms x and u;
//   2. computes its router rows (staged by bulk copy during the previous step with the layer's
//      slot-table row, logit bias and descriptor) and publishes the logits as epoch-tagged
//      (epoch, value) pairs;
//   3. shared-expert blocks: their gate/up rows (fetched during the previous step) -> h, published;
//      routed blocks: poll the logits and take the top-k (every block, the same result; bounds from
//      the warps' maxima, then at most a short bisection), then issue every byte they read of their
//      expert in one go from the lanes of one warp (launch-time copy plan: gate and up rows in
//      column-block pieces, each on its own mbarrier, down rows, scale spans);
//   4. turn their gate/up rows into h as the pieces land and publish h to their group;
//   5. poll their group's h and compute their down rows;
//   6. add w_j y_j (gamma y_shared for the shared group) into the step's output words: each word
//      collects exactly k + 1 contributions as fixed-point integers with a contribution count in
//      its low byte, so the sum is exact and order independent. The output words rotate over three
//      buffers: a block clears its slice of the next step's buffer, which every block last read
//      two steps before (the step counter orders the clear after those reads and before the next
//      step's adds). Then the block counts the step done and queues the next step's dense copies
//      (and, in the shared group, the next layer's shared rows).
// int4 codes become fp16 values 1024 + q in registers (one lop3 per pair) and meet the activations
// on the tensor cores (mma.m16n8k16, fp32 accumulate), one 64-field chunk at a time; the offset
// and the affine dequantisation are applied per chunk as s * (sum q u) + b * (sum u). Every sum
// runs in a fixed order, so the result depends neither on arrival order nor on pool placement.
// Every wait has an iteration limit: on expiry the block records a timeout status and the launch
// ends (nothing spins forever).
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

__device__ __forceinline__ uint16_t f2h(float v)
{
    __half h = __float2half_rn(v);
    return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(*reinterpret_cast<const __half*>(&b)); }

// Order-preserving map of a float onto uint32 (larger float -> larger key; finite keys > 0).
__device__ __forceinline__ uint32_t ord_key(float f)
{
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// SM cycle counter: waits check their limit on it. A limit of t ns is taken as 2 t cycles (about
// t ns at the 2.03 GHz maximum SM clock, longer at lower clocks).
__device__ __forceinline__ long long cycles() { return clock64(); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

#define TID ((int)threadIdx.x)
#define WARP ((int)threadIdx.x >> 5)
#define LANE ((int)threadIdx.x & 31)
#define CTA ((int)blockIdx.x)
#define GRID ((int)gridDim.x)

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
    const uint32_t w8 = __umulhi(w, 1u << 24);  // w >> 8, as a multiply (off the integer-logic pipe)
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

__device__ __forceinline__ void red_add_u64(long long* p, long long v)
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

__device__ __forceinline__ void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
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

__device__ __forceinline__ void mbar_expect_at(uint32_t m, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(m), "r"(bytes) : "memory");
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

// 4D tiled TMA load (coordinates: byte in the column block, row, column block, slot)
__device__ __forceinline__ void tma4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w, uint64_t* m)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(m))
        : "memory");
}

// The same two copies with the shared-memory addresses given as such.
__device__ __forceinline__ void bulk_g2s_at(uint32_t dst, const void* src, uint32_t bytes, uint32_t m)
{
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(m)
                 : "memory");
}
__device__ __forceinline__ void tma4d_at(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w, uint32_t m)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(m)
        : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ------------------------------------------------------------------------------------------
// per-block context
// ------------------------------------------------------------------------------------------

// Block-uniform constants of a launch: shape, the expert group this block serves, its rows, its
// copies and the shared-memory carve-up. One copy per block in shared memory, written by thread 0
// at start; the phases below copy what they need into registers at their start.
// Division by a launch constant d (1 <= d < 2^16) of x (0 <= x < 2^16): with m = ceil(2^32 / d),
// floor(x * m / 2^32) = floor(x / d) exactly (the error x (m - 2^32 / d) / 2^32 < x / 2^32 < 1 / d
// cannot carry the quotient past the next integer). d = 1 (m = 2^32 does not fit) is m = 0.
__host__ __device__ __forceinline__ uint32_t div_magic(int d)
{
    return d <= 1 ? 0u : (uint32_t)((0x100000000ull + (uint64_t)d - 1) / (uint64_t)d);
}
__device__ __forceinline__ int div_by(int x, uint32_t m) { return m ? (int)__umulhi((uint32_t)x, m) : x; }

// One planned copy of a block's expert bytes: a tile of one of the expert's code maps (b < 0:
// map index in bits 24..30, column-block coordinate in bits 0..23; a: row coordinate) or a span
// of its scale rows (a: byte offset in the blob; b: bytes).
struct CopyOp {
    uint32_t dst;   // shared-memory address
    uint32_t mbar;  // shared-memory address of the copy's mbarrier
    int32_t a, b;
};
static_assert(sizeof(CopyOp) == 16, "one 16-byte load per planned copy");

struct Ctx {
    int H, E, k, I, Is, xp, KU, NCu, ngu;
    int j;            // group rank: the routed expert of rank j (j < k) or the shared expert (j = k)
    int sh;           // 1 when this block serves the shared expert
    int Ie, KD, NCd, ngd;  // intermediate size of the served expert and the derived sizes
    int e0, e1;       // router rows
    int o0, o1;       // the slice of the output words this block clears
    int r0, r1;       // gate/up rows of the served expert
    int d0, d1;       // down rows
    StageGeo g;       // staging geometry of the served expert
    uint32_t sc_src[6], sc_bytes[6];  // scale spans: offset in the blob, bytes (16-byte aligned)
    int sc_off[6];    // offset of the first row inside each span
    float invH;
    uint64_t* mbar;
    int* sel_idx;     // [kMaxK]
    float* sel_w;     // [kMaxK]
    int* sel_slot;    // [kMaxK]
    float* red;       // [64]
    float* misc;      // [32]: [0] gamma
    float* sx;        // [H] layer input x (fp32)
    uint16_t* su;     // [H] u (bf16)
    uint16_t* sup;    // [KU] B operand of u (fp16, permuted blocks)
    float2* scs;      // [NCu] per chunk: sum of u, 1024 * sum of B
    float* slg;       // [E] logits
    uint32_t* tk;     // top-k scratch
    uint16_t* srt;    // [Rr][H] router rows
    uint16_t* swsg;   // [H] shared gate vector
    int32_t* stab;    // the layer's slot-table row (16-byte aligned superset of [E])
    float* sbias;     // the layer's logit bias [E] (when staged)
    LayerDesc* ld;    // [2] layer descriptors of the steps, by step parity
    const LayerDesc* cur;  // the step's
    int tab_off;      // offset (entries) of the row inside stab
    int bias_staged;  // 1: sbias holds the bias, 0: read it from global memory
    uint8_t* ring;    // gate/up slots [nslot][2][nr_gu][gu_copy], then down [nr_d][d_copy]
    uint8_t* rsb;     // 4 spans: gate.s, gate.b, up.s, up.b rows
    uint8_t* rdsb;    // 2 spans: down.s, down.b rows
    uint16_t* shj;    // [2][KD] B operand of h
    float2* chj;      // [NCd]
    float* hv;        // [Ie] polled h values
    float* sp;        // gate/up partials [rows][2 * ncb_gu]
    float* spd;       // down partials [rows][ncb_d]
    float* rp;        // router partials [Rr][kRouterParts]
    uint32_t span_gu, span_d;  // bytes per staged scale span
    // work items of the gate/up and down loops (launch constants; divisors as div_by magics)
    int nrc_gu, per_m;            // gate/up row boxes; items per matrix of a column group
    int nrc_d, tpi_d, ntg_d, n_dn;  // down row boxes, tiles per item, tile groups, items
    uint32_t mg_cpg_gu, mg_cpp_gu, mg_ntg_d, mg_cpg_d;
    CopyOp* cops;     // [kMaxCopies] the copies of one step's expert bytes (planned at launch)
    uint2* cexp;      // [kMaxExpects] their mbarriers {address, bytes expected}
    int ncop, nexp;   // counts (ncop < 0: too many to plan; the copies are issued one by one)
};

static_assert(sizeof(Ctx) <= kCtxBytes, "the block context outgrew its shared-memory slot");

__device__ __noinline__ void make_ctx(const StepParams& P, Ctx& C, uint8_t* base)
{
    C.H = P.H;
    C.E = P.E;
    C.k = P.k;
    C.I = P.I;
    C.Is = P.Is;
    C.xp = P.bits == 8 ? 2 : 1;
    C.KU = P.H * C.xp;
    C.NCu = C.KU / kChunk;
    C.ngu = P.H / 64;
    C.invH = 1.f / (float)P.H;
    const int G = GRID, b = CTA, ng = P.k + 1;
    C.e0 = part(P.E, G, b);
    C.e1 = part(P.E, G, b + 1);
    C.o0 = part(P.H, G, b);
    C.o1 = part(P.H, G, b + 1);
    C.j = grp_of(b, G, ng);
    C.sh = C.j == P.k;
    C.g = C.sh ? P.sgs : P.sg;
    const BlobGeo& bg = C.sh ? P.geo_s : P.geo;
    C.Ie = C.sh ? P.Is : P.I;
    C.KD = C.Ie * C.xp;
    C.NCd = C.KD / kChunk;
    C.ngd = C.Ie / 64;
    const int gi = b - grp_start(C.j, G, ng);
    C.r0 = imin(gi * C.g.SRgu, C.Ie);
    C.r1 = imin(C.r0 + C.g.SRgu, C.Ie);
    C.d0 = imin(gi * C.g.SRd, P.H);
    C.d1 = imin(C.d0 + C.g.SRd, P.H);
    // scale spans of the block's rows: gate.s, gate.b, up.s, up.b, down.s, down.b (blob bases are
    // 16-byte aligned, so the spans' alignment does not depend on the blob)
#pragma unroll 1
    for (int i = 0; i < 6; ++i) {
        const bool d = i >= 4;
        const uint64_t sec = (i & 1) ? bg.b_off[i >> 1] : bg.s_off[i >> 1];
        const int rb = d ? C.ngd * 2 : C.ngu * 2, r0 = d ? C.d0 : C.r0, r1 = d ? C.d1 : C.r1;
        if (r1 <= r0) {
            C.sc_src[i] = C.sc_bytes[i] = 0;
            C.sc_off[i] = 0;
            continue;
        }
        const uint64_t a = sec + (uint64_t)r0 * rb, e = sec + (uint64_t)r1 * rb;
        const uint64_t a16 = a & ~(uint64_t)15, e16 = (e + 15) & ~(uint64_t)15;
        C.sc_src[i] = (uint32_t)a16;
        C.sc_bytes[i] = (uint32_t)(e16 - a16);
        C.sc_off[i] = (int)(a - a16);
    }
    const SmemPlan s = smem_plan(P.H, P.E, P.I, P.Is, P.bits, G, P.sg, P.sgs);
    C.mbar = (uint64_t*)(base + s.mbar);
    int* ctl = (int*)(base + s.ctl);
    C.sel_idx = ctl;
    C.sel_w = (float*)(ctl + kMaxK);
    C.sel_slot = ctl + 2 * kMaxK;
    C.red = (float*)(ctl + 3 * kMaxK);
    C.misc = (float*)(ctl + 3 * kMaxK + 64);
    C.sx = (float*)(base + s.x);
    C.su = (uint16_t*)(base + s.u);
    C.sup = (uint16_t*)(base + s.up);
    C.scs = (float2*)(base + s.uc);
    C.slg = (float*)(base + s.lg);
    C.tk = (uint32_t*)(base + s.tk);
    C.srt = (uint16_t*)(base + s.rt);
    C.swsg = (uint16_t*)(base + s.wsg);
    C.stab = (int32_t*)(base + s.tab);
    C.ld = (LayerDesc*)(base + s.ld);
    C.sbias = (float*)(base + s.bias);
    C.ring = base + s.ring;
    C.rsb = base + s.rsb;
    C.rdsb = base + s.rdsb;
    C.shj = (uint16_t*)(base + s.hj);
    C.chj = (float2*)(base + s.uhj);
    C.hv = (float*)(base + s.hv);
    C.sp = (float*)(base + s.sp);
    C.spd = (float*)(base + s.spd);
    C.rp = (float*)(base + s.rp);
    const int Im = imax(P.I, P.Is);
    C.span_gu = sb_span_max(imax(P.sg.SRgu, P.sgs.SRgu), 2 * C.ngu);
    C.span_d = sb_span_max(imax(P.sg.SRd, P.sgs.SRd), 2 * (Im / 64));
    {
        const StageGeo& g = C.g;
        C.nrc_gu = cdiv(imax(C.r1 - C.r0, 0), g.bh_gu);
        C.per_m = C.nrc_gu * g.cpg_gu;
        C.nrc_d = cdiv(imax(C.d1 - C.d0, 0), g.bh_d);
        const int tb = cdiv(g.bh_d, 16);
        C.tpi_d = imax(1, cdiv(C.nrc_d * g.cpg_d * tb, kWarps));
        C.ntg_d = cdiv(tb, C.tpi_d);
        C.n_dn = C.nrc_d * g.cpg_d * C.ntg_d;
        C.mg_cpg_gu = div_magic(g.cpg_gu);
        C.mg_cpp_gu = div_magic(g.cpp_gu);
        C.mg_ntg_d = div_magic(C.ntg_d);
        C.mg_cpg_d = div_magic(g.cpg_d);
    }
    C.cops = (CopyOp*)(base + s.cp);
    C.cexp = (uint2*)(base + s.cp + 16u * kMaxCopies);
}

// ------------------------------------------------------------------------------------------
// copies
// ------------------------------------------------------------------------------------------

// One thread: what a step reads of layer l besides its experts: the router rows [e0, e1), the
// layer's slot-table row and logit bias (rt), the shared gate vector (wsg), and the descriptor of
// the layer after (ln) into the other descriptor slot. Layer l's descriptor is in slot par: it
// landed with the previous step's copies (or was written at launch).
__device__ __noinline__ void issue_dense(const StepParams& P, Ctx& C, int l, int par, int ln, bool rt, bool wsg)
{
    uint64_t* m = C.mbar + kMbDense;
    const LayerDesc& L = C.ld[par];
    C.cur = &C.ld[par];
    const int H = C.H, E = C.E;
    const bool rr = rt && C.e1 > C.e0;
    uint32_t bytes = (rr ? (uint32_t)(C.e1 - C.e0) * H * 2 : 0u) + (wsg ? (uint32_t)H * 2 : 0u) +
                     (uint32_t)sizeof(LayerDesc);
    // the slot-table row: its 16-byte aligned superset (inside the table's buffer)
    const int32_t* row = P.table + (size_t)l * E;
    const uintptr_t ta = reinterpret_cast<uintptr_t>(row) & ~(uintptr_t)15;
    const uint32_t tb = (uint32_t)(((reinterpret_cast<uintptr_t>(row + E) + 15) & ~(uintptr_t)15) - ta);
    C.tab_off = (int)((reinterpret_cast<uintptr_t>(row) - ta) / 4);
    C.bias_staged = rt && L.logit_bias && (reinterpret_cast<uintptr_t>(L.logit_bias) & 15) == 0 && (E & 3) == 0;
    if (rt)
        bytes += tb + (C.bias_staged ? (uint32_t)E * 4 : 0u);
    mbar_expect(m, bytes);
    bulk_g2s(&C.ld[par ^ 1], P.layers + ln, (uint32_t)sizeof(LayerDesc), m);
    if (rr)
        bulk_g2s(C.srt, L.router + (size_t)C.e0 * H, (uint32_t)(C.e1 - C.e0) * H * 2, m);
    if (wsg)
        bulk_g2s(C.swsg, L.shared_gate, (uint32_t)H * 2, m);
    if (rt) {
        bulk_g2s(C.stab, reinterpret_cast<const void*>(ta), tb, m);
        if (C.bias_staged)
            bulk_g2s(C.sbias, L.logit_bias, (uint32_t)E * 4, m);
    }
}

// Staging address of gate/up copy (slot sl, matrix m, row box rc) and of down copy rc.
__device__ __forceinline__ uint8_t* gu_copy_at(const Ctx& C, int sl, int m, int rc)
{
    return C.ring + (size_t)((sl * 2 + m) * C.g.nr_gu + rc) * C.g.gu_copy;
}
__device__ __forceinline__ uint8_t* d_copy_at(const Ctx& C, int rc)
{
    return C.ring + (size_t)C.g.nslot_gu * 2 * C.g.nr_gu * C.g.gu_copy + (size_t)rc * C.g.d_copy;
}

// Mbarrier bit of gate/up piece p of matrix m in slot sl.
__device__ __forceinline__ int gu_bar(const StageGeo& g, int sl, int m, int p) { return (2 * sl + m) * g.npc_gu + p; }
// Mask of n low bits (n <= 32).
__device__ __forceinline__ uint32_t low_bits(int n) { return n >= 32 ? 0xFFFFFFFFu : (1u << n) - 1u; }

// One thread: the gate (m = 0) or up (m = 1) copy of column group cg of the block's gate/up rows,
// into slot sl, piece by piece; with the matrix's scale and bias rows (on piece 0) when `scales`
// (the first group). maps: the expert's gate/up/down maps; w: the blob's coordinate in them;
// blob: the blob itself.
__device__ __noinline__ void issue_gu(const Ctx& C, const uint8_t* blob, const CUtensorMap* maps, int w, int cg, int sl,
                                      int m, bool scales)
{
    const StageGeo& g = C.g;
    const int nrc = cdiv(C.r1 - C.r0, g.bh_gu);
    const uint32_t pbytes = (uint32_t)g.cbw_gu * g.bh_gu * g.cpp_gu;
#pragma unroll 1
    for (int p = 0; p < g.npc_gu; ++p) {
        uint64_t* mb = C.mbar + gu_bar(g, sl, m, p);
        mbar_expect(mb, (uint32_t)nrc * pbytes + ((scales && p == 0) ? C.sc_bytes[2 * m] + C.sc_bytes[2 * m + 1] : 0u));
#pragma unroll 1
        for (int rc = 0; rc < nrc; ++rc)
            tma4d(gu_copy_at(C, sl, m, rc) + p * pbytes, maps + m, 0, C.r0 + rc * g.bh_gu, cg * g.cpg_gu + p * g.cpp_gu,
                  w, mb);
        if (scales && p == 0)
#pragma unroll 1
            for (int i = 2 * m; i < 2 * m + 2; ++i)
                if (C.sc_bytes[i])
                    bulk_g2s(C.rsb + i * C.span_gu, blob + C.sc_src[i], C.sc_bytes[i], mb);
    }
}

// One thread: every byte the block reads of its expert in a step, gate rows first, then up rows,
// then down rows (the copy engine takes copies in order), each matrix's codes and scales on one
// mbarrier; gate/up rows of the first column groups only when the groups take turns.
__device__ __noinline__ void issue_expert(const Ctx& C, const uint8_t* blob, const CUtensorMap* maps, int w)
{
    const StageGeo& g = C.g;
    if (C.r1 > C.r0)
#pragma unroll 1
        for (int cg = 0; cg < g.nslot_gu; ++cg)
#pragma unroll 1
            for (int m = 0; m < 2; ++m)
                issue_gu(C, blob, maps, w, cg, cg, m, cg == 0);
    if (C.d1 > C.d0) {
        const int nrc = cdiv(C.d1 - C.d0, g.bh_d);
        uint64_t* md = C.mbar + kMbDown;
        mbar_expect(md, (uint32_t)nrc * g.cbw_d * g.bh_d * g.cpg_d + C.sc_bytes[4] + C.sc_bytes[5]);
#pragma unroll 1
        for (int rc = 0; rc < nrc; ++rc)
            tma4d(d_copy_at(C, rc), maps + 2, 0, C.d0 + rc * g.bh_d, 0, w, md);
#pragma unroll 1
        for (int i = 4; i < 6; ++i)
            if (C.sc_bytes[i])
                bulk_g2s(C.rdsb + (i - 4) * C.span_d, blob + C.sc_src[i], C.sc_bytes[i], md);
    }
}

// One thread, at launch: the copies issue_expert makes, as a table (the same for every step but
// for the blob and its coordinate), so that a warp can issue them side by side.
__device__ __noinline__ void plan_copies(Ctx& C)
{
    const StageGeo& g = C.g;
    int nc = 0, ne = 0;
    auto add = [&](uint32_t dst, uint32_t mb, int a, int b) {
        if (nc < kMaxCopies)
            C.cops[nc] = CopyOp{dst, mb, a, b};
        ++nc;
    };
    if (C.r1 > C.r0) {
        // piece by piece, gate and up side by side, so that both matrices land progressively
        const int nrc = cdiv(C.r1 - C.r0, g.bh_gu);
        const uint32_t pbytes = (uint32_t)g.cbw_gu * g.bh_gu * g.cpp_gu;
#pragma unroll 1
        for (int cg = 0; cg < g.nslot_gu; ++cg)
#pragma unroll 1
            for (int p = 0; p < g.npc_gu; ++p)
#pragma unroll 1
                for (int m = 0; m < 2; ++m) {
                    const uint32_t mb = smem_u32(C.mbar + gu_bar(g, cg, m, p));
                    const bool sc = cg == 0 && p == 0;
                    if (ne < kMaxExpects)
                        C.cexp[ne] = make_uint2(mb, (uint32_t)nrc * pbytes +
                                                        (sc ? C.sc_bytes[2 * m] + C.sc_bytes[2 * m + 1] : 0u));
                    ++ne;
#pragma unroll 1
                    for (int rc = 0; rc < nrc; ++rc)
                        add(smem_u32(gu_copy_at(C, cg, m, rc)) + p * pbytes, mb, C.r0 + rc * g.bh_gu,
                            (int)(0x80000000u | ((uint32_t)m << 24) | (uint32_t)(cg * g.cpg_gu + p * g.cpp_gu)));
                    if (sc)
#pragma unroll 1
                        for (int i = 2 * m; i < 2 * m + 2; ++i)
                            if (C.sc_bytes[i])
                                add(smem_u32(C.rsb + i * C.span_gu), mb, (int)C.sc_src[i], (int)C.sc_bytes[i]);
                }
    }
    if (C.d1 > C.d0) {
        const int nrc = cdiv(C.d1 - C.d0, g.bh_d);
        const uint32_t mb = smem_u32(C.mbar + kMbDown);
        if (ne < kMaxExpects)
            C.cexp[ne] = make_uint2(mb, (uint32_t)nrc * g.cbw_d * g.bh_d * g.cpg_d + C.sc_bytes[4] + C.sc_bytes[5]);
        ++ne;
#pragma unroll 1
        for (int rc = 0; rc < nrc; ++rc)
            add(smem_u32(d_copy_at(C, rc)), mb, C.d0 + rc * g.bh_d, (int)(0x80000000u | (2u << 24)));
#pragma unroll 1
        for (int i = 4; i < 6; ++i)
            if (C.sc_bytes[i])
                add(smem_u32(C.rdsb + (i - 4) * C.span_d), mb, (int)C.sc_src[i], (int)C.sc_bytes[i]);
    }
    C.ncop = (nc <= kMaxCopies && ne <= kMaxExpects) ? nc : -1;
    C.nexp = ne;
}

// One warp: every byte the block reads of its expert in a step (blob: the expert's bytes; w: its
// coordinate in maps), the planned copies issued by the lanes side by side; one by one by lane 0
// when the plan did not fit.
__device__ __forceinline__ void issue_expert_warp(const Ctx& C, const uint8_t* blob, const CUtensorMap* maps, int w)
{
    const int nc = C.ncop;
    if (nc < 0) {
        if (LANE == 0)
            issue_expert(C, blob, maps, w);
        return;
    }
#pragma unroll 1
    for (int i = LANE; i < C.nexp; i += 32) {
        const uint2 e = C.cexp[i];
        mbar_expect_at(e.x, e.y);
    }
#pragma unroll 1
    for (int i = LANE; i < nc; i += 32) {
        const CopyOp op = C.cops[i];
        if (op.b < 0)
            tma4d_at(op.dst, maps + ((op.b >> 24) & 0x7F), 0, op.a, op.b & 0xFFFFFF, w, op.mbar);
        else
            bulk_g2s_at(op.dst, blob + (uint32_t)op.a, (uint32_t)op.b, op.mbar);
    }
}

// ------------------------------------------------------------------------------------------
// waits and exchanges
// ------------------------------------------------------------------------------------------

// Block-uniform wait for a block-level mbarrier phase (all threads).
__device__ __forceinline__ bool wait_block(uint64_t* m, uint32_t parity, long long limit, int* status)
{
    const long long t0 = cycles();
    bool ok = true;
    while (!mbar_try(m, parity))
        if (cycles() - t0 > limit) {
            ok = false;
            break;
        }
    if (__syncthreads_or(!ok)) {
        if (TID == 0)
            set_status(status, kStatusTimeout);
        return false;
    }
    return true;
}

// Warp-uniform wait for an mbarrier phase; false after the limit.
__device__ __forceinline__ bool wait_warp(uint64_t* m, uint32_t parity, long long limit)
{
    const long long t0 = cycles();
    while (true) {
        if (__all_sync(0xffffffffu, mbar_try(m, parity)))
            return true;
        if (__any_sync(0xffffffffu, cycles() - t0 > limit))
            return false;
    }
}

// Poll n epoch-tagged pairs until each carries `epoch`; values -> dst (fp32). Each thread spins on
// its own 16-byte pieces, so only stale pieces are read again (a pair carries its own value: no
// ordering beyond the pair is needed). Block-uniform.
__device__ __forceinline__ bool poll_pairs(const unsigned long long* src, int n, uint32_t epoch, float* dst,
                                        long long limit, int* status)
{
    const long long t0 = cycles();
    bool ok = true;
#pragma unroll 1
    for (int e = 2 * TID; ok && e < n; e += 2 * kThreads) {
        unsigned long long a, b;
        while (true) {
            ld_pair2(src + e, a, b);
            if ((uint32_t)(a >> 32) == epoch && (e + 1 >= n || (uint32_t)(b >> 32) == epoch))
                break;
            if (cycles() - t0 > limit) {
                ok = false;
                break;
            }
        }
        dst[e] = __uint_as_float((uint32_t)a);
        if (e + 1 < n)
            dst[e + 1] = __uint_as_float((uint32_t)b);
    }
    if (__syncthreads_or(!ok)) {
        if (TID == 0)
            set_status(status, kStatusTimeout);
        return false;
    }
    return true;
}

// Wait until the step counter (one release-add per block and step) reaches `target` (thread 0
// polls it with acquire loads; the block then reads what every counted block stored before its
// add). Block-uniform.
__device__ __forceinline__ bool wait_steps(const unsigned long long* counter, unsigned long long target,
                                           long long limit, int* status)
{
    bool ok = true;
    if (TID == 0) {
        const long long t0 = cycles();
        while (true) {
            unsigned long long v;
            asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(counter) : "memory");
            if (v >= target)
                break;
            if (cycles() - t0 > limit) {
                ok = false;
                break;
            }
        }
    }
    if (__syncthreads_or(!ok)) {
        if (TID == 0)
            set_status(status, kStatusTimeout);
        return false;
    }
    return true;
}

// Output words of element pairs qa and qb (16 bytes each) once each holds `want` contributions
// (the two loads go out together); false after the limit. A warp reading pairs q0 + lane reads
// 512 contiguous bytes: one request per 128-byte line.
__device__ __forceinline__ bool poll_out2x2(const long long* X, int qa, int qb, bool hb, int want, long long t0,
                                            long long limit, float2& ya, float2& yb)
{
    long long v[4] = {0, 0, 0, 0};
    while (true) {
        ld_s64x2(X + 2 * qa, v[0], v[1]);
        if (hb)
            ld_s64x2(X + 2 * qb, v[2], v[3]);
        const bool all = (int)(v[0] & 0xFF) == want && (int)(v[1] & 0xFF) == want &&
                         (!hb || ((int)(v[2] & 0xFF) == want && (int)(v[3] & 0xFF) == want));
        if (all)
            break;
        if (cycles() - t0 > limit)
            return false;
    }
    ya = make_float2(__ll2float_rn(v[0] >> kCountBits) * kFixInv, __ll2float_rn(v[1] >> kCountBits) * kFixInv);
    yb = make_float2(__ll2float_rn(v[2] >> kCountBits) * kFixInv, __ll2float_rn(v[3] >> kCountBits) * kFixInv);
    return true;
}

// One contribution v to output word p (count + 1, value in fixed point).
__device__ __forceinline__ void add_out(long long* p, float v, int* status)
{
    long long fx = 0;
    if (fabsf(v) < kFixMax)
        fx = __float2ll_rn(v * kFix);
    else
        set_status(status, kStatusInvalid);
    red_add_u64(p, (long long)((unsigned long long)fx << kCountBits) + 1);
}

// Launch-start barrier on a monotonically increasing counter (a multiple of the grid between
// launches).
__device__ __noinline__ bool grid_barrier(const StepParams& P, long long limit)
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
            if (cycles() - t0 > limit) {
                ok = 0;
                set_status(P.status, kStatusTimeout);
                break;
            }
        }
    }
    return __syncthreads_or(!ok) == 0;
}

// ------------------------------------------------------------------------------------------
// the GEMV tiles
// ------------------------------------------------------------------------------------------

// One 16-row tile: A fragments of the nch chunks (rows Ra, Rb present when ha / hb), scales sv / bv
// of the thread's row, the four MMA chains, and the thread's row partial.
__device__ __forceinline__ float tile_mma(uint32_t aa, uint32_t ab, bool ha, bool hb, int nch, const uint32_t (&off)[4],
                                          const uint4 (&Bx)[4], const uint4 (&By)[4], const float2 (&cs)[4],
                                          const float (&sv)[4], const float (&bv)[4], int gsh, bool lo, int tq)
{
    uint2 ra[4], rb[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const bool on = c < nch;
        ra[c] = (on && ha) ? lds64(aa + off[c]) : make_uint2(0, 0);
        rb[c] = (on && hb) ? lds64(ab + off[c]) : make_uint2(0, 0);
    }
    float acc[4][4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
        acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
    // first 32 fields of each chunk, then the second 32: four independent chains
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t a[4], b[4];
        deq8(ra[c].x, a);
        deq8(rb[c].x, b);
        mma_f16(acc[c], a[0], b[0], a[1], b[1], Bx[c].x, Bx[c].y);
        mma_f16(acc[c], a[2], b[2], a[3], b[3], Bx[c].z, Bx[c].w);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t a[4], b[4];
        deq8(ra[c].y, a);
        deq8(rb[c].y, b);
        mma_f16(acc[c], a[0], b[0], a[1], b[1], By[c].x, By[c].y);
        mma_f16(acc[c], a[2], b[2], a[3], b[3], By[c].z, By[c].w);
    }
    float part = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float v = tq == 0 ? acc[c][0] : acc[c][2];
        if (lo)
            v += tq == 0 ? acc[c][1] : acc[c][3];
        part = fmaf(sv[c >> gsh], v - cs[c].y, fmaf(bv[c >> gsh], cs[c].x, part));
    }
    return part;
}

// Tiles [t0, t1) (16 rows each) of one staged column block, of which rows [0, nvalid) are real: row
// R at base + R * width. With swz = 7 the rows are 128-byte swizzled TMA rows (16-byte piece q of
// a row at shared address bits 7..9 XOR q; the copy's destination is 1024-byte aligned); with
// swz = 0 they are linear. Chunks c0 .. c0 + nch - 1 (nch <= 4) of the B operand start at byte
// 32 (cofs + c - c0) of a row. For each real row R this writes out[R * ostride] = sum over the
// chunks (in chunk order) of s * (sum q v) + b * (sum v), with v the activation: the B operand
// `bsrc` (lo_off = 0: u, every column the same) or h (lo_off = KD: hi parts in the even columns, lo
// parts at bsrc + KD in the odd ones). Scales: sc / bi + R * sbrow, one bf16 per group (a group is
// one chunk at int4, two at int8: gsh). The B fragments and chunk sums are loaded once for all
// tiles; the chunks run as independent MMA chains. Rows g and g + 8 of every tile share one
// swizzle key (a tile is 16 rows), so each thread's four piece offsets are fixed for the call.
__device__ __forceinline__ void box_mma(const uint8_t* base, uint32_t swz, int width, int nvalid, int t0, int t1,
                                        int c0, int nch, const uint16_t* bsrc, int lo_off, const float2* csum,
                                        const uint8_t* sc, const uint8_t* bi, int sbrow, int gsh, float* out,
                                        int ostride, int cofs = 0)
{
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    const uint16_t* bb = bsrc + (size_t)(g & 1) * lo_off;
    const uint32_t b0 = smem_u32(base);
    uint4 Bx[4], By[4];
    float2 cs[4];
    uint32_t off[4];
    const uint32_t key = ((b0 >> 7) + (uint32_t)(t0 * 16 + g) * ((uint32_t)width >> 7)) & swz;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int cc = c0 + (c < nch ? c : 0);
        const uint4* bp = reinterpret_cast<const uint4*>(bb + kChunk * cc + 16 * tq);
        Bx[c] = bp[0];
        By[c] = bp[1];
        cs[c] = csum[cc];
        off[c] = ((((uint32_t)(2 * (cofs + c) + (tq >> 1))) ^ key) << 4) | (uint32_t)(8 * (tq & 1));
    }
    const int nsc = (nch + (1 << gsh) - 1) >> gsh;  // scale groups the chunks touch
    const int q0 = c0 >> gsh;
    // 8-byte scale loads when the four groups of every row are 8-byte aligned
    const bool vec = gsh == 0 && nch == 4 && ((reinterpret_cast<uintptr_t>(sc) | reinterpret_cast<uintptr_t>(bi) |
                                               (uintptr_t)sbrow | (uintptr_t)(2 * q0)) & 7) == 0;
#pragma unroll 1
    for (int tile = t0; tile < t1; ++tile) {
        const int Ra = tile * 16 + g, Rb = Ra + 8;
        const int R = tq == 0 ? Ra : Rb;
        const bool mine = tq < 2 && R < nvalid;
        const uint32_t aa = b0 + (uint32_t)Ra * (uint32_t)width, ab = aa + 8u * (uint32_t)width;
        float sv[4], bv[4];
        if (vec) {
            uint2 s2 = make_uint2(0, 0), b2 = make_uint2(0, 0);
            if (mine) {
                s2 = *reinterpret_cast<const uint2*>(sc + R * sbrow + 2 * q0);
                b2 = *reinterpret_cast<const uint2*>(bi + R * sbrow + 2 * q0);
            }
            sv[0] = __uint_as_float(s2.x << 16);
            sv[1] = __uint_as_float(s2.x & 0xFFFF0000u);
            sv[2] = __uint_as_float(s2.y << 16);
            sv[3] = __uint_as_float(s2.y & 0xFFFF0000u);
            bv[0] = __uint_as_float(b2.x << 16);
            bv[1] = __uint_as_float(b2.x & 0xFFFF0000u);
            bv[2] = __uint_as_float(b2.y << 16);
            bv[3] = __uint_as_float(b2.y & 0xFFFF0000u);
        } else {
            const uint16_t* sp = reinterpret_cast<const uint16_t*>(sc + R * sbrow) + q0;
            const uint16_t* bp = reinterpret_cast<const uint16_t*>(bi + R * sbrow) + q0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool on = mine && q < nsc;
                sv[q] = on ? bf16f(sp[q]) : 0.f;
                bv[q] = on ? bf16f(bp[q]) : 0.f;
            }
        }
        float part;
        if (tile * 16 + 16 <= nvalid && nch == 4)  // a full tile: no per-load checks
            part = tile_mma(aa, ab, true, true, 4, off, Bx, By, cs, sv, bv, gsh, lo_off != 0, tq);
        else
            part = tile_mma(aa, ab, Ra < nvalid, Rb < nvalid, nch, off, Bx, By, cs, sv, bv, gsh, lo_off != 0, tq);
        if (mine)
            out[R * ostride] = part;
    }
}

// ------------------------------------------------------------------------------------------
// layer input, u, h operands
// ------------------------------------------------------------------------------------------

// The B operand of a chunk: fp16 activations in the MMA's register order (pslot).

// Eight fp16 B entries of elements [8o, 8o + 8) in pslot order (see put_b8): int4 at positions [8o, 8o + 8) in the order 0,4,1,5,2,6,3,7;
// int8 (two fields per code) at [16o, 16o + 16).
__device__ __forceinline__ void store_b8(uint16_t* __restrict__ bop, int xp, int o, const uint32_t (&hb)[8])
{
    if (xp == 1) {
        reinterpret_cast<uint4*>(bop)[o] = make_uint4(hb[0] | (hb[4] << 16), hb[1] | (hb[5] << 16), hb[2] | (hb[6] << 16),
                                                      hb[3] | (hb[7] << 16));
    } else {
        const uint32_t w0 = hb[0] | (hb[2] << 16), w1 = hb[1] | (hb[3] << 16), w2 = hb[4] | (hb[6] << 16),
                       w3 = hb[5] | (hb[7] << 16);
        reinterpret_cast<uint4*>(bop)[2 * o] = make_uint4(w0, w0, w1, w1);
        reinterpret_cast<uint4*>(bop)[2 * o + 1] = make_uint4(w2, w2, w3, w3);
    }
}

// The B operand entries of the eight activations v of elements [8o, 8o + 8) and their chunk-sum
// contributions {sum v, sum B}. For int4 the odd fields of a code word enter A multiplied by 16,
// so their activations are divided by 16; an int8 code is read as two fields (low, 16 x high),
// both paired with the code's activation.
__device__ __forceinline__ float2 put_b8(uint16_t* __restrict__ bop, int xp, int o, const float (&v)[8])
{
    float us = 0.f, bs = 0.f;
    uint32_t hb[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        us += v[j];
        hb[j] = f2h((xp == 1 && (j & 1)) ? v[j] * 0.0625f : v[j]);
        bs += h2f((uint16_t)hb[j]);
    }
    store_b8(bop, xp, o, hb);
    return make_float2(us, xp == 1 ? bs : 2.f * bs);
}

// Chunk sums of a chunk whose elements are held by lpc consecutive lanes.
__device__ __forceinline__ float2 chunk_reduce(float2 v, int lpc)
{
#pragma unroll 1
    for (int o = lpc / 2; o; o >>= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
    }
    return v;
}

// Layer input of a step. When the previous step exists, waits for its output words (want
// contributions each) and forms its output xo = (x if residual) + y. x becomes xo, or the next
// token's input x_in (fp32, or bf16 bits) when `fresh`. Block 0 writes xo to out_prev (the
// previous token's output, when non-null) and to trace_prev, and x to trace_cur. Then u =
// bf16(x / rms(x)) (norm), bf16(x) (from_x) or the bf16 input bits as given, its B operand and
// chunk sums. x is formed in element pairs (coalesced reads of the output words), u and its B
// operand from 8 consecutive elements per thread. Block-uniform; false (status set) after the
// limit.
__device__ __forceinline__ bool layer_input(const Ctx& C, const long long* Xprev, int want, bool residual, bool fresh,
                                            const void* x_in, bool in_f32, bool from_x, bool norm, float* out_prev,
                                            float* trace_prev, float* trace_cur, long long limit, int* status)
{
    const int H = C.H, xp = C.xp, n8 = H / 8;
    const float4* sx = reinterpret_cast<const float4*>(C.sx);
    uint16_t* __restrict__ su = C.su;
    uint16_t* __restrict__ bop = C.sup;
    float2* __restrict__ scs = C.scs;
    float* __restrict__ red = C.red;
    const bool w0 = CTA == 0;
    const long long t0 = cycles();
    bool ok = true;
    float ss = 0.f;
    // element pairs: thread TID takes pairs q0 + TID and q0 + kThreads + TID (coalesced)
    float2* sx2 = reinterpret_cast<float2*>(C.sx);
    const int n2 = H / 2;
#pragma unroll 1
    for (int q0 = 0; q0 < n2; q0 += 2 * kThreads) {
        const int qa = q0 + TID, qb = qa + kThreads;
        if (qa >= n2)
            break;
        const bool hb = qb < n2;
        float2 xa = sx2[qa], xb = hb ? sx2[qb] : make_float2(0.f, 0.f);
        if (Xprev) {
            float2 ya, yb;
            if (!poll_out2x2(Xprev, qa, qb, hb, want, t0, limit, ya, yb)) {
                ok = false;
                break;
            }
            xa = residual ? make_float2(xa.x + ya.x, xa.y + ya.y) : ya;
            xb = residual ? make_float2(xb.x + yb.x, xb.y + yb.y) : yb;
            if (w0 && out_prev) {
                reinterpret_cast<float2*>(out_prev)[qa] = xa;
                if (hb)
                    reinterpret_cast<float2*>(out_prev)[qb] = xb;
            }
            if (w0 && trace_prev) {
                reinterpret_cast<float2*>(trace_prev)[qa] = xa;
                if (hb)
                    reinterpret_cast<float2*>(trace_prev)[qb] = xb;
            }
        }
        if (fresh) {
            if (in_f32) {
                xa = reinterpret_cast<const float2*>(x_in)[qa];
                if (hb)
                    xb = reinterpret_cast<const float2*>(x_in)[qb];
            } else {
                const uint32_t ba = reinterpret_cast<const uint32_t*>(x_in)[qa];
                xa = make_float2(bf16f((uint16_t)ba), bf16f((uint16_t)(ba >> 16)));
                if (hb) {
                    const uint32_t bb = reinterpret_cast<const uint32_t*>(x_in)[qb];
                    xb = make_float2(bf16f((uint16_t)bb), bf16f((uint16_t)(bb >> 16)));
                }
            }
        }
        sx2[qa] = xa;
        if (hb)
            sx2[qb] = xb;
        if (w0 && trace_cur) {
            reinterpret_cast<float2*>(trace_cur)[qa] = xa;
            if (hb)
                reinterpret_cast<float2*>(trace_cur)[qb] = xb;
        }
        ss = fmaf(xa.x, xa.x, fmaf(xa.y, xa.y, ss));
        if (hb)
            ss = fmaf(xb.x, xb.x, fmaf(xb.y, xb.y, ss));
    }
    if (__syncthreads_or(!ok)) {
        if (TID == 0)
            set_status(status, kStatusTimeout);
        return false;
    }
    float rinv = 1.f;
    if (norm) {
        ss = warp_sum(ss);
        if ((TID & 31) == 0)
            red[TID >> 5] = ss;
        __syncthreads();
        const float4* r4 = reinterpret_cast<const float4*>(red);
        const float4 a = r4[0], b = r4[1], c = r4[2], d = r4[3];
        const float tot = ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w)) + ((c.x + c.y) + (c.z + c.w)) +
                          ((d.x + d.y) + (d.z + d.w));
        rinv = rsqrtf(tot * C.invH + 1e-6f);
    }
    const int lsh = 4 - xp, lpc = 1 << lsh;  // lanes per chunk (a chunk is 64 fields): 8 at int4, 4 at int8
    bool big = false;
    // every lane of a warp runs every iteration: the chunk sums are shuffled across lanes
#pragma unroll 1
    for (int o0 = 0; o0 < n8; o0 += kThreads) {
        const int o = o0 + TID;
        const bool on = o < n8;
        float2 part = make_float2(0.f, 0.f);
        if (on) {
            const float4 x0 = sx[2 * o], x1 = sx[2 * o + 1];
            uint16_t ub[8];
            if (from_x) {
                const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    ub[j] = f2bf(xs[j] * rinv);
            } else {
                const uint4 bits = reinterpret_cast<const uint4*>(x_in)[o];
                const uint32_t bw[4] = {bits.x, bits.y, bits.z, bits.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ub[2 * j] = (uint16_t)bw[j];
                    ub[2 * j + 1] = (uint16_t)(bw[j] >> 16);
                }
            }
            reinterpret_cast<uint4*>(su)[o] =
                make_uint4((uint32_t)ub[0] | ((uint32_t)ub[1] << 16), (uint32_t)ub[2] | ((uint32_t)ub[3] << 16),
                           (uint32_t)ub[4] | ((uint32_t)ub[5] << 16), (uint32_t)ub[6] | ((uint32_t)ub[7] << 16));
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v[j] = bf16f(ub[j]);
                big |= !(fabsf(v[j]) <= 65504.f);  // the fp16 B operand would overflow
            }
            part = put_b8(bop, xp, o, v);
        }
        const float2 cs = chunk_reduce(part, lpc);
        if (on && (o & (lpc - 1)) == 0)
            scs[o >> lsh] = make_float2(cs.x, 1024.f * cs.y);
    }
    if (big)
        set_status(status, kStatusRange);
    __syncthreads();
    return true;
}

// h values hv[0, n) -> B operand hi/lo parts (sh: [2][n * xp]) and per chunk {sum of h, 1024 *
// sum of (hi + lo)}; hi + lo carries h to about 22 bits. Each thread takes 8 consecutive values.
__device__ __forceinline__ void stage_h(int xp, const float* __restrict__ hv, int n, uint16_t* __restrict__ sh,
                                        float2* __restrict__ chs, int* status)
{
    bool big = false;
    const int n8 = n >> 3, lsh = 4 - xp, lpc = 1 << lsh;
    uint16_t* __restrict__ hi = sh;
    uint16_t* __restrict__ lo = sh + n * xp;
    // every lane of a warp runs every iteration: the chunk sums are shuffled across lanes
#pragma unroll 1
    for (int o0 = 0; o0 < n8; o0 += kThreads) {
        const int o = o0 + TID;
        const bool on = o < n8;
        float hs = 0.f, bs = 0.f;
        if (on) {
            const float4 a = reinterpret_cast<const float4*>(hv)[2 * o], b = reinterpret_cast<const float4*>(hv)[2 * o + 1];
            const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint32_t hb[8], lb[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                hs += v[j];
                big |= !(fabsf(v[j]) <= 65504.f);  // the fp16 hi part would overflow
                const float e = (xp == 1 && (j & 1)) ? v[j] * 0.0625f : v[j];
                hb[j] = f2h(e);
                lb[j] = f2h(e - h2f((uint16_t)hb[j]));
                bs += h2f((uint16_t)hb[j]) + h2f((uint16_t)lb[j]);
            }
            if (xp == 2)
                bs *= 2.f;
            store_b8(hi, xp, o, hb);
            store_b8(lo, xp, o, lb);
        }
        const float2 cs = chunk_reduce(make_float2(hs, bs), lpc);
        if (on && (o & (lpc - 1)) == 0)
            chs[o >> lsh] = make_float2(cs.x, 1024.f * cs.y);
    }
    if (big)
        set_status(status, kStatusRange);
    __syncthreads();
}

// ------------------------------------------------------------------------------------------
// routing
// ------------------------------------------------------------------------------------------

// This block's router rows -> logits, published as epoch-tagged pairs. Each row's dot product is
// cut into kRouterParts fixed parts (one warp each, lane-strided bf16 FMAs, butterfly sum) added
// in part order, so a logit does not depend on the grid.
__device__ __forceinline__ void router_rows(const Ctx& C, unsigned long long* xlog, uint32_t epoch)
{
    const int nr = C.e1 - C.e0, H = C.H, e0 = C.e0;
    const uint16_t* __restrict__ srt = C.srt;
    const uint16_t* __restrict__ su = C.su;
    float* __restrict__ rp = C.rp;
    const int nv = H / 8;  // 16-byte vectors per row
#pragma unroll 1
    for (int it = WARP; it < nr * kRouterParts; it += kWarps) {
        const int r = it / kRouterParts, p = it - r * kRouterParts;
        const uint16_t* row = srt + (size_t)r * H;
        const int v1 = part(nv, kRouterParts, p + 1);
        float acc = 0.f;
#pragma unroll 2
        for (int v = part(nv, kRouterParts, p) + LANE; v < v1; v += 32)
            acc = dot8_bf16(*reinterpret_cast<const uint4*>(row + 8 * v), *reinterpret_cast<const uint4*>(su + 8 * v),
                            acc);
        acc = warp_sum(acc);
        if (LANE == 0)
            rp[it] = acc;
    }
    __syncthreads();
    if (TID < nr) {
        const float4 p4 = reinterpret_cast<const float4*>(rp)[TID];
        float bias = 0.f;
        if (C.cur->logit_bias)
            bias = C.bias_staged ? C.sbias[e0 + TID] : __ldg(C.cur->logit_bias + e0 + TID);
        st_pair(xlog + e0 + TID, epoch, (((p4.x + p4.y) + p4.z) + p4.w) + bias);
    }
}

// One warp: the combine weights of the ranked selection sel_idx (softmax over the k selected
// logits with renorm, else over all E).
__device__ __forceinline__ void topk_weights(const Ctx& C, bool renorm)
{
    const int E = C.E, k = C.k;
    const float* __restrict__ slg = C.slg;
    const int isel = LANE < k ? C.sel_idx[LANE] : 0;
    const float lsel = LANE < k ? slg[isel] : 0.f;
    const float lmax = __shfl_sync(0xffffffffu, lsel, 0);
    const float pj = LANE < k ? __expf(lsel - lmax) : 0.f;
    float denom;
    if (renorm) {
        denom = warp_sum(pj);
    } else {
        float sum = 0.f;
#pragma unroll 1
        for (int e2 = LANE; e2 < E; e2 += 32)
            sum += __expf(slg[e2] - lmax);
        denom = warp_sum(sum);
    }
    if (LANE < k)
        C.sel_w[LANE] = __fdividef(pj, denom);
}

// slg (logits) -> sel_idx / sel_w / sel_slot (rank order: larger fp32 logit first, equal logits ->
// lower index). Thread e holds expert e's order-preserving key. Bounds first: the k-th largest of
// the warps' maximum keys is a lower bound lo with at least k keys >= lo (k warps hold one), and
// one past the largest key an upper bound hi with none. While more than 32 keys are >= lo, a
// bisection of [lo, hi) on the key value (one block-wide count per step) raises lo, ending at the
// k-th largest key itself at worst. The keys >= lo hold the top k; they are gathered and each is
// ranked by counting the larger ones (composite keys: the logit key above, the complement of the
// index below, so that equal logits rank by index). slots: look the selected experts' pool slots up
// in the staged slot-table row. The combine weights are left to topk_weights (needed only when
// the block adds its output, so they are computed off the path to the expert copies).
__device__ __forceinline__ void topk_select(const Ctx& C, bool slots)
{
    const int E = C.E, k = C.k;
    int* __restrict__ scnt = reinterpret_cast<int*>(C.tk);                                     // [1]
    unsigned long long* __restrict__ skey = reinterpret_cast<unsigned long long*>(C.tk + 4);  // [E]
    uint32_t* __restrict__ wmax = C.tk + 4 + 2 * kMaxE;                                        // [kWarps]
    const int e = TID;
    const bool valid = e < E;
    const uint32_t key = valid ? ord_key(C.slg[e]) : 0u;
    const int nl = (E + 31) / 32;  // warps holding keys
    if (WARP < nl) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, key);
        if (LANE == 0)
            wmax[WARP] = m;
    }
    if (TID == 0)
        *scnt = 0;
    __syncthreads();
    // every warp alike: the largest maximum, and the k-th largest (equal maxima ranked by warp)
    unsigned long long hi;
    uint32_t lo = 0;
    {
        const uint32_t mine = LANE < nl ? wmax[LANE] : 0u;
        int rank = 0;
#pragma unroll
        for (int i = 0; i < kWarps; ++i) {
            const uint32_t o = wmax[i];
            rank += i < nl && (o > mine || (o == mine && i < LANE));
        }
        hi = (unsigned long long)__reduce_max_sync(0xffffffffu, mine) + 1ull;
        const unsigned at = __ballot_sync(0xffffffffu, LANE < nl && rank == k - 1);
        if (nl >= k && at)
            lo = __shfl_sync(0xffffffffu, mine, __ffs(at) - 1);
    }
    int ns = __syncthreads_count(valid && key >= lo);
#pragma unroll 1
    while (ns > 32 && hi - lo > 1ull) {
        const uint32_t mid = (uint32_t)(lo + (hi - lo) / 2);
        const int c = __syncthreads_count(valid && key >= mid);
        if (c >= k) {
            lo = mid;
            ns = c;
        } else {
            hi = mid;
        }
    }
    if (valid && key >= lo)
        skey[atomicAdd(scnt, 1)] = ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)e);
    __syncthreads();
    if (ns <= 32) {
        if (WARP == 0) {
            if (LANE < ns) {
                const unsigned long long mine = skey[LANE];
                int rank = 0;
#pragma unroll 4
                for (int q = 0; q < ns; ++q)
                    rank += skey[q] > mine;
                if (rank < k)
                    C.sel_idx[rank] = (int)(0xFFFFFFFFu - (uint32_t)mine);
            }
            __syncwarp();
            if (LANE < k)
                C.sel_slot[LANE] = slots ? C.stab[C.tab_off + C.sel_idx[LANE]] : -1;
        }
    } else {
        // many equal keys at the k-th: every survivor ranked by its own thread
        if (TID < ns) {
            const unsigned long long mine = skey[TID];
            int rank = 0;
#pragma unroll 4
            for (int q = 0; q < ns; ++q)
                rank += skey[q] > mine;
            if (rank < k)
                C.sel_idx[rank] = (int)(0xFFFFFFFFu - (uint32_t)mine);
        }
        __syncthreads();
        if (WARP == 0 && LANE < k)
            C.sel_slot[LANE] = slots ? C.stab[C.tab_off + C.sel_idx[LANE]] : -1;
    }
    __syncthreads();
}

}  // namespace

// Dynamic shared memory of the fused kernel: the plan plus 1024 bytes to align the staging slots.
__host__ __device__ uint32_t decode_smem_bytes(const StepParams& P, int grid)
{
    return smem_plan(P.H, P.E, P.I, P.Is, P.bits, grid, P.sg, P.sgs).total + 1024;
}

__global__ void __launch_bounds__(kThreads, 1) moe_decode_kernel(const __grid_constant__ StepParams P)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Ctx& C = *reinterpret_cast<Ctx*>(base);  // the plan puts the context first
    if (TID == 0)
        make_ctx(P, C, base);
    __syncthreads();
    const bool route = P.mode != kModeExperts;
    const bool experts = P.mode != kModeRoute;
    const bool prenorm = (P.flags & kPrenorm) != 0;
    const bool residual = (P.flags & kResidual) != 0;
    const int n_steps = P.mode == kModeFull ? P.n_tokens * P.n_layers : 1;
    const long long limit = (long long)(2 * P.timeout_ns);
    const int H = C.H, K = C.k, hdim = xh_stride(C.I, C.Is);
    const bool shb = experts && C.sh;  // this block serves the shared expert
    const StageGeo& g = C.g;
    // the warp that clears this block's slice of the output words
    constexpr int kClearWarp = kWarps - 2;

    if (TID == 0) {
#pragma unroll 1
        for (int i = 0; i < kNumMbar; ++i)
            mbar_init(C.mbar + i, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (experts)
#pragma unroll 1
            for (int i = 0; i < 3; ++i)
                prefetch_map(&P.tmap[i]);
        // the first step's descriptor: written here, then overwritten by bulk copies (ordered after
        // this write by the proxy fence)
        C.ld[0] = P.layers[P.layer0];
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue_dense(P, C, P.layer0, 0, P.layer0 + (1 % P.n_layers), route, shb);
        if (experts)
            plan_copies(C);
    }
    __syncwarp();
    if (shb && WARP == 0)
        issue_expert_warp(C, C.cur->shared_blob, P.smaps + 3 * P.layer0, 0);
    // this block's slice of the first step's output words starts at zero
    if (experts && WARP == kClearWarp) {
#pragma unroll 1
        for (int o = C.o0 + LANE; o < C.o1; o += 32)
            st_s64(P.xacc + o, 0);
        fence_gpu();
    }

    // mbarrier phases (block-uniform)
    uint32_t ph_dense = 0, ph_down = 0, ph_gu = 0;  // ph_gu: bit gu_bar(slot, matrix, piece)
    bool dense_pending = true, down_pending = shb && C.d1 > C.d0;
    uint32_t gu_pending = (shb && C.r1 > C.r0) ? low_bits(2 * g.nslot_gu * g.npc_gu) : 0u;

    // the step counter before this launch's first add: no block adds before every block has
    // passed the launch barrier, so every block reads the same value here
    unsigned long long done0 = 0;
    if (TID == 0)
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(done0) : "l"(P.xflag) : "memory");
    bool ok = grid_barrier(P, limit);

    // token t, layer li of the step; the layers of the next two steps; the step's output buffer
    int t = 0, li = 0, xb = 0;
#pragma unroll 1
    for (int step = 0; ok && step < n_steps;
         ++step, xb = (xb == 2) ? 0 : xb + 1, t += (li + 1 == P.n_layers), li = (li + 1 == P.n_layers) ? 0 : li + 1) {
        const int l = P.layer0 + li;
        const int li1 = (li + 1 == P.n_layers) ? 0 : li + 1, li2 = (li1 + 1 == P.n_layers) ? 0 : li1 + 1;
        const int ln = P.layer0 + li1;
        const uint32_t epoch = P.epoch0 + (uint32_t)step;
        long long* X = P.xacc + (size_t)xb * H;

        // ---------------- 1. layer input, u ----------------
        {
            const bool fresh = li == 0;
            const size_t trow = (size_t)P.n_layers + 1;
            if (step > 0 && experts && !(ok = wait_steps(P.xflag, done0 + (unsigned long long)GRID * step, limit, P.status)))
                break;
            float* tr_prev = (step > 0 && fresh && P.trace) ? P.trace + ((size_t)(t - 1) * trow + P.n_layers) * H : nullptr;
            float* tr_cur = P.trace ? P.trace + ((size_t)t * trow + li) * H : nullptr;
            const char* xin = (const char*)P.x_in + (size_t)t * H * (prenorm ? 4 : 2);
            if (!(ok = layer_input(C, (step > 0 && experts) ? P.xacc + (size_t)(xb == 0 ? 2 : xb - 1) * H : nullptr, K + 1,
                                   residual, fresh, xin, prenorm, prenorm || li > 0, prenorm,
                                   (step > 0 && fresh) ? P.y_out + (size_t)(t - 1) * H : nullptr, tr_prev, tr_cur,
                                   limit, P.status)))
                break;
        }

        // ---------------- 2. router rows -> logits; gamma ----------------
        if (!(ok = wait_block(C.mbar + kMbDense, ph_dense & 1, limit, P.status)))
            break;
        ++ph_dense;
        dense_pending = false;
        if (route)
            router_rows(C, P.xlog, epoch);
        if (shb && WARP == 1) {
            float z = 0.f;
#pragma unroll 2
            for (int v = LANE; v < H / 8; v += 32)
                z = dot8_bf16(*reinterpret_cast<const uint4*>(C.swsg + 8 * v), *reinterpret_cast<const uint4*>(C.su + 8 * v),
                              z);
            z = warp_sum(z);
            if (LANE == 0)
                C.misc[0] = __fdividef(1.f, 1.f + __expf(-z));
        }

        // ---------------- 3. the expert's gate/up rows -> h (shared expert: now) ----------------
        // (the routed experts' come after the top-k; the code is shared through this lambda-free
        // loop body, run at most once per step)
        bool blob = false;
        int rslot = -1;
        const CUtensorMap* maps = nullptr;
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            if (pass == 1) {
                // ---------------- 4. top-k ----------------
                if (route) {
                    if (!(ok = poll_pairs(P.xlog, C.E, epoch, C.slg, limit, P.status)))
                        break;
                    topk_select(C, P.mode == kModeFull);
                    // the combine weights (one warp, beside warp 0's expert copies below) and block
                    // 0's selection outputs
                    if (WARP == 1) {
                        topk_weights(C, (P.flags & kRenorm) != 0);
                        __syncwarp();
                        if (CTA == 0 && LANE < K) {
                            const size_t o = ((size_t)t * P.n_layers + li) * K + LANE;
                            if (P.topk_idx)
                                P.topk_idx[o] = C.sel_idx[LANE];
                            if (P.topk_w)
                                P.topk_w[o] = C.sel_w[LANE];
                        }
                    }
                    if (!experts)
                        break;  // a route-only launch has one step
                    if (TID < K && C.sel_slot[TID] < 0)
                        set_status(P.status, kStatusNotResident);
                } else {
                    if (TID < K) {
                        C.sel_w[TID] = P.topk_w[TID];
                        C.sel_slot[TID] = P.slots[TID];
                        C.sel_idx[TID] = -1;
                    }
                    __syncthreads();
                }
                // the next step's output words (three buffers, by step): every block read them
                // last in the step before the previous one, which the step counter says is done;
                // clear this block's slice of them. This block's count of this step, which the
                // next step's adders wait for, is ordered after the clear.
                if (step + 1 < n_steps) {
                    if (WARP == kClearWarp) {
#pragma unroll 1
                        for (int o = C.o0 + LANE; o < C.o1; o += 32)
                            st_s64(P.xacc + (size_t)(xb == 2 ? 0 : xb + 1) * H + o, 0);
                    }
                }
                if (shb)
                    break;  // the shared expert's rows are done
                // this block's routed expert: every byte it reads of it, issued now
                rslot = C.sel_slot[C.j];
                blob = rslot >= 0;
                maps = P.tmap;
                if (blob && WARP == 0)
                    issue_expert_warp(C, P.arena + (uint64_t)rslot * P.stride, maps, rslot);
                down_pending = blob && C.d1 > C.d0;
                if (blob && C.r1 > C.r0)
                    gu_pending = low_bits(2 * g.nslot_gu * g.npc_gu);
            } else {
                if (!shb)
                    continue;
                blob = true;
                maps = P.smaps + 3 * l;
            }
            const bool have_gu = blob && C.r1 > C.r0;
            if (have_gu) {
                const int cpb = g.cbw_gu >> 5;
                const int per_m = C.per_m;  // items per matrix of a column group: (row box, column block)
                bool wok = true;
                int sl = 0;
#pragma unroll 1
                for (int cg = 0; cg < g.ncs_gu; ++cg, sl = (sl + 1 == g.nslot_gu) ? 0 : sl + 1) {
#pragma unroll 1
                    for (int it = WARP; wok && it < 2 * per_m; it += kWarps) {
                        const int m = it >= per_m, q = it - m * per_m;
                        const int rc = div_by(q, C.mg_cpg_gu), cbl = q - rc * g.cpg_gu;
                        const int cb = cg * g.cpg_gu + cbl;
                        const int nvalid = imin(g.bh_gu, C.r1 - C.r0 - rc * g.bh_gu);
                        if (cb >= g.ncb_gu)
                            continue;
                        // the item's piece (and, for the first group, piece 0 with the scales)
                        const int pb = gu_bar(g, sl, m, div_by(cbl, C.mg_cpp_gu)), p0 = gu_bar(g, sl, m, 0);
                        if (!(wok = wait_warp(C.mbar + pb, (ph_gu >> pb) & 1, limit)))
                            break;
                        if (cg == 0 && pb != p0 && !(wok = wait_warp(C.mbar + p0, (ph_gu >> p0) & 1, limit)))
                            break;
                        const int c0 = cb * cpb;
                        box_mma(gu_copy_at(C, sl, m, rc) + (size_t)cbl * g.bh_gu * g.cbw_gu, g.swz_gu ? 7u : 0u, g.cbw_gu,
                                nvalid, 0, cdiv(nvalid, 16), c0, imin(cpb, C.NCu - c0), C.sup, 0, C.scs,
                                C.rsb + (2 * m) * C.span_gu + C.sc_off[2 * m] + rc * g.bh_gu * C.ngu * 2,
                                C.rsb + (2 * m + 1) * C.span_gu + C.sc_off[2 * m + 1] + rc * g.bh_gu * C.ngu * 2,
                                C.ngu * 2, C.xp - 1, C.sp + (rc * g.bh_gu) * 2 * g.ncb_gu + m * g.ncb_gu + cb,
                                2 * g.ncb_gu);
                    }
                    if (__syncthreads_or(!wok)) {
                        if (TID == 0)
                            set_status(P.status, kStatusTimeout);
                        ok = false;
                        break;
                    }
                    const uint32_t slot_bits = low_bits(2 * g.npc_gu) << (2 * sl * g.npc_gu);
                    ph_gu ^= slot_bits;
                    gu_pending &= ~slot_bits;
                    // slot sl is free again: its next column group (when the groups take turns)
                    if (cg + g.nslot_gu < g.ncs_gu) {
                        if (TID == 0)
#pragma unroll 1
                            for (int m = 0; m < 2; ++m)
                                issue_gu(C, shb ? C.cur->shared_blob : P.arena + (uint64_t)rslot * P.stride, maps,
                                         shb ? 0 : rslot, cg + g.nslot_gu, sl, m, false);
                        gu_pending |= slot_bits;
                    }
                }
                if (!ok)
                    break;
            }
            __syncthreads();
            unsigned long long* xh = P.xh + (size_t)C.j * hdim;
#pragma unroll 1
            for (int r = TID; r < C.r1 - C.r0; r += kThreads) {
                float h = 0.f;
                if (blob) {
                    const int ncb = g.ncb_gu;
                    const float* pg = C.sp + r * 2 * ncb;
                    float gg = 0.f, vv = 0.f;
#pragma unroll 4
                    for (int cb = 0; cb < ncb; ++cb) {
                        gg += pg[cb];
                        vv += pg[ncb + cb];
                    }
                    h = __fdividef(gg, 1.f + __expf(-gg)) * vv;
                }
                st_pair(xh + C.r0 + r, epoch, h);
            }
        }
        if (!ok || !experts)
            break;

        // ---------------- 5. the group's h, down rows, contributions ----------------
        const bool have_d = blob && C.d1 > C.d0;
        if (C.d1 > C.d0) {
            unsigned long long* xh = P.xh + (size_t)C.j * hdim;
            if (!(ok = poll_pairs(xh, C.Ie, epoch, C.hv, limit, P.status)))
                break;
            if (have_d) {
                stage_h(C.xp, C.hv, C.Ie, C.shj, C.chj, P.status);
                const int cpd = g.cbw_d >> 5, tpi = C.tpi_d;
                // items (row box, column block, group of tpi tiles), about one per warp
                bool wok = true;
#pragma unroll 1
                for (int it = WARP; it < C.n_dn; it += kWarps) {
                    const int q = div_by(it, C.mg_ntg_d), tg = it - q * C.ntg_d;
                    const int rc = div_by(q, C.mg_cpg_d), cb = q - rc * g.cpg_d;
                    const int nvalid = imin(g.bh_d, C.d1 - C.d0 - rc * g.bh_d);
                    const int tt0 = tg * tpi, tt1 = imin(tt0 + tpi, (nvalid + 15) >> 4);
                    if (tt0 >= tt1)
                        continue;
                    if (!(wok = wait_warp(C.mbar + kMbDown, ph_down & 1, limit)))
                        break;
                    const int c0 = cb * cpd;
                    box_mma(d_copy_at(C, rc) + (size_t)cb * g.bh_d * g.cbw_d, g.swz_d ? 7u : 0u, g.cbw_d, nvalid, tt0, tt1,
                            c0, imin(cpd, C.NCd - c0), C.shj, C.KD, C.chj, C.rdsb + C.sc_off[4] + rc * g.bh_d * C.ngd * 2,
                            C.rdsb + C.span_d + C.sc_off[5] + rc * g.bh_d * C.ngd * 2, C.ngd * 2, C.xp - 1,
                            C.spd + (rc * g.bh_d) * g.ncb_d + cb, g.ncb_d);
                }
                if (__syncthreads_or(!wok)) {
                    if (TID == 0)
                        set_status(P.status, kStatusTimeout);
                    ok = false;
                    break;
                }
                ++ph_down;
                down_pending = false;
            }
            const float wj = C.sh ? C.misc[0] : C.sel_w[C.j];
#pragma unroll 1
            for (int r = TID; r < C.d1 - C.d0; r += kThreads) {
                float yj = 0.f;
                if (have_d)
#pragma unroll 1
                    for (int cb = 0; cb < g.ncb_d; ++cb)
                        yj += C.spd[r * g.ncb_d + cb];
                add_out(X + C.d0 + r, wj * yj, P.status);
            }
        }
        __syncthreads();
        // this block's contributions to the step's output words are in: its count, first (the other
        // blocks wait for it)
        if (TID == 0)
            asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(P.xflag) : "memory");
        // the next step's router rows, slot-table row, bias, gate vector and (the shared expert's
        // blocks) shared rows: the staging is free again
        // (warp 1: thread 0 is held by its release)
        if (step + 1 < n_steps) {
            if (WARP == 1) {
                if (LANE == 0)
                    issue_dense(P, C, ln, (step + 1) & 1, P.layer0 + li2, route, shb);
                __syncwarp();
                if (shb)
                    issue_expert_warp(C, C.cur->shared_blob, P.smaps + 3 * ln, 0);
            }
            dense_pending = true;
        }
        if (shb && step + 1 < n_steps) {
            down_pending = C.d1 > C.d0;
            if (C.r1 > C.r0)
                gu_pending = low_bits(2 * g.nslot_gu * g.npc_gu);
        }
    }

    // the last step's output
    if (ok && experts) {
        const int s = n_steps - 1, t = s / P.n_layers;
        ok = wait_steps(P.xflag, done0 + (unsigned long long)GRID * n_steps, limit, P.status) &&
             layer_input(C, P.xacc + (size_t)(s % 3) * H, K + 1, residual, false, nullptr, false, true, false,
                         P.y_out + (size_t)t * H,
                         P.trace ? P.trace + ((size_t)t * (P.n_layers + 1) + P.n_layers) * H : nullptr, nullptr, limit,
                         P.status);
    }

    // drain: copies still in flight into this block's shared memory finish before it exits
    if (TID == 0) {
        const long long t0 = cycles();
        auto drain = [&](uint64_t* m, uint32_t parity) {
            while (!mbar_try(m, parity) && cycles() - t0 < 4 * limit) {
            }
        };
#pragma unroll 1
        for (int i = 0; i < kMaxGuBars; ++i)
            if (gu_pending & (1u << i))
                drain(C.mbar + i, (ph_gu >> i) & 1);
        if (down_pending)
            drain(C.mbar + kMbDown, ph_down & 1);
        if (dense_pending)
            drain(C.mbar + kMbDense, ph_dense & 1);
    }
}

}  // namespace moe
