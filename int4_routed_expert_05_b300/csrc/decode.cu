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
// Design (one cooperative launch covers every layer and token of a call; grid = one 512-thread
// block per SM):
//   phase A  every block: input -> u (bf16) in shared memory; a slice of the router rows -> logits;
//            a slice of the shared expert's gate/up rows -> h_shared; the shared gate.
//   barrier  (logits complete)
//   phase B  every block redundantly: top-k + weights; then a slice of the routed experts'
//            gate/up rows -> h_j. The block's down-projection rows are prefetched to L2 at once and
//            loaded into registers before the next barrier.
//   barrier  (all h complete)
//   phase C  every block: its slice of output rows for all k + 1 experts, combined in rank order
//            then the shared term, plus the residual.
//   barrier  (next step reads the new residual)
// Expert weights stream once from HBM with 64-bit coalesced loads (a warp reads 32 contiguous bytes
// of 8 rows per instruction). int4 codes become exact bf16 integers in registers (mask + bf16x2
// fma) and meet the activations on the tensor cores (mma.m16n8k16, fp32 accumulate), one
// 64-element chunk (one quantisation group) at a time; per chunk and row the affine dequantisation
// is applied exactly as  s * (sum q u) + b * (sum u). Partial sums are added in a fixed order, so
// the result does not depend on the grid size or on where the experts sit in the pool.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "layout.h"

namespace moe {
namespace {

constexpr int NBG = 16;  // gate/up items held in flight per warp
constexpr int NBD = 8;   // down items held in flight per warp (across the barrier)
constexpr int kRouterRegs = 8;  // 16-byte router loads held per lane (hidden <= 2048 in one go)

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

// Position of element n of the expanded activation vector inside its permuted 16-element block
// (register order 0,4,1,5,2,6,3,7, 8,12,9,13,10,14,11,15 of the B fragments).
__device__ __forceinline__ int pslot(int n)
{
    const int e = n & 15;
    return (n & ~15) | (e & 8) | ((e & 3) << 1) | ((e >> 2) & 1);
}

__device__ __forceinline__ uint2 ldg_stream(const void* p)
{
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg_stream4(const void* p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// loads of data written by other blocks of the same launch: L2 only, never hoisted
__device__ __forceinline__ float ld_cg(const float* p)
{
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

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

__device__ __forceinline__ void set_status(int* status, int code) { atomicCAS(status, 0, code); }

// ------------------------------------------------------------------------------------------
// per-block context
// ------------------------------------------------------------------------------------------

struct Ctx {
    int H, E, k, I, Is, xp, KU, NCu, Imax, KDmax, NCdmax, ngu, ngdmax;
    int G, cta, tid, warp, lane, g, tq;
    float* sx;            // [H] layer input (fp32)
    uint16_t* su;         // [H] u (bf16)
    uint16_t* sup;        // [KU] expanded u, permuted blocks
    float* suc;           // [NCu] chunk sums of u
    float* sp;            // [kGuRows][2][NCu] gate/up partials
    uint16_t* ssb;        // [kGuRows][2][2][ngu] gate/up scale, bias
    uint16_t* shp;        // [k+1][2][KDmax] h hi/lo, permuted blocks
    float* suh;           // [k+1][NCdmax] chunk sums of h
    float* spd;           // [k+1][kDnRows][NCdmax] down partials
    uint16_t* ssbd;       // [k+1][kDnRows][2][ngdmax] down scale, bias
    float* slg;           // [E] logits
    uint32_t* lkey;       // [kWarps][kMaxK]
    int* lidx;            // [kWarps][kMaxK]
    int* sel_idx;         // [kMaxK]
    float* sel_w;         // [kMaxK]
    int* sel_slot;        // [kMaxK]
    float* red;           // [64]
    float* misc;          // [0] gamma, [1] rms
    const uint8_t** gptr; // [kGuRows] blob of each gate/up row (null: skip)
    int* grow;            // [kGuRows] row inside its expert
    int* gj;              // [kGuRows] expert rank (k = shared)
    const uint8_t** dptr; // [kMaxK + 1] blob of each expert rank for the down rows
};

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

// Grid-wide barrier on a monotonically increasing ticket counter (starts at a multiple of the
// grid size). Bounded: after timeout_ns of waiting it records kStatusTimeout and returns false.
__device__ bool grid_barrier(const StepParams& P, const Ctx& C)
{
    __shared__ int s_ok;
    __syncthreads();
    if (C.tid == 0) {
        int ok = 1;
        const unsigned long long G = gridDim.x;
        __threadfence();
        unsigned long long ticket;
        asm volatile("atom.release.gpu.global.add.u64 %0, [%1], 1;" : "=l"(ticket) : "l"(P.bar) : "memory");
        const unsigned long long target = (ticket / G + 1) * G;
        uint64_t t0 = 0;
        uint32_t spins = 0;
        while (true) {
            unsigned long long v;
            asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(P.bar) : "memory");
            if (v >= target)
                break;
            if ((++spins & 63u) == 0) {
                const uint64_t now = globaltimer();
                if (t0 == 0)
                    t0 = now;
                else if (now - t0 > P.timeout_ns) {
                    ok = 0;
                    set_status(P.status, kStatusTimeout);
                    break;
                }
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// ------------------------------------------------------------------------------------------
// phase A pieces
// ------------------------------------------------------------------------------------------

// Input of layer li of token t -> sx (fp32), su (bf16 u), sup (expanded, permuted), suc.
__device__ void load_input(const StepParams& P, const Ctx& C, int t, int li)
{
    const int H = C.H;
    if (P.flags & kPrenorm) {
        const float* src = li == 0 ? (const float*)P.x_in + (size_t)t * H : P.xbuf;
        float ss = 0.f;
        for (int i = C.tid; i < H; i += kThreads) {
            const float v = li == 0 ? __ldg(src + i) : ld_cg(src + i);
            C.sx[i] = v;
            ss = fmaf(v, v, ss);
        }
        ss = block_sum(C, ss);
        const float r = sqrtf(ss / (float)H + 1e-6f);
        for (int i = C.tid; i < H; i += kThreads)
            C.su[i] = f2bf(C.sx[i] / r);
    } else {
        const uint16_t* src = (const uint16_t*)P.x_in + (size_t)t * H;
        for (int i = C.tid; i < H; i += kThreads) {
            const uint16_t b = __ldg(src + i);
            C.su[i] = b;
            C.sx[i] = bf16f(b);
        }
    }
    if (P.trace && C.cta == 0)
        for (int i = C.tid; i < H; i += kThreads)
            P.trace[((size_t)t * (P.n_layers + 1) + li) * H + i] = C.sx[i];
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

// ------------------------------------------------------------------------------------------
// gate/up rows (flattened over experts) -> h
// ------------------------------------------------------------------------------------------

struct GuJob {
    int f0, nrows;   // flattened rows [f0, f0 + nrows), nrows <= kGuRows
    bool shared;     // shared expert (rows of one blob) or routed (rows f -> rank f / I)
};

__device__ void gu_setup(const StepParams& P, const Ctx& C, const LayerDesc& L, const GuJob& J)
{
    if (C.tid < J.nrows) {
        const int f = J.f0 + C.tid;
        const uint8_t* base;
        int r, j;
        if (J.shared) {
            base = L.shared_blob;
            r = f;
            j = C.k;
        } else {
            j = f / C.I;
            r = f - j * C.I;
            const int s = C.sel_slot[j];
            base = s >= 0 ? P.arena + (uint64_t)s * P.stride : nullptr;
        }
        C.gptr[C.tid] = base;
        C.grow[C.tid] = r;
        C.gj[C.tid] = j;
    }
    __syncthreads();
}

__device__ __forceinline__ int gu_items(const Ctx& C, const GuJob& J)
{
    const int ntiles = (J.nrows + 15) >> 4;
    const int nch = C.warp < C.NCu ? (C.NCu - C.warp + kWarps - 1) / kWarps : 0;
    return nch * ntiles * 2;
}

// item it of this warp -> chunk c, tile, matrix m (chunk-major order)
__device__ __forceinline__ void gu_item(const Ctx& C, const GuJob& J, int it, int& c, int& tile, int& m)
{
    const int ntiles = (J.nrows + 15) >> 4;
    const int cs = it / (ntiles * 2);
    const int rem = it - cs * ntiles * 2;
    tile = rem >> 1;
    m = rem & 1;
    c = C.warp + kWarps * cs;
}

__device__ __forceinline__ void gu_issue(const StepParams& P, const Ctx& C, const GuJob& J, int base,
                                         uint2 (&ra)[NBG], uint2 (&rb)[NBG])
{
    const BlobGeo& geo = J.shared ? P.geo_s : P.geo;
    const int nit = gu_items(C, J);
#pragma unroll
    for (int i = 0; i < NBG; ++i) {
        ra[i] = make_uint2(0, 0);
        rb[i] = make_uint2(0, 0);
        const int it = base + i;
        if (it < nit) {
            int c, tile, m;
            gu_item(C, J, it, c, tile, m);
            const int rowa = tile * 16 + C.g, rowb = rowa + 8;
            const uint64_t off = geo.q_off[m] + 32ull * c + 8ull * C.tq;
            if (rowa < J.nrows && C.gptr[rowa])
                ra[i] = ldg_stream(C.gptr[rowa] + off + (uint64_t)C.grow[rowa] * geo.row_bytes[m]);
            if (rowb < J.nrows && C.gptr[rowb])
                rb[i] = ldg_stream(C.gptr[rowb] + off + (uint64_t)C.grow[rowb] * geo.row_bytes[m]);
        }
    }
}

// scale and bias of the job's rows -> ssb[row][m][s|b][group]
__device__ void gu_stage_scales(const StepParams& P, const Ctx& C, const GuJob& J)
{
    const BlobGeo& geo = J.shared ? P.geo_s : P.geo;
    const int nq = C.ngu / 4;  // 8-byte words per row section
    const int total = J.nrows * 2 * 2 * nq;
    for (int e = C.tid; e < total; e += kThreads) {
        const int wq = e % nq;
        const int rest = e / nq;
        const int sb = rest & 1, m = (rest >> 1) & 1, row = rest >> 2;
        if (!C.gptr[row])
            continue;
        const uint64_t off = (sb ? geo.b_off[m] : geo.s_off[m]) + ((uint64_t)C.grow[row] * C.ngu + 4 * wq) * 2;
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(C.gptr[row] + off));
        *reinterpret_cast<uint2*>(C.ssb + ((row * 2 + m) * 2 + sb) * C.ngu + 4 * wq) = v;
    }
}

__device__ __forceinline__ void gu_compute(const Ctx& C, const GuJob& J, int base, const uint2 (&ra)[NBG],
                                           const uint2 (&rb)[NBG])
{
    const int nit = gu_items(C, J);
#pragma unroll
    for (int i = 0; i < NBG; ++i) {
        const int it = base + i;
        if (it < nit) {
            int c, tile, m;
            gu_item(C, J, it, c, tile, m);
            const uint4* bp = reinterpret_cast<const uint4*>(C.sup + kChunk * c + 16 * C.tq);
            float acc[4];
            chunk_mma(acc, ra[i], rb[i], bp[0], bp[1]);
            const int gi = c / C.xp;
            const int rowa = tile * 16 + C.g, rowb = rowa + 8;
            if (C.tq == 0 && rowa < J.nrows) {
                const uint16_t* sb = C.ssb + (rowa * 2 + m) * 2 * C.ngu;
                C.sp[(rowa * 2 + m) * C.NCu + c] = fmaf(bf16f(sb[gi]), acc[0], bf16f(sb[C.ngu + gi]) * C.suc[c]);
            }
            if (C.tq == 1 && rowb < J.nrows) {
                const uint16_t* sb = C.ssb + (rowb * 2 + m) * 2 * C.ngu;
                C.sp[(rowb * 2 + m) * C.NCu + c] = fmaf(bf16f(sb[gi]), acc[2], bf16f(sb[C.ngu + gi]) * C.suc[c]);
            }
        }
    }
}

__device__ void gu_finalize(const StepParams& P, const Ctx& C, const GuJob& J)
{
    if (C.tid < J.nrows && C.gptr[C.tid]) {
        const float* pg = C.sp + (C.tid * 2 + 0) * C.NCu;
        const float* pv = C.sp + (C.tid * 2 + 1) * C.NCu;
        float g = 0.f, v = 0.f;
        for (int c = 0; c < C.NCu; ++c) {
            g += pg[c];
            v += pv[c];
        }
        const float h = g / (1.f + expf(-g)) * v;
        P.hbuf[(size_t)C.gj[C.tid] * C.Imax + C.grow[C.tid]] = h;
    }
}

// Whole gate/up job (all batches of at most kGuRows rows). The first batch's loads may have been
// issued by the caller (pre_ra/pre_rb) before shared data they do not depend on was ready.
__device__ void gu_run(const StepParams& P, const Ctx& C, const LayerDesc& L, int f0, int nrows_total, bool shared)
{
    for (int b0 = 0; b0 < nrows_total; b0 += kGuRows) {
        GuJob J{f0 + b0, min(kGuRows, nrows_total - b0), shared};
        gu_setup(P, C, L, J);
        uint2 ra[NBG], rb[NBG];
        gu_issue(P, C, J, 0, ra, rb);
        gu_stage_scales(P, C, J);
        __syncthreads();
        gu_compute(C, J, 0, ra, rb);
        const int nit = gu_items(C, J);
        for (int base = NBG; base < nit; base += NBG) {
            gu_issue(P, C, J, base, ra, rb);
            gu_compute(C, J, base, ra, rb);
        }
        __syncthreads();
        gu_finalize(P, C, J);
        __syncthreads();
    }
}

// ------------------------------------------------------------------------------------------
// down rows of all k + 1 experts -> combined output
// ------------------------------------------------------------------------------------------

struct DnJob {
    int o0, nr;  // output rows [o0, o0 + nr), nr <= kDnRows
};

__device__ __forceinline__ int dn_nch(const StepParams& P, const Ctx& C, int j)
{
    return (j < C.k ? C.I : C.Is) * C.xp / kChunk;
}

__device__ __forceinline__ int dn_total(const StepParams& P, const Ctx& C)
{
    return C.k * dn_nch(P, C, 0) + dn_nch(P, C, C.k);
}

__device__ __forceinline__ void dn_item(const StepParams& P, const Ctx& C, int it, int& j, int& c)
{
    const int ncr = dn_nch(P, C, 0);
    if (it < C.k * ncr) {
        j = it / ncr;
        c = it - j * ncr;
    } else {
        j = C.k;
        c = it - C.k * ncr;
    }
}

__device__ __forceinline__ void dn_issue(const StepParams& P, const Ctx& C, const DnJob& J, int base,
                                         uint2 (&ra)[NBD], uint2 (&rb)[NBD])
{
    const int tot = dn_total(P, C);
#pragma unroll
    for (int i = 0; i < NBD; ++i) {
        ra[i] = make_uint2(0, 0);
        rb[i] = make_uint2(0, 0);
        const int it = C.warp + kWarps * (base + i);
        if (it < tot) {
            int j, c;
            dn_item(P, C, it, j, c);
            const uint8_t* blob = C.dptr[j];
            if (blob) {
                const BlobGeo& geo = j < C.k ? P.geo : P.geo_s;
                const uint64_t off = geo.q_off[2] + 32ull * c + 8ull * C.tq;
                const int rowa = C.g, rowb = C.g + 8;
                if (rowa < J.nr)
                    ra[i] = ldg_stream(blob + off + (uint64_t)(J.o0 + rowa) * geo.row_bytes[2]);
                if (rowb < J.nr)
                    rb[i] = ldg_stream(blob + off + (uint64_t)(J.o0 + rowb) * geo.row_bytes[2]);
            }
        }
    }
}

__device__ void dn_stage_scales(const StepParams& P, const Ctx& C, const DnJob& J)
{
    const int per_j = J.nr * 2 * C.ngdmax;
    const int total = (C.k + 1) * per_j;
    for (int e = C.tid; e < total; e += kThreads) {
        const int j = e / per_j;
        int rest = e - j * per_j;
        const int gi = rest % C.ngdmax;
        rest /= C.ngdmax;
        const int sb = rest & 1, row = rest >> 1;
        const BlobGeo& geo = j < C.k ? P.geo : P.geo_s;
        const uint8_t* blob = C.dptr[j];
        if (!blob || gi >= geo.groups[2])
            continue;
        const uint64_t off = (sb ? geo.b_off[2] : geo.s_off[2]) + ((uint64_t)(J.o0 + row) * geo.groups[2] + gi) * 2;
        C.ssbd[((j * kDnRows + row) * 2 + sb) * C.ngdmax + gi] = __ldg(reinterpret_cast<const uint16_t*>(blob + off));
    }
}

// all h (written by every block) -> shp hi/lo permuted, suh chunk sums
__device__ void dn_stage_h(const StepParams& P, const Ctx& C)
{
    for (int j = 0; j <= C.k; ++j) {
        if (!C.dptr[j])
            continue;
        const int Ij = j < C.k ? C.I : C.Is;
        const int KD = Ij * C.xp;
        uint16_t* hi = C.shp + (size_t)(j * 2 + 0) * C.KDmax;
        uint16_t* lo = C.shp + (size_t)(j * 2 + 1) * C.KDmax;
        const float* hsrc = P.hbuf + (size_t)j * C.Imax;
        for (int n = C.tid; n < KD; n += kThreads) {
            float v = ld_cg(hsrc + (C.xp == 1 ? n : (n >> 1)));
            if (C.xp == 2 && (n & 1))
                v *= 16.f;
            const uint16_t h = f2bf(v);
            hi[pslot(n)] = h;
            lo[pslot(n)] = f2bf(v - bf16f(h));
        }
        const int cpc = kChunk / C.xp;
        const int nch = KD / kChunk;
        for (int c = C.warp; c < nch; c += kWarps) {
            float s = 0.f;
            for (int i = C.lane; i < cpc; i += 32)
                s += ld_cg(hsrc + c * cpc + i);
            s = warp_sum(s);
            if (C.lane == 0)
                C.suh[j * C.NCdmax + c] = s;
        }
    }
}

__device__ __forceinline__ void dn_compute(const StepParams& P, const Ctx& C, const DnJob& J, int base,
                                           const uint2 (&ra)[NBD], const uint2 (&rb)[NBD])
{
    const int tot = dn_total(P, C);
#pragma unroll
    for (int i = 0; i < NBD; ++i) {
        const int it = C.warp + kWarps * (base + i);
        if (it < tot) {
            int j, c;
            dn_item(P, C, it, j, c);
            if (!C.dptr[j])
                continue;
            const uint4* bp = reinterpret_cast<const uint4*>(C.shp + (size_t)(j * 2 + (C.g & 1)) * C.KDmax +
                                                             kChunk * c + 16 * C.tq);
            float acc[4];
            chunk_mma(acc, ra[i], rb[i], bp[0], bp[1]);
            const int gi = c / C.xp;
            const float uh = C.suh[j * C.NCdmax + c];
            const int rowa = C.g, rowb = C.g + 8;
            if (C.tq == 0 && rowa < J.nr) {
                const uint16_t* sb = C.ssbd + (j * kDnRows + rowa) * 2 * C.ngdmax;
                C.spd[(j * kDnRows + rowa) * C.NCdmax + c] = fmaf(bf16f(sb[gi]), acc[0] + acc[1], bf16f(sb[C.ngdmax + gi]) * uh);
            }
            if (C.tq == 1 && rowb < J.nr) {
                const uint16_t* sb = C.ssbd + (j * kDnRows + rowb) * 2 * C.ngdmax;
                C.spd[(j * kDnRows + rowb) * C.NCdmax + c] = fmaf(bf16f(sb[gi]), acc[2] + acc[3], bf16f(sb[C.ngdmax + gi]) * uh);
            }
        }
    }
}

__device__ void dn_finalize(const StepParams& P, const Ctx& C, const DnJob& J, int t, int li)
{
    if (C.tid < J.nr) {
        const int row = C.tid;
        float y = 0.f;
        for (int j = 0; j < C.k; ++j) {
            if (!C.dptr[j])
                continue;
            const float* pd = C.spd + (j * kDnRows + row) * C.NCdmax;
            const int nch = dn_nch(P, C, j);
            float yj = 0.f;
            for (int c = 0; c < nch; ++c)
                yj += pd[c];
            y = fmaf(C.sel_w[j], yj, y);
        }
        {
            const float* pd = C.spd + (C.k * kDnRows + row) * C.NCdmax;
            const int nch = dn_nch(P, C, C.k);
            float ys = 0.f;
            for (int c = 0; c < nch; ++c)
                ys += pd[c];
            y = fmaf(C.misc[0], ys, y);
        }
        const int o = J.o0 + row;
        const float out = (P.flags & kResidual) ? C.sx[o] + y : y;
        const bool last_layer = li == P.n_layers - 1;
        if (last_layer)
            P.y_out[(size_t)t * C.H + o] = out;
        else
            P.xbuf[o] = out;
        if (P.trace)
            P.trace[((size_t)t * (P.n_layers + 1) + li + 1) * C.H + o] = out;
    }
}

// ------------------------------------------------------------------------------------------
// routing
// ------------------------------------------------------------------------------------------

// logits (global) -> sel_idx / sel_w (rank order: larger fp32 logit first, ties -> lower index).
__device__ void topk_select(const StepParams& P, const Ctx& C)
{
    const int E = C.E, k = C.k;
    for (int e = C.tid; e < E; e += kThreads)
        C.slg[e] = ld_cg(P.logits + e);
    __syncthreads();
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
// the kernel
// ------------------------------------------------------------------------------------------

__device__ void make_ctx(const StepParams& P, Ctx& C, uint8_t* smem)
{
    C.H = P.H;
    C.E = P.E;
    C.k = P.k;
    C.I = P.I;
    C.Is = P.Is;
    C.xp = P.bits == 8 ? 2 : 1;
    C.KU = P.H * C.xp;
    C.NCu = C.KU / kChunk;
    C.Imax = P.I > P.Is ? P.I : P.Is;
    C.KDmax = C.Imax * C.xp;
    C.NCdmax = C.KDmax / kChunk;
    C.ngu = P.H / P.group;
    C.ngdmax = C.Imax / P.group;
    C.G = gridDim.x;
    C.cta = blockIdx.x;
    C.tid = threadIdx.x;
    C.warp = C.tid >> 5;
    C.lane = C.tid & 31;
    C.g = C.lane >> 2;
    C.tq = C.lane & 3;
    const SmemPlan sp = smem_plan(P.H, P.E, P.k, P.I, P.Is, P.bits, P.group);
    C.sx = (float*)(smem + sp.x);
    C.su = (uint16_t*)(smem + sp.u);
    C.sup = (uint16_t*)(smem + sp.up);
    C.suc = (float*)(smem + sp.uc);
    C.sp = (float*)(smem + sp.p);
    C.ssb = (uint16_t*)(smem + sp.sb);
    C.shp = (uint16_t*)(smem + sp.hp);
    C.suh = (float*)(smem + sp.uh);
    C.spd = (float*)(smem + sp.pd);
    C.ssbd = (uint16_t*)(smem + sp.sbd);
    C.slg = (float*)(smem + sp.lg);
    C.lkey = (uint32_t*)(smem + sp.lkey);
    C.lidx = (int*)(smem + sp.lidx);
    C.sel_idx = (int*)(smem + sp.sel_idx);
    C.sel_w = (float*)(smem + sp.sel_w);
    C.sel_slot = (int*)(smem + sp.sel_slot);
    C.red = (float*)(smem + sp.red);
    C.misc = (float*)(smem + sp.misc);
    C.gptr = (const uint8_t**)(smem + sp.total);
    C.grow = (int*)(smem + sp.total + 8 * kGuRows);
    C.gj = (int*)(smem + sp.total + 12 * kGuRows);
    C.dptr = (const uint8_t**)(smem + sp.total + 16 * kGuRows);
}

__device__ __forceinline__ int split(int n, int parts, int i) { return (int)(((long long)n * i) / parts); }

}  // namespace

// Extra shared memory beyond the plan: per-row blob pointers of the gate/up batch and the
// per-rank blob pointers of the down rows.
__host__ __device__ uint32_t decode_smem_bytes(const StepParams& P)
{
    const SmemPlan sp = smem_plan(P.H, P.E, P.k, P.I, P.Is, P.bits, P.group);
    return sp.total + 16 * kGuRows + 8 * (kMaxK + 1);
}

__global__ void __launch_bounds__(kThreads, 1) moe_decode_kernel(const __grid_constant__ StepParams P)
{
    extern __shared__ __align__(16) uint8_t smem[];
    Ctx C;
    make_ctx(P, C, smem);
    const bool route = P.mode != kModeExperts;
    const bool experts = P.mode != kModeRoute;

    for (int t = 0; t < P.n_tokens; ++t) {
        for (int li = 0; li < P.n_layers; ++li) {
            const int l = P.layer0 + li;
            const LayerDesc L = P.layers[l];

            // ---------------- phase A ----------------
            // router row of this warp: issue its loads before the input is ready
            const int e_first = C.cta + C.G * C.warp;
            uint4 rw[kRouterRegs];
            const int nreg = C.H / 256;
#pragma unroll
            for (int i = 0; i < kRouterRegs; ++i)
                rw[i] = make_uint4(0, 0, 0, 0);
            if (route && e_first < C.E) {
                const uint16_t* row = L.router + (size_t)e_first * C.H;
#pragma unroll
                for (int i = 0; i < kRouterRegs; ++i)
                    if (i < nreg)
                        rw[i] = ldg_stream4(row + 256 * i + 8 * C.lane);
            }
            load_input(P, C, t, li);
            if (route) {
                for (int m = 0;; ++m) {
                    const int e = C.cta + C.G * (C.warp + kWarps * m);
                    if (e >= C.E)
                        break;
                    const uint16_t* row = L.router + (size_t)e * C.H;
                    float acc = 0.f;
#pragma unroll
                    for (int i = 0; i < kRouterRegs; ++i) {
                        if (i < nreg) {
                            const uint4 w = m == 0 ? rw[i] : ldg_stream4(row + 256 * i + 8 * C.lane);
                            const uint4 x = *reinterpret_cast<const uint4*>(C.su + 256 * i + 8 * C.lane);
                            acc = dot8_bf16(w, x, acc);
                        }
                    }
                    for (int i = kRouterRegs; i < nreg; ++i) {
                        const uint4 w = ldg_stream4(row + 256 * i + 8 * C.lane);
                        const uint4 x = *reinterpret_cast<const uint4*>(C.su + 256 * i + 8 * C.lane);
                        acc = dot8_bf16(w, x, acc);
                    }
                    acc = warp_sum(acc);
                    if (C.lane == 0)
                        P.logits[e] = L.logit_bias ? acc + __ldg(L.logit_bias + e) : acc;
                }
            }
            if (experts) {
                // shared gate sigmoid(w_sg . u), computed by every block for its own combine
                if (C.warp == kWarps - 1) {
                    float z = 0.f;
                    for (int i = 0; i < nreg; ++i) {
                        const uint4 w = __ldg(reinterpret_cast<const uint4*>(L.shared_gate + 256 * i + 8 * C.lane));
                        const uint4 x = *reinterpret_cast<const uint4*>(C.su + 256 * i + 8 * C.lane);
                        z = dot8_bf16(w, x, z);
                    }
                    z = warp_sum(z);
                    if (C.lane == 0)
                        C.misc[0] = 1.f / (1.f + expf(-z));
                }
                // this block's slice of the shared expert's gate/up rows
                const int s0 = split(C.Is, C.G, C.cta), s1 = split(C.Is, C.G, C.cta + 1);
                gu_run(P, C, L, s0, s1 - s0, true);
            }

            // ---------------- routing ----------------
            if (route) {
                if (!grid_barrier(P, C))
                    return;
                topk_select(P, C);
                if (C.cta == 0 && C.tid < C.k) {
                    const size_t o = ((size_t)t * P.n_layers + li) * C.k + C.tid;
                    if (P.topk_idx)
                        P.topk_idx[o] = C.sel_idx[C.tid];
                    if (P.topk_w)
                        P.topk_w[o] = C.sel_w[C.tid];
                }
                if (!experts)
                    continue;  // one step per route-only launch
                if (C.tid < C.k) {
                    const int s = P.table[(size_t)l * C.E + C.sel_idx[C.tid]];
                    C.sel_slot[C.tid] = s;
                    if (s < 0)
                        set_status(P.status, kStatusNotResident);
                }
            } else {
                if (C.tid < C.k) {
                    C.sel_w[C.tid] = __ldg(P.topk_w + C.tid);
                    C.sel_slot[C.tid] = P.slots[C.tid];
                    C.sel_idx[C.tid] = -1;
                }
            }
            if (C.tid <= C.k) {
                if (C.tid < C.k) {
                    const int s = C.sel_slot[C.tid];
                    C.dptr[C.tid] = s >= 0 ? P.arena + (uint64_t)s * P.stride : nullptr;
                } else {
                    C.dptr[C.k] = L.shared_blob;
                }
            }
            __syncthreads();

            // ---------------- phase B ----------------
            const int o0 = split(C.H, C.G, C.cta), o1 = split(C.H, C.G, C.cta + 1);
            // prefetch this block's down rows of the routed experts into L2
            if (C.tid < C.k && C.dptr[C.tid] && o1 > o0) {
                const uint8_t* blob = C.dptr[C.tid];
                const BlobGeo& geo = P.geo;
                const uint64_t a = geo.q_off[2] + (uint64_t)o0 * geo.row_bytes[2];
                const uint64_t b = geo.q_off[2] + (uint64_t)o1 * geo.row_bytes[2];
                const uint64_t a16 = a & ~15ull, b16 = (b + 15) & ~15ull;
                prefetch_l2(blob + a16, (uint32_t)(b16 - a16));
                for (int sb = 0; sb < 2; ++sb) {
                    const uint64_t base = sb ? geo.b_off[2] : geo.s_off[2];
                    const uint64_t sa = (base + (uint64_t)o0 * geo.groups[2] * 2) & ~15ull;
                    const uint64_t se = (base + (uint64_t)o1 * geo.groups[2] * 2 + 15) & ~15ull;
                    prefetch_l2(blob + sa, (uint32_t)(se - sa));
                }
            }
            {
                const int kI = C.k * C.I;
                const int f0 = split(kI, C.G, C.cta), f1 = split(kI, C.G, C.cta + 1);
                gu_run(P, C, L, f0, f1 - f0, false);
            }

            // first batch of down rows: loads and scales before the barrier
            uint2 ra[NBD], rb[NBD];
            DnJob J0{o0, min(kDnRows, o1 - o0)};
            if (J0.nr > 0) {
                dn_issue(P, C, J0, 0, ra, rb);
                dn_stage_scales(P, C, J0);
            }
            if (!grid_barrier(P, C))
                return;

            // ---------------- phase C ----------------
            dn_stage_h(P, C);
            __syncthreads();
            for (int ob = o0; ob < o1; ob += kDnRows) {
                DnJob J{ob, min(kDnRows, o1 - ob)};
                if (ob != o0) {
                    dn_issue(P, C, J, 0, ra, rb);
                    dn_stage_scales(P, C, J);
                    __syncthreads();
                }
                dn_compute(P, C, J, 0, ra, rb);
                const int tot = dn_total(P, C);
                for (int base = NBD; C.warp + kWarps * base < tot; base += NBD) {
                    dn_issue(P, C, J, base, ra, rb);
                    dn_compute(P, C, J, base, ra, rb);
                }
                __syncthreads();
                dn_finalize(P, C, J, t, li);
                __syncthreads();
            }
            const bool last_step = (t == P.n_tokens - 1) && (li == P.n_layers - 1);
            if (!last_step && !grid_barrier(P, C))
                return;
        }
    }
}

}  // namespace moe
