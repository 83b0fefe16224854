// layout.h -- blob geometry, launch parameters, work split and shared-memory plan of the decode
// kernels.
//
// Blob format (one expert = one contiguous blob fetched at arena + slot * stride; paotong.dev
// commentary on Swiftlet, the fixed-stride .qpack container): sections gate.q | up.q | down.q |
// gate.s | gate.b | up.s | up.b | down.s | down.b. gate/up are [I][H], down is [H][I], codes
// packed along the input dimension (int4: element c in byte c/2, low nibble for even c), bf16
// scale and bias per 64 consecutive inputs (cheshm.ai item on Swiftlet: MLX-style int4/int8
// group quantisation). Stride = bytes rounded up to 4096.
#pragma once
#include <cuda.h>  // CUtensorMap (the type only; maps are encoded through the runtime's driver entry point)

#include <cstddef>
#include <cstdint>

#ifdef __CUDACC__
#define MOE_HD __host__ __device__ __forceinline__
#else
#define MOE_HD inline
#endif

namespace moe {

constexpr int kThreads = 512;   // threads per block of the fused decode kernel
constexpr int kWarps = kThreads / 32;
constexpr int kMaxK = 16;       // top-k limit
constexpr int kMaxE = 512;      // experts per layer limit
constexpr int kChunk = 64;      // nibbles per MMA chunk (one int4 quantisation group)
constexpr int kCb = 128;        // bytes of one staged column block (the 128-byte swizzle span)
constexpr int kMaxBoxRows = 256;
constexpr uint64_t kStrideAlign = 4096;
constexpr int kMaxGrid = 512;   // most blocks a decode launch may have (one per SM)

// Row stride (in pairs) of the h exchange buffer: rows 0..k-1 hold the routed experts' h, row k the
// shared expert's h followed by one step flag per block.
MOE_HD int xh_stride(int I, int Is) { return I > Is + kMaxGrid ? I : Is + kMaxGrid; }
constexpr float kFix = 4294967296.f;       // fixed-point scale of the output accumulator (2^32)
constexpr float kFixInv = 2.3283064365386963e-10f;
constexpr float kFixMax = 1073741824.f;    // largest |contribution| accepted (2^30)

// device status codes (same values as moe_status)
constexpr int kStatusInvalid = 1;
constexpr int kStatusNotResident = 3;
constexpr int kStatusTimeout = 6;

enum Mode : int { kModeFull = 0, kModeRoute = 1, kModeExperts = 2 };
enum Flags : int { kRenorm = 1, kPrenorm = 2, kResidual = 4 };

struct BlobGeo {
    uint64_t q_off[3];     // code sections: gate, up, down
    uint64_t s_off[3];     // bf16 scale sections
    uint64_t b_off[3];     // bf16 bias sections
    int32_t rows[3];       // output dimension of each matrix
    int32_t cols[3];       // input dimension of each matrix
    int32_t row_bytes[3];  // bytes of codes per row
    int32_t groups[3];     // scale groups per row
    uint64_t bytes;        // blob size
    uint64_t stride;       // bytes rounded up to kStrideAlign
};

MOE_HD BlobGeo blob_geo(int H, int I, int bits, int group)
{
    BlobGeo g{};
    const int rows[3] = {I, I, H};
    const int cols[3] = {H, H, I};
    uint64_t o = 0;
    for (int m = 0; m < 3; ++m) {
        g.rows[m] = rows[m];
        g.cols[m] = cols[m];
        g.row_bytes[m] = cols[m] * bits / 8;
        g.groups[m] = cols[m] / group;
        g.q_off[m] = o;
        o += (uint64_t)rows[m] * g.row_bytes[m];
    }
    for (int m = 0; m < 3; ++m) {
        const uint64_t sb = (uint64_t)rows[m] * g.groups[m] * 2;
        g.s_off[m] = o;
        o += sb;
        g.b_off[m] = o;
        o += sb;
    }
    g.bytes = o;
    g.stride = (o + kStrideAlign - 1) / kStrideAlign * kStrideAlign;
    return g;
}

// One layer's resident dense weights, as the kernels read them (device table [L]).
struct LayerDesc {
    const uint16_t* router;       // bf16 [E][H]
    const uint8_t* shared_blob;   // shared expert blob
    const uint16_t* shared_gate;  // bf16 [H]
    const float* logit_bias;      // fp32 [E] or null
};

// ------------------------------------------------------------------------------------------
// Work split (identical on host and device)
// ------------------------------------------------------------------------------------------

// [part(n, p, i), part(n, p, i + 1)) is part i of [0, n) cut into p nearly equal ranges
// (n * p < 2^32 for every shape the kernels take).
MOE_HD int part(int n, int parts, int i) { return (int)(((unsigned)n * (unsigned)i) / (unsigned)parts); }
// Routed expert of rank j is served by the blocks [grp_start(j), grp_start(j + 1)).
MOE_HD int grp_of(int b, int G, int k) { return (int)(((unsigned)b * (unsigned)k) / (unsigned)G); }
MOE_HD int grp_start(int j, int G, int k) { return (int)(((unsigned)j * (unsigned)G + (unsigned)k - 1u) / (unsigned)k); }
MOE_HD int cdiv(int a, int b) { return (a + b - 1) / b; }

// How one block's share of the routed experts is staged: row ranges of gate/up and down rows
// are fetched as TMA boxes of SR rows x one 128-byte column block (or the whole row when a row
// is narrower), one box per stage, through a ring of kWarps slots.
struct StageGeo {
    int SR;              // box rows
    int nrc_gu, nrc_d;   // row chunks of a block's gate/up rows / down rows
    int ncb_gu, ncb_d;   // column blocks per gate/up row / down row
    int cbw_gu, cbw_d;   // bytes per column block
    int swz_gu, swz_d;   // 1: 128-byte swizzled boxes, 0: linear boxes
    int n_gu, n_stages;  // gate/up stages, all stages
    int Rgu, Rd;         // most gate/up rows / down rows one block owns
    int Rr, Rs, Rsd;     // most router rows, shared gate/up rows, shared down rows per block
    uint32_t slot_bytes; // one ring slot (1024-byte multiple)
};

MOE_HD StageGeo stage_geo(int H, int E, int k, int I, int Is, int bits, int G)
{
    StageGeo s{};
    const int nmin = G / k;  // smallest group
    s.Rgu = cdiv(I, nmin);
    s.Rd = cdiv(H, nmin);
    s.SR = s.Rgu < kMaxBoxRows ? s.Rgu : kMaxBoxRows;
    if (s.SR < 1)
        s.SR = 1;
    s.nrc_gu = cdiv(s.Rgu, s.SR);
    s.nrc_d = cdiv(s.Rd, s.SR);
    const int rb_gu = H * bits / 8, rb_d = I * bits / 8;
    s.swz_gu = rb_gu >= kCb;
    s.swz_d = rb_d >= kCb;
    s.cbw_gu = s.swz_gu ? kCb : rb_gu;
    s.cbw_d = s.swz_d ? kCb : rb_d;
    s.ncb_gu = cdiv(rb_gu, s.cbw_gu);
    s.ncb_d = cdiv(rb_d, s.cbw_d);
    s.n_gu = 2 * s.ncb_gu * s.nrc_gu;
    s.n_stages = s.n_gu + s.ncb_d * s.nrc_d;
    s.Rr = cdiv(E, G);
    s.Rs = cdiv(Is, G);
    s.Rsd = cdiv(H, G);
    const uint32_t box = (uint32_t)s.SR * kCb;
    s.slot_bytes = (box + 1023u) & ~1023u;
    return s;
}

// Shared-memory room for the scale or bias rows [r0, r0 + n) of a section whose rows hold row_b
// bytes: the 16-byte aligned superset a 1D bulk copy fetches, rounded up to 16 bytes so that
// consecutive spans stay valid bulk-copy destinations.
MOE_HD uint32_t sb_span_max(int nrows, int row_b) { return ((uint32_t)(nrows * row_b + 32) + 15u) & ~15u; }

// ------------------------------------------------------------------------------------------
// Launch parameters
// ------------------------------------------------------------------------------------------

struct StepParams {
    // 3D TMA maps over the arena: bytes of a row x rows x slots, for gate.q, up.q and down.q
    CUtensorMap tmap[3];
    int H, E, k, I, Is, bits, group, flags;
    BlobGeo geo, geo_s;           // routed / shared blob geometry
    StageGeo sg;
    const uint8_t* arena;
    uint64_t stride;
    const int32_t* table;         // [L][E] slot of (layer, expert), -1 if absent
    const LayerDesc* layers;      // [L]
    int layer0, n_layers, n_tokens, mode;
    const void* x_in;             // [T][H]: bf16 layer input, or fp32 residual with kPrenorm
    float* y_out;                 // [T][H]
    float* trace;                 // [T][n_layers + 1][H] or null
    int32_t* topk_idx;            // [T][n_layers][k] or null (output)
    float* topk_w;                // [T][n_layers][k] or null (output; input in kModeExperts)
    int32_t slots[kMaxK];         // kModeExperts: slot of the expert of rank j
    // exchange buffers (workspace)
    unsigned long long* xlog;     // [E] (epoch << 32 | fp32 logit)
    unsigned long long* xh;       // [k + 1][max(I, Is)] (epoch << 32 | fp32 h); row k: shared expert
    long long* xacc;              // [2][H] fixed-point output accumulators (token parity)
    unsigned long long* bar;      // grid-barrier counter (a multiple of the grid between launches)
    int* status;
    uint32_t epoch0;              // epoch of the launch's first step (>= 1)
    unsigned long long timeout_ns;
    // scalar reference path only
    float* logits;                // [E]
    float* hbuf;                  // [k + 1][max(I, Is)]
};

// ------------------------------------------------------------------------------------------
// Shared-memory plan of the fused kernel (byte offsets)
// ------------------------------------------------------------------------------------------

struct SmemPlan {
    uint32_t ctx, mbar, ctl, x, u, up, uc, lg, lkey, lidx;
    uint32_t rt, wsg, sgq, ssb, sdq, sdsb;
    uint32_t ring, rsb, rdsb;
    uint32_t hs, uhs, hj, uhj, hv, sp, spd;
    uint32_t total;
};

constexpr uint32_t kCtxBytes = 1024;  // room for the kernel's block context
constexpr int kNumMbar = kWarps + 3;  // ring slots, routed scales, dense prefetch, shared down
// control words: sel_idx[kMaxK], sel_w[kMaxK], sel_slot[kMaxK], red[64], misc[16], imisc[16]
constexpr int kCtlWords = 3 * kMaxK + 64 + 16 + 16;

MOE_HD uint32_t align_to(uint32_t v, uint32_t a) { return (v + a - 1) & ~(a - 1); }

MOE_HD SmemPlan smem_plan(int H, int E, int k, int I, int Is, int bits, int G)
{
    const StageGeo sg = stage_geo(H, E, k, I, Is, bits, G);
    const int xp = (bits == 8) ? 2 : 1;           // int8 codes are read as two nibbles
    const int KU = H * xp;                         // expanded length of u
    const int NCu = KU / kChunk;
    const int KD = I * xp, KDs = Is * xp;
    const int NCd = KD / kChunk, NCds = KDs / kChunk;
    const int ngu = H / 64, ngd = I / 64, ngds = Is / 64;
    const int rb_gu = H * bits / 8, rb_ds = Is * bits / 8;
    SmemPlan s{};
    uint32_t o = 0;
    auto take = [&](uint32_t& field, uint32_t bytes, uint32_t a) {
        o = align_to(o, a);
        field = o;
        o += bytes;
    };
    take(s.ctx, kCtxBytes, 16);
    take(s.mbar, 8u * kNumMbar, 16);
    take(s.ctl, 4u * kCtlWords, 16);
    take(s.x, 4u * H, 16);
    take(s.u, 2u * H, 16);
    take(s.up, 2u * KU, 16);
    take(s.uc, 8u * NCu, 16);
    take(s.lg, 4u * (E > 32 ? E : 32), 16);
    take(s.lkey, 4u * (kMaxE + 2 * kWarps + 8), 16);
    take(s.lidx, 4u * (kMaxE + 2 * kWarps + 8), 16);
    take(s.rt, 2u * sg.Rr * H, 128);
    take(s.wsg, 2u * H, 16);
    take(s.sgq, 2u * sg.Rs * rb_gu, 128);
    take(s.ssb, 4u * sb_span_max(sg.Rs, 2 * ngu), 16);
    take(s.sdq, (uint32_t)sg.Rsd * rb_ds, 128);
    take(s.sdsb, 2u * sb_span_max(sg.Rsd, 2 * ngds), 16);
    take(s.ring, (uint32_t)kWarps * sg.slot_bytes, 1024);
    take(s.rsb, 4u * sb_span_max(sg.Rgu, 2 * ngu), 16);
    take(s.rdsb, 2u * sb_span_max(sg.Rd, 2 * ngd), 16);
    take(s.hs, 2u * 2 * KDs, 16);
    take(s.uhs, 8u * NCds, 16);
    take(s.hj, 2u * 2 * KD, 16);
    take(s.uhj, 8u * NCd, 16);
    take(s.hv, 4u * xh_stride(I, Is), 16);
    const int spr = sg.Rgu > sg.Rs ? sg.Rgu : sg.Rs;
    take(s.sp, 4u * spr * 2 * sg.ncb_gu, 16);
    const int sdr = sg.Rd > sg.Rsd ? sg.Rd : sg.Rsd;
    const int ncb_ds = cdiv(NCds, 4);
    const int sdc = sg.ncb_d > ncb_ds ? sg.ncb_d : ncb_ds;
    take(s.spd, 4u * sdr * sdc, 16);
    s.total = align_to(o, 16);
    return s;
}

}  // namespace moe
