// layout.h -- blob geometry, launch parameters, work split and shared-memory plan of the decode
// kernel.
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
constexpr int kChunk = 64;      // 4-bit fields per MMA chunk (one int4 quantisation group)
constexpr int kCb = 128;        // bytes of one staged column block (the 128-byte swizzle span)
constexpr int kMaxBoxRows = 256;
constexpr uint64_t kStrideAlign = 4096;
constexpr int kMaxGrid = 512;   // most blocks a decode launch may have (one per SM)
constexpr int kRouterParts = 4; // a router row's dot product is cut into this many fixed parts

// Row stride (in pairs) of the h exchange buffer: rows 0..k-1 hold the routed experts' h, row k
// the shared expert's.
MOE_HD int xh_stride(int I, int Is) { return I > Is ? I : Is; }

// Output words: each of the k + 1 expert contributions to output element o adds
// (round(v * 2^32) << 8) + 1 to word o, so the low byte counts the contributions that have
// landed and the upper 56 bits hold their exact fixed-point sum, whatever the arrival order.
constexpr float kFix = 4294967296.f;       // 2^32
constexpr float kFixInv = 2.3283064365386963e-10f;
constexpr float kFixMax = 4194304.f;       // largest |contribution| accepted (2^22)
constexpr int kCountBits = 8;

// device status codes (same values as moe_status)
constexpr int kStatusInvalid = 1;
constexpr int kStatusNotResident = 3;
constexpr int kStatusTimeout = 6;
constexpr int kStatusRange = 8;

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
MOE_HD int imin(int a, int b) { return a < b ? a : b; }
MOE_HD int imax(int a, int b) { return a > b ? a : b; }

constexpr int kMaxCopies = 64;         // planned copies of a block's expert bytes per step
constexpr int kMaxExpects = 64;        // their mbarriers
// mbarriers: gate/up copy pieces [kMaxGuBars] (slot s, matrix m (gate 0, up 1), piece p: bit
// (2s + m) * npc + p), then down copies, then the dense copies.
constexpr int kMaxGuSlots = 8;
// Pieces per gate/up copy. Measured on the 80B-shaped stack: with every block's copies in flight at
// once, a block's first 10 KB piece landed no earlier than its whole 43 KB gate copy did (the
// memory system serves all blocks' requests interleaved), while 8 pieces per matrix raised the
// copies per block from 9 to 23 and the issue time from 0.6 to 1.3 us. So one piece.
constexpr int kMaxPieces = 1;
constexpr int kMaxGuBars = 32;
constexpr int kMbDown = kMaxGuBars, kMbDense = kMbDown + 1;
constexpr int kNumMbar = kMbDown + 2;

// The k routed experts of a step and the shared expert are served by k + 1 groups of blocks:
// group j < k serves the expert of rank j, group k the shared expert.
// How one block's share of an expert is staged. Block i of a group owns gate/up rows
// [i * SRgu, (i + 1) * SRgu) and down rows [i * SRd, (i + 1) * SRd), clipped to the matrix. They
// are fetched by a few large tensor copies: a copy is a box of bh rows by cpg column blocks (a
// column block is 128 bytes, 128-byte swizzled, or the whole row when rows are narrower) and lands
// as [column block][row][column-block bytes]. Rows a box reads beyond the block's range lie past
// the end of the matrix (zero-filled by the copy engine, no memory traffic), because SRgu and SRd
// are whole multiples of the box heights. Gate and up rows are fetched in ncs_gu column groups; a
// slot holds the gate and the up copies of one group, and with fewer slots than groups
// (nslot_gu < ncs_gu) the groups take turns (a slot is refilled once the block is done with it).
// A gate or up copy goes out as npc_gu pieces of cpp_gu column blocks, each on its own mbarrier,
// so that the work on a piece starts as soon as it lands. Down rows are fetched all at once. Routed and shared experts have one geometry each (their
// intermediate sizes may differ).
struct StageGeo {
    int SRgu, SRd;         // gate/up rows and down rows per block of a group
    int bh_gu, bh_d;       // box rows (<= 256)
    int nr_gu, nr_d;       // boxes along the rows: SRgu = nr_gu * bh_gu, SRd = nr_d * bh_d
    int cbw_gu, cbw_d;     // bytes per column block
    int swz_gu, swz_d;     // 1: 128-byte swizzled boxes, 0: linear boxes
    int ncb_gu, ncb_d;     // column blocks per gate/up row / down row
    int cpg_gu, cpg_d;     // column blocks per copy
    int ncs_gu, ncs_d;     // column groups
    int nslot_gu;          // gate/up column-group slots
    int cpp_gu, npc_gu;    // a gate/up copy in npc_gu pieces of cpp_gu column blocks, each on its own mbarrier
    uint32_t gu_copy;      // shared-memory bytes of one gate (or up) copy, 1024-aligned
    uint32_t d_copy;       // shared-memory bytes of one down copy, 1024-aligned
};

MOE_HD uint32_t align1k(uint32_t v) { return (v + 1023u) & ~1023u; }

// Geometry of an expert with intermediate size Ie served by groups of at least G / ngroups
// blocks. ncs_gu / nslot_gu: column groups and slots of the gate/up rows (1 / 1 fetches every
// gate/up byte of the block at once).
MOE_HD StageGeo stage_geo(int H, int Ie, int bits, int G, int ngroups, int ncs_gu, int nslot_gu)
{
    StageGeo s{};
    const int nmin = imax(1, G / ngroups);  // smallest group
    const int rgu = cdiv(Ie, nmin), rd = cdiv(H, nmin);
    s.nr_gu = cdiv(rgu, kMaxBoxRows);
    s.bh_gu = cdiv(rgu, s.nr_gu);
    s.SRgu = s.nr_gu * s.bh_gu;
    s.nr_d = cdiv(rd, kMaxBoxRows);
    s.bh_d = cdiv(rd, s.nr_d);
    s.SRd = s.nr_d * s.bh_d;
    const int rb_gu = H * bits / 8, rb_d = Ie * bits / 8;
    s.swz_gu = rb_gu >= kCb;
    s.swz_d = rb_d >= kCb;
    s.cbw_gu = s.swz_gu ? kCb : rb_gu;
    s.cbw_d = s.swz_d ? kCb : rb_d;
    s.ncb_gu = cdiv(rb_gu, s.cbw_gu);
    s.ncb_d = cdiv(rb_d, s.cbw_d);
    s.ncs_gu = imax(1, imin(ncs_gu, s.ncb_gu));
    s.cpg_gu = cdiv(s.ncb_gu, s.ncs_gu);
    s.ncs_gu = cdiv(s.ncb_gu, s.cpg_gu);
    s.nslot_gu = imax(1, imin(nslot_gu, s.ncs_gu));
    s.ncs_d = 1;
    s.cpg_d = s.ncb_d;
    // pieces: the most (up to kMaxPieces) that divide the copy's column blocks evenly, fit the
    // mbarriers, and start on the swizzle period (1024 bytes) when the rows are swizzled
    s.npc_gu = 1;
    for (int n = imin(kMaxPieces, s.cpg_gu); n > 1; --n)
        if (s.cpg_gu % n == 0 && 2 * s.nslot_gu * n <= kMaxGuBars &&
            (!s.swz_gu || ((s.cpg_gu / n) * s.bh_gu * s.cbw_gu) % 1024 == 0)) {
            s.npc_gu = n;
            break;
        }
    s.cpp_gu = s.cpg_gu / s.npc_gu;
    s.gu_copy = align1k((uint32_t)s.cbw_gu * s.bh_gu * s.cpg_gu);
    s.d_copy = align1k((uint32_t)s.cbw_d * s.bh_d * s.cpg_d);
    return s;
}

// Staging bytes of a geometry: its gate/up slots and its down copies.
MOE_HD uint32_t stage_bytes(const StageGeo& g)
{
    return (uint32_t)g.nslot_gu * 2 * g.nr_gu * g.gu_copy + (uint32_t)g.nr_d * g.d_copy;
}

// Shared-memory room for the scale or bias rows [r0, r0 + n) of a section whose rows hold row_b
// bytes: the 16-byte aligned superset a 1D bulk copy fetches, rounded up to 16 bytes so that
// consecutive spans stay valid bulk-copy destinations.
MOE_HD uint32_t sb_span_max(int nrows, int row_b) { return ((uint32_t)(nrows * row_b + 32) + 15u) & ~15u; }

// ------------------------------------------------------------------------------------------
// Launch parameters
// ------------------------------------------------------------------------------------------

struct StepParams {
    // 4D TMA maps over the arena: bytes of a column block x rows x column blocks x slots, for
    // gate.q, up.q and down.q
    CUtensorMap tmap[3];
    int H, E, k, I, Is, bits, group, flags;
    BlobGeo geo, geo_s;           // routed / shared blob geometry
    StageGeo sg, sgs;             // staging of a routed / the shared expert's rows
    const CUtensorMap* smaps;     // [L][3] the same maps over each layer's shared-expert blob (workspace)
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
    long long* xacc;              // [3][H] counted fixed-point output words (step % 3)
    unsigned long long* xflag;    // step counter: every block adds 1 once its contributions to a step's output words are in
    unsigned long long* bar;      // launch-start barrier counter (a multiple of the grid between launches)
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
    uint32_t ctx, mbar, ctl, x, u, up, uc, lg, tk;
    uint32_t rt, wsg, tab, bias, ld, cp;
    uint32_t ring, rsb, rdsb;
    uint32_t hj, uhj, hv, sp, spd, rp;
    uint32_t total;
};

constexpr uint32_t kCtxBytes = 1024;   // room for the kernel's block context
// control words: sel_idx[kMaxK], sel_w[kMaxK], sel_slot[kMaxK], red[64], misc[32], imisc[16]
constexpr int kCtlWords = 3 * kMaxK + 64 + 32 + 16;

MOE_HD uint32_t align_to(uint32_t v, uint32_t a) { return (v + a - 1) & ~(a - 1); }

MOE_HD SmemPlan smem_plan(int H, int E, int I, int Is, int bits, int G, const StageGeo& sg, const StageGeo& sgs)
{
    const int xp = (bits == 8) ? 2 : 1;           // int8 codes are read as two 4-bit fields
    const int KU = H * xp;                         // expanded length of u
    const int NCu = KU / kChunk;
    const int Im = imax(I, Is);
    const int KD = Im * xp, NCd = KD / kChunk;
    const int ngu = H / 64, ngd = Im / 64;
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
    take(s.lg, 4u * imax(E, 32), 16);
    take(s.tk, 16u + 8u * kMaxE + 4u * kWarps, 16);
    take(s.rt, 2u * cdiv(E, G) * H, 128);
    take(s.wsg, 2u * H, 16);
    take(s.tab, 4u * E + 32, 16);
    take(s.ld, 2u * (uint32_t)sizeof(LayerDesc), 16);
    take(s.cp, 16u * kMaxCopies + 8u * kMaxExpects, 16);
    take(s.bias, 4u * E, 16);
    take(s.ring, imax((int)stage_bytes(sg), (int)stage_bytes(sgs)), 1024);
    const int srgu = imax(sg.SRgu, sgs.SRgu), srd = imax(sg.SRd, sgs.SRd);
    take(s.rsb, 4u * sb_span_max(srgu, 2 * ngu), 16);
    take(s.rdsb, 2u * sb_span_max(srd, 2 * ngd), 16);
    take(s.hj, 2u * 2 * KD, 16);
    take(s.uhj, 8u * NCd, 16);
    take(s.hv, 4u * Im, 16);
    take(s.sp, 4u * srgu * 2 * imax(sg.ncb_gu, sgs.ncb_gu), 16);
    take(s.spd, 4u * srd * imax(sg.ncb_d, sgs.ncb_d), 16);
    take(s.rp, 4u * imax(cdiv(E, G), 1) * kRouterParts, 16);
    s.total = align_to(o, 16);
    return s;
}

}  // namespace moe
