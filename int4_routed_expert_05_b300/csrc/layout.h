// layout.h -- blob geometry, kernel parameters and shared-memory plan of the decode kernels.
//
// Blob format (one expert = one contiguous blob fetched at arena + slot * stride; paotong.dev
// commentary on Swiftlet, the fixed-stride .qpack container): sections gate.q | up.q | down.q |
// gate.s | gate.b | up.s | up.b | down.s | down.b. gate/up are [I][H], down is [H][I], codes
// packed along the input dimension (int4: element c in byte c/2, low nibble for even c), bf16
// scale and bias per 64 consecutive inputs (cheshm.ai item on Swiftlet: MLX-style int4/int8
// group quantisation). Stride = bytes rounded up to 4096.
#pragma once
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
constexpr int kMaxE = 512;      // experts per layer limit (one per thread of the top-k)
constexpr int kGuRows = 64;     // gate/up rows per batch (four 16-row MMA tiles)
constexpr int kDnRows = 16;     // down output rows per batch (one MMA tile)
constexpr int kChunk = 64;      // nibbles per MMA chunk (four m16n8k16 steps)
constexpr uint64_t kStrideAlign = 4096;

// device status codes (same values as moe_status)
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

// Parameters of one launch of the fused decode kernel (passed by value).
struct StepParams {
    int H, E, k, I, Is, bits, group, flags;
    BlobGeo geo, geo_s;           // routed / shared blob geometry
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
    float* logits;                // workspace [E]
    float* hbuf;                  // workspace [k + 1][max(I, Is)]
    float* xbuf;                  // workspace [H]
    unsigned long long* bar;      // workspace grid-barrier counter
    int* status;                  // workspace status word
    unsigned long long timeout_ns;
};

// Shared-memory plan of the fused kernel (byte offsets, 16-byte aligned).
struct SmemPlan {
    uint32_t x, u, up, uc, p, sb, hp, uh, pd, sbd, lg, lkey, lidx, sel_idx, sel_w, sel_slot, red, misc;
    uint32_t total;
};

MOE_HD uint32_t align16(uint32_t v) { return (v + 15u) & ~15u; }

MOE_HD SmemPlan smem_plan(int H, int E, int k, int I, int Is, int bits, int group)
{
    const int xp = (bits == 8) ? 2 : 1;          // int8 codes are read as two nibbles
    const int KU = H * xp;                        // expanded length of u
    const int NCu = KU / kChunk;                  // chunks along a gate/up row
    const int Imax = I > Is ? I : Is;
    const int KD = Imax * xp;
    const int NCd = KD / kChunk;
    const int ngu = H / group;
    const int ngd = Imax / group;
    SmemPlan s{};
    uint32_t o = 0;
    auto take = [&](uint32_t& field, uint32_t bytes) { field = o; o = align16(o + bytes); };
    take(s.x, 4u * H);
    take(s.u, 2u * H);
    take(s.up, 2u * KU);
    take(s.uc, 4u * NCu);
    take(s.p, 4u * kGuRows * 2 * NCu);
    take(s.sb, 2u * kGuRows * 2 * 2 * ngu);
    take(s.hp, 2u * (k + 1) * 2 * KD);
    take(s.uh, 4u * (k + 1) * NCd);
    take(s.pd, 4u * (k + 1) * kDnRows * NCd);
    take(s.sbd, 2u * (k + 1) * kDnRows * 2 * ngd);
    take(s.lg, 4u * (E > 32 ? E : 32));
    take(s.lkey, 4u * kWarps * kMaxK);
    take(s.lidx, 4u * kWarps * kMaxK);
    take(s.sel_idx, 4u * kMaxK);
    take(s.sel_w, 4u * kMaxK);
    take(s.sel_slot, 4u * kMaxK);
    take(s.red, 4u * 64);
    take(s.misc, 64u);
    s.total = o;
    return s;
}

}  // namespace moe
