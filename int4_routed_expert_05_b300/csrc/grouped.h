// grouped.h -- parameters of the batched layer's tensor-core GEMMs (tcgen05), shared by the host
// entry point and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "layout.h"

namespace moe {
namespace tc {

constexpr int kNT = 128;          // tokens per task at most (the N of one MMA tile)
constexpr int kKS = 64;           // K elements of one operand sub-tile: one quantisation group, one 128-byte row
constexpr int kTiles = 4;         // operand sub-tiles of A (and of B) in shared memory, grouped into stages
constexpr int kCodeRow = 64;      // bytes of one row's codes in one pipeline slice (one TMA box row)
// Expert-GEMM pipeline slice: 64 bytes of codes per row, i.e. 128 K elements (two sub-tiles) at
// int4 and 64 (one sub-tile) at int8; kTiles / sub stages of sub sub-tiles each.
__host__ __device__ constexpr int slice_sub(int bits) { return bits == 4 ? 2 : 1; }
constexpr int kStagesR = 6;       // A/B operand stages of the router GEMM
constexpr int kTileBytes = 128 * 128;  // one 128-row x 64-element fp16/bf16 operand tile
constexpr int kCodeRing = 32768;  // bytes of the staged-code ring
constexpr int kThreadsX = 480;    // expert kernel: 8 dequant, 4 epilogue, code TMA, MMA, operand-B TMA warps
constexpr int kBRows = 16;        // rows of one B-operand TMA box
constexpr int kThreadsR = 192;    // router kernel: 4 epilogue, 1 TMA, 1 MMA warps
constexpr int kTmemCols = 256;    // two accumulators of kNT fp32 columns

struct GroupedArgs {
    CUtensorMap map_q[2][3];  // codes of gate, up, down: [0] over the arena's slots, [1] over the shared blob
    CUtensorMap map_wr;       // router weights bf16 [E][H], 128B-swizzled boxes of 128 rows x 64
    CUtensorMap map_u;        // layer input bf16 [T][H], boxes of 128 tokens x 64
    CUtensorMap map_b[2];     // expert B operands, fp16 rows of 64 elements in boxes of 16 rows:
                              // [0] input rows in assignment order [A][H], [1] h rows [A][Imax]
    BlobGeo geo, geo_s;
    int T, H, E, k, I, Is, bits, Imax;
    const uint8_t* arena;
    uint64_t stride;
    const int32_t* table;     // [E] slot of each routed expert of this layer
    const uint8_t* shared_blob;
    const int32_t* list;      // [A] token of each assignment, grouped by expert
    const float* aw;          // [A] combine weight of each assignment
    const __half* us;         // [A][H] input rows in assignment order, K-permuted (the small-T path
                              // reads them directly; the GEMMs through map_b[0])
    __half* hbuf;             // [A][Imax] SwiGLU output, K-permuted (see kperm)
    float* y;                 // [T][H] output, zeroed before the down GEMM (fp32 reductions)
    float* ypart;             // [A][H] weighted down rows per assignment (deterministic combine), or null
    float* logits;            // [T][E]
    const int4* tasks;        // {expert, m0, n0, n} per task
    const int32_t* n_tasks;   // device count of tasks
    int* status;
    long long timeout_cycles;
};

// Position of element j (0..7) of an 8-element K block in the fp16 operand rows: the dequantiser
// emits code pairs in the order the packed words hold them (int4: nibbles j and j+4 of a 32-bit
// word; int8: bytes j and j+2 of a 16-bit pair), so activations are stored in that same order.
__host__ __device__ inline int kperm(int j, int bits)
{
    return bits == 4 ? (((j & 3) << 1) | (j >> 2)) : ((j & 4) | ((j & 1) << 1) | ((j >> 1) & 1));
}

// Dynamic shared memory of the expert kernel.
struct XPlan {
    uint32_t a, b, code, code_stage, n_code, sc, sc_bytes, xch, bar, total;
};

__host__ __device__ inline XPlan xplan(int H, int Imax, int bits)
{
    XPlan p{};
    uint32_t o = 0;
    p.a = o;
    o += kTiles * kTileBytes;
    p.b = o;
    o += kTiles * kTileBytes;
    p.code = o;
    p.code_stage = 128 * kCodeRow;
    (void)bits;
    p.n_code = kCodeRing / p.code_stage;
    o += kCodeRing;
    p.sc = o;
    const int gmax = (H > Imax ? H : Imax) / kKS;
    p.sc_bytes = (uint32_t)(128 * gmax * 4 + 15) / 16 * 16;
    o += 2 * p.sc_bytes;
    p.xch = o;
    o += 64 * 17 * 4;
    p.bar = (o + 15) / 16 * 16;
    o = p.bar + 64 * 8 + 16;
    p.total = o;
    return p;
}

void launch_router_gemm(const GroupedArgs& A, int grid, cudaStream_t st);
void launch_expert_gemm(int kind, const GroupedArgs& A, const int4* tasks, const int32_t* n_tasks, int grid,
                        cudaStream_t st);
size_t router_smem_bytes();
size_t expert_smem_bytes(int H, int Imax, int bits);

}  // namespace tc
namespace gv {
// The small-token path (gemv.cu): the two expert products as matrix-vector products for token
// counts up to kMaxTokens, on the same task lists and buffers as the GEMMs.
constexpr int kMaxTokens = 64;
size_t smem_bytes(int H, int Imax, int bits);
bool geometry_ok(const BlobGeo& g);  // every section and row 16-byte aligned (row bulk copies)
void launch(int kind, const tc::GroupedArgs& A, const int4* tasks, const int32_t* n_tasks, int grid, cudaStream_t st);
}  // namespace gv

}  // namespace moe
