// host.h -- host-side helpers shared by the entry points: TMA map encoding over an expert arena
// and the epoch bookkeeping of the exchange buffers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "layout.h"

namespace moe {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link against libcuda).
inline EncodeTiledFn encode_tiled_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// The three code sections (gate.q, up.q, down.q) of every blob of an arena of n_slots blobs as 4D
// byte tensors: (byte in a column block, row, column block, slot) with strides (row bytes, column
// block bytes, blob stride); a box is the decode kernel's copy of bh rows by cpg (down) or cpp
// (a gate/up piece) column blocks, 128-byte swizzled when rows are at least 128 bytes wide. Returns 0 or a CUresult (-1: no driver
// entry point).
inline int encode_arena_maps(CUtensorMap (&maps)[3], const uint8_t* arena, int n_slots, const BlobGeo& geo,
                             const StageGeo& sg)
{
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn)
        return -1;
    for (int m = 0; m < 3; ++m) {
        const bool dn = m == 2;
        const int cbw = dn ? sg.cbw_d : sg.cbw_gu, ncb = dn ? sg.ncb_d : sg.ncb_gu;
        const cuuint64_t dims[4] = {(cuuint64_t)cbw, (cuuint64_t)geo.rows[m], (cuuint64_t)ncb, (cuuint64_t)n_slots};
        const cuuint64_t strides[3] = {(cuuint64_t)geo.row_bytes[m], (cuuint64_t)cbw, (cuuint64_t)geo.stride};
        const cuuint32_t box[4] = {(cuuint32_t)cbw, (cuuint32_t)(dn ? sg.bh_d : sg.bh_gu),
                                   (cuuint32_t)(dn ? sg.cpg_d : sg.cpp_gu), 1};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        const CUtensorMapSwizzle swz = (dn ? sg.swz_d : sg.swz_gu) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
        const CUresult r = fn(&maps[m], CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, (void*)(arena + geo.q_off[m]), dims, strides,
                              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return (int)r;
    }
    return 0;
}

// Code sections (gate, up, down) as 3D byte tensors [slots][rows][row bytes] with boxes of one
// pipeline slice (64 bytes of codes: 128 elements at int4, 64 at int8) by 64 rows (gate, up) or
// 128 rows (down), 64-byte swizzled (16-byte chunk c of row r lands at chunk c ^ ((r >> 1) & 3), so
// the dequantising threads, one row each, read without bank conflicts):
// the tiles the batched path's dequantising warps read. `base` is the arena (n_slots blobs at
// `stride`) or one blob (n_slots = 1).
inline int encode_slice_maps(CUtensorMap (&maps)[3], const uint8_t* base, int n_slots, uint64_t stride,
                             const BlobGeo& geo, int /*bits*/)
{
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn)
        return -1;
    for (int m = 0; m < 3; ++m) {
        const cuuint64_t dims[3] = {(cuuint64_t)geo.row_bytes[m], (cuuint64_t)geo.rows[m], (cuuint64_t)n_slots};
        const cuuint64_t strides[2] = {(cuuint64_t)geo.row_bytes[m], (cuuint64_t)stride};
        const cuuint32_t box[3] = {64u, m == 2 ? 128u : 64u, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        const CUresult r = fn(&maps[m], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, (void*)(base + geo.q_off[m]), dims, strides,
                              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return (int)r;
    }
    return 0;
}

// A row-major 16-bit matrix [rows][cols] (bf16 or fp16) with boxes of 64 columns (128 bytes) x
// box_rows rows, 128-byte swizzled: the K-major operand tiles of the tensor cores.
inline int encode_tiles16(CUtensorMap* map, const void* ptr, int cols, int rows, int box_rows, bool fp16)
{
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn)
        return -1;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = fn(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(ptr), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : (int)r;
}

// Staging plan of the fused kernel for a shape on `grid` blocks (one per SM): k + 1 groups of
// blocks (the routed experts and the shared expert); every byte a block reads of its expert
// fetched at once when that fits in shared memory, else the gate/up rows in column groups that
// take turns in fewer slots. Returns the dynamic shared memory bytes and the two geometries, or 0
// when the shape cannot be staged (fewer blocks than groups, or too little shared memory).
inline uint32_t plan_decode(int H, int E, int k, int I, int Is, int bits, int grid, int smem_optin, StageGeo* sg,
                            StageGeo* sgs)
{
    if (grid < k + 1 || grid > kMaxGrid)
        return 0;
    for (int ncs = 1; ncs <= 16; ncs *= 2)
        for (int nslot = ncs; nslot >= 1; nslot /= 2) {
            const StageGeo g = stage_geo(H, I, bits, grid, k + 1, ncs, nslot);
            const StageGeo gs = stage_geo(H, Is, bits, grid, k + 1, ncs, nslot);
            if (g.nslot_gu > kMaxGuSlots || gs.nslot_gu > kMaxGuSlots || g.ncs_gu != ncs)
                continue;
            const uint32_t bytes = smem_plan(H, E, I, Is, bits, grid, g, gs).total + 1024;
            if (bytes <= (uint32_t)smem_optin) {
                *sg = g;
                *sgs = gs;
                return bytes;
            }
        }
    return 0;
}

// Epochs of the exchange buffers: a launch of n steps takes [epoch0, epoch0 + n). When the 32-bit
// counter would wrap, the caller clears the buffers (so no stale pair can match) and starts at 1.
inline bool next_epochs(uint32_t& counter, uint32_t n, uint32_t* epoch0)
{
    bool reset = false;
    if (counter == 0 || (uint64_t)counter + n >= 0xFFFFFFF0ull) {
        counter = 1;
        reset = true;
    }
    *epoch0 = counter;
    counter += n;
    return reset;
}

}  // namespace moe
