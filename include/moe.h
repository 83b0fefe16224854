/*
 * moe.h -- C ABI of libmoe: the routed-expert Mixture-of-Experts FFN for batch-1 decode on
 * B300 (sm_103a), with a fixed-stride pool of int4/int8 group-quantised expert blobs.
 *
 * Per token and layer the library computes
 *     logits = Wr u (+ bias);  idx, w = top-k(logits) with renormalised softmax weights
 *     y      = sum_j w_j * Wd_j (silu(Wg_j u) * (Wu_j u))  +  sigmoid(w_sg . u) * S(u)
 * where expert j's gate/up/down matrices sit in one blob at  arena + slot * stride  and S is the
 * always-on shared expert in the same blob format.
 *
 * Sources (web pages about the Swiftlet runtime; no code is printed on them):
 *  [qpack]  paotong.dev commentary on Swiftlet (paotong.dev/a/b3a48bd74abb1ebf): routed experts
 *           are repacked into one fixed-stride blob each and fetched with one read at
 *           blobBase + expertIndex * expertStride; a bounded pool caches hot experts with LFU
 *           plus recency eviction (reported hit rate 43-70%).
 *  [route]  cheshm.ai, "Swiftlet fits an 80B-level Qwen giant into Mac", paragraph on scheduling:
 *           each layer routes a token to 10 of 512 (80B) or 8 of 256 (35B) experts; router and
 *           shared experts stay resident; popular experts are cached in a bounded pool with LFU
 *           and recency.
 *  [quant]  same item, closing paragraph: MLX-style int4/int8 group quantisation, byte-addressed
 *           kernels with 64-bit offsets, high-sparsity MoE with shared experts.
 *  [renorm] alphalab.site, "Swiftlet 實測資料解讀", section on the 35B correctness fix: top-k
 *           routing weights are renormalised (norm_topk_prob = true).
 *  [size]   same page, section on SSD reads: with no cache hits the 80B model requests at most
 *           480 experts (about 810 MiB) per token, i.e. 1,769,472 bytes per expert.
 *
 * Conventions for every entry point:
 *  - Pointers named d_* are device pointers owned by the caller (for instance PyTorch tensors);
 *    pointers named h_* are host pointers owned by the caller. The library never frees them.
 *  - Streams are cudaStream_t values passed as void*; NULL is the legacy default stream.
 *  - Work is enqueued on the given stream and the call returns without waiting for it, unless
 *    the entry point says otherwise. No entry point allocates device memory after
 *    moe_pool_create.
 *  - Errors are returned as moe_status codes; moe_last_error() gives a message (per thread).
 *    Nothing throws across the ABI, exits, or traps on the device. Problems found by a kernel
 *    (an expert that is not resident, a device-side wait that timed out, a value the fp16
 *    operands cannot hold) are written to a device status word that moe_device_status() reads.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_E_INVALID = 1,       /* bad argument (null pointer, out-of-range index, misalignment) */
    MOE_E_SHAPE = 2,         /* shape outside what the kernels support */
    MOE_E_NOT_RESIDENT = 3,  /* a selected expert has no slot in the pool */
    MOE_E_POOL_FULL = 4,     /* every slot is pinned by the step in flight */
    MOE_E_CUDA = 5,          /* a CUDA runtime call failed (message in moe_last_error) */
    MOE_E_TIMEOUT = 6,       /* a device-side wait ran past its limit */
    MOE_E_NOMEM = 7,         /* workspace or arena too small */
    MOE_E_RANGE = 8          /* a value outside what the kernels' fp16 operands hold (device status):
                              * an input, activation or h value above 65504 in magnitude; on the
                              * batched path's GEMMs also a scale below fp16's normal range (2^-14)
                              * or a weight s q + b that would overflow fp16 (the MOE_GEMV path
                              * applies scales in fp32 and has no such limit) */
} moe_status;

/* flags of moe_shape.flags */
#define MOE_RENORM   1  /* renormalise the top-k weights ([renorm]); off: full-softmax weights */
#define MOE_PRENORM  2  /* stack layer: u = bf16(x / sqrt(mean(x^2) + 1e-6)) from an fp32 residual */
#define MOE_RESIDUAL 4  /* stack layer: output x + y instead of y */
#define MOE_DETERMINISTIC 8 /* batched path: each token's k + 1 contributions summed in rank order,
                             * then the shared expert's, from a per-assignment buffer (bit for bit
                             * reproducible; 4 T (k + 1) H more workspace bytes) instead of fp32
                             * reductions in tile completion order. The decode kernels are always
                             * deterministic and ignore it. */
#define MOE_GEMV 16 /* batched path, T <= 64: the two expert products as matrix-vector products
                     * (each touched expert's rows streamed once into mma.sync fragments) instead
                     * of the tensor-core GEMMs. The weights enter exactly (codes as 1024 + q, the
                     * affine dequantisation per group in fp32), so any bf16 scale is exact here;
                     * results agree with the GEMMs within the path's tolerance. Off by default
                     * (measured on B300 against the GEMMs). The decode kernels ignore it. */

/* One MoE FFN layer. hidden H, n_experts E, top_k k, inter I (routed expert), shared_inter Is,
 * bits 4 or 8, group 64. Supported: H % 256 == 0, I % 64 == 0, Is % 64 == 0, 1 <= k <= 16,
 * k <= E <= 512, group == 64. */
typedef struct {
    int32_t hidden, n_experts, top_k, inter, shared_inter, bits, group, flags;
} moe_shape;

/* ----------------------------------------------------------------------------------------- */
/* Blob format ([qpack], [quant], [size])                                                     */
/* ----------------------------------------------------------------------------------------- */
/*
 * One expert = one contiguous blob, sections in this order with no gaps:
 *   gate.q | up.q | down.q | gate.s | gate.b | up.s | up.b | down.s | down.b
 * gate, up: [I][H] (out x in); down: [H][I]. Codes row-major, packed along the input dimension:
 * int4 element c of a row is in byte c/2 of the row, low nibble for even c, high nibble for odd c;
 * int8 codes take one byte. Scale s and bias b: bf16, row-major [out][in/64]; the weight is
 * w = s * q + b with q the unsigned code. Blobs sit stride bytes apart, stride = blob bytes
 * rounded up to 4096. For hidden 2048, inter 512, int4 both are 1,769,472 bytes ([size]).
 */

/* Bytes of one blob (shared = 1: the shared expert, whose inter is shape->shared_inter); 0 for a
 * NULL shape or one without a blob (bits not 4 or 8, sizes not whole positive groups). */
size_t moe_expert_bytes(const moe_shape* shape, int shared);
/* Distance between consecutive blobs in a pool or host store (0 as for moe_expert_bytes). */
size_t moe_expert_stride(const moe_shape* shape, int shared);

/* Write one blob into h_blob (moe_expert_stride bytes, host; the padding is zeroed).
 * h_codes[m]: uint8 [out][in] codes of matrix m (0 gate, 1 up, 2 down), each < 2^bits;
 * h_scale[m], h_bias[m]: bf16 bit patterns [out][in/64]. Host-only, synchronous. */
moe_status moe_pack_expert(const moe_shape* shape, int shared, const uint8_t* const h_codes[3],
                           const uint16_t* const h_scale[3], const uint16_t* const h_bias[3],
                           void* h_blob);

/* ----------------------------------------------------------------------------------------- */
/* Expert pool ([qpack], [route])                                                             */
/* ----------------------------------------------------------------------------------------- */
/*
 * A pool is host metadata over a caller-owned device arena of n_slots blobs at a fixed stride,
 * plus a caller-owned device workspace (size from moe_workspace_bytes) that holds the
 * (layer, expert) -> slot table, the per-layer weight pointers and the kernels' scratch.
 * It serves both modes:
 *  - resident: every expert of every layer is placed once (moe_pool_place) and the fused kernels
 *    look slots up on the device, with no host round trip inside a step;
 *  - bounded: fewer slots than experts; per layer the caller routes (moe_route), looks up the
 *    selected experts (moe_pool_lookup), fills misses from a pinned host store
 *    (moe_pool_load_slot), runs moe_experts with the returned slots, then moe_pool_release.
 */
typedef struct moe_pool moe_pool;

/* One layer's resident dense weights (device pointers, caller-owned, 16-byte aligned). */
typedef struct {
    const void* router;        /* bf16 [E][H] */
    const void* shared_blob;   /* one blob of the shared expert (moe_expert_stride(shape, 1)) */
    const void* shared_gate;   /* bf16 [H], the shared expert's gate vector w_sg */
    const float* logit_bias;   /* fp32 [E] added to the router logits, or NULL. Not part of the
                                  method: a hook for synthetic routing-popularity workloads. */
} moe_layer_weights;

/* Device workspace bytes for a pool over n_layers layers of this shape. */
size_t moe_workspace_bytes(const moe_shape* shape, int32_t n_layers);

/* Create a pool. d_arena: n_slots * moe_expert_stride(shape, 0) bytes (4096-aligned);
 * d_workspace: moe_workspace_bytes bytes (256-aligned). Both stay owned by the caller and must
 * outlive the pool. Initialises the workspace on the current device (synchronous). */
moe_status moe_pool_create(const moe_shape* shape, int32_t n_layers, int32_t n_slots,
                           void* d_arena, size_t arena_bytes, void* d_workspace,
                           size_t workspace_bytes, moe_pool** out);
void moe_pool_destroy(moe_pool* pool);

/* Device address of a slot (arena + slot * stride), NULL if out of range. */
void* moe_pool_slot_ptr(const moe_pool* pool, int32_t slot);

/* Register layer `layer`'s dense weights (pointers are copied; takes effect at moe_pool_sync). */
moe_status moe_pool_set_layer(moe_pool* pool, int32_t layer, const moe_layer_weights* w);

/* Resident mode: declare that `slot` holds expert (layer, expert) (the caller wrote the blob).
 * A slot holds at most one expert; placing over an occupied slot evicts its previous expert. */
moe_status moe_pool_place(moe_pool* pool, int32_t layer, int32_t expert, int32_t slot);

/* Upload the slot table and layer weights to the workspace (enqueued on `stream`; the host
 * copies are staged before return). Call after set_layer/place and before forward calls. */
moe_status moe_pool_sync(moe_pool* pool, void* stream);

/* Bounded mode: look up n experts of `layer`. h_slots_out[i] = slot, or -1 on a miss.
 * Every call advances the pool's tick by one. A hit counts one more use of the slot and stamps
 * it with the tick; every expert passed (hit or later loaded) is pinned until moe_pool_release. */
moe_status moe_pool_lookup(moe_pool* pool, int32_t layer, const int32_t* h_experts, int32_t n,
                           int32_t* h_slots_out);

/* Bounded mode: place expert (layer, expert) in a slot and copy its blob from pinned host memory
 * h_blob (moe_expert_stride bytes) with cudaMemcpyAsync on copy_stream. The slot is the lowest
 * free one, else the unpinned slot with the smallest (use count, last tick, slot index): LFU with
 * recency as the tie-break. The copy waits (on copy_stream) for the last kernel that read the
 * evicted slot. The new entry has use count 1 and the current tick, and is pinned.
 * MOE_E_POOL_FULL if every slot is pinned. Returns the slot in *slot_out. */
moe_status moe_pool_load_slot(moe_pool* pool, int32_t layer, int32_t expert, const void* h_blob,
                              void* copy_stream, int32_t* slot_out);

/* Make `compute_stream` wait for the copies issued by moe_pool_load_slot since the last call. */
moe_status moe_pool_wait_loads(moe_pool* pool, void* compute_stream);

/* Record the end of the work enqueued so far on compute_stream as the last use of every pinned
 * slot, then unpin them all. */
moe_status moe_pool_release(moe_pool* pool, void* compute_stream);

/* Speculative copies in moe_stack_forward_streamed: the next layer's n best predicted experts (in
 * rank order; n >= top_k: all of them) that are not resident are copied ahead; 0 (the default)
 * turns it off. A guess costs link time when wrong and takes a slot, so it pays when the link has
 * room (a pool smaller than a token's working set) and costs when the link is already the limit.
 * Host-side setting, takes effect at the next call; MOE_E_INVALID for n < 0. */
moe_status moe_pool_set_prefetch(moe_pool* pool, int32_t n);

/* Counters since creation: lookups that hit, lookups that missed, bytes copied by load_slot. */
moe_status moe_pool_stats(const moe_pool* pool, int64_t* hits, int64_t* misses, int64_t* bytes_loaded);

/* ----------------------------------------------------------------------------------------- */
/* Forward passes                                                                             */
/* ----------------------------------------------------------------------------------------- */

/* One layer for n_tokens tokens taken one after another ([route], [quant], [renorm]).
 * d_x: bf16 [T][H] layer input u (or fp32 [T][H] residual x when the shape has MOE_PRENORM).
 * d_y: fp32 [T][H] layer output (y, or x + y with MOE_RESIDUAL).
 * d_topk_idx (int32 [T][k]) and d_topk_w (fp32 [T][k]): selected experts in rank order (largest
 * logit first, equal fp32 logits to the lower index) and their weights; either may be NULL.
 * Every selected expert must be placed (resident mode); one that is not sets the device status
 * MOE_E_NOT_RESIDENT and contributes nothing; an input or intermediate value above 65504 in
 * magnitude (the kernel's fp16 operands) sets MOE_E_RANGE. The sum over the k + 1 experts is exact
 * fixed-point integer arithmetic, so the output does not depend on pool placement or timing. One
 * cooperative kernel launch. */
moe_status moe_layer_forward(moe_pool* pool, int32_t layer, const void* d_x, int32_t n_tokens,
                             float* d_y, int32_t* d_topk_idx, float* d_topk_w, void* stream);

/* Layers [layer0, layer0 + n_layers) applied in order to one token, as a pre-norm residual
 * stack: x <- x + MoE_l(bf16(rmsnorm(x))) (the shape needs MOE_PRENORM | MOE_RESIDUAL).
 * d_x: fp32 [H] input residual; d_x_out: fp32 [H] final residual. d_trace (fp32
 * [n_layers + 1][H], or NULL) receives each layer's input and the final residual.
 * d_topk_idx / d_topk_w: [n_layers][k] or NULL. One cooperative kernel launch for all layers. */
moe_status moe_stack_forward(moe_pool* pool, int32_t layer0, int32_t n_layers, const float* d_x,
                             float* d_x_out, float* d_trace, int32_t* d_topk_idx, float* d_topk_w,
                             void* stream);

/* Bounded mode, first half of a layer: router and top-k only. d_x as for moe_layer_forward
 * (one token); writes d_topk_idx [k] and d_topk_w [k]. */
moe_status moe_route(moe_pool* pool, int32_t layer, const void* d_x, int32_t* d_topk_idx,
                     float* d_topk_w, void* stream);

/* Bounded mode, second half: experts and combine for one token given the selection.
 * d_topk_w: fp32 [k] weights from moe_route; h_slots: host int32 [k], the pool slot of each
 * selected expert in rank order (copied into the launch, so the array may be reused at once). */
moe_status moe_experts(moe_pool* pool, int32_t layer, const void* d_x, const float* d_topk_w,
                       const int32_t* h_slots, float* d_y, void* stream);

/* Bounded mode, a whole pre-norm residual stack for one token, driven on the host ([qpack],
 * [route]): per layer moe_route, a device-to-host read of the k selected experts (synchronous),
 * moe_pool_lookup, moe_pool_load_slot for every miss from h_blobs on copy_stream, moe_pool_wait_loads,
 * moe_experts and moe_pool_release. With prefetch set (moe_pool_set_prefetch, off by default) the
 * next layer is also routed on this layer's input, in the same synchronous read, and its best
 * predicted experts that are not resident are loaded behind this layer's misses while this layer
 * runs;
 * the next layer's real selection is looked up as usual, so the result does not depend on the
 * guess (a wrong one costs link time and slots). h_blobs: host array of pinned host blob pointers
 * indexed by absolute layer, entry [l * n_experts + e] for layer l (layers layer0 .. layer0 +
 * n_layers - 1 must be filled; moe_expert_stride bytes each; entries may repeat).
 * d_x: fp32 [H] input residual; d_x_out: fp32 [H] final residual (the pool workspace holds the
 * residuals in between). h_topk_idx: host int32 [n_layers][k] receiving the selections, or NULL.
 * Returns when the last layer has been enqueued on compute_stream. */
moe_status moe_stack_forward_streamed(moe_pool* pool, int32_t layer0, int32_t n_layers, const float* d_x,
                                      float* d_x_out, const void* const* h_blobs, void* compute_stream,
                                      void* copy_stream, int32_t* h_topk_idx);

/* Batched tokens (prefill or batched decode), one layer, resident experts: the same layer as
 * moe_layer_forward for each of n_tokens tokens (cheshm.ai item "Swiftlet fits an 80B-level Qwen
 * giant into Mac", scheduling and quantisation paragraphs; alphalab.site benchmark article, TTFT
 * sections: batched prefill is what the pages' runtime lacks), computed as GEMMs on the tensor
 * cores: router GEMM, per-token top-k (ties to the lower index) with renormalised weights and the
 * shared gate, a sort of the token-expert assignments by expert (the shared expert takes every
 * token), grouped gate/up GEMMs with SwiGLU and grouped down GEMMs whose weighted results are
 * added into d_y. Weights are dequantised to fp16 (w = s*q + b, one rounding); accumulation fp32.
 * The k + 1 contributions of a token are summed by fp32 reductions in tile completion order, so
 * d_y agrees run to run to fp32 rounding, not bit for bit.
 *   d_x        bf16 [T][H] device, 16-byte aligned (read only)
 *   d_y        fp32 [T][H] device, 16-byte aligned (overwritten)
 *   d_topk_idx int32 [T][k] device or NULL; d_topk_w fp32 [T][k] device or NULL
 *   d_work     caller-owned device workspace of at least moe_batched_workspace_bytes(shape, T)
 *              bytes, 256-byte aligned; its contents need no initialisation
 *   stream     cudaStream_t (as void*); all work is enqueued on it, no host synchronisation
 * Errors: MOE_E_SHAPE if the shape has MOE_PRENORM or MOE_RESIDUAL, if hidden, inter or
 * shared_inter is not a multiple of 64, or if the staging for `hidden` does not fit in shared
 * memory; MOE_E_NOMEM if work_bytes is too small; MOE_E_INVALID for T <= 0, misaligned pointers or
 * a device other than the pool's; MOE_E_CUDA for a launch or tensor-map failure. Device-side
 * problems (non-resident expert, wait timeout) go to the status word (moe_device_status).
 * moe_batched_workspace_bytes returns 0 for a NULL shape or n_tokens <= 0; it needs no GPU. */
size_t moe_batched_workspace_bytes(const moe_shape* shape, int32_t n_tokens);
/* Timing of the batched path's expert GEMMs (a measurement hook; the pages have no counterpart):
 * moe_pool_time_batched(pool, n) makes each following moe_layer_forward_batched call record a CUDA
 * event pair on its stream around its two expert-GEMM launches, in a ring of n pairs owned by the
 * pool (n = 0 turns it off); moe_pool_batched_gemm_ms waits for the recorded pairs and returns the
 * sum of their elapsed times (ms) and their count (at most n, the latest calls), then clears them. */
moe_status moe_pool_time_batched(moe_pool* pool, int32_t n_calls);
moe_status moe_pool_batched_gemm_ms(moe_pool* pool, float* h_total_ms, int32_t* h_calls);
moe_status moe_layer_forward_batched(moe_pool* pool, int32_t layer, const void* d_x, int32_t n_tokens, float* d_y,
                                     int32_t* d_topk_idx, float* d_topk_w, void* d_work, size_t work_bytes,
                                     void* stream);

/* Reference path: the same layer for one token with plain kernels (one thread per logit, one
 * thread per selection, one thread per output row, fp32 sums in index order). Used to cross-check
 * the fused kernel. Same arguments as moe_layer_forward with n_tokens = 1. */
moe_status moe_layer_forward_scalar(moe_pool* pool, int32_t layer, const void* d_x, float* d_y,
                                    int32_t* d_topk_idx, float* d_topk_w, void* stream);

/* ----------------------------------------------------------------------------------------- */
/* Expert container on disk ([qpack], [size])                                                  */
/* ----------------------------------------------------------------------------------------- */
/*
 * One file holds every routed expert of a stack as a fixed-stride blob, so that a miss costs one
 * positioned read and no index lookup: a 4096-byte header (magic "MOEQPCK1", version 1, the
 * moe_shape, layers, experts, blob bytes, stride, data offset 4096, file bytes), then blob
 * (layer l, expert e) at 4096 + (l * n_experts + e) * moe_expert_stride(shape, 0). Every blob
 * starts on a 4096-byte boundary, so a reader can bypass the page cache (O_DIRECT). Host-only;
 * no call needs a GPU. All calls are synchronous.
 */
typedef struct moe_qpack moe_qpack;
#define MOE_QPACK_DIRECT 1 /* open flag: read with O_DIRECT when the file system allows it */

/* Create (or truncate) the container at `path` for n_layers layers of `shape`'s routed experts,
 * write its header and size the file (unwritten blobs read as zeros). MOE_E_INVALID if the file
 * cannot be written; MOE_E_SHAPE for a shape without a blob size. */
moe_status moe_qpack_create(const char* path, const moe_shape* shape, int32_t n_layers, moe_qpack** out);
/* Open a container for reading. flags: MOE_QPACK_DIRECT or 0. n_threads: reader threads for the
 * parallel reads of moe_stack_forward_qpack (0: reads run on the calling thread). MOE_E_INVALID if
 * the file is missing, truncated or not of this format. */
moe_status moe_qpack_open(const char* path, int32_t flags, int32_t n_threads, moe_qpack** out);
/* The container's shape, layer count, blob stride, and whether it is read with O_DIRECT (1/0);
 * any output may be NULL. */
moe_status moe_qpack_info(const moe_qpack* q, moe_shape* shape, int32_t* n_layers, uint64_t* stride,
                          int32_t* direct);
/* Write one blob (moe_expert_stride bytes from h_blob, host memory) of a container opened by
 * moe_qpack_create. MOE_E_INVALID for a layer or expert out of range. */
moe_status moe_qpack_write(moe_qpack* q, int32_t layer, int32_t expert, const void* h_blob);
/* Read one blob (moe_expert_stride bytes) into h_dst (host memory; 4096-byte aligned when the
 * container reads with O_DIRECT). One positioned read. */
moe_status moe_qpack_read(moe_qpack* q, int32_t layer, int32_t expert, void* h_dst);
/* Close (a written container is flushed to the device first). NULL is a no-op. */
moe_status moe_qpack_close(moe_qpack* q);

/* Bounded mode as moe_stack_forward_streamed, with the misses read from the container `q` (which
 * must hold the pool's shape and layers layer0 .. layer0 + n_layers - 1) instead of a pinned host
 * store: per layer, the misses are read in parallel (one positioned read each, on the container's
 * reader threads) into slots of h_staging, a caller-owned pinned host buffer of n_staging blobs
 * (n_staging >= top_k, 4096-byte aligned), then copied to their pool slots on copy_stream. A
 * staging slot is reused only after its previous copy has completed. The speculative copies of
 * moe_pool_set_prefetch do not apply. MOE_E_INVALID for a container of another shape, too few
 * staging slots or a failed read. */
moe_status moe_stack_forward_qpack(moe_pool* pool, int32_t layer0, int32_t n_layers, const float* d_x, float* d_x_out,
                                   moe_qpack* q, void* h_staging, int32_t n_staging, void* compute_stream,
                                   void* copy_stream, int32_t* h_topk_idx);

/* ----------------------------------------------------------------------------------------- */
/* Forward pass that allocates nothing                                                         */
/* ----------------------------------------------------------------------------------------- */
/*
 * The pages have no counterpart of this entry point; it exists for callers that may not allocate
 * device memory at all: a plugin running inside a host application that owns every device
 * allocation, or a latency-critical loop that must never call cudaMalloc (which can synchronise
 * the device). Such a caller cannot provide the workspace that moe_pool_create needs.
 *
 * moe_layer_forward_static computes the same layer as moe_layer_forward (same kernel, same
 * arguments d_x, n_tokens, d_y, d_topk_idx, d_topk_w, same results) without a pool. Its scratch
 * (launch-barrier and step counters, status word, expert table, layer descriptor, the shared
 * expert's tensor maps, exchanged logits and intermediate activations, output words) is a
 * file-scope device array of MOE_STATIC_SCRATCH_BYTES that every GPU which loads the library
 * keeps until the process exits. It calls no cudaMalloc, cudaFree or other allocating routine.
 *  - d_experts: the n_experts routed blobs in the fixed-stride container layout, expert e at
 *    d_experts + e * moe_expert_stride(shape, 0) (256-byte aligned); w: the layer's resident
 *    weights as for moe_pool_set_layer. All caller-owned, device memory.
 *  - d_status (required, 4-byte aligned): a device int32 that receives the layer's device status
 *    (MOE_OK; MOE_E_TIMEOUT if a device-side wait ran past 2 s; MOE_E_RANGE as for
 *    moe_layer_forward); it is reset to MOE_OK by the call. NULL returns MOE_E_INVALID.
 *  - A shape whose scratch does not fit returns MOE_E_NOMEM (message in moe_last_error); other
 *    argument errors return MOE_E_INVALID or MOE_E_SHAPE before anything is enqueued.
 *  - The first call on a device does a one-time set-up with that device current (the scratch
 *    array's device address via cudaGetSymbolAddress, the SM count). Make that first call before
 *    any stream capture.
 *  - Every call on a device shares the one scratch array, which keeps the previous call's
 *    contents; each call resets the parts that must start at zero, and a call whose shape lays
 *    the array out differently from the previous call's clears its exchange buffers first.
 *    Calls that overlap on the GPU (issued on different streams without ordering) race on the
 *    array and give wrong results.
 * Enqueues a set-up kernel and the decode kernel (and a clear when the layout changed) on
 * `stream` and returns. */
#define MOE_STATIC_SCRATCH_BYTES (128 * 1024)
moe_status moe_layer_forward_static(const moe_shape* shape, const void* d_experts, const moe_layer_weights* w,
                                    const void* d_x, int32_t n_tokens, float* d_y, int32_t* d_topk_idx,
                                    float* d_topk_w, int32_t* d_status, void* stream);

/* ----------------------------------------------------------------------------------------- */
/* Status                                                                                      */
/* ----------------------------------------------------------------------------------------- */

/* Wait for `stream`, read and clear the pool's device status word into *h_status (a moe_status
 * value, MOE_OK if no kernel reported a problem). After MOE_E_TIMEOUT the launch-barrier counter
 * is reset too. Synchronous. */
moe_status moe_device_status(moe_pool* pool, void* stream, int32_t* h_status);

/* Limit, in nanoseconds, of every device-side wait of this pool's kernels (default 2 s). A wait
 * that runs past it sets MOE_E_TIMEOUT in the device status and the kernel returns. */
moe_status moe_pool_set_timeout(moe_pool* pool, uint64_t timeout_ns);

/* Number of thread blocks the cooperative kernels of this pool launch (one per SM). */
int32_t moe_pool_grid(const moe_pool* pool);

/* Message of the last error on the calling thread ("" if none). */
const char* moe_last_error(void);

/* ----------------------------------------------------------------------------------------- */
/* Inspection and test hooks                                                                  */
/* ----------------------------------------------------------------------------------------- */

/* Slot currently holding (layer, expert), -1 if none (host metadata; no device access). */
moe_status moe_pool_slot_of(const moe_pool* pool, int32_t layer, int32_t expert, int32_t* slot);

/* Replace the device copy of moe_pool_load_slot by a host callback fn(user, slot, h_blob, bytes)
 * (fn = NULL restores the copy). A nonzero return makes load_slot fail with MOE_E_CUDA and leave
 * the pool unchanged. Lets the slot policy and its failure handling run without a GPU on a
 * host-only pool (moe_pool_create with d_workspace = NULL). */
moe_status moe_pool_set_copy_hook(moe_pool* pool, int (*fn)(void* user, int32_t slot, const void* h_blob, size_t bytes),
                                  void* user);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
