// noalloc.cu -- moe_layer_forward_static: one MoE layer whose scratch lives in a file-scope device
// array, for callers that must not allocate device memory (see include/moe.h).
//
// The fused decode kernel needs scratch beyond its inputs and outputs: a grid-barrier counter, a
// status word, the expert -> blob table, the layer descriptor, the exchange buffers through which
// blocks share router logits and intermediate activations, and the output accumulators.
// moe_layer_forward takes
// that scratch from a caller-allocated workspace. This entry point takes it from
// g_static_scratch instead, a fixed-size array that every device loading the library holds until
// the process exits. The experts are read where the fixed-stride container puts them: expert e at
// d_experts + e * stride.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "../../include/moe.h"
#include "host.h"
#include "layout.h"

namespace moe {
__global__ void moe_decode_kernel(const __grid_constant__ StepParams P);
void set_last_error(const char* msg);
}  // namespace moe

using namespace moe;

namespace {

constexpr size_t kStaticScratchBytes = 128 * 1024;  // MOE_STATIC_SCRATCH_BYTES in moe.h
constexpr int kMaxDevices = 64;
constexpr unsigned long long kStaticTimeoutNs = 2000000000ull;

static_assert(kStaticScratchBytes == MOE_STATIC_SCRATCH_BYTES, "moe.h states the scratch size");

}  // namespace

// Shared by every call on a device. In host code this name is only a stand-in for the symbol:
// the device address comes from cudaGetSymbolAddress in device_setup().
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

namespace {

struct StaticLayout {
    size_t bar, status, table, layer, smaps, xlog, xh, xflag, xacc, total;
};

size_t round256(size_t v) { return (v + 255) & ~(size_t)255; }

StaticLayout static_layout(const moe_shape& s)
{
    StaticLayout l{};
    size_t o = 0;
    l.bar = o;
    o += 256;
    l.status = o;
    o += 256;
    l.table = o;
    o = round256(o + sizeof(int32_t) * (size_t)s.n_experts);
    l.layer = o;
    o = round256(o + sizeof(LayerDesc));
    l.smaps = o;
    o = round256(o + 3 * sizeof(CUtensorMap));
    l.xlog = o;
    o = round256(o + sizeof(unsigned long long) * (size_t)s.n_experts);
    l.xh = o;
    o = round256(o + sizeof(unsigned long long) * (size_t)(s.top_k + 1) * xh_stride(s.inter, s.shared_inter));
    l.xflag = o;  // the step counter
    o = round256(o + sizeof(unsigned long long));
    l.xacc = o;
    o = round256(o + sizeof(long long) * 3 * (size_t)s.hidden);
    l.total = o;
    return l;
}

moe_status fail_static(moe_status st, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    set_last_error(buf);
    return st;
}

struct DeviceSetup {
    bool ready;
    uint8_t* scratch;  // device address of g_static_scratch on this device
    int sms;
    int smem_optin;
    uint32_t epoch;    // next exchange-buffer epoch on this device (0: buffers not yet cleared)
    StaticLayout last; // layout of the previous call on this device (all zero before the first)
};

bool same_layout(const StaticLayout& a, const StaticLayout& b)
{
    return a.bar == b.bar && a.status == b.status && a.table == b.table && a.layer == b.layer && a.smaps == b.smaps &&
           a.xlog == b.xlog && a.xh == b.xh && a.xflag == b.xflag && a.xacc == b.xacc && a.total == b.total;
}

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

// Once per device, with that device current: the device address of the scratch array and the
// SM count (the cooperative grid).
moe_status device_setup(int dev, DeviceSetup* out)
{
    if (dev < 0 || dev >= kMaxDevices)
        return fail_static(MOE_E_INVALID, "device %d outside the %d devices this entry point serves", dev,
                           kMaxDevices);
    std::lock_guard<std::mutex> lock(g_setup_mu);
    DeviceSetup& d = g_setup[dev];
    if (!d.ready) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess)
            return fail_static(MOE_E_CUDA, "cudaGetSymbolAddress(g_static_scratch) failed: %s", cudaGetErrorString(e));
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess || sms <= 0)
            return fail_static(MOE_E_CUDA, "cudaDeviceGetAttribute(SM count) failed: %s", cudaGetErrorString(e));
        int optin = 0;
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess)
            return fail_static(MOE_E_CUDA, "cudaDeviceGetAttribute(shared memory) failed: %s", cudaGetErrorString(e));
        d.scratch = static_cast<uint8_t*>(ptr);
        d.sms = sms;
        d.smem_optin = optin;
        d.epoch = 0;
        d.last = StaticLayout{};
        d.ready = true;
    }
    *out = d;
    return MOE_OK;
}

struct SharedMaps {
    CUtensorMap m[3];
};

// Resets what must start at zero (barrier counter, status words) and writes the identity
// expert table, the layer descriptor and the maps over the shared blob into the scratch array.
__global__ void static_prepare(uint8_t* scratch, StaticLayout sl, int n_experts, LayerDesc desc,
                               const __grid_constant__ SharedMaps maps, int* status_out)
{
    if (threadIdx.x == 0) {
        *reinterpret_cast<unsigned long long*>(scratch + sl.bar) = 0ull;
        *reinterpret_cast<int*>(scratch + sl.status) = 0;
        *reinterpret_cast<LayerDesc*>(scratch + sl.layer) = desc;
        if (status_out)
            *status_out = 0;
    }
    if (threadIdx.x < 3 * sizeof(CUtensorMap) / 8)
        reinterpret_cast<unsigned long long*>(scratch + sl.smaps)[threadIdx.x] =
            reinterpret_cast<const unsigned long long*>(maps.m)[threadIdx.x];
    int32_t* table = reinterpret_cast<int32_t*>(scratch + sl.table);
    for (int e = threadIdx.x; e < n_experts; e += blockDim.x)
        table[e] = e;
}

moe_status check_static_shape(const moe_shape* s)
{
    if (!s)
        return fail_static(MOE_E_INVALID, "shape is NULL");
    if (s->group != 64 || (s->bits != 4 && s->bits != 8))
        return fail_static(MOE_E_SHAPE, "group must be 64 and bits 4 or 8");
    if (s->hidden <= 0 || s->hidden % 256 != 0 || s->hidden > 8192)
        return fail_static(MOE_E_SHAPE, "hidden must be a positive multiple of 256, at most 8192 (got %d)", s->hidden);
    if (s->inter <= 0 || s->inter % 64 != 0 || s->shared_inter <= 0 || s->shared_inter % 64 != 0 ||
        s->inter > 4096 || s->shared_inter > 4096)
        return fail_static(MOE_E_SHAPE, "inter and shared_inter must be positive multiples of 64, at most 4096");
    if (s->top_k < 1 || s->top_k > kMaxK || s->n_experts < s->top_k || s->n_experts > kMaxE)
        return fail_static(MOE_E_SHAPE, "need 1 <= top_k <= %d and top_k <= n_experts <= %d", kMaxK, kMaxE);
    if (s->flags & ~(MOE_RENORM | MOE_PRENORM | MOE_RESIDUAL))
        return fail_static(MOE_E_SHAPE, "unknown flag bits 0x%x", s->flags);
    return MOE_OK;
}

bool misaligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a != 0; }

}  // namespace

extern "C" moe_status moe_layer_forward_static(const moe_shape* shape, const void* d_experts,
                                               const moe_layer_weights* w, const void* d_x, int32_t n_tokens,
                                               float* d_y, int32_t* d_topk_idx, float* d_topk_w,
                                               int32_t* d_status, void* stream)
{
    moe_status st = check_static_shape(shape);
    if (st != MOE_OK)
        return st;
    const StaticLayout sl = static_layout(*shape);
    if (sl.total > kStaticScratchBytes)
        return fail_static(MOE_E_NOMEM,
                           "this shape needs %zu bytes of scratch; the static scratch array holds %zu "
                           "(MOE_STATIC_SCRATCH_BYTES): use moe_layer_forward with a workspace instead",
                           sl.total, kStaticScratchBytes);
    if (!d_experts || !w || !w->router || !w->shared_blob || !w->shared_gate || !d_x || !d_y || !d_status)
        return fail_static(MOE_E_INVALID, "d_experts, the layer weights, d_x, d_y and d_status are required");
    if (misaligned(d_status, 4))
        return fail_static(MOE_E_INVALID, "d_status must be 4-byte aligned");
    if (misaligned(d_experts, 256) || misaligned(w->router, 16) || misaligned(w->shared_blob, 16) ||
        misaligned(w->shared_gate, 16) || misaligned(d_x, 16) || misaligned(d_y, 16))
        return fail_static(MOE_E_INVALID, "d_experts must be 256-byte aligned; weights, d_x and d_y 16-byte aligned");
    if (n_tokens <= 0)
        return fail_static(MOE_E_INVALID, "n_tokens must be positive");

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail_static(MOE_E_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    DeviceSetup ds{};
    if ((st = device_setup(dev, &ds)) != MOE_OK)
        return st;
    if (ds.sms > kMaxGrid)
        return fail_static(MOE_E_SHAPE, "%d SMs exceed the %d blocks a decode launch supports", ds.sms, kMaxGrid);
    StageGeo sg{}, sgs{};
    const uint32_t smem = plan_decode(shape->hidden, shape->n_experts, shape->top_k, shape->inter,
                                      shape->shared_inter, shape->bits, ds.sms, ds.smem_optin, &sg, &sgs);
    if (smem == 0)
        return fail_static(MOE_E_SHAPE, "the fused decode kernel cannot stage this shape on this GPU");

    StepParams P{};
    P.H = shape->hidden;
    P.E = shape->n_experts;
    P.k = shape->top_k;
    P.I = shape->inter;
    P.Is = shape->shared_inter;
    P.bits = shape->bits;
    P.group = shape->group;
    P.flags = shape->flags;
    P.geo = blob_geo(P.H, P.I, P.bits, P.group);
    P.geo_s = blob_geo(P.H, P.Is, P.bits, P.group);
    P.sg = sg;
    P.sgs = sgs;
    SharedMaps smaps{};
    if (encode_arena_maps(smaps.m, static_cast<const uint8_t*>(w->shared_blob), 1, P.geo_s, sgs) != 0)
        return fail_static(MOE_E_CUDA, "cuTensorMapEncodeTiled over the shared blob failed");
    const int rc = encode_arena_maps(P.tmap, static_cast<const uint8_t*>(d_experts), P.E, P.geo, P.sg);
    if (rc != 0)
        return fail_static(MOE_E_CUDA, "cuTensorMapEncodeTiled over the expert blobs failed (%d)", rc);
    P.arena = static_cast<const uint8_t*>(d_experts);
    P.stride = P.geo.stride;
    uint8_t* s = ds.scratch;
    P.table = reinterpret_cast<const int32_t*>(s + sl.table);
    P.layers = reinterpret_cast<const LayerDesc*>(s + sl.layer);
    P.xlog = reinterpret_cast<unsigned long long*>(s + sl.xlog);
    P.xh = reinterpret_cast<unsigned long long*>(s + sl.xh);
    P.xacc = reinterpret_cast<long long*>(s + sl.xacc);
    P.xflag = reinterpret_cast<unsigned long long*>(s + sl.xflag);
    P.smaps = reinterpret_cast<const CUtensorMap*>(s + sl.smaps);
    P.bar = reinterpret_cast<unsigned long long*>(s + sl.bar);
    P.status = reinterpret_cast<int*>(d_status);
    P.timeout_ns = kStaticTimeoutNs;
    for (int j = 0; j < kMaxK; ++j)
        P.slots[j] = -1;
    P.mode = kModeFull;
    P.layer0 = 0;
    P.n_layers = 1;
    P.n_tokens = n_tokens;
    P.x_in = d_x;
    P.y_out = d_y;
    P.topk_idx = d_topk_idx;
    P.topk_w = d_topk_w;

    cudaFuncAttributes fa{};
    if ((e = cudaFuncGetAttributes(&fa, moe_decode_kernel)) != cudaSuccess)
        return fail_static(MOE_E_CUDA, "cudaFuncGetAttributes failed: %s", cudaGetErrorString(e));
    if ((uint32_t)fa.maxDynamicSharedSizeBytes < smem &&
        (e = cudaFuncSetAttribute(moe_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
            cudaSuccess)
        return fail_static(MOE_E_CUDA, "cudaFuncSetAttribute(%u bytes) failed: %s", smem, cudaGetErrorString(e));

    const LayerDesc desc{static_cast<const uint16_t*>(w->router), static_cast<const uint8_t*>(w->shared_blob),
                         static_cast<const uint16_t*>(w->shared_gate), w->logit_bias};
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    bool clear;
    {
        // The exchange buffers are cleared when the epoch counter starts over and whenever this
        // call's layout differs from the previous call's: the buffers then sit on bytes that the
        // previous call used for something else (output words, the expert table), which could
        // read as a pair carrying one of this call's epochs.
        std::lock_guard<std::mutex> lock(g_setup_mu);
        DeviceSetup& d = g_setup[dev];
        clear = next_epochs(d.epoch, (uint32_t)n_tokens, &P.epoch0);
        if (!same_layout(d.last, sl)) {
            clear = true;
            d.last = sl;
        }
    }
    if (clear) {  // no earlier pair may carry an epoch of this call
        if ((e = cudaMemsetAsync(s + sl.xlog, 0, sl.xacc - sl.xlog, cs)) != cudaSuccess)
            return fail_static(MOE_E_CUDA, "clearing the exchange buffers failed: %s", cudaGetErrorString(e));
    }
    static_prepare<<<1, 256, 0, cs>>>(s, sl, P.E, desc, smaps, reinterpret_cast<int*>(d_status));
    if ((e = cudaGetLastError()) != cudaSuccess)
        return fail_static(MOE_E_CUDA, "scratch preparation launch failed: %s", cudaGetErrorString(e));
    void* args[] = {&P};
    e = cudaLaunchCooperativeKernel((const void*)moe_decode_kernel, dim3(ds.sms), dim3(kThreads), args, smem, cs);
    if (e != cudaSuccess)
        return fail_static(MOE_E_CUDA, "decode kernel launch failed: %s", cudaGetErrorString(e));
    return MOE_OK;
}
