// api.cu -- the C ABI declared in include/moe.h: argument checks, the expert pool, launches.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/moe.h"
#include "host.h"
#include "layout.h"
#include "policy.h"

#include <cuda_fp16.h>

#include "grouped.h"
#include "qpack.h"

namespace moe {
__global__ void moe_decode_kernel(const __grid_constant__ StepParams P);
namespace bat {
void launch_gather_rows(const uint16_t* x, const int32_t* list, int A, int H, int bits, __half* us, int* status,
                        cudaStream_t st);
void launch_topk(const float* logits, const float* bias, int T, int E, int k, int renorm, const uint16_t* u,
                 const uint16_t* wsg, int H, int32_t* idx, float* w, float* gamma, int32_t* counts, cudaStream_t st);
void launch_plan(const int32_t* counts, int E, int T, int I, int Is, int H, int32_t* offs, int32_t* cursor,
                 int4* tasks_gu, int4* tasks_dn, int32_t* n_tasks, cudaStream_t st);
void launch_place(const int32_t* idx, const float* w, const float* gamma, int T, int E, int k, int32_t* cursor,
                  int32_t* list, float* aw, int32_t* apos, cudaStream_t st);
void launch_combine(const float* ypart, const int32_t* apos, int T, int k, int H, float* y, cudaStream_t st);
}  // namespace bat
__global__ void scalar_router(const StepParams P);
__global__ void scalar_topk(const StepParams P, int32_t* sel);
__global__ void scalar_gateup(const StepParams P, const int32_t* sel);
__global__ void scalar_down(const StepParams P, const int32_t* sel);
}  // namespace moe

using namespace moe;

namespace {

thread_local std::string g_err;

moe_status fail(moe_status st, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

#define CUDA_TRY(call)                                                                         \
    do {                                                                                       \
        cudaError_t e_ = (call);                                                               \
        if (e_ != cudaSuccess)                                                                 \
            return fail(MOE_E_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_));           \
    } while (0)

size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

struct WsLayout {
    size_t bar, status, table, layers, smaps, logits, hbuf, sel, xlog, xh, xflag, xacc, xbuf, total;
};

WsLayout ws_layout(const moe_shape& s, int L)
{
    WsLayout w{};
    const int Imax = s.inter > s.shared_inter ? s.inter : s.shared_inter;
    size_t o = 0;
    auto take = [&](size_t& field, size_t bytes) {
        field = o;
        o = up256(o + bytes);
    };
    take(w.bar, 256);
    take(w.status, 256);
    take(w.table, sizeof(int32_t) * (size_t)L * s.n_experts);
    take(w.layers, sizeof(LayerDesc) * (size_t)L);
    take(w.smaps, sizeof(CUtensorMap) * 3 * (size_t)L);
    take(w.logits, sizeof(float) * (size_t)s.n_experts);
    take(w.hbuf, sizeof(float) * (size_t)(s.top_k + 1) * Imax);
    take(w.sel, sizeof(int32_t) * 5 * kMaxK);
    take(w.xlog, sizeof(unsigned long long) * (size_t)s.n_experts);
    take(w.xh, sizeof(unsigned long long) * (size_t)(s.top_k + 1) * xh_stride(s.inter, s.shared_inter));
    take(w.xflag, sizeof(unsigned long long));  // the step counter
    take(w.xacc, sizeof(long long) * 3 * (size_t)s.hidden);
    take(w.xbuf, sizeof(float) * 2 * (size_t)s.hidden);
    w.total = o;
    return w;
}

moe_status check_shape(const moe_shape* s)
{
    if (!s)
        return fail(MOE_E_INVALID, "shape is NULL");
    if (s->group != 64)
        return fail(MOE_E_SHAPE, "group must be 64 (got %d)", s->group);
    if (s->bits != 4 && s->bits != 8)
        return fail(MOE_E_SHAPE, "bits must be 4 or 8 (got %d)", s->bits);
    if (s->hidden <= 0 || s->hidden % 256 != 0 || s->hidden > 8192)
        return fail(MOE_E_SHAPE, "hidden must be a positive multiple of 256, at most 8192 (got %d)", s->hidden);
    if (s->inter <= 0 || s->inter % 64 != 0 || s->shared_inter <= 0 || s->shared_inter % 64 != 0)
        return fail(MOE_E_SHAPE, "inter and shared_inter must be positive multiples of 64");
    if (s->inter > 4096 || s->shared_inter > 4096)
        return fail(MOE_E_SHAPE, "inter and shared_inter must be at most 4096");
    if (s->top_k < 1 || s->top_k > kMaxK)
        return fail(MOE_E_SHAPE, "top_k must be in [1, %d] (got %d)", kMaxK, s->top_k);
    if (s->n_experts < s->top_k || s->n_experts > kMaxE)
        return fail(MOE_E_SHAPE, "n_experts must be in [top_k, %d] (got %d)", kMaxE, s->n_experts);
    if (s->flags & ~(MOE_RENORM | MOE_PRENORM | MOE_RESIDUAL | MOE_DETERMINISTIC | MOE_GEMV))
        return fail(MOE_E_SHAPE, "unknown flag bits 0x%x", s->flags);
    return MOE_OK;
}

}  // namespace

namespace moe {
// Message for moe_last_error() from entry points defined in other files of the library.
void set_last_error(const char* msg) { g_err = msg; }
}  // namespace moe

struct moe_pool {
    moe_shape shape{};
    int L = 0, S = 0;
    uint8_t* arena = nullptr;
    size_t arena_bytes = 0;
    uint8_t* ws = nullptr;
    size_t ws_bytes = 0;
    WsLayout wl{};
    BlobGeo geo{}, geo_s{};
    StageGeo sg{}, sgs{};
    CUtensorMap tmap[3];
    std::vector<CUtensorMap> smaps;  // [L][3] decode-kernel maps over each layer's shared blob
    uint32_t epoch_next = 1;  // exchange-buffer epochs (the workspace starts zeroed)
    std::vector<LayerDesc> layers;
    SlotPolicy policy;
    int64_t hits = 0, misses = 0, bytes_loaded = 0;
    int device = -1, grid = 0;
    uint32_t smem = 0;
    int smem_optin = 0;
    uint64_t timeout_ns = 2000000000ull;
    int prefetch = 0;  // bounded stacks: copy ahead the next layer's top `prefetch` predicted experts
    // bounded mode: events
    std::vector<cudaEvent_t> ring;   // last-use events, reused round robin
    size_t ring_next = 0;
    std::vector<cudaEvent_t> slot_last_use;  // per slot, nullptr if never read
    cudaEvent_t loads_done = nullptr;
    cudaStream_t last_copy_stream = nullptr;
    bool loads_pending = false;
    std::vector<cudaEvent_t> stage_ev;  // moe_stack_forward_qpack: last copy out of each staging slot
    std::vector<char> stage_used;
    int stage_next = 0;
    // test hook replacing the device copy of load_slot
    int (*copy_hook)(void*, int32_t, const void*, size_t) = nullptr;
    void* copy_user = nullptr;
    // batched-path timing: event pairs around the expert GEMMs of each call, round robin
    std::vector<cudaEvent_t> gemm_ev;  // [2 * n]
    int gemm_next = 0, gemm_used = 0;
    // batched-path tensor maps, re-encoded only when the memory they describe changes
    struct MapKey {
        const void* ptr = nullptr;
        int64_t a = -1, b = -1;
        bool same(const void* p, int64_t x, int64_t y) const { return ptr == p && a == x && b == y; }
    };
    MapKey k_arena, k_u, k_b0, k_b1;
    CUtensorMap m_arena[3], m_u, m_b0, m_b1;
    std::vector<MapKey> k_shared, k_router;   // per layer
    std::vector<CUtensorMap> m_shared, m_router;  // [L][3], [L]
};

extern "C" {

const char* moe_last_error(void) { return g_err.c_str(); }

// A shape whose blob is defined: positive sizes that are whole groups and a code width of 4 or 8.
static bool blob_defined(const moe_shape* s, int shared)
{
    const int I = shared ? s->shared_inter : s->inter;
    return (s->bits == 4 || s->bits == 8) && s->group > 0 && s->hidden > 0 && I > 0 && s->hidden % s->group == 0 &&
           I % s->group == 0;
}

size_t moe_expert_bytes(const moe_shape* s, int shared)
{
    if (!s || !blob_defined(s, shared))
        return 0;
    return blob_geo(s->hidden, shared ? s->shared_inter : s->inter, s->bits, s->group).bytes;
}

size_t moe_expert_stride(const moe_shape* s, int shared)
{
    if (!s || !blob_defined(s, shared))
        return 0;
    return blob_geo(s->hidden, shared ? s->shared_inter : s->inter, s->bits, s->group).stride;
}

moe_status moe_pack_expert(const moe_shape* s, int shared, const uint8_t* const codes[3],
                           const uint16_t* const scale[3], const uint16_t* const bias[3], void* h_blob)
{
    moe_status st = check_shape(s);
    if (st != MOE_OK)
        return st;
    if (!codes || !scale || !bias || !h_blob)
        return fail(MOE_E_INVALID, "NULL argument to moe_pack_expert");
    const BlobGeo g = blob_geo(s->hidden, shared ? s->shared_inter : s->inter, s->bits, s->group);
    uint8_t* out = static_cast<uint8_t*>(h_blob);
    memset(out, 0, g.stride);
    for (int m = 0; m < 3; ++m) {
        if (!codes[m] || !scale[m] || !bias[m])
            return fail(MOE_E_INVALID, "NULL array for matrix %d", m);
        const int rows = g.rows[m], cols = g.cols[m];
        const uint8_t* q = codes[m];
        uint8_t* dst = out + g.q_off[m];
        const int maxq = (1 << s->bits) - 1;
        for (size_t i = 0; i < (size_t)rows * cols; ++i)
            if (q[i] > maxq)
                return fail(MOE_E_INVALID, "code %d out of range in matrix %d", (int)q[i], m);
        if (s->bits == 8) {
            memcpy(dst, q, (size_t)rows * cols);
        } else {
            // two codes per byte: the even-indexed one in the low nibble
            const size_t nbytes = (size_t)rows * cols / 2;
            for (size_t b = 0; b < nbytes; ++b)
                dst[b] = (uint8_t)(q[2 * b] | (q[2 * b + 1] << 4));
        }
        const size_t n = (size_t)rows * g.groups[m];
        for (size_t i = 0; i < n; ++i) {
            out[g.s_off[m] + 2 * i] = (uint8_t)(scale[m][i] & 0xFF);
            out[g.s_off[m] + 2 * i + 1] = (uint8_t)(scale[m][i] >> 8);
            out[g.b_off[m] + 2 * i] = (uint8_t)(bias[m][i] & 0xFF);
            out[g.b_off[m] + 2 * i + 1] = (uint8_t)(bias[m][i] >> 8);
        }
    }
    return MOE_OK;
}

size_t moe_workspace_bytes(const moe_shape* s, int32_t n_layers)
{
    if (!s || n_layers <= 0)
        return 0;
    return ws_layout(*s, n_layers).total;
}

moe_status moe_pool_create(const moe_shape* s, int32_t n_layers, int32_t n_slots, void* d_arena,
                           size_t arena_bytes, void* d_workspace, size_t workspace_bytes, moe_pool** out)
{
    moe_status st = check_shape(s);
    if (st != MOE_OK)
        return st;
    if (!out)
        return fail(MOE_E_INVALID, "out is NULL");
    *out = nullptr;
    if (n_layers <= 0 || n_slots <= 0)
        return fail(MOE_E_INVALID, "n_layers and n_slots must be positive");
    const BlobGeo geo = blob_geo(s->hidden, s->inter, s->bits, s->group);
    if (d_workspace) {
        if (!d_arena)
            return fail(MOE_E_INVALID, "d_arena is NULL");
        if (reinterpret_cast<uintptr_t>(d_arena) % 256 || reinterpret_cast<uintptr_t>(d_workspace) % 256)
            return fail(MOE_E_INVALID, "arena and workspace must be 256-byte aligned");
        if (arena_bytes < (size_t)n_slots * geo.stride)
            return fail(MOE_E_NOMEM, "arena holds %zu bytes, %d slots need %zu", arena_bytes, n_slots,
                        (size_t)n_slots * geo.stride);
        if (workspace_bytes < ws_layout(*s, n_layers).total)
            return fail(MOE_E_NOMEM, "workspace holds %zu bytes, needs %zu", workspace_bytes,
                        ws_layout(*s, n_layers).total);
    }
    moe_pool* p = new moe_pool();
    p->shape = *s;
    p->L = n_layers;
    p->S = n_slots;
    p->arena = static_cast<uint8_t*>(d_arena);
    p->arena_bytes = arena_bytes;
    p->ws = static_cast<uint8_t*>(d_workspace);
    p->ws_bytes = workspace_bytes;
    p->wl = ws_layout(*s, n_layers);
    p->geo = geo;
    p->geo_s = blob_geo(s->hidden, s->shared_inter, s->bits, s->group);
    p->layers.assign(n_layers, LayerDesc{nullptr, nullptr, nullptr, nullptr});
    p->smaps.assign(3 * (size_t)n_layers, CUtensorMap{});
    p->policy = SlotPolicy(n_layers, s->n_experts, n_slots);
    p->slot_last_use.assign(n_slots, nullptr);
    if (!d_workspace) {  // host-only pool: slot policy without a device
        *out = p;
        return MOE_OK;
    }
    auto cleanup = [&](moe_status r) {
        delete p;
        return r;
    };
    if (cudaGetDevice(&p->device) != cudaSuccess)
        return cleanup(fail(MOE_E_CUDA, "no CUDA device"));
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess)
        return cleanup(fail(MOE_E_CUDA, "cudaDeviceGetAttribute failed"));
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device) != cudaSuccess)
        return cleanup(fail(MOE_E_CUDA, "cudaDeviceGetAttribute failed"));
    p->smem = plan_decode(s->hidden, s->n_experts, s->top_k, s->inter, s->shared_inter, s->bits, sms, optin, &p->sg,
                          &p->sgs);
    if (p->smem == 0)
        return cleanup(fail(MOE_E_SHAPE, "the fused decode kernel cannot stage this shape on %d SMs with %d bytes of "
                            "shared memory per block", sms, optin));
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, moe_decode_kernel);
    if (e == cudaSuccess && (uint32_t)fa.maxDynamicSharedSizeBytes < p->smem)
        e = cudaFuncSetAttribute(moe_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p->smem);
    if (e != cudaSuccess)
        return cleanup(fail(MOE_E_CUDA, "cudaFuncSetAttribute(%u bytes): %s", p->smem, cudaGetErrorString(e)));
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, moe_decode_kernel, kThreads, p->smem);
    if (e != cudaSuccess || per_sm < 1)
        return cleanup(fail(MOE_E_CUDA, "decode kernel cannot be resident (%d per SM): %s", per_sm,
                            cudaGetErrorString(e)));
    const int rc = encode_arena_maps(p->tmap, p->arena, n_slots, p->geo, p->sg);
    if (rc != 0)
        return cleanup(fail(MOE_E_CUDA, "cuTensorMapEncodeTiled over the arena failed (%d)", rc));
    if (sms > kMaxGrid)
        return cleanup(fail(MOE_E_SHAPE, "%d SMs exceed the %d blocks a decode launch supports", sms, kMaxGrid));
    p->grid = sms;  // one block per SM
    p->smem_optin = optin;
    if (cudaMemset(p->ws, 0, p->wl.total) != cudaSuccess ||
        cudaMemset(p->ws + p->wl.table, 0xFF, sizeof(int32_t) * (size_t)n_layers * s->n_experts) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
        return cleanup(fail(MOE_E_CUDA, "workspace initialisation failed"));
    *out = p;
    return MOE_OK;
}

void moe_pool_destroy(moe_pool* p)
{
    if (!p)
        return;
    for (cudaEvent_t ev : p->ring)
        cudaEventDestroy(ev);
    for (cudaEvent_t ev : p->gemm_ev)
        cudaEventDestroy(ev);
    if (p->loads_done)
        cudaEventDestroy(p->loads_done);
    for (cudaEvent_t ev : p->stage_ev)
        cudaEventDestroy(ev);
    delete p;
}

void* moe_pool_slot_ptr(const moe_pool* p, int32_t slot)
{
    if (!p || !p->arena || slot < 0 || slot >= p->S)
        return nullptr;
    return p->arena + (size_t)slot * p->geo.stride;
}

int32_t moe_pool_grid(const moe_pool* p) { return p ? p->grid : 0; }

moe_status moe_pool_time_batched(moe_pool* p, int32_t n_calls)
{
    if (!p || n_calls < 0 || n_calls > 100000)
        return fail(MOE_E_INVALID, "bad pool or call count");
    for (cudaEvent_t ev : p->gemm_ev)
        cudaEventDestroy(ev);
    p->gemm_ev.assign(2 * (size_t)n_calls, nullptr);
    for (auto& ev : p->gemm_ev)
        CUDA_TRY(cudaEventCreate(&ev));
    p->gemm_next = p->gemm_used = 0;
    return MOE_OK;
}

moe_status moe_pool_batched_gemm_ms(moe_pool* p, float* h_total_ms, int32_t* h_calls)
{
    if (!p || !h_total_ms || !h_calls)
        return fail(MOE_E_INVALID, "NULL argument");
    float total = 0.f;
    const int n = (int)p->gemm_ev.size() / 2;
    const int used = p->gemm_used < n ? p->gemm_used : n;
    for (int i = 0; i < used; ++i) {
        CUDA_TRY(cudaEventSynchronize(p->gemm_ev[2 * i + 1]));
        float ms = 0.f;
        CUDA_TRY(cudaEventElapsedTime(&ms, p->gemm_ev[2 * i], p->gemm_ev[2 * i + 1]));
        total += ms;
    }
    *h_total_ms = total;
    *h_calls = used;
    p->gemm_next = p->gemm_used = 0;
    return MOE_OK;
}

moe_status moe_pool_set_timeout(moe_pool* p, uint64_t timeout_ns)
{
    if (!p || timeout_ns == 0)
        return fail(MOE_E_INVALID, "bad pool or zero timeout");
    p->timeout_ns = timeout_ns;
    return MOE_OK;
}

moe_status moe_pool_set_prefetch(moe_pool* p, int32_t n)
{
    if (!p || n < 0)
        return fail(MOE_E_INVALID, "bad pool or negative prefetch depth");
    p->prefetch = n;
    return MOE_OK;
}

moe_status moe_pool_set_layer(moe_pool* p, int32_t layer, const moe_layer_weights* w)
{
    if (!p || !w)
        return fail(MOE_E_INVALID, "NULL pool or weights");
    if (layer < 0 || layer >= p->L)
        return fail(MOE_E_INVALID, "layer %d out of range [0, %d)", layer, p->L);
    if (!w->router || !w->shared_blob || !w->shared_gate)
        return fail(MOE_E_INVALID, "router, shared_blob and shared_gate are required");
    if (reinterpret_cast<uintptr_t>(w->router) % 16 || reinterpret_cast<uintptr_t>(w->shared_blob) % 16 ||
        reinterpret_cast<uintptr_t>(w->shared_gate) % 16)
        return fail(MOE_E_INVALID, "layer weights must be 16-byte aligned");
    if (p->ws) {  // the decode kernel's maps over this layer's shared blob
        CUtensorMap m[3];
        const int rc = encode_arena_maps(m, static_cast<const uint8_t*>(w->shared_blob), 1, p->geo_s, p->sgs);
        if (rc != 0)
            return fail(MOE_E_CUDA, "cuTensorMapEncodeTiled over the shared blob of layer %d failed (%d)", layer, rc);
        for (int i = 0; i < 3; ++i)
            p->smaps[3 * (size_t)layer + i] = m[i];
    }
    p->layers[layer] = LayerDesc{static_cast<const uint16_t*>(w->router), static_cast<const uint8_t*>(w->shared_blob),
                                 static_cast<const uint16_t*>(w->shared_gate), w->logit_bias};
    return MOE_OK;
}

moe_status moe_pool_place(moe_pool* p, int32_t layer, int32_t expert, int32_t slot)
{
    if (!p)
        return fail(MOE_E_INVALID, "NULL pool");
    if (layer < 0 || layer >= p->L || expert < 0 || expert >= p->shape.n_experts || slot < 0 || slot >= p->S)
        return fail(MOE_E_INVALID, "place(%d, %d, %d) out of range", layer, expert, slot);
    p->policy.place(layer, expert, slot);
    return MOE_OK;
}

moe_status moe_pool_sync(moe_pool* p, void* stream)
{
    if (!p || !p->ws)
        return fail(MOE_E_INVALID, "pool has no device workspace");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const auto& t = p->policy.table();
    CUDA_TRY(cudaMemcpyAsync(p->ws + p->wl.table, t.data(), sizeof(int32_t) * t.size(), cudaMemcpyHostToDevice, st));
    CUDA_TRY(cudaMemcpyAsync(p->ws + p->wl.layers, p->layers.data(), sizeof(LayerDesc) * p->layers.size(),
                             cudaMemcpyHostToDevice, st));
    CUDA_TRY(cudaMemcpyAsync(p->ws + p->wl.smaps, p->smaps.data(), sizeof(CUtensorMap) * p->smaps.size(),
                             cudaMemcpyHostToDevice, st));
    return MOE_OK;
}

moe_status moe_pool_lookup(moe_pool* p, int32_t layer, const int32_t* experts, int32_t n, int32_t* slots_out)
{
    if (!p || !experts || !slots_out || n < 0)
        return fail(MOE_E_INVALID, "bad lookup arguments");
    if (layer < 0 || layer >= p->L)
        return fail(MOE_E_INVALID, "layer %d out of range", layer);
    for (int i = 0; i < n; ++i)
        if (experts[i] < 0 || experts[i] >= p->shape.n_experts)
            return fail(MOE_E_INVALID, "expert %d out of range", experts[i]);
    p->policy.lookup(layer, experts, n, slots_out, &p->hits, &p->misses);
    return MOE_OK;
}

moe_status moe_pool_load_slot(moe_pool* p, int32_t layer, int32_t expert, const void* h_blob, void* copy_stream,
                              int32_t* slot_out)
{
    if (!p || !h_blob || !slot_out)
        return fail(MOE_E_INVALID, "bad load_slot arguments");
    if (layer < 0 || layer >= p->L || expert < 0 || expert >= p->shape.n_experts)
        return fail(MOE_E_INVALID, "load_slot(%d, %d) out of range", layer, expert);
    const int have = p->policy.slot_of(layer, expert);
    if (have >= 0) {  // already resident: nothing to copy
        int64_t h = 0, m = 0;
        int32_t s;
        p->policy.lookup(layer, &expert, 1, &s, &h, &m);
        *slot_out = have;
        return MOE_OK;
    }
    int victim = -1;
    const int s = p->policy.choose(&victim);
    if (s < 0)
        return fail(MOE_E_POOL_FULL, "every one of the %d slots is pinned", p->S);
    const size_t bytes = p->geo.stride;
    if (p->copy_hook) {
        if (p->copy_hook(p->copy_user, s, h_blob, bytes) != 0)
            return fail(MOE_E_CUDA, "copy into slot %d failed (copy hook)", s);
    } else {
        if (!p->arena)
            return fail(MOE_E_INVALID, "host-only pool cannot copy");
        cudaStream_t cs = static_cast<cudaStream_t>(copy_stream);
        if (p->slot_last_use[s])
            CUDA_TRY(cudaStreamWaitEvent(cs, p->slot_last_use[s], 0));
        CUDA_TRY(cudaMemcpyAsync(p->arena + (size_t)s * bytes, h_blob, bytes, cudaMemcpyHostToDevice, cs));
        p->last_copy_stream = cs;
        p->loads_pending = true;
    }
    p->policy.install(layer, expert, s);
    p->bytes_loaded += (int64_t)bytes;
    *slot_out = s;
    return MOE_OK;
}

moe_status moe_pool_wait_loads(moe_pool* p, void* compute_stream)
{
    if (!p)
        return fail(MOE_E_INVALID, "NULL pool");
    if (!p->loads_pending)
        return MOE_OK;
    if (!p->loads_done)
        CUDA_TRY(cudaEventCreateWithFlags(&p->loads_done, cudaEventDisableTiming));
    CUDA_TRY(cudaEventRecord(p->loads_done, p->last_copy_stream));
    CUDA_TRY(cudaStreamWaitEvent(static_cast<cudaStream_t>(compute_stream), p->loads_done, 0));
    p->loads_pending = false;
    return MOE_OK;
}

moe_status moe_pool_release(moe_pool* p, void* compute_stream)
{
    if (!p)
        return fail(MOE_E_INVALID, "NULL pool");
    if (p->arena && !p->copy_hook && !p->policy.pinned_list().empty()) {
        const size_t kRing = 256;
        if (p->ring.size() < kRing) {
            cudaEvent_t ev;
            CUDA_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
            p->ring.push_back(ev);
        }
        cudaEvent_t ev = p->ring[p->ring_next % p->ring.size()];
        ++p->ring_next;
        // A ring event recorded again later only makes a wait on it later (still safe).
        CUDA_TRY(cudaEventRecord(ev, static_cast<cudaStream_t>(compute_stream)));
        for (int s : p->policy.pinned_list())
            p->slot_last_use[s] = ev;
    }
    p->policy.release();
    return MOE_OK;
}

moe_status moe_pool_stats(const moe_pool* p, int64_t* hits, int64_t* misses, int64_t* bytes_loaded)
{
    if (!p)
        return fail(MOE_E_INVALID, "NULL pool");
    if (hits)
        *hits = p->hits;
    if (misses)
        *misses = p->misses;
    if (bytes_loaded)
        *bytes_loaded = p->bytes_loaded;
    return MOE_OK;
}

// test hook (declared in moe_test.h): replace the device copy of load_slot by a host callback
moe_status moe_pool_set_copy_hook(moe_pool* p, int (*fn)(void*, int32_t, const void*, size_t), void* user)
{
    if (!p)
        return fail(MOE_E_INVALID, "NULL pool");
    p->copy_hook = fn;
    p->copy_user = user;
    return MOE_OK;
}

moe_status moe_pool_slot_of(const moe_pool* p, int32_t layer, int32_t expert, int32_t* slot)
{
    if (!p || !slot || layer < 0 || layer >= p->L || expert < 0 || expert >= p->shape.n_experts)
        return fail(MOE_E_INVALID, "bad slot_of arguments");
    *slot = p->policy.slot_of(layer, expert);
    return MOE_OK;
}

}  // extern "C"

namespace {

StepParams base_params(const moe_pool* p)
{
    StepParams P{};
    const moe_shape& s = p->shape;
    P.H = s.hidden;
    P.E = s.n_experts;
    P.k = s.top_k;
    P.I = s.inter;
    P.Is = s.shared_inter;
    P.bits = s.bits;
    P.group = s.group;
    P.flags = s.flags;
    P.geo = p->geo;
    P.geo_s = p->geo_s;
    P.sg = p->sg;
    P.sgs = p->sgs;
    P.smaps = reinterpret_cast<const CUtensorMap*>(p->ws + p->wl.smaps);
    P.xflag = reinterpret_cast<unsigned long long*>(p->ws + p->wl.xflag);
    for (int m = 0; m < 3; ++m)
        P.tmap[m] = p->tmap[m];
    P.arena = p->arena;
    P.stride = p->geo.stride;
    P.table = reinterpret_cast<const int32_t*>(p->ws + p->wl.table);
    P.layers = reinterpret_cast<const LayerDesc*>(p->ws + p->wl.layers);
    P.logits = reinterpret_cast<float*>(p->ws + p->wl.logits);
    P.hbuf = reinterpret_cast<float*>(p->ws + p->wl.hbuf);
    P.xlog = reinterpret_cast<unsigned long long*>(p->ws + p->wl.xlog);
    P.xh = reinterpret_cast<unsigned long long*>(p->ws + p->wl.xh);
    P.xacc = reinterpret_cast<long long*>(p->ws + p->wl.xacc);
    P.bar = reinterpret_cast<unsigned long long*>(p->ws + p->wl.bar);
    P.status = reinterpret_cast<int*>(p->ws + p->wl.status);
    P.timeout_ns = p->timeout_ns;
    for (int j = 0; j < kMaxK; ++j)
        P.slots[j] = -1;
    return P;
}

moe_status check_layers(const moe_pool* p, int layer0, int n)
{
    if (!p || !p->ws)
        return fail(MOE_E_INVALID, "pool has no device workspace");
    if (layer0 < 0 || n <= 0 || layer0 + n > p->L)
        return fail(MOE_E_INVALID, "layers [%d, %d) out of range [0, %d)", layer0, layer0 + n, p->L);
    for (int l = layer0; l < layer0 + n; ++l)
        if (!p->layers[l].router)
            return fail(MOE_E_INVALID, "layer %d has no weights (moe_pool_set_layer)", l);
    return MOE_OK;
}

moe_status launch(moe_pool* p, StepParams& P, cudaStream_t st)
{
    int dev = -1;
    CUDA_TRY(cudaGetDevice(&dev));
    if (dev != p->device)
        return fail(MOE_E_INVALID, "current device %d differs from the pool's device %d", dev, p->device);
    const uint32_t steps = P.mode == kModeFull ? (uint32_t)(P.n_tokens * P.n_layers) : 1u;
    if (next_epochs(p->epoch_next, steps, &P.epoch0)) {
        CUDA_TRY(cudaMemsetAsync(p->ws + p->wl.xlog, 0, p->wl.xh - p->wl.xlog, st));
        CUDA_TRY(cudaMemsetAsync(p->ws + p->wl.xh, 0, p->wl.xacc - p->wl.xh, st));
    }
    void* args[] = {&P};
    CUDA_TRY(cudaLaunchCooperativeKernel((const void*)moe_decode_kernel, dim3(p->grid), dim3(kThreads), args,
                                         p->smem, st));
    return MOE_OK;
}

moe_status check_ptr(const void* ptr, size_t align, const char* what)
{
    if (!ptr)
        return fail(MOE_E_INVALID, "%s is NULL", what);
    if (reinterpret_cast<uintptr_t>(ptr) % align)
        return fail(MOE_E_INVALID, "%s must be %zu-byte aligned", what, align);
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_layer_forward(moe_pool* p, int32_t layer, const void* d_x, int32_t n_tokens, float* d_y,
                             int32_t* d_topk_idx, float* d_topk_w, void* stream)
{
    moe_status st = check_layers(p, layer, 1);
    if (st != MOE_OK)
        return st;
    if (n_tokens <= 0)
        return fail(MOE_E_INVALID, "n_tokens must be positive");
    if ((st = check_ptr(d_x, 16, "d_x")) != MOE_OK || (st = check_ptr(d_y, 16, "d_y")) != MOE_OK)
        return st;
    StepParams P = base_params(p);
    P.mode = kModeFull;
    P.layer0 = layer;
    P.n_layers = 1;
    P.n_tokens = n_tokens;
    P.x_in = d_x;
    P.y_out = d_y;
    P.topk_idx = d_topk_idx;
    P.topk_w = d_topk_w;
    return launch(p, P, static_cast<cudaStream_t>(stream));
}

moe_status moe_stack_forward(moe_pool* p, int32_t layer0, int32_t n_layers, const float* d_x, float* d_x_out,
                             float* d_trace, int32_t* d_topk_idx, float* d_topk_w, void* stream)
{
    moe_status st = check_layers(p, layer0, n_layers);
    if (st != MOE_OK)
        return st;
    if ((p->shape.flags & (MOE_PRENORM | MOE_RESIDUAL)) != (MOE_PRENORM | MOE_RESIDUAL))
        return fail(MOE_E_SHAPE, "a stack needs MOE_PRENORM | MOE_RESIDUAL in the shape flags");
    if ((st = check_ptr(d_x, 16, "d_x")) != MOE_OK || (st = check_ptr(d_x_out, 16, "d_x_out")) != MOE_OK)
        return st;
    StepParams P = base_params(p);
    P.mode = kModeFull;
    P.layer0 = layer0;
    P.n_layers = n_layers;
    P.n_tokens = 1;
    P.x_in = d_x;
    P.y_out = d_x_out;
    P.trace = d_trace;
    P.topk_idx = d_topk_idx;
    P.topk_w = d_topk_w;
    return launch(p, P, static_cast<cudaStream_t>(stream));
}

moe_status moe_route(moe_pool* p, int32_t layer, const void* d_x, int32_t* d_topk_idx, float* d_topk_w, void* stream)
{
    moe_status st = check_layers(p, layer, 1);
    if (st != MOE_OK)
        return st;
    if ((st = check_ptr(d_x, 16, "d_x")) != MOE_OK || (st = check_ptr(d_topk_idx, 4, "d_topk_idx")) != MOE_OK ||
        (st = check_ptr(d_topk_w, 4, "d_topk_w")) != MOE_OK)
        return st;
    StepParams P = base_params(p);
    P.mode = kModeRoute;
    P.layer0 = layer;
    P.n_layers = 1;
    P.n_tokens = 1;
    P.x_in = d_x;
    P.topk_idx = d_topk_idx;
    P.topk_w = d_topk_w;
    return launch(p, P, static_cast<cudaStream_t>(stream));
}

moe_status moe_experts(moe_pool* p, int32_t layer, const void* d_x, const float* d_topk_w, const int32_t* h_slots,
                       float* d_y, void* stream)
{
    moe_status st = check_layers(p, layer, 1);
    if (st != MOE_OK)
        return st;
    if ((st = check_ptr(d_x, 16, "d_x")) != MOE_OK || (st = check_ptr(d_y, 16, "d_y")) != MOE_OK ||
        (st = check_ptr(d_topk_w, 4, "d_topk_w")) != MOE_OK || (st = check_ptr(h_slots, 4, "h_slots")) != MOE_OK)
        return st;
    StepParams P = base_params(p);
    for (int j = 0; j < p->shape.top_k; ++j) {
        if (h_slots[j] < 0 || h_slots[j] >= p->S)
            return fail(MOE_E_INVALID, "slot %d of rank %d out of range [0, %d)", h_slots[j], j, p->S);
        P.slots[j] = h_slots[j];
    }
    P.mode = kModeExperts;
    P.layer0 = layer;
    P.n_layers = 1;
    P.n_tokens = 1;
    P.x_in = d_x;
    P.y_out = d_y;
    P.topk_w = const_cast<float*>(d_topk_w);
    return launch(p, P, static_cast<cudaStream_t>(stream));
}

moe_status moe_layer_forward_scalar(moe_pool* p, int32_t layer, const void* d_x, float* d_y, int32_t* d_topk_idx,
                                    float* d_topk_w, void* stream)
{
    moe_status st = check_layers(p, layer, 1);
    if (st != MOE_OK)
        return st;
    if (p->shape.flags & (MOE_PRENORM | MOE_RESIDUAL))
        return fail(MOE_E_SHAPE, "the scalar reference path takes a bf16 layer input (no pre-norm, no residual)");
    if ((st = check_ptr(d_x, 16, "d_x")) != MOE_OK || (st = check_ptr(d_y, 16, "d_y")) != MOE_OK)
        return st;
    StepParams P = base_params(p);
    P.mode = kModeFull;
    P.layer0 = layer;
    P.n_layers = 1;
    P.n_tokens = 1;
    P.x_in = d_x;
    P.y_out = d_y;
    P.topk_idx = d_topk_idx;
    P.topk_w = d_topk_w;
    int32_t* sel = reinterpret_cast<int32_t*>(p->ws + p->wl.sel);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int Imax = P.I > P.Is ? P.I : P.Is;
    scalar_router<<<(P.E + 127) / 128, 128, 0, cs>>>(P);
    scalar_topk<<<1, 32, 0, cs>>>(P, sel);
    scalar_gateup<<<((P.k + 1) * Imax + 127) / 128, 128, 0, cs>>>(P, sel);
    scalar_down<<<(P.H + 127) / 128, 128, 0, cs>>>(P, sel);
    CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

moe_status moe_device_status(moe_pool* p, void* stream, int32_t* h_status)
{
    if (!p || !p->ws || !h_status)
        return fail(MOE_E_INVALID, "bad device_status arguments");
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    CUDA_TRY(cudaStreamSynchronize(cs));
    int32_t v = 0;
    CUDA_TRY(cudaMemcpy(&v, p->ws + p->wl.status, sizeof v, cudaMemcpyDeviceToHost));
    if (v != 0) {
        CUDA_TRY(cudaMemset(p->ws + p->wl.status, 0, sizeof(int32_t)));
        if (v == MOE_E_TIMEOUT)
            CUDA_TRY(cudaMemset(p->ws + p->wl.bar, 0, sizeof(unsigned long long)));
        CUDA_TRY(cudaDeviceSynchronize());
    }
    *h_status = v;
    return MOE_OK;
}

moe_status moe_stack_forward_streamed(moe_pool* p, int32_t layer0, int32_t n_layers, const float* d_x, float* d_x_out,
                                      const void* const* h_blobs, void* compute_stream, void* copy_stream,
                                      int32_t* h_topk_idx)
{
    moe_status st = check_layers(p, layer0, n_layers);
    if (st != MOE_OK)
        return st;
    if ((p->shape.flags & (MOE_PRENORM | MOE_RESIDUAL)) != (MOE_PRENORM | MOE_RESIDUAL))
        return fail(MOE_E_SHAPE, "a stack needs MOE_PRENORM | MOE_RESIDUAL in the shape flags");
    if ((st = check_ptr(d_x, 16, "d_x")) != MOE_OK || (st = check_ptr(d_x_out, 16, "d_x_out")) != MOE_OK)
        return st;
    if (!h_blobs)
        return fail(MOE_E_INVALID, "h_blobs is NULL");
    const int E = p->shape.n_experts, k = p->shape.top_k, H = p->shape.hidden;
    cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
    int32_t* d_idx = reinterpret_cast<int32_t*>(p->ws + p->wl.sel);
    float* d_w = reinterpret_cast<float*>(d_idx + kMaxK);
    int32_t* d_spec = d_idx + 3 * kMaxK;  // the next layer routed on this layer's input
    float* d_spec_w = reinterpret_cast<float*>(d_idx + 4 * kMaxK);
    float* bufs[2] = {reinterpret_cast<float*>(p->ws + p->wl.xbuf), reinterpret_cast<float*>(p->ws + p->wl.xbuf) + H};
    const float* cur = d_x;
    int32_t idx[kMaxK], slots[kMaxK], spec[kMaxK];
    for (int li = 0; li < n_layers; ++li) {
        const int l = layer0 + li;
        float* out = li == n_layers - 1 ? d_x_out : bufs[li & 1];
        // speculation: the next layer's router on this layer's input (the residual changes by one
        // layer's output in between), so that its likely misses can travel while this layer runs
        const bool spec_on = p->prefetch > 0 && li + 1 < n_layers;
        if ((st = moe_route(p, l, cur, d_idx, d_w, cs)) != MOE_OK)
            return st;
        if (spec_on && (st = moe_route(p, l + 1, cur, d_spec, d_spec_w, cs)) != MOE_OK)
            return st;
        CUDA_TRY(cudaMemcpyAsync(idx, d_idx, sizeof(int32_t) * k, cudaMemcpyDeviceToHost, cs));
        if (spec_on)
            CUDA_TRY(cudaMemcpyAsync(spec, d_spec, sizeof(int32_t) * k, cudaMemcpyDeviceToHost, cs));
        CUDA_TRY(cudaStreamSynchronize(cs));
        for (int j = 0; j < k; ++j)
            if (idx[j] < 0 || idx[j] >= E)
                return fail(MOE_E_CUDA, "routing returned expert %d at layer %d (device status %s)", idx[j], l,
                            "unknown: read it with moe_device_status");
        if ((st = moe_pool_lookup(p, l, idx, k, slots)) != MOE_OK)
            return st;
        for (int j = 0; j < k; ++j) {
            if (slots[j] >= 0)
                continue;
            const void* blob = h_blobs[(size_t)l * E + idx[j]];
            if (!blob)
                return fail(MOE_E_INVALID, "no host blob for expert %d of layer %d", idx[j], l);
            if ((st = moe_pool_load_slot(p, l, idx[j], blob, copy_stream, &slots[j])) != MOE_OK)
                return st;
        }
        if ((st = moe_pool_wait_loads(p, compute_stream)) != MOE_OK)
            return st;
        // the next layer's top predicted experts that are not resident: copied behind this
        // layer's misses on the copy stream (the next layer's own lookup decides what is used; a
        // wrong guess only costs link time). A full pool skips the rest of the guesses.
        if (spec_on)
            for (int j = 0; j < k && j < p->prefetch; ++j) {
                int32_t s_ = -1;
                if (spec[j] < 0 || spec[j] >= E || moe_pool_slot_of(p, l + 1, spec[j], &s_) != MOE_OK || s_ >= 0)
                    continue;
                const void* blob = h_blobs[(size_t)(l + 1) * E + spec[j]];
                if (!blob || moe_pool_load_slot(p, l + 1, spec[j], blob, copy_stream, &s_) != MOE_OK)
                    break;
            }
        if ((st = moe_experts(p, l, cur, d_w, slots, out, compute_stream)) != MOE_OK)
            return st;
        if ((st = moe_pool_release(p, compute_stream)) != MOE_OK)
            return st;
        if (h_topk_idx)
            for (int j = 0; j < k; ++j)
                h_topk_idx[(size_t)li * k + j] = idx[j];
        cur = out;
    }
    return MOE_OK;
}

moe_status moe_stack_forward_qpack(moe_pool* p, int32_t layer0, int32_t n_layers, const float* d_x, float* d_x_out,
                                   moe_qpack* q, void* h_staging, int32_t n_staging, void* compute_stream,
                                   void* copy_stream, int32_t* h_topk_idx)
{
    moe_status st = check_layers(p, layer0, n_layers);
    if (st != MOE_OK)
        return st;
    if ((p->shape.flags & (MOE_PRENORM | MOE_RESIDUAL)) != (MOE_PRENORM | MOE_RESIDUAL))
        return fail(MOE_E_SHAPE, "a stack needs MOE_PRENORM | MOE_RESIDUAL in the shape flags");
    if ((st = check_ptr(d_x, 16, "d_x")) != MOE_OK || (st = check_ptr(d_x_out, 16, "d_x_out")) != MOE_OK)
        return st;
    const int E = p->shape.n_experts, k = p->shape.top_k, H = p->shape.hidden;
    if (!q || !h_staging)
        return fail(MOE_E_INVALID, "container or staging buffer is NULL");
    const moe_shape& qs = moe::qp::shape(q);
    if (qs.hidden != H || qs.n_experts != E || qs.inter != p->shape.inter || qs.bits != p->shape.bits ||
        qs.group != p->shape.group || moe::qp::stride(q) != p->geo.stride || layer0 + n_layers > moe::qp::n_layers(q))
        return fail(MOE_E_INVALID, "the container holds another shape or fewer layers than the pool's");
    if (n_staging < k)
        return fail(MOE_E_INVALID, "%d staging slots for top-%d", n_staging, k);
    if (reinterpret_cast<uintptr_t>(h_staging) & 4095)
        return fail(MOE_E_INVALID, "h_staging must be 4096-byte aligned");
    if ((int)p->stage_ev.size() < n_staging) {
        for (int i = (int)p->stage_ev.size(); i < n_staging; ++i) {
            cudaEvent_t ev;
            CUDA_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
            p->stage_ev.push_back(ev);
            p->stage_used.push_back(0);
        }
    }
    const uint64_t stride = p->geo.stride;
    uint8_t* stage = static_cast<uint8_t*>(h_staging);
    cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
    cudaStream_t ys = static_cast<cudaStream_t>(copy_stream);
    int32_t* d_idx = reinterpret_cast<int32_t*>(p->ws + p->wl.sel);
    float* d_w = reinterpret_cast<float*>(d_idx + kMaxK);
    float* bufs[2] = {reinterpret_cast<float*>(p->ws + p->wl.xbuf), reinterpret_cast<float*>(p->ws + p->wl.xbuf) + H};
    const float* cur = d_x;
    int32_t idx[kMaxK], slots[kMaxK], mlayer[kMaxK], mexpert[kMaxK], mj[kMaxK], ms[kMaxK];
    void* mdst[kMaxK];
    for (int li = 0; li < n_layers; ++li) {
        const int l = layer0 + li;
        float* out = li == n_layers - 1 ? d_x_out : bufs[li & 1];
        if ((st = moe_route(p, l, cur, d_idx, d_w, cs)) != MOE_OK)
            return st;
        CUDA_TRY(cudaMemcpyAsync(idx, d_idx, sizeof(int32_t) * k, cudaMemcpyDeviceToHost, cs));
        CUDA_TRY(cudaStreamSynchronize(cs));
        for (int j = 0; j < k; ++j)
            if (idx[j] < 0 || idx[j] >= E)
                return fail(MOE_E_CUDA, "routing returned expert %d at layer %d (device status %s)", idx[j], l,
                            "unknown: read it with moe_device_status");
        if ((st = moe_pool_lookup(p, l, idx, k, slots)) != MOE_OK)
            return st;
        // the misses: staging slots (each free once its previous copy is done), parallel reads
        int nm = 0;
        for (int j = 0; j < k; ++j) {
            if (slots[j] >= 0)
                continue;
            const int s = p->stage_next;
            p->stage_next = (p->stage_next + 1) % n_staging;
            if (p->stage_used[s])
                CUDA_TRY(cudaEventSynchronize(p->stage_ev[s]));
            mlayer[nm] = l;
            mexpert[nm] = idx[j];
            mdst[nm] = stage + (size_t)s * stride;
            mj[nm] = j;
            ms[nm] = s;
            ++nm;
        }
        if (nm) {
            const int e = moe::qp::read_many(q, nm, mlayer, mexpert, mdst);
            if (e)
                return fail(MOE_E_INVALID, "reading layer %d's experts from the container failed (%s)", l, strerror(e));
        }
        for (int i = 0; i < nm; ++i) {
            if ((st = moe_pool_load_slot(p, l, mexpert[i], mdst[i], copy_stream, &slots[mj[i]])) != MOE_OK)
                return st;
            CUDA_TRY(cudaEventRecord(p->stage_ev[ms[i]], ys));
            p->stage_used[ms[i]] = 1;
        }
        if ((st = moe_pool_wait_loads(p, compute_stream)) != MOE_OK)
            return st;
        if ((st = moe_experts(p, l, cur, d_w, slots, out, compute_stream)) != MOE_OK)
            return st;
        if ((st = moe_pool_release(p, compute_stream)) != MOE_OK)
            return st;
        if (h_topk_idx)
            for (int j = 0; j < k; ++j)
                h_topk_idx[(size_t)li * k + j] = idx[j];
        cur = out;
    }
    return MOE_OK;
}

}  // extern "C"

namespace {

struct BatLayout {
    size_t us, logits, idx, w, gamma, counts, offs, cursor, list, aw, apos, ypart, hbuf, tasks_gu, tasks_dn, n_tasks,
        total;
    size_t max_gu, max_dn;
};

BatLayout bat_layout(const moe_shape& s, int T)
{
    BatLayout b{};
    const size_t H = s.hidden, E = s.n_experts, k = s.top_k;
    const size_t Imax = s.inter > s.shared_inter ? s.inter : s.shared_inter;
    const size_t A = (size_t)T * (k + 1);
    size_t o = 0;
    auto take = [&](size_t& f, size_t bytes) {
        f = o;
        o = up256(o + bytes);
    };
    take(b.us, 2 * A * H);
    take(b.logits, 4 * (size_t)T * E);
    take(b.idx, 4 * (size_t)T * k);
    take(b.w, 4 * (size_t)T * k);
    take(b.gamma, 4 * (size_t)T);
    take(b.counts, 4 * (E + 2));
    take(b.offs, 4 * (E + 2));
    take(b.cursor, 4 * (E + 2));
    take(b.list, 4 * A);
    take(b.aw, 4 * A);
    take(b.apos, 4 * A);
    take(b.ypart, (s.flags & MOE_DETERMINISTIC) ? 4 * A * H : 0);
    take(b.hbuf, 2 * A * Imax);
    const size_t chunks = A / tc::kNT + E + 1;  // 128-token chunks over all experts (one partial each)
    b.max_gu = chunks * (Imax / 64);
    b.max_dn = chunks * ((H + 127) / 128);
    take(b.tasks_gu, 16 * b.max_gu);
    take(b.tasks_dn, 16 * b.max_dn);
    take(b.n_tasks, 16);
    b.total = o;
    return b;
}

}  // namespace

extern "C" {

size_t moe_batched_workspace_bytes(const moe_shape* s, int32_t n_tokens)
{
    if (!s || n_tokens <= 0)
        return 0;
    return bat_layout(*s, n_tokens).total;
}

moe_status moe_layer_forward_batched(moe_pool* p, int32_t layer, const void* d_x, int32_t T, float* d_y,
                                     int32_t* d_topk_idx, float* d_topk_w, void* d_work, size_t work_bytes,
                                     void* stream)
{
    moe_status st = check_layers(p, layer, 1);
    if (st != MOE_OK)
        return st;
    if (p->shape.flags & (MOE_PRENORM | MOE_RESIDUAL))
        return fail(MOE_E_SHAPE, "the batched path takes a bf16 layer input (no pre-norm, no residual)");
    if (T <= 0)
        return fail(MOE_E_INVALID, "n_tokens must be positive");
    if ((st = check_ptr(d_x, 16, "d_x")) != MOE_OK || (st = check_ptr(d_y, 16, "d_y")) != MOE_OK ||
        (st = check_ptr(d_work, 256, "d_work")) != MOE_OK)
        return st;
    const moe_shape& sh = p->shape;
    const int H = sh.hidden, E = sh.n_experts, k = sh.top_k, I = sh.inter, Is = sh.shared_inter;
    const int Imax = I > Is ? I : Is;
    if (H % 64 != 0 || I % 64 != 0 || Is % 64 != 0)
        return fail(MOE_E_SHAPE, "batched path needs hidden, inter and shared_inter multiples of 64");
    if (tc::expert_smem_bytes(H, Imax, sh.bits) > (size_t)p->smem_optin)
        return fail(MOE_E_SHAPE, "batched path: staging for hidden %d does not fit in shared memory", H);
    const BatLayout bl = bat_layout(sh, T);
    if (work_bytes < bl.total)
        return fail(MOE_E_NOMEM, "batched workspace holds %zu bytes, needs %zu (moe_batched_workspace_bytes)",
                    work_bytes, bl.total);
    int dev = -1;
    CUDA_TRY(cudaGetDevice(&dev));
    if (dev != p->device)
        return fail(MOE_E_INVALID, "current device %d differs from the pool's device %d", dev, p->device);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(d_work);
    const LayerDesc& L = p->layers[layer];

    tc::GroupedArgs A{};
    const int nA = T * (k + 1);
    if ((int)p->k_shared.size() != p->L) {
        p->k_shared.assign(p->L, {});
        p->k_router.assign(p->L, {});
        p->m_shared.resize(3 * (size_t)p->L);
        p->m_router.resize(p->L);
    }
    int rc = 0;
    if (!p->k_arena.same(p->arena, p->S, sh.bits)) {
        p->k_arena = {};
        rc = encode_slice_maps(p->m_arena, p->arena, p->S, p->geo.stride, p->geo, sh.bits);
        if (rc == 0)
            p->k_arena = {p->arena, p->S, sh.bits};
    }
    auto& ks = p->k_shared[layer];
    if (rc == 0 && !ks.same(L.shared_blob, sh.bits, 0)) {
        ks = {};
        CUtensorMap tmp[3];
        rc = encode_slice_maps(tmp, L.shared_blob, 1, p->geo_s.stride, p->geo_s, sh.bits);
        if (rc == 0) {
            for (int m = 0; m < 3; ++m)
                p->m_shared[3 * (size_t)layer + m] = tmp[m];
            ks = {L.shared_blob, sh.bits, 0};
        }
    }
    auto& kr = p->k_router[layer];
    if (rc == 0 && !kr.same(L.router, H, E)) {
        kr = {};
        rc = encode_tiles16(&p->m_router[layer], L.router, H, E, 128, false);
        if (rc == 0)
            kr = {L.router, H, E};
    }
    if (rc == 0 && !p->k_u.same(d_x, T, H)) {
        p->k_u = {};
        rc = encode_tiles16(&p->m_u, d_x, H, T, tc::kNT, false);
        if (rc == 0)
            p->k_u = {d_x, T, H};
    }
    if (rc == 0 && !p->k_b0.same(w + bl.us, nA, H)) {
        p->k_b0 = {};
        rc = encode_tiles16(&p->m_b0, w + bl.us, H, nA, tc::kBRows, true);
        if (rc == 0)
            p->k_b0 = {w + bl.us, nA, H};
    }
    if (rc == 0 && !p->k_b1.same(w + bl.hbuf, nA, Imax)) {
        p->k_b1 = {};
        rc = encode_tiles16(&p->m_b1, w + bl.hbuf, Imax, nA, tc::kBRows, true);
        if (rc == 0)
            p->k_b1 = {w + bl.hbuf, nA, Imax};
    }
    if (rc != 0)
        return fail(MOE_E_CUDA, "tensor map encoding failed (%d)", rc);
    for (int m = 0; m < 3; ++m) {
        A.map_q[0][m] = p->m_arena[m];
        A.map_q[1][m] = p->m_shared[3 * (size_t)layer + m];
    }
    A.map_wr = p->m_router[layer];
    A.map_u = p->m_u;
    A.map_b[0] = p->m_b0;
    A.map_b[1] = p->m_b1;
    A.geo = p->geo;
    A.geo_s = p->geo_s;
    A.T = T;
    A.H = H;
    A.E = E;
    A.k = k;
    A.I = I;
    A.Is = Is;
    A.bits = sh.bits;
    A.Imax = Imax;
    A.arena = p->arena;
    A.stride = p->geo.stride;
    A.table = reinterpret_cast<const int32_t*>(p->ws + p->wl.table) + (size_t)layer * E;
    A.shared_blob = L.shared_blob;
    A.list = reinterpret_cast<const int32_t*>(w + bl.list);
    A.aw = reinterpret_cast<const float*>(w + bl.aw);
    A.us = reinterpret_cast<const __half*>(w + bl.us);
    A.hbuf = reinterpret_cast<__half*>(w + bl.hbuf);
    A.y = d_y;
    const bool det = (sh.flags & MOE_DETERMINISTIC) != 0;
    A.ypart = det ? reinterpret_cast<float*>(w + bl.ypart) : nullptr;
    A.logits = reinterpret_cast<float*>(w + bl.logits);
    A.status = reinterpret_cast<int*>(p->ws + p->wl.status);
    A.timeout_cycles = 2 * (long long)p->timeout_ns;

    int32_t* idx = d_topk_idx ? d_topk_idx : reinterpret_cast<int32_t*>(w + bl.idx);
    float* wts = d_topk_w ? d_topk_w : reinterpret_cast<float*>(w + bl.w);
    float* gamma = reinterpret_cast<float*>(w + bl.gamma);
    int32_t* counts = reinterpret_cast<int32_t*>(w + bl.counts);
    int32_t* offs = reinterpret_cast<int32_t*>(w + bl.offs);
    int32_t* cursor = reinterpret_cast<int32_t*>(w + bl.cursor);
    int4* tgu = reinterpret_cast<int4*>(w + bl.tasks_gu);
    int4* tdn = reinterpret_cast<int4*>(w + bl.tasks_dn);
    int32_t* ntasks = reinterpret_cast<int32_t*>(w + bl.n_tasks);
    const int grid = p->grid;

    CUDA_TRY(cudaMemsetAsync(counts, 0, sizeof(int32_t) * (E + 2), cs));
    if (!det)
        CUDA_TRY(cudaMemsetAsync(d_y, 0, sizeof(float) * (size_t)T * H, cs));
    const int r_tasks = ((E + 127) / 128) * ((T + tc::kNT - 1) / tc::kNT);
    tc::launch_router_gemm(A, r_tasks < grid ? r_tasks : grid, cs);
    bat::launch_topk(A.logits, L.logit_bias, T, E, k, (sh.flags & MOE_RENORM) ? 1 : 0,
                     static_cast<const uint16_t*>(d_x), L.shared_gate, H, idx, wts, gamma, counts, cs);
    bat::launch_plan(counts, E, T, I, Is, H, offs, cursor, tgu, tdn, ntasks, cs);
    int32_t* apos = reinterpret_cast<int32_t*>(w + bl.apos);
    bat::launch_place(idx, wts, gamma, T, E, k, cursor, const_cast<int32_t*>(A.list), const_cast<float*>(A.aw), apos, cs);
    bat::launch_gather_rows(static_cast<const uint16_t*>(d_x), A.list, nA, H, sh.bits, reinterpret_cast<__half*>(w + bl.us),
                            A.status, cs);
    const int nev = (int)p->gemm_ev.size() / 2;
    const int ei = nev ? p->gemm_next : -1;
    if (ei >= 0)
        CUDA_TRY(cudaEventRecord(p->gemm_ev[2 * ei], cs));
    // MOE_GEMV and few tokens: the experts' weights streamed once through matrix-vector products;
    // else (the default) the tensor-core GEMMs
    if ((sh.flags & MOE_GEMV) && T <= gv::kMaxTokens && gv::geometry_ok(p->geo) && gv::geometry_ok(p->geo_s) &&
        gv::smem_bytes(H, Imax, sh.bits) <= (size_t)p->smem_optin) {
        gv::launch(1, A, tgu, ntasks, 2 * grid, cs);
        gv::launch(2, A, tdn, ntasks + 1, 2 * grid, cs);
    } else {
        tc::launch_expert_gemm(1, A, tgu, ntasks, grid, cs);
        tc::launch_expert_gemm(2, A, tdn, ntasks + 1, grid, cs);
    }
    if (det)
        bat::launch_combine(A.ypart, apos, T, k, H, d_y, cs);
    if (ei >= 0) {
        CUDA_TRY(cudaEventRecord(p->gemm_ev[2 * ei + 1], cs));
        p->gemm_next = (p->gemm_next + 1) % nev;
        p->gemm_used += 1;
    }
    CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

}  // extern "C"
