// hybrid.cu -- the two per-layer decode steps that precede the MoE FFN in the 80B hybrid stack
// (include/hybrid.h): the Gated DeltaNet decode step and gated grouped-query attention decode.
//
// Both are bandwidth-bound: the DeltaNet step reads and writes each state element once (8 bytes
// for 2 multiply-adds of the update and 1 of the read-out), and decode attention reads each cached
// K and V element once (4 bytes each for G multiply-adds, G = query heads per K/V head). Neither
// is a dense contraction with reuse, so both run on the FP32 pipes with coalesced 16-byte loads;
// what matters is bytes in flight and how the work is spread over the 148 SMs.
//
// Gated DeltaNet step. One cluster of 8 CTAs per (sequence, value head); CTA j owns dv/8 rows of
// the head's dv x dk state, each warp dv/32 of them, each lane one float4 of a 128-wide row. A row
// update needs only the row, k^ and q^ (the gated delta rule is rank one along k):
//     d = S_r . k^,  S_r <- alpha S_r + beta (v_r - alpha d) k^,  o_r = S_r . q^,
// so each state element is loaded once, updated in registers and stored once. The head's RMS norm
// needs the sum of o_r^2 over all dv rows: each CTA writes its partial sum into slot `rank` of every
// CTA's shared memory (distributed shared memory), one cluster barrier later every CTA adds its
// eight slots in rank order (so all compute the same total).
//
// Gated GQA decode. Split-K ("flash decoding"): the positions of each (sequence, K/V head) are
// cut into n_split ranges, about one CTA per SM in all. A CTA streams its range in chunks of 32
// positions through a three-stage shared-memory ring filled by 1D bulk copies (K rows and V rows of a
// chunk are contiguous in the cache), computes the G heads' scores, keeps a running softmax
// (maximum, sum) per head and accumulates the weighted V rows; it leaves (m, l, o) per head in the
// workspace. A second kernel merges the ranges of each query head in range order and applies the
// output gate. The new token's k and v enter the cache from the CTA whose range holds position pos.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdarg>
#include <cstdint>
#include <cstdio>

#include "attr.h"
#include "hybrid.h"

namespace cg = cooperative_groups;

namespace moe {
void set_last_error(const char* msg);
}

namespace {

moe_status hfail(moe_status st, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    moe::set_last_error(buf);
    return st;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ float4 bf4(const uint16_t* p)  // 4 bf16 at an 8-byte aligned address
{
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xFFFF0000u));
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Sums G per-lane values (one per head) over the warp's 32 lanes with one butterfly: at each of the
// first log2(G) levels a lane keeps the half of its values its partner does not and adds the
// partner's copy of it (G/2, G/4, ... shuffles), then the last levels sum the single remaining
// value. Lane l ends with the full sum for head head_of<G>(l); 2^(5 - log2 G) lanes hold each head.
// G + log2(32 / G) - 1 shuffles instead of 5 G.
template <int G>
__device__ __forceinline__ float reduce_scatter(float (&v)[G], int lane)
{
    int off = 16;
#pragma unroll
    for (int w = G / 2; w >= 1; w /= 2, off /= 2) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float send = upper ? v[i] : v[i + w];
            const float keep = upper ? v[i + w] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float r = v[0];
    for (; off >= 1; off /= 2)
        r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
}

template <int G>
__device__ __forceinline__ int head_of(int lane)
{
    int h = 0, off = 16;
#pragma unroll
    for (int w = G / 2; w >= 1; w /= 2, off /= 2)
        if (lane & off)
            h += w;
    return h;
}

__device__ __forceinline__ float dot4(float4 a, float4 b) { return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w; }

__device__ __forceinline__ float sigmoidf(float x) { return 1.0f / (1.0f + expf(-x)); }

// Programmatic dependent launch: the kernels are launched so that they may start while the
// previous kernel in the stream finishes; each waits for that kernel's completion (and the
// visibility of its writes) before its first global-memory access, and lets the next kernel start
// once its own work is under way. Without the launch attribute both are no-ops.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------------------------------
// Gated DeltaNet decode step
// ------------------------------------------------------------------------------------------

constexpr int kGdnCluster = 8;    // CTAs per (sequence, value head)
constexpr int kGdnThreads = 128;  // 4 warps
constexpr int kGdnDk = 128;       // key_dim: one float4 of each state row per lane

struct GdnArgs {
    int Hk, Hv, dv, rep;
    float* state;
    const uint16_t *q, *k, *v, *z;
    const float *a, *b, *A_log, *dt_bias, *norm_w;
    float scale;
    float *o, *y;
};

template <int RPW>  // state rows per warp: dv = 32 * RPW
__global__ void __cluster_dims__(kGdnCluster, 1, 1) __launch_bounds__(kGdnThreads)
    gdn_step_kernel(const GdnArgs A)
{
    __shared__ float warp_ss[kGdnThreads / 32];
    __shared__ float cta_ss[kGdnCluster];  // slot j: the partial sum of the cluster's CTA j
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int head = blockIdx.x / kGdnCluster;  // sequence * Hv + value head
    const int seq = head / A.Hv, h = head - seq * A.Hv;
    const int g = h / A.rep;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int dv = A.dv;
    const int row0 = rank * (4 * RPW) + warp * RPW;
    // first half of a cluster barrier: no CTA writes into a peer's shared memory before every CTA
    // of the cluster is running; the wait half comes after the loads, so it costs nothing
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    grid_dep_wait();

    // the state rows go out first: they are the step's bytes
    float* Sh = A.state + (size_t)head * dv * kGdnDk;
    float4 s[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i)
        s[i] = *reinterpret_cast<const float4*>(Sh + (size_t)(row0 + i) * kGdnDk + 4 * lane);
    float vr[RPW], zr[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        vr[i] = bf(A.v[(size_t)head * dv + row0 + i]);
        zr[i] = bf(A.z[(size_t)head * dv + row0 + i]);
    }
    const size_t kq = ((size_t)seq * A.Hk + g) * kGdnDk + 4 * lane;
    float4 kk = bf4(A.k + kq), qq = bf4(A.q + kq);
    // the per-head scalars and the norm weight of this lane's output row: all loads in one round trip
    const float a_in = A.a[head], b_in = A.b[head], A_log = A.A_log[h], dt_bias = A.dt_bias[h];
    const float nw = lane < RPW ? A.norm_w[row0 + lane] : 0.0f;
    const float kinv = 1.0f / sqrtf(warp_sum(dot4(kk, kk)) + MOE_GDN_L2_EPS);
    const float qmul = A.scale / sqrtf(warp_sum(dot4(qq, qq)) + MOE_GDN_L2_EPS);
    kk = make_float4(kk.x * kinv, kk.y * kinv, kk.z * kinv, kk.w * kinv);
    qq = make_float4(qq.x * qmul, qq.y * qmul, qq.z * qmul, qq.w * qmul);

    grid_dep_launch();
    const float x = a_in + dt_bias;
    const float sp = x > 0.0f ? x + log1pf(expf(-x)) : log1pf(expf(x));
    const float alpha = expf(-expf(A_log) * sp);
    const float beta = sigmoidf(b_in);

    float o[RPW];
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const float d = warp_sum(dot4(s[i], kk));
        const float c = beta * (vr[i] - alpha * d);
        const float4 n = make_float4(alpha * s[i].x + c * kk.x, alpha * s[i].y + c * kk.y, alpha * s[i].z + c * kk.z,
                                     alpha * s[i].w + c * kk.w);
        *reinterpret_cast<float4*>(Sh + (size_t)(row0 + i) * kGdnDk + 4 * lane) = n;
        o[i] = warp_sum(dot4(n, qq));
        ss += o[i] * o[i];
    }
    if (lane == 0)
        warp_ss[warp] = ss;
    __syncthreads();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (threadIdx.x < kGdnCluster)  // this CTA's partial into slot `rank` of every CTA of the cluster
        *cluster.map_shared_rank(&cta_ss[rank], threadIdx.x) = (warp_ss[0] + warp_ss[1]) + (warp_ss[2] + warp_ss[3]);
    cluster.sync();  // release/acquire: every slot written before any is read (and no CTA exits
                     // while a peer may still write into it)
    float tot = 0.0f;
#pragma unroll
    for (int j = 0; j < kGdnCluster; ++j)
        tot += cta_ss[j];
    const float rinv = 1.0f / sqrtf(tot / (float)dv + MOE_GDN_NORM_EPS);
    if (lane < RPW) {
        // lane i writes row i of the warp (o[] indexed by a lane-dependent value: pick by unrolled select)
        float oi = o[0], zi = zr[0];
#pragma unroll
        for (int i = 1; i < RPW; ++i)
            if (lane == i) {
                oi = o[i];
                zi = zr[i];
            }
        const int r = row0 + lane;
        if (A.o)
            A.o[(size_t)head * dv + r] = oi;
        A.y[(size_t)head * dv + r] = oi * rinv * nw * (zi * sigmoidf(zi));
    }
}

// ------------------------------------------------------------------------------------------
// Gated GQA decode attention
// ------------------------------------------------------------------------------------------

constexpr int kGqaChunk = 32;       // positions per bulk copy
constexpr int kGqaStages = 3;       // shared-memory ring depth (3 x 64 KiB at D = 256)
constexpr int kGqaThreads = 256;    // 8 warps
constexpr int kGqaWarps = kGqaThreads / 32;
constexpr int kGqaCtaTarget = 148;  // split CTAs per launch aimed at (one per SM of a B300)
constexpr long long kGqaWaitLimit = 2000000000LL;  // cycles (about a second) per copy wait

struct GqaArgs {
    int Hq, Hkv, L, max_pos, n_split, per_split;
    float *kc, *vc;
    const int* pos;
    const uint16_t *q, *k, *v, *gate;
    float scale;
    float *part_o, *part_ml;
    float *o, *y;
    int* status;
};

struct GqaSplit {
    int n_split, per_split;
};

// Ranges per (sequence, K/V head): about one CTA per SM over all of them, never more ranges than
// chunks of positions; then the range length, and the count of ranges that length actually needs.
GqaSplit gqa_split(int batch, int Hkv, int max_pos)
{
    const int by_chunks = (max_pos + kGqaChunk - 1) / kGqaChunk;
    const int by_sms = std::max(1, kGqaCtaTarget / (batch * Hkv));
    const int n = std::min(by_chunks, by_sms);
    const int per = (max_pos + n - 1) / n;
    return {(max_pos + per - 1) / per, per};
}

size_t gqa_work_bytes(int batch, int Hq, int Hkv, int D, int max_pos)
{
    const GqaSplit s = gqa_split(batch, Hkv, max_pos);
    const size_t parts = (size_t)batch * Hkv * s.n_split * (Hq / Hkv);
    return parts * D * sizeof(float) + parts * 2 * sizeof(float);
}

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* m, int n)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(m)), "r"(n) : "memory");
}

__device__ __forceinline__ void mbar_expect(uint64_t* m, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(m)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t* m, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(su32(m)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// 1D bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* m)
{
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(su32(dst)),
                 "l"(src), "r"(bytes), "r"(su32(m))
                 : "memory");
}

// Wait for an mbarrier phase with a cycle limit (one thread).
__device__ __forceinline__ bool mbar_wait(uint64_t* m, uint32_t parity, long long limit)
{
    const long long t0 = clock64();
    while (!mbar_try(m, parity))
        if (clock64() - t0 > limit)
            return false;
    return true;
}

template <int G>
constexpr int gqa_groups() { return G >= 4 ? 2 : 1; }  // warp groups, each with G / groups heads

template <int D, int G>
__global__ void __launch_bounds__(kGqaThreads * gqa_groups<G>(), 1) gqa_split_kernel(const GqaArgs A)
{
    constexpr int HG = gqa_groups<G>();
    constexpr int GH = G / HG;  // heads of a warp group
    constexpr int NT = kGqaThreads * HG;
    constexpr int NV = D / 128;  // float4 pieces of a row per lane: dims 128 j + 4 lane + 0..3
    constexpr int kStage = 2 * kGqaChunk * D;  // floats: K rows then V rows
    extern __shared__ __align__(128) float smem[];
    float* p_s = smem + kGqaStages * kStage;  // [G][kGqaChunk] scores, then weights
    float* m_s = p_s + G * kGqaChunk;         // running maximum per head
    float* l_s = m_s + G;                     // running sum per head
    float* c_s = l_s + G;                     // this chunk's rescale factor per head
    uint64_t* bar = reinterpret_cast<uint64_t*>(c_s + ((G + 1) & ~1));

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // warps are (head group, position lane): group hg owns heads hg * GH ..; position lane pw takes
    // positions pw, pw + 8, ... of each chunk, for its group's heads
    const int hb = (warp / kGqaWarps) * GH, pw = warp % kGqaWarps;
    grid_dep_wait();
    const int pos = A.pos[b];
    if (pos < 0 || pos >= A.max_pos) {
        if (tid == 0 && split == 0 && g == 0)
            atomicCAS(A.status, 0, (int)MOE_E_RANGE);
        grid_dep_launch();
        return;
    }
    const int len = pos + 1;
    const int t0 = split * A.per_split;
    const int t1 = min(len, t0 + A.per_split);
    if (t0 >= t1) {
        grid_dep_launch();
        return;  // past this sequence's end: the merge reads only ranges below len
    }
    const size_t kvrow0 = (size_t)(b * A.Hkv + g) * A.L;  // row of position 0 in the caches
    const float* Kg = A.kc + kvrow0 * D;
    const float* Vg = A.vc + kvrow0 * D;
    const int nchunk = (t1 - t0 + kGqaChunk - 1) / kGqaChunk;

    if (tid == 0) {
        for (int s = 0; s < kGqaStages; ++s)
            mbar_init(&bar[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < G) {
        m_s[tid] = -INFINITY;
        l_s[tid] = 0.0f;
    }
    __syncthreads();
    auto issue = [&](int c) {
        const int s = c % kGqaStages;
        const int a0 = t0 + c * kGqaChunk;
        const int n = min(kGqaChunk, t1 - a0);
        const uint32_t bytes = (uint32_t)n * D * sizeof(float);
        float* st = smem + s * kStage;
        mbar_expect(&bar[s], 2 * bytes);
        bulk_g2s(st, Kg + (size_t)a0 * D, bytes, &bar[s]);
        bulk_g2s(st + kGqaChunk * D, Vg + (size_t)a0 * D, bytes, &bar[s]);
    };
    if (tid == 0)
        for (int c = 0; c < nchunk && c < kGqaStages; ++c)
            issue(c);
    grid_dep_launch();

    // this warp group's GH query rows, pre-scaled, in registers
    float4 qr[GH][NV];
#pragma unroll
    for (int h = 0; h < GH; ++h)
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const float4 t = bf4(A.q + ((size_t)b * A.Hq + g * G + hb + h) * D + 128 * j + 4 * lane);
            qr[h][j] = make_float4(t.x * A.scale, t.y * A.scale, t.z * A.scale, t.w * A.scale);
        }
    float4 acc[GH][NV];
#pragma unroll
    for (int h = 0; h < GH; ++h)
#pragma unroll
        for (int j = 0; j < NV; ++j)
            acc[h][j] = make_float4(0.f, 0.f, 0.f, 0.f);

    bool failed = false;
    int c = 0;
    for (; c < nchunk; ++c) {
        const int s = c % kGqaStages;
        // every thread observes the copy's completion itself (that is what makes the bytes visible)
        const bool ok = mbar_wait(&bar[s], (uint32_t)(c / kGqaStages) & 1u, kGqaWaitLimit);
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        float* Ks = smem + s * kStage;
        float* Vs = Ks + kGqaChunk * D;
        const int a0 = t0 + c * kGqaChunk;
        const int n = min(kGqaChunk, t1 - a0);
        if (pos >= a0 && pos < a0 + n) {
            // the new token: its row comes from the inputs, into shared memory and the cache
            const int r = pos - a0;
            const size_t src = ((size_t)b * A.Hkv + g) * D;
            for (int d = tid; d < D; d += NT) {
                const float kv = bf(A.k[src + d]), vv = bf(A.v[src + d]);
                Ks[r * D + d] = kv;
                Vs[r * D + d] = vv;
                A.kc[(kvrow0 + pos) * D + d] = kv;
                A.vc[(kvrow0 + pos) * D + d] = vv;
            }
            // these generic writes come before a later bulk copy into the same stage
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncthreads();
        }
        // scores of the group's heads at positions pw, pw + 8, ... (unrolled: the chains interleave)
#pragma unroll
        for (int i = 0; i < kGqaChunk / kGqaWarps; ++i) {
            const int t = pw + i * kGqaWarps;
            if (t < n) {
                float4 kr[NV];
#pragma unroll
                for (int j = 0; j < NV; ++j)
                    kr[j] = *reinterpret_cast<const float4*>(Ks + t * D + 128 * j + 4 * lane);
                float d[GH];
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    d[h] = 0.0f;
#pragma unroll
                    for (int j = 0; j < NV; ++j)
                        d[h] += dot4(qr[h][j], kr[j]);
                }
                const float r = reduce_scatter<GH>(d, lane);
                if ((lane & (32 / GH - 1)) == 0)
                    p_s[(hb + head_of<GH>(lane)) * kGqaChunk + t] = r;
            }
        }
        __syncthreads();
        // running softmax per head (warp h): new maximum, weights exp(s - m), rescale of the old sum
        for (int h = warp; h < G; h += NT / 32) {
            const float sc = lane < n ? p_s[h * kGqaChunk + lane] : -INFINITY;
            const float mo = m_s[h];
            const float mn = fmaxf(mo, warp_max(sc));
            const float pe = lane < n ? expf(sc - mn) : 0.0f;
            const float sum = warp_sum(pe);
            p_s[h * kGqaChunk + lane] = pe;
            if (lane == 0) {
                const float cr = expf(mo - mn);  // 0 on the first chunk (mo = -inf)
                c_s[h] = cr;
                l_s[h] = l_s[h] * cr + sum;
                m_s[h] = mn;
            }
        }
        __syncthreads();
        // values: rescale this warp's sums, then add its positions' weighted V rows
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            const float cr = c_s[hb + h];
#pragma unroll
            for (int j = 0; j < NV; ++j)
                acc[h][j] = make_float4(acc[h][j].x * cr, acc[h][j].y * cr, acc[h][j].z * cr, acc[h][j].w * cr);
        }
#pragma unroll
        for (int i = 0; i < kGqaChunk / kGqaWarps; ++i) {
            const int t = pw + i * kGqaWarps;
            if (t >= n)
                break;
            float4 vr[NV];
#pragma unroll
            for (int j = 0; j < NV; ++j)
                vr[j] = *reinterpret_cast<const float4*>(Vs + t * D + 128 * j + 4 * lane);
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                const float p = p_s[(hb + h) * kGqaChunk + t];
#pragma unroll
                for (int j = 0; j < NV; ++j) {
                    acc[h][j].x += p * vr[j].x;
                    acc[h][j].y += p * vr[j].y;
                    acc[h][j].z += p * vr[j].z;
                    acc[h][j].w += p * vr[j].w;
                }
            }
        }
        __syncthreads();  // the stage and the weights are free again
        if (tid == 0 && c + kGqaStages < nchunk)
            issue(c + kGqaStages);
    }
    if (failed) {
        if (tid == 0) {
            atomicCAS(A.status, 0, (int)MOE_E_TIMEOUT);
            // copies still in flight into this CTA's shared memory land before it exits (bounded)
            for (int cc = c; cc < nchunk && cc < c + kGqaStages; ++cc)
                mbar_wait(&bar[cc % kGqaStages], (uint32_t)(cc / kGqaStages) & 1u, kGqaWaitLimit);
        }
        return;
    }
    // the position lanes' sums into one, in lane order, through the (now idle) ring
    float* red = smem;  // [kGqaWarps][G][D]: kGqaWarps * G <= 2 * kGqaStages * kGqaChunk
#pragma unroll
    for (int h = 0; h < GH; ++h)
#pragma unroll
        for (int j = 0; j < NV; ++j)
            *reinterpret_cast<float4*>(red + ((size_t)pw * G + hb + h) * D + 128 * j + 4 * lane) = acc[h][j];
    __syncthreads();
    const size_t part = ((size_t)(b * A.Hkv + g) * A.n_split + split) * G;
    float* po = A.part_o + part * D;
    for (int e = 4 * tid; e < G * D; e += 4 * NT) {
        float4 t = *reinterpret_cast<const float4*>(red + e);
#pragma unroll
        for (int w = 1; w < kGqaWarps; ++w) {
            const float4 u = *reinterpret_cast<const float4*>(red + (size_t)w * G * D + e);
            t.x += u.x;
            t.y += u.y;
            t.z += u.z;
            t.w += u.w;
        }
        *reinterpret_cast<float4*>(po + e) = t;
    }
    if (tid < G) {
        A.part_ml[(part + tid) * 2] = m_s[tid];
        A.part_ml[(part + tid) * 2 + 1] = l_s[tid];
    }
}

// Merge of the ranges of one query head (block = one (head, sequence), thread = one dimension):
// M = max_s m_s, w_s = exp(m_s - M), o = sum_s w_s o_s / sum_s w_s l_s. Every reduction runs in a
// fixed order for a given number of ranges, so the result does not depend on timing.
constexpr int kMergeThreads = 256;

template <int NT>  // block size
__device__ __forceinline__ float block_reduce(float v, bool is_max, float* scratch)
{
    v = is_max ? warp_max(v) : warp_sum(v);
    const int warp = threadIdx.x >> 5;
    __syncthreads();  // scratch free (an earlier reduction may still be reading it)
    if ((threadIdx.x & 31) == 0)
        scratch[warp] = v;
    __syncthreads();
    float r = scratch[0];
#pragma unroll
    for (int w = 1; w < NT / 32; ++w)
        r = is_max ? fmaxf(r, scratch[w]) : r + scratch[w];
    return r;
}

template <int D, int G>
__global__ void __launch_bounds__(kMergeThreads) gqa_merge_kernel(const GqaArgs A)
{
    constexpr int kQuads = D / 4;                     // float4 columns of a head
    constexpr int kGroups = kMergeThreads / kQuads;   // range groups summed separately, then in order
    constexpr int kPer = (kGqaCtaTarget + kGroups - 1) / kGroups;  // ranges per group at most
    __shared__ float wgt[kGqaCtaTarget];
    __shared__ float scratch[kMergeThreads / 32];
    __shared__ float4 gsum[kGroups][kQuads];
    const int h = blockIdx.x, b = blockIdx.y;
    const int g = h / G, hh = h - g * G;
    grid_dep_wait();
    grid_dep_launch();
    const int pos = A.pos[b];
    if (pos < 0 || pos >= A.max_pos)
        return;
    const int nsp = (pos + 1 + A.per_split - 1) / A.per_split;
    const size_t part0 = (size_t)(b * A.Hkv + g) * A.n_split * G + hh;  // range s at part0 + s * G
    const int tid = threadIdx.x;
    const int quad = tid % kQuads, grp = tid / kQuads;
    // this thread's ranges s = grp + kGroups * i: their values first, all loads in flight together
    float4 v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int s = grp + kGroups * i;
        v[i] = s < nsp ? *reinterpret_cast<const float4*>(A.part_o + (part0 + (size_t)s * G) * D + 4 * quad)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float m = -INFINITY;
    for (int s = tid; s < nsp; s += kMergeThreads)
        m = fmaxf(m, A.part_ml[(part0 + (size_t)s * G) * 2]);
    const float M = block_reduce<kMergeThreads>(m, true, scratch);
    float l = 0.0f;
    for (int s = tid; s < nsp; s += kMergeThreads) {
        const float w = expf(A.part_ml[(part0 + (size_t)s * G) * 2] - M);
        wgt[s] = w;
        l += A.part_ml[(part0 + (size_t)s * G) * 2 + 1] * w;
    }
    const float Lsum = block_reduce<kMergeThreads>(l, false, scratch);  // its barriers also publish wgt[]
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int s = grp + kGroups * i;
        if (s < nsp) {
            const float w = wgt[s];
            acc.x += w * v[i].x;
            acc.y += w * v[i].y;
            acc.z += w * v[i].z;
            acc.w += w * v[i].w;
        }
    }
    gsum[grp][quad] = acc;
    __syncthreads();
    if (grp == 0) {
        float4 o = gsum[0][quad];
#pragma unroll
        for (int q = 1; q < kGroups; ++q) {
            o.x += gsum[q][quad].x;
            o.y += gsum[q][quad].y;
            o.z += gsum[q][quad].z;
            o.w += gsum[q][quad].w;
        }
        const float inv = 1.0f / Lsum;
        o = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
        const size_t i = ((size_t)b * A.Hq + h) * D + 4 * quad;
        if (A.o)
            *reinterpret_cast<float4*>(A.o + i) = o;
        const float4 gt = bf4(A.gate + i);
        *reinterpret_cast<float4*>(A.y + i) =
            make_float4(o.x * sigmoidf(gt.x), o.y * sigmoidf(gt.y), o.z * sigmoidf(gt.z), o.w * sigmoidf(gt.w));
    }
}

// Launch with programmatic stream serialization (the kernel may start before the previous one in
// the stream has finished; it waits for it with griddepcontrol.wait).
template <typename Args>
cudaError_t launch_pdl(void (*kernel)(Args), dim3 grid, dim3 block, size_t smem, cudaStream_t st, const Args& a)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <int D, int G>
moe_status gqa_launch(const GqaArgs& A, int batch, cudaStream_t st)
{
    constexpr size_t smem = (size_t)kGqaStages * 2 * kGqaChunk * D * sizeof(float) +
                            ((size_t)G * kGqaChunk + 3 * G + 2) * sizeof(float) + kGqaStages * sizeof(uint64_t) + 16;
    static std::atomic<int> done[moe::kMaxDevices];  // per instantiation and device
    cudaError_t e = moe::raise_smem_limit(gqa_split_kernel<D, G>, (int)smem, done);
    if (e != cudaSuccess)
        return hfail(MOE_E_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    e = launch_pdl(gqa_split_kernel<D, G>, dim3(A.n_split, A.Hkv, batch), dim3(kGqaThreads * gqa_groups<G>()),
                               smem, st, A);
    if (e == cudaSuccess)
        e = launch_pdl(gqa_merge_kernel<D, G>, dim3(A.Hq, batch), dim3(kMergeThreads), 0, st, A);
    if (e == cudaSuccess)
        e = cudaGetLastError();
    return e == cudaSuccess ? MOE_OK : hfail(MOE_E_CUDA, "gqa launch: %s", cudaGetErrorString(e));
}

}  // namespace

extern "C" moe_status moe_gdn_step(const moe_gdn_shape* shape, int32_t batch, float* d_state, const uint16_t* d_q,
                                   const uint16_t* d_k, const uint16_t* d_v, const uint16_t* d_z, const float* d_a,
                                   const float* d_b, const float* d_A_log, const float* d_dt_bias,
                                   const float* d_norm_w, float scale, float* d_o, float* d_y, void* stream)
{
    if (!shape)
        return hfail(MOE_E_INVALID, "moe_gdn_step: null shape");
    const int Hk = shape->n_key_heads, Hv = shape->n_value_heads, dk = shape->key_dim, dv = shape->value_dim;
    if (dk != kGdnDk || !(dv == 32 || dv == 64 || dv == 128 || dv == 256) || Hk < 1 || Hv < Hk || Hv % Hk)
        return hfail(MOE_E_SHAPE, "moe_gdn_step: unsupported shape Hk=%d Hv=%d dk=%d dv=%d", Hk, Hv, dk, dv);
    if (batch < 1 || (long long)batch * Hv * kGdnCluster > INT_MAX)
        return hfail(MOE_E_INVALID, "moe_gdn_step: batch %d out of range", batch);
    const void* ptrs[] = {d_state, d_q, d_k, d_v, d_z, d_a, d_b, d_A_log, d_dt_bias, d_norm_w, d_y};
    for (const void* p : ptrs)
        if (!aligned16(p))
            return hfail(MOE_E_INVALID, "moe_gdn_step: null or misaligned pointer");
    if (d_o && !aligned16(d_o))
        return hfail(MOE_E_INVALID, "moe_gdn_step: misaligned d_o");
    GdnArgs A{Hk, Hv, dv, Hv / Hk, d_state, d_q, d_k, d_v, d_z, d_a, d_b, d_A_log, d_dt_bias, d_norm_w, scale, d_o, d_y};
    const dim3 grid(batch * Hv * kGdnCluster);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (dv) {
    case 32: e = launch_pdl(gdn_step_kernel<1>, grid, dim3(kGdnThreads), 0, st, A); break;
    case 64: e = launch_pdl(gdn_step_kernel<2>, grid, dim3(kGdnThreads), 0, st, A); break;
    case 128: e = launch_pdl(gdn_step_kernel<4>, grid, dim3(kGdnThreads), 0, st, A); break;
    default: e = launch_pdl(gdn_step_kernel<8>, grid, dim3(kGdnThreads), 0, st, A); break;
    }
    if (e == cudaSuccess)
        e = cudaGetLastError();
    return e == cudaSuccess ? MOE_OK : hfail(MOE_E_CUDA, "moe_gdn_step launch: %s", cudaGetErrorString(e));
}

namespace {
bool gqa_supported(const moe_gqa_shape* s)
{
    if (!s || s->n_kv_heads < 1 || s->n_q_heads < s->n_kv_heads || s->n_q_heads % s->n_kv_heads || s->max_len < 1)
        return false;
    const int G = s->n_q_heads / s->n_kv_heads;
    if (s->head_dim == 256)
        return G == 1 || G == 2 || G == 4 || G == 8;
    if (s->head_dim == 128)
        return G == 1 || G == 2 || G == 4 || G == 8 || G == 16;
    return false;
}
}  // namespace

extern "C" size_t moe_gqa_workspace_bytes(const moe_gqa_shape* shape, int32_t batch, int32_t max_pos)
{
    if (!gqa_supported(shape) || batch < 1 || max_pos < 1 || max_pos > shape->max_len)
        return 0;
    return gqa_work_bytes(batch, shape->n_q_heads, shape->n_kv_heads, shape->head_dim, max_pos);
}

extern "C" moe_status moe_gqa_decode(const moe_gqa_shape* shape, int32_t batch, int32_t max_pos, float* d_k_cache,
                                     float* d_v_cache, const int32_t* d_pos, const uint16_t* d_q, const uint16_t* d_k,
                                     const uint16_t* d_v, const uint16_t* d_gate, float scale, void* d_work,
                                     size_t work_bytes, float* d_o, float* d_y, int32_t* d_status, void* stream)
{
    if (!gqa_supported(shape))
        return hfail(MOE_E_SHAPE, "moe_gqa_decode: unsupported shape");
    const int Hq = shape->n_q_heads, Hkv = shape->n_kv_heads, D = shape->head_dim;
    if (batch < 1 || batch > 65535 || (long long)batch * Hkv > 65535)
        return hfail(MOE_E_INVALID, "moe_gqa_decode: batch %d out of range", batch);
    if (max_pos < 1 || max_pos > shape->max_len)
        return hfail(MOE_E_INVALID, "moe_gqa_decode: max_pos %d outside 1..%d", max_pos, shape->max_len);
    const void* ptrs[] = {d_k_cache, d_v_cache, d_pos, d_q, d_k, d_v, d_gate, d_work, d_y, d_status};
    for (const void* p : ptrs)
        if (!aligned16(p))
            return hfail(MOE_E_INVALID, "moe_gqa_decode: null or misaligned pointer");
    if (d_o && !aligned16(d_o))
        return hfail(MOE_E_INVALID, "moe_gqa_decode: misaligned d_o");
    const size_t need = gqa_work_bytes(batch, Hq, Hkv, D, max_pos);
    if (work_bytes < need)
        return hfail(MOE_E_NOMEM, "moe_gqa_decode: workspace %zu bytes, %zu needed", work_bytes, need);
    const GqaSplit sp = gqa_split(batch, Hkv, max_pos);
    const int G = Hq / Hkv;
    const size_t parts = (size_t)batch * Hkv * sp.n_split * G;
    float* part_o = static_cast<float*>(d_work);
    GqaArgs A{Hq, Hkv, shape->max_len, max_pos, sp.n_split, sp.per_split, d_k_cache, d_v_cache, d_pos, d_q, d_k, d_v,
              d_gate, scale, part_o, part_o + parts * D, d_o, d_y, d_status};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (D == 256) {
        switch (G) {
        case 1: return gqa_launch<256, 1>(A, batch, st);
        case 2: return gqa_launch<256, 2>(A, batch, st);
        case 4: return gqa_launch<256, 4>(A, batch, st);
        default: return gqa_launch<256, 8>(A, batch, st);
        }
    }
    switch (G) {
    case 1: return gqa_launch<128, 1>(A, batch, st);
    case 2: return gqa_launch<128, 2>(A, batch, st);
    case 4: return gqa_launch<128, 4>(A, batch, st);
    case 8: return gqa_launch<128, 8>(A, batch, st);
    default: return gqa_launch<128, 16>(A, batch, st);
    }
}
