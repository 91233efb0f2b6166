// gdn_internal.cuh -- types and device helpers shared by the libgdn translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "gdn.h"

namespace gdn {

// ----------------------------------------------------------------- pool ----

struct LayerParams {
    const float* conv_w = nullptr;
    const float* A_log = nullptr;
    const float* dt_bias = nullptr;
    const float* norm_w = nullptr;
    bool set() const { return conv_w && A_log && dt_bias && norm_w; }
};

// Prefill workspace.  The recurrent path (d < 128) keeps per-token intermediates in fp32;
// the chunked tensor-core path (d = 128) forms q, k, v and the gates inside its pre-pass
// and keeps only per-chunk records.
struct PrefillWorkspace {
    float* qh = nullptr;     // [T][Hqk*dk] normalised q, scaled by dk^-1/2   (recurrent path)
    float* kh = nullptr;     // [T][Hqk*dk] normalised k                      (recurrent path)
    float* vc = nullptr;     // [T][Hv*dv]  conv + SiLU v                     (recurrent path)
    float* g = nullptr;      // [T][Hv]     log decay                         (recurrent path)
    float* beta = nullptr;   // [T][Hv]                                       (recurrent path)
    float* o = nullptr;      // [T][Hv*dv]  delta-rule output before the norm (recurrent path)
    float* kq = nullptr;     // [T][Hqk]    k_hat . q_hat                     (recurrent path)
    int* order = nullptr;    // [T + 64] sequences ranked by length, longest first
    int* lcnt = nullptr;     // [T + 2] validation scratch (length histogram; many sequences)
    int* ltie = nullptr;     // [T + 2] validation scratch (ties of equal lengths)
    // Chunked path: the call's chunk records are numbered chunk-index-major -- every sequence's
    // chunk 0 (in length order), then every chunk 1, ... -- so that a segment of records holds a
    // stretch of chunks of all the sequences still running.  Chunk c of the sequence of rank p is
    // record coff[c] + p.
    int* coff = nullptr;     // [ceil(T / 64) + 2] records of chunk index < c; coff[nc] = all records
    int* ctmp = nullptr;     // [ceil(T / 64) + 2] scratch of the validation kernel
    int2* rec_cp = nullptr;  // [ceil(T / 64) + T + 64] record -> (chunk index c, rank p)
    unsigned char* rec = nullptr;  // [chunk_cap][Hv] per-(chunk, v-head) records of the chunked path
    unsigned char* kimg = nullptr; // [chunk_cap][Hqk] per-(chunk, q/k head) K images
    int chunk_cap = 0;             // chunk records the workspace holds
    int* valid = nullptr;    // [0] 1 when the call's cu_seqlens / slot ids passed validation;
                             // [1] chunks of the longest sequence (nc); [8 .. 15] the sequences
                             // of a segment, by segment parity (chunked path, several segments)
    void* base = nullptr;
    size_t bytes = 0;
};

// A pool's second stream for the chunked prefill's segments: the state pass of segment g runs on
// it (high priority) while the caller's stream runs the pre-pass of segment g + 1 into the other
// half of the workspace; events order the two.
struct SegStreams {
    cudaStream_t side = nullptr;
    cudaEvent_t prep[2] = {nullptr, nullptr}, state[2] = {nullptr, nullptr};
};

struct Pool {
    gdn_shape shape{};
    int num_slots = 0, num_layers = 0;
    int C = 0, r = 0, io_size = 0;
    size_t state_bytes = 0, conv_bytes = 0, slot_bytes = 0, total_bytes = 0;
    char* base = nullptr;
    unsigned char* live_dev = nullptr;   // [num_slots] 1 = allocated (read by device-side checks)
    int* mark_dev = nullptr;             // [num_slots] zero between calls (prefill id check, many sequences)
    unsigned int* status_dev = nullptr;  // device status word (GDN_DEV_* bits)
    int* gate_dev = nullptr;             // [1] set when a mixed step's two parts name a common slot
    std::vector<int> free_list;          // free slot ids, popped from the back (lowest id first)
    std::vector<unsigned char> live;     // host mirror of live_dev
    std::vector<LayerParams> params;
    PrefillWorkspace ws;
    int device = 0, num_sms = 0;
    int debug_flags = 0;  // GDN_DEBUG_FLAGS at creation (timeout tests): bit 0: the decode producer fills
                          // no stage; bit 1: the chunked state pass does not fetch its first record
    SegStreams seg;       // chunked prefill (d = 128, max_prefill_tokens > 0) only
};

// Everything the prefill kernels of one call need (device pointers and sizes).
struct PrefillArgs {
    const int* cu;
    const int* ids;
    int n, T;
    const void *q, *k, *v, *a, *b, *z;
    void* out;
    const float *conv_w, *A_log, *dt_bias, *norm_w;
    char* base;
    uint64_t slot_bytes;
    uint32_t state_bytes;
    int num_layers, layer, num_slots;
    const unsigned char* live;
    int* mark;  // [num_slots] zero between calls: the distinct-id check of calls with many sequences
    unsigned int* status;
    int hqk, hv, r, D, W, C;
    float l2_eps, norm_eps;
    PrefillWorkspace ws;
    float* kq;  // [T][Hqk] k_hat . q_hat (workspace)
    const int* gate;  // when non-null and *gate != 0 the call does nothing (a mixed step's overlap check)
    int chunk;        // chunk length of the d < 128 chunked kernel (8, 16, 32 or 64)
    // chunked path (d = 128): the window of global chunk records [seg_lo, seg_hi) that this
    // pre-pass / state-pass launch pair handles (seg_hi = INT_MAX: all of them, the call being one
    // segment); record gc is stored at workspace position gc - seg_lo (< ws.chunk_cap)
    int seg_lo = 0, seg_hi = 0;
    int stall_fetch = 0;  // test hook: the state pass does not fetch its first chunk's record (timeout test)
};

// ------------------------------------------------------- checked builds ----
// A checked build (compiled with GDN_CHECKED into libgdn_checked.so) has the chunked prefill and
// projection kernels test every computed global and shared-memory range against the region it
// belongs to before the access: a failed test sets GDN_DEV_BOUNDS in the call's status word and the
// access is skipped.  It stands in for a device memory checker.  In normal builds kChecked is false
// and the tests compile away.
#ifdef GDN_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// [p, p + bytes) inside [lo, lo + region)
__device__ __forceinline__ bool within(const void* p, size_t bytes, const void* lo, size_t region)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(lo);
    return a >= b && a - b <= region && bytes <= region - (a - b);
}

// true when the access may go ahead: always in normal builds; in checked builds when ok, else the
// status bit is set
__device__ __forceinline__ bool chk(bool ok, unsigned int* status)
{
    if constexpr (kChecked) {
        if (!ok) atomicOr(status, GDN_DEV_BOUNDS);
        return ok;
    } else {
        return true;
    }
}

// Facts every kernel needs to check a slot pointer before touching memory.
struct SlotCheck {
    uint64_t base, total_bytes, slot_bytes;
    int num_layers, layer;
};

__device__ __forceinline__ bool slot_ptr_ok(uint64_t p, const SlotCheck& c)
{
    if (p < c.base) return false;
    uint64_t off = p - c.base;
    if (off >= c.total_bytes || off % c.slot_bytes) return false;
    return (int)((off / c.slot_bytes) % (uint64_t)c.num_layers) == c.layer;
}

// ----------------------------------------------------------- io dtypes ----

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// ------------------------------------------------------------- scalars ----

// x * sigmoid(x) with the fast exponential and division (a few ulp; the layer's tolerances are 1e-3)
__device__ __forceinline__ float silu_f(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// softplus(x) = log(1 + e^x); above 20 the correction log1p(e^-x) is below 2.1e-9 and dropped.
__device__ __forceinline__ float softplus_f(float x) { return x > 20.0f ? x : log1pf(expf(x)); }

__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

// g = -exp(A_log) * softplus(a + dt_bias): the log of the per-token decay alpha.
__device__ __forceinline__ float log_decay(float A_log, float a, float dt_bias)
{
    return -expf(A_log) * softplus_f(a + dt_bias);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    __half2 p = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}

// ----------------------------------------------------------- mbarriers ----

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per pipeline wait

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Programmatic dependent launch (a kernel launched with the programmatic stream serialization
// attribute may start before the previous kernel on its stream has finished): block until every
// prerequisite grid has completed and its memory operations are visible.  Code before this call
// must touch no global memory that a previous kernel writes or reads.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the next kernel on the stream, if launched with that attribute, to start its CTAs (they
// still wait in grid_dependency_wait for this grid to complete).
__device__ __forceinline__ void grid_dependents_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity.  Gives up after kWaitLimitNs,
// or as soon as *abort is set by another thread; returns false in both cases.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort && *abort) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// ---- packed fp32 pairs: f32x2 arithmetic, round to nearest (each lane equals the scalar op)
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

// the hardware's base-2 exponential and reciprocal approximations (PTX ex2.approx / rcp.approx)
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// SiLU of a pair: x sigma(x), sigma(x) = 1 / (1 + 2^(-x log2(e)))
__device__ __forceinline__ float2 silu2(float2 x)
{
    constexpr float kLog2e = 1.44269504088896340736f;
    const float2 t = mul2(x, make_float2(-kLog2e, -kLog2e));
    const float2 d = add2(make_float2(ex2_approx(t.x), ex2_approx(t.y)), make_float2(1.f, 1.f));
    return mul2(x, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

// ---- thread-block clusters: distributed shared memory between the CTAs of a cluster
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of the same shared-memory location in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// asynchronous 16-B store into another CTA's shared memory that completes 16 transaction bytes
// on that CTA's mbarrier (both addresses shared::cluster); the issuing thread does not wait
__device__ __forceinline__ void st_async_cluster_v4(uint32_t caddr, float4 v, uint32_t cbar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     caddr),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(cbar)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// bounded wait (kWaitLimitNs) with cluster-scope acquire, for phases completed by another CTA
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity)
{
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// all threads of all CTAs of the cluster
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 1-D bulk copy global -> shared (the TMA engine), completing on an mbarrier.
// dst, src 16-B aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 1-D bulk copy shared -> global (the TMA engine), tracked by the issuing thread's bulk
// async-group; dst, src 16-B aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until every bulk store this thread committed has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

__device__ __forceinline__ void named_bar_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void st_global_v4(void* p, float4 v)
{
    asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// ------------------------------------------------- shared layer arithmetic ----
// The decode kernel and the recurrent prefill kernels use these same routines,
// with the same reduction orders, so a prefill over L tokens reproduces L decode
// steps bit for bit.

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// sum_i x[i] * y[i] over n values by one warp (lane-strided partial sums, then a butterfly)
__device__ __forceinline__ float warp_dot(const float* x, const float* y, int n, int lane)
{
    float s = 0.0f;
    for (int i = lane; i < n; i += 32) s = fmaf(x[i], y[i], s);
    return warp_sum(s);
}

// q and k scales: q_hat = q * rsqrt(|q|^2 + eps) * D^-1/2, k_hat = k * rsqrt(|k|^2 + eps)
__device__ __forceinline__ float q_scale(float ssq, float eps, int D) { return rsqrtf(ssq + eps) * rsqrtf((float)D); }
__device__ __forceinline__ float k_scale(float ssk, float eps) { return rsqrtf(ssk + eps); }

// gated RMSNorm factor 1 / sqrt(mean(o^2) + eps)
__device__ __forceinline__ float rms_scale(float sso, float eps, int D) { return rsqrtf(sso / (float)D + eps); }

// One row i of one head's state S (d_k columns spread over LPR lanes, 16 per lane) for one token:
//   u_i = alpha (S_i . k);  delta_i = beta (v_i - u_i);  S_i <- alpha S_i + delta_i k;
//   o_i = S_i(new) . q = alpha (S_i . q) + delta_i (k . q)
// kq is k . q over the whole head.  All LPR lanes of the row get the same o.
template <int LPR>
__device__ __forceinline__ float row_update(float (&s)[16], const float (&kr)[16], const float (&qr)[16], float alpha,
                                            float beta, float v, float kq)
{
    float k0 = 0.f, k1 = 0.f, k2 = 0.f, k3 = 0.f, q0 = 0.f, q1 = 0.f, q2 = 0.f, q3 = 0.f;
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
        k0 = fmaf(s[j], kr[j], k0);
        k1 = fmaf(s[j + 1], kr[j + 1], k1);
        k2 = fmaf(s[j + 2], kr[j + 2], k2);
        k3 = fmaf(s[j + 3], kr[j + 3], k3);
        q0 = fmaf(s[j], qr[j], q0);
        q1 = fmaf(s[j + 1], qr[j + 1], q1);
        q2 = fmaf(s[j + 2], qr[j + 2], q2);
        q3 = fmaf(s[j + 3], qr[j + 3], q3);
    }
    float dk = (k0 + k1) + (k2 + k3);
    float dq = (q0 + q1) + (q2 + q3);
#pragma unroll
    for (int off = LPR / 2; off >= 1; off >>= 1) {
        dk += __shfl_xor_sync(0xffffffffu, dk, off);
        dq += __shfl_xor_sync(0xffffffffu, dq, off);
    }
    const float u = alpha * dk;
    const float delta = beta * (v - u);
#pragma unroll
    for (int j = 0; j < 16; ++j) s[j] = fmaf(delta, kr[j], alpha * s[j]);
    return fmaf(delta, kq, alpha * dq);
}

// Column j (0..15) of lane cl in a row spread over LPR lanes: float4 groups interleaved
// across the row's lanes, so a quarter-warp touches 128 contiguous bytes.
template <int LPR>
__device__ __forceinline__ int row_col(int j, int cl) { return (j >> 2) * 4 * LPR + 4 * cl + (j & 3); }

// --------------------------------------------------------- launchers ----

// Each returns cudaSuccess or the launch error.
// `gate` (device, may be null): when *gate != 0 at run time the launch does nothing
cudaError_t launch_decode(const Pool& P, int layer, const uint64_t* slot_ptrs, int m, const void* q, const void* k,
                          const void* v, const void* a, const void* b, const void* z, void* out, cudaStream_t st,
                          const int* gate = nullptr, int sms = 0);  // sms > 0: size the launch for that many SMs

// the pool's segment stream (highest priority) and events; destroy_seg_streams accepts a partial set
cudaError_t create_seg_streams(SegStreams* ss);
void destroy_seg_streams(SegStreams* ss);

cudaError_t launch_prefill(const Pool& P, int layer, const int* cu_seqlens, const int* slot_ids, int n_seqs,
                           int total_tokens, const void* q, const void* k, const void* v, const void* a,
                           const void* b, const void* z, void* out, cudaStream_t st, const int* gate = nullptr,
                           cudaEvent_t prep_done = nullptr, bool* split = nullptr);
// With prep_done (a mixed step): when the call is one chunked segment, the state pass runs on the
// pool's segment stream (highest priority) after prep_done, recorded on st once the pre-pass is
// enqueued, and st then waits for it; *split tells whether that happened.

// the row tensors of a prefill call are read and written in 16-B pieces (and by tensor copies)
inline bool rows_aligned16(const void* q, const void* k, const void* v, const void* z, const void* out)
{
    const uintptr_t m = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(z) |
                        reinterpret_cast<uintptr_t>(out);
    return (m & 15u) == 0;
}

// workspace of a prefill call of up to max_tokens tokens and chunk_cap chunk records
size_t prefill_workspace_bytes(const gdn_shape& s, int max_tokens, int chunk_cap);
// sequences a call may carry for a workspace of max_tokens tokens
inline int prefill_max_seqs(int max_tokens) { return max_tokens + 64; }
// up to this many sequences a prefill call's validation compares ids pairwise and ranks lengths by
// counting (O(n^2), fast for few); more use per-slot marks and a length histogram
constexpr int kPairwiseSeqs = 512;
// chunk records a pool reserves for calls of up to max_tokens tokens (chunked path, d = 128):
// a call needs ceil(T / 64) + n_seqs of them at most
inline bool prefill_chunked(const gdn_shape& s) { return s.dk == 128 && s.dv == 128; }
// A call whose records exceed the workspace runs in segments of chunk_cap records (prefill_segments),
// so a pool holds at most kPrefillMaxRecords of them, whatever max_tokens is.
constexpr int kPrefillMaxRecords = 512;  // also the most records of one segment (the state pass's table)
inline int prefill_pool_chunk_cap(const gdn_shape& s, int max_tokens)
{
    return prefill_chunked(s) ? std::min(2 * ((max_tokens + 63) / 64) + 64, kPrefillMaxRecords) : 0;
}
inline int prefill_call_chunks(int total_tokens, int n_seqs) { return (total_tokens + 63) / 64 + n_seqs; }
// segments (launch pairs) a call of that size takes with chunk_cap records per segment
inline int prefill_segments(int total_tokens, int n_seqs, int chunk_cap)
{
    return chunk_cap > 0 ? (prefill_call_chunks(total_tokens, n_seqs) + chunk_cap - 1) / chunk_cap : 0;
}
// bytes of one chunk record set (all v-heads and q/k heads of one chunk)
size_t chunk_record_bytes(int hv, int hqk);

// chunked tensor-core prefill of the delta rule + gated RMSNorm (d_k = d_v = 128), in two
// launches: the parallel pre-pass (conv, norms, gates and the chunk-local products; it reads
// the slots' conv buffers, so it runs before they are updated) and the state pass
// chunked prefill of the delta rule at d < 128 in fp32 on the CUDA cores (pre-norm output into
// ws.o and the final states), from the prep kernel's per-token rows
cudaError_t launch_chunk_small(const PrefillArgs& A, int chunk, cudaStream_t st);
template <typename TIn>
cudaError_t launch_chunk_prep(const PrefillArgs& A, cudaStream_t st);
template <typename TIn, typename TOut>
cudaError_t launch_chunk_state(const PrefillArgs& A, cudaStream_t st);
// lays the parts out from ws.base; false if they would not fit in ws.bytes
bool prefill_workspace_carve(PrefillWorkspace& ws, const gdn_shape& s, int max_tokens, int chunk_cap);

inline SlotCheck slot_check(const Pool& P, int layer)
{
    return SlotCheck{reinterpret_cast<uint64_t>(P.base), (uint64_t)P.total_bytes, (uint64_t)P.slot_bytes,
                     P.num_layers, layer};
}

}  // namespace gdn
