// gdn_decode.cu -- batched GDN decode: one launch advances m slots by one token.
//
// This is the batched decode step that issue #5279 asks for (phase P5: the GDN conv1d
// and delta rule gain a slot dimension, one launch over a device u64 array of per-slot
// state pointers), computing the decode branch of the System Design page's "GDN Kernel
// Dispatch Detail" (conv1d state update, temporal_state decay + delta write, Query @
// state) plus the gated RMSNorm that both branches end with.
//
// Work unit ("item"): one (batch row, q/k head) pair, i.e. the r = Hv/Hqk v-heads that
// share a q/k head.  The item owns its q, k and v conv channels exclusively, so it can
// read the old conv buffer and write the shifted one without racing other CTAs.
//
// Kernel shape: persistent CTAs, 8 consumer warps + 1 producer warp.  The producer
// streams each item's r*D*D fp32 state (contiguous, 128 KiB at D=128, r=2) from HBM
// into a shared-memory ring of 16 KiB stages with 1-D bulk copies (TMA engine) completing
// on mbarriers; it runs ahead across items.  Many items: 4 stages, 3 CTAs per SM.  Fewer
// items at D = 128: 6 stages at 2 CTAs per SM, or 8 at 1 when each item has an SM of its
// own, so that more of an item's state is in flight at once.  Consumers fuse the item's conv + SiLU, L2
// norms and gates (while the first stages land), then per S row compute both dot
// products (S.k, S.q) from one read, apply the rank-1 update and store the new row
// with 128-bit global stores -- one HBM read and one write of S per step.  The row
// outputs feed the gated RMSNorm epilogue of the item.
//
// Every result of an item depends only on that item's inputs and state: no atomics,
// fixed reduction orders, no m-dependent choices, so batched output equals m = 1 output
// bit for bit.
#include <algorithm>
#include <mutex>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kStageBytes = 16384;
constexpr int kStages = 4;      // ring depth with 3 CTAs per SM (batches of many items)
constexpr int kMidStages = 6;   // ring depth with 2 CTAs per SM
constexpr int kDeepStages = 8;  // ring depth with 1 CTA per SM (an item per SM: the whole item in flight)

struct DecodeArgs {
    const uint64_t* slot_ptrs;
    int m;
    const void *q, *k, *v, *a, *b, *z;
    void* out;
    const float *conv_w, *A_log, *dt_bias, *norm_w;
    SlotCheck chk;
    unsigned int* status;
    int hqk, hv, r, W, C;
    uint32_t state_bytes;
    float l2_eps, norm_eps;
    int stall_producer;  // test hook: the producer fills no stage, so the consumers' waits run out
    const int* gate;     // when non-null and *gate != 0 the launch does nothing (mixed-step overlap check)
    int sms;             // SMs the launch is sized for (host side: the pool's SM count, or fewer)
};

size_t decode_smem_bytes(int D, int r, int stages)
{
    size_t bytes = (size_t)stages * kStageBytes;      // stage ring
    bytes += 2 * stages * sizeof(uint64_t);             // full / empty barriers
    bytes += (size_t)(2 * D + 2 * r * D + 3 * r + 4) * sizeof(float);  // qs, ks, vs, obuf, alpha, beta, rms, red
    bytes += 16;                                        // abort flag
    return bytes;
}

template <int D, typename TIn, typename TOut, int STAGES>
__global__ void __launch_bounds__(kThreads, STAGES == kStages ? 3 : STAGES == kMidStages ? 2 : 1)
    decode_kernel(const DecodeArgs A)
{
    constexpr int LPR = D / 16;    // lanes per S row (16 columns per lane)
    constexpr int RPW = 32 / LPR;  // rows per warp per stage
    static_assert(kStageBytes / (D * 4) == kConsumerWarps * RPW, "one warp-step per stage");

    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * kStageBytes);
    uint64_t* empty = full + STAGES;
    const int r = A.r;
    float* qs = reinterpret_cast<float*>(empty + STAGES);
    float* ks = qs + D;
    float* vs = ks + D;       // [r][D] conv + SiLU v of the item's v-heads
    float* obuf = vs + r * D;  // [r][D] delta-rule output before the norm
    float* gal = obuf + r * D; // [r] alpha
    float* gbe = gal + r;      // [r] beta
    float* rms = gbe + r;      // [r] RMSNorm factor
    float* red = rms + r;      // [4] q scale, k scale, k.q
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int items = A.m * A.hqk;
    const uint32_t item_bytes = (uint32_t)r * D * D * 4;
    const int stages_per_item = (int)((item_bytes + kStageBytes - 1) / kStageBytes);
    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    // The launch is programmatic (see launch_t): the setup above touches only this CTA's shared
    // memory and may overlap the end of the previous kernel on the stream; every global access
    // (slot pointers, states, inputs, the gate) comes after the wait.  The next decode launch may
    // then start its own setup as soon as this grid's CTAs are all running.
    grid_dependency_wait();
    grid_dependents_launch();
    if (A.gate && *A.gate) return;  // a mixed step whose parts name a common slot: nothing runs
    __syncthreads();

    // ------------------------------------------------------------ producer ----
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            int slot = 0;
            uint32_t phase = 0, issued = 0, last_parity = 0;
            for (int item = blockIdx.x; item < items && !*abort_flag && !A.stall_producer; item += gridDim.x) {
                const int row = item / A.hqk, hk = item % A.hqk;
                const uint64_t p = A.slot_ptrs[row];
                if (!slot_ptr_ok(p, A.chk)) continue;
                const char* src = reinterpret_cast<const char*>(p) + (size_t)hk * item_bytes;
                for (int s = 0; s < stages_per_item; ++s) {
                    const uint32_t bytes = min((uint32_t)kStageBytes, item_bytes - (uint32_t)s * kStageBytes);
                    if (!mbar_wait_bounded(&empty[slot], phase ^ 1u, abort_flag)) {
                        if (!*abort_flag) atomicOr(A.status, GDN_DEV_TIMEOUT);
                        *abort_flag = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[slot], bytes);
                    bulk_g2s(ring + slot * kStageBytes, src + (size_t)s * kStageBytes, bytes, &full[slot]);
                    issued |= 1u << slot;
                    last_parity = (last_parity & ~(1u << slot)) | (phase << slot);
                    if (++slot == STAGES) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every issued copy must have landed before the CTA's shared memory goes away
            for (int i = 0; i < STAGES; ++i)
                if ((issued >> i) & 1u) mbar_wait_bounded(&full[i], (last_parity >> i) & 1u, nullptr);
        }
        return;
    }

    // ----------------------------------------------------------- consumers ----
    const TIn* qin = static_cast<const TIn*>(A.q);
    const TIn* kin = static_cast<const TIn*>(A.k);
    const TIn* vin = static_cast<const TIn*>(A.v);
    const TIn* ain = static_cast<const TIn*>(A.a);
    const TIn* bin = static_cast<const TIn*>(A.b);
    const TIn* zin = static_cast<const TIn*>(A.z);
    TOut* out = static_cast<TOut*>(A.out);
    const int Dq = A.hqk * D, Dv = A.hv * D, W = A.W, C = A.C;
    const int rsub = lane / LPR, cl = lane % LPR;
    int slot = 0;
    uint32_t phase = 0;

    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int row = item / A.hqk, hk = item % A.hqk;
        const uint64_t p = A.slot_ptrs[row];
        if (!slot_ptr_ok(p, A.chk)) {  // same decision as the producer: the item is skipped
            if (tid == 0) atomicOr(A.status, GDN_DEV_BAD_SLOT_PTR);
            continue;
        }
        float* S = reinterpret_cast<float*>(p) + (size_t)hk * r * D * D;
        TIn* cbuf = reinterpret_cast<TIn*>(p + A.state_bytes);  // [W-1][C]
        // With the deeper rings (few items; latency-bound), requested now and used at the end:
        // this thread's z of the epilogue (one element when r * D == kConsumers) and, for the
        // first r threads, the gate inputs of v-head hk*r + tid (at 4 stages, 3 CTAs per SM,
        // the registers they hold cost more than the round trips they save: measured)
        constexpr bool kEarly = STAGES != kStages;
        TIn zpre = TIn(0.f);
        if (kEarly && r * D <= kConsumers && tid < r * D) zpre = zin[(size_t)row * Dv + (size_t)hk * r * D + tid];
        float g_in = 0.f, b_in = 0.f;
        if (kEarly && tid < r) {
            const int h = hk * r + tid;
            g_in = log_decay(A.A_log[h], to_f(ain[(size_t)row * A.hv + h]), A.dt_bias[h]);
            b_in = to_f(bin[(size_t)row * A.hv + h]);
        }

        // conv + SiLU of the item's q, k and v channels; shift the conv buffer by one token
        const int nch = (2 + r) * D;
        for (int c = tid; c < nch; c += kConsumers) {
            int ch;
            TIn xraw;
            float* dst;
            if (c < D) {
                ch = hk * D + c;
                xraw = qin[(size_t)row * Dq + hk * D + c];
                dst = qs + c;
            } else if (c < 2 * D) {
                ch = Dq + hk * D + (c - D);
                xraw = kin[(size_t)row * Dq + hk * D + (c - D)];
                dst = ks + (c - D);
            } else {
                const int vc = hk * r * D + (c - 2 * D);
                ch = 2 * Dq + vc;
                xraw = vin[(size_t)row * Dv + vc];
                dst = vs + (c - 2 * D);
            }
            const float* w = A.conv_w + (size_t)ch * W;
            TIn prev[8];
            float acc = 0.0f;
#pragma unroll
            for (int j = 0; j < 7; ++j) {
                if (j < W - 1) {
                    prev[j] = cbuf[(size_t)j * C + ch];
                    acc = fmaf(w[j], to_f(prev[j]), acc);
                }
            }
            acc = fmaf(w[W - 1], to_f(xraw), acc);
#pragma unroll
            for (int j = 0; j < 6; ++j)
                if (j < W - 2) cbuf[(size_t)j * C + ch] = prev[j + 1];
            if (W > 1) cbuf[(size_t)(W - 2) * C + ch] = xraw;
            *dst = silu_f(acc);
        }
        named_bar_sync(1, kConsumers);

        // L2 scales, k.q and the gates of the item's v-heads
        if (warp == 0) {
            const float ss = warp_dot(qs, qs, D, lane);
            if (lane == 0) red[0] = q_scale(ss, A.l2_eps, D);
        } else if (warp == 1) {
            const float ss = warp_dot(ks, ks, D, lane);
            if (lane == 0) red[1] = k_scale(ss, A.l2_eps);
        } else if (warp == 2) {
            const float d = warp_dot(qs, ks, D, lane);
            if (lane == 0) red[2] = d;
        } else if (!kEarly) {
            for (int rr = (warp - 3) * 32 + lane; rr < r; rr += 5 * 32) {
                const int h = hk * r + rr;
                const float g = log_decay(A.A_log[h], to_f(ain[(size_t)row * A.hv + h]), A.dt_bias[h]);
                gal[rr] = expf(g);
                gbe[rr] = sigmoid_f(to_f(bin[(size_t)row * A.hv + h]));
            }
        }
        if (kEarly && tid < r) {
            gal[tid] = expf(g_in);
            gbe[tid] = sigmoid_f(b_in);
        }
        named_bar_sync(1, kConsumers);

        const float sq = red[0], sk = red[1];
        const float kq = red[2] * sq * sk;
        float kr[16], qr[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int col = row_col<LPR>(j, cl);
            kr[j] = ks[col] * sk;
            qr[j] = qs[col] * sq;
        }

        // stream the item's S rows through the ring
        for (int s = 0; s < stages_per_item; ++s) {
            const uint32_t bytes = min((uint32_t)kStageBytes, item_bytes - (uint32_t)s * kStageBytes);
            const int rows_here = (int)(bytes / (D * 4));
            if (!*abort_flag && !mbar_wait_bounded(&full[slot], phase, abort_flag)) {
                if (lane == 0) {
                    if (!*abort_flag) atomicOr(A.status, GDN_DEV_TIMEOUT);
                    *abort_flag = 1;
                }
            }
            const int lr = warp * RPW + rsub;
            const int grow = s * (kStageBytes / (D * 4)) + lr;  // row within the item: head * D + i
            const bool rv = lr < rows_here && !*abort_flag;
            const float* srow = reinterpret_cast<const float*>(ring + slot * kStageBytes) + lr * D;
            float sv[16];
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
                float4 t = rv ? *reinterpret_cast<const float4*>(srow + row_col<LPR>(j, cl))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
                sv[j] = t.x;
                sv[j + 1] = t.y;
                sv[j + 2] = t.z;
                sv[j + 3] = t.w;
            }
            const int hr = rv ? grow / D : 0;
            const float al = gal[hr], be = gbe[hr], vi = rv ? vs[grow] : 0.0f;
            const float o = row_update<LPR>(sv, kr, qr, al, be, vi, kq);
            if (rv) {
                float* grow_ptr = S + (size_t)grow * D;
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    st_global_v4(grow_ptr + row_col<LPR>(j, cl), make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]));
                if (cl == 0) obuf[grow] = o;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (++slot == STAGES) {
                slot = 0;
                phase ^= 1u;
            }
        }
        named_bar_sync(1, kConsumers);

        // gated RMSNorm epilogue of the item's v-heads
        for (int rr = warp; rr < r; rr += kConsumerWarps) {
            const float ss = warp_dot(obuf + rr * D, obuf + rr * D, D, lane);
            if (lane == 0) rms[rr] = rms_scale(ss, A.norm_eps, D);
        }
        named_bar_sync(1, kConsumers);
        if (!*abort_flag) {
            for (int c = tid; c < r * D; c += kConsumers) {
                const int rr = c / D, i = c % D, h = hk * r + rr;
                const size_t o_idx = (size_t)row * Dv + (size_t)h * D + i;
                const TIn zv = (kEarly && r * D <= kConsumers) ? zpre : zin[o_idx];
                const float y = obuf[c] * rms[rr] * A.norm_w[i] * silu_f(to_f(zv));
                out[o_idx] = from_f<TOut>(y);
            }
        }
    }
}

template <int D, typename TIn, typename TOut, int STAGES>
cudaError_t launch_t(const Pool& P, const DecodeArgs& A, cudaStream_t st)
{
    auto kern = decode_kernel<D, TIn, TOut, STAGES>;
    const size_t smem = decode_smem_bytes(D, A.r, STAGES);
    // resident CTAs per SM for this instantiation and shared-memory size, per device (the
    // attribute is a per-device setting; cached; calls from several host threads are serialised here)
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static int cached_per_sm[kMaxDevices] = {};
    static size_t cached_smem[kMaxDevices] = {};
    const int dev = P.device;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (cached_per_sm[dev] <= 0 || cached_smem[dev] != smem) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            int n = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem);
            if (e != cudaSuccess) return e;
            cached_per_sm[dev] = std::max(n, 1);
            cached_smem[dev] = smem;
        }
        per_sm = cached_per_sm[dev];
    }
    const int items = A.m * A.hqk;
    const int grid = std::max(1, std::min(items, per_sm * A.sms));
    // Programmatic stream serialization: the CTAs may be scheduled while the previous kernel on the
    // stream finishes (at small m the launch and setup are a large part of a step); the kernel
    // waits for that kernel's completion before its first global access.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, A);
}

template <typename TIn, typename TOut>
cudaError_t launch_d(const Pool& P, const DecodeArgs& A, cudaStream_t st)
{
    switch (P.shape.dk) {
        case 16: return launch_t<16, TIn, TOut, kStages>(P, A, st);
        case 32: return launch_t<32, TIn, TOut, kStages>(P, A, st);
        case 64: return launch_t<64, TIn, TOut, kStages>(P, A, st);
        case 128: {
            // Ring depth by batch size (measured at 16 q/k heads): an item per SM -> 8 stages at
            // 1 CTA per SM, so an item's state streams in about one round trip; up to 8 items per
            // SM -> 6 stages at 2 CTAs per SM (m = 16 / 32 / 64: 12.4 -> 10.6, 24.4 -> 20.8,
            // 56.2 -> 53.7 us); more -> 4 stages at 3 CTAs per SM.  The arithmetic is the same.
            const size_t items = (size_t)A.m * P.shape.hqk;
            if (items <= (size_t)A.sms) return launch_t<128, TIn, TOut, kDeepStages>(P, A, st);
            if (items <= 8 * (size_t)A.sms) return launch_t<128, TIn, TOut, kMidStages>(P, A, st);
            return launch_t<128, TIn, TOut, kStages>(P, A, st);
        }
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_decode(const Pool& P, int layer, const uint64_t* slot_ptrs, int m, const void* q, const void* k,
                          const void* v, const void* a, const void* b, const void* z, void* out, cudaStream_t st,
                          const int* gate, int sms)
{
    const LayerParams& L = P.params[(size_t)layer];
    DecodeArgs A;
    A.slot_ptrs = slot_ptrs;
    A.m = m;
    A.q = q;
    A.k = k;
    A.v = v;
    A.a = a;
    A.b = b;
    A.z = z;
    A.out = out;
    A.conv_w = L.conv_w;
    A.A_log = L.A_log;
    A.dt_bias = L.dt_bias;
    A.norm_w = L.norm_w;
    A.chk = slot_check(P, layer);
    A.status = P.status_dev;
    A.hqk = P.shape.hqk;
    A.hv = P.shape.hv;
    A.r = P.r;
    A.W = P.shape.conv_w;
    A.C = P.C;
    A.state_bytes = (uint32_t)P.state_bytes;
    A.l2_eps = P.shape.l2_eps;
    A.norm_eps = P.shape.norm_eps;
    A.stall_producer = P.debug_flags & 1;
    A.gate = gate;
    A.sms = sms > 0 ? std::min(sms, P.num_sms) : P.num_sms;
    const bool in_bf16 = P.shape.io_dtype == 1, out_bf16 = P.shape.out_dtype == 1;
    if (in_bf16 && out_bf16) return launch_d<__nv_bfloat16, __nv_bfloat16>(P, A, st);
    if (in_bf16) return launch_d<__nv_bfloat16, float>(P, A, st);
    if (out_bf16) return launch_d<float, __nv_bfloat16>(P, A, st);
    return launch_d<float, float>(P, A, st);
}

}  // namespace gdn
