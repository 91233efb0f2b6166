// gdn_chunk.cu -- chunked (WY / UT-transform) gated delta rule for the varlen prefill, on
// tcgen05 tensor cores with TMEM accumulators, d_k = d_v = 128, chunks of 64 tokens.
//
// The prefill branch of the System Design page's "GDN Kernel Dispatch Detail" runs a
// chunked gated delta rule over the prompt with the sequence's state, then updates the
// temporal state and applies the gated RMSNorm.  Within a chunk of n <= 64 tokens (local
// i, j), with G_i = g_0 + ... + g_i (g = log decay), beta the write strengths, q_hat, k_hat
// the normalised (q scaled) vectors and v the values, the recurrence
//     S <- e^{g_t} S;  S <- S + beta_t (v_t - S k_t) k_t^T;  o_t = S q_t
// equals, in exact arithmetic (the derivation writes S_t = e^{G_t} S0 + sum_{j<=t}
// e^{G_t - G_j} delta_j k_j^T and solves for the deltas):
//     A_ij   = beta_i e^{G_i - G_j} (k_i . k_j)       (i > j)
//     T      = (I + A)^-1                              (unit lower triangular)
//     W      = T diag(beta e^G) K,     U = T diag(beta) V
//     P_ij   = e^{G_i - G_j} (q_i . k_j)               (i >= j)
//     Q'     = diag(e^G) Q - P W,      O0 = P U        (independent of S0)
//     Delta  = U - W S0^T,             O  = Q' S0^T + O0
//     S_end  = e^{G_last} S0 + Delta^T diag(e^{G_last - G_j}) K
// Only the last three lines depend on the incoming state.  Every product runs on the
// tensor cores as a 128-row MMA:
//     MMA1  [K; Q]  x K^T      -> K K^T (rows 0-63) and Q K^T (rows 64-127)      128 x 64  x 128
//     MMA3  [T2; T1] x [K|V]   -> U = T2 V (rows 0-63), W = T1 K (rows 64-127)     128 x 256 x 64
//     MMA5  [P; P]  x W, U     -> P W, P U                                        2 x 128 x 128 x 64
//     MMA4  [W; Q'] x S0^T     -> W S0^T (rows 0-63), Q' S0^T (rows 64-127)      128 x 128 x 128
//     MMA6  S += Delta~^T x K  (S pre-scaled by e^{G_last} in TMEM)              128 x 128 x 64
// with fp16 operands and fp32 accumulation; the state S itself stays fp32 in TMEM for the
// whole sequence.  The triangular inverse, the decay factors, Delta, and the gated RMSNorm
// of each output row run on the CUDA cores (one thread per TMEM lane = one token or one
// d_v row).  One CTA (4 warps, 1 per SM) owns one (sequence, v-head); CTAs are ordered so
// that the longest sequences start first.
#include <algorithm>

#include "gdn_internal.cuh"
#include "gdn_tcgen05.cuh"

namespace gdn {
namespace {

constexpr int D = 128, CH = 64, NT = 128;
// MMA operand type: fp16 (11-bit significand) -- bf16 operands (8-bit) put the chunked
// result at ~5e-3 of the recurrent definition; fp16 runs at the same tensor-core rate.
using Op = __half;

// shared memory (offsets from a 1024-aligned base); every operand tile is swizzled K-major fp16
constexpr uint32_t OFF_A1 = 0;         // [K; Q] (MMA1 A), then [W; Q'] (MMA4 A): 2 K-tiles x 128 rows
constexpr uint32_t OFF_KT = 32768;     // K^T: 128 dk rows x 64 tokens (MMA3 B rows 0-127, MMA6 B)
constexpr uint32_t OFF_VT = 49152;     // V^T: 128 dv rows x 64 tokens (MMA3 B rows 128-255)
constexpr uint32_t OFF_AP = 65536;     // [P; P] (MMA5 A), then Delta~^T (MMA6 A): 128 rows x 64
constexpr uint32_t OFF_AT = 81920;     // [T2; T1] (MMA3 A): 128 rows x 64
constexpr uint32_t OFF_BWU = 98304;    // [W^T; U^T] (MMA5 B): 256 rows x 64
constexpr uint32_t OFF_B4 = 131072;    // S0 in fp16 (MMA4 B): 2 K-tiles x 128 rows
constexpr uint32_t OFF_FA = 163840;    // fp32 A, 64 x 64
constexpr uint32_t OFF_FT = 180224;    // fp32 T, 64 x 64
constexpr uint32_t OFF_SMALL = 196608; // per-chunk scalars, barrier, TMEM slot
constexpr size_t SMEM_BYTES = OFF_SMALL + 2048 + 1024;

// TMEM columns (512 allocated): S lives in [0, 128) for the whole sequence
constexpr uint32_t TM_S = 0;
constexpr uint32_t TM_D1 = 128;   // MMA1
constexpr uint32_t TM_D3 = 128;   // MMA3, 256 columns: W at rows 64-127 cols 128-255, U at rows 0-63 cols 256-383
constexpr uint32_t TM_U = 256;
constexpr uint32_t TM_PW = 128;   // MMA5 first half
constexpr uint32_t TM_PU = 384;   // MMA5 second half
constexpr uint32_t TM_D4 = 128;   // MMA4

__device__ __forceinline__ void sync_all()
{
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
}

__device__ __forceinline__ void load8(const float* p, float* v)
{
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(NT, 1) chunk_kernel(PrefillArgs A)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    float* sGraw = reinterpret_cast<float*>(sm + OFF_SMALL);  // [64] g of the chunk
    float* sG = sGraw + 64;    // [64] inclusive prefix sums G_i
    float* sB = sG + 64;       // [64] beta (0 past the chunk's end)
    float* sEG = sB + 64;      // [64] e^{G_i}
    float* sGam = sEG + 64;    // [64] e^{G_last - G_i} (0 past the end)
    float* sMisc = sGam + 64;  // [8] e^{G_last}
    uint64_t* bar = reinterpret_cast<uint64_t*>(sMisc + 8);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);

    if (!*A.ws.valid) return;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int s = A.ws.order[blockIdx.x / A.hv], h = blockIdx.x % A.hv;
    const int t0 = A.cu[s], L = A.cu[s + 1] - t0;
    if (L <= 0) return;
    const int hk = h / A.r, Dq = A.hqk * D, Dv = A.hv * D;
    float* Sg = reinterpret_cast<float*>(A.base + ((uint64_t)A.ids[s] * A.num_layers + A.layer) * A.slot_bytes) +
                (size_t)h * D * D;
    const TIn* zin = static_cast<const TIn*>(A.z);
    TOut* out = static_cast<TOut*>(A.out);

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) tc::alloc(tmem_slot, 512);
    sync_all();
    const uint32_t tm = *tmem_slot;
    uint32_t phase = 0;
    bool ok = true;

    // issue + wait helper: thread 0 issues, everyone waits for the commit
    auto mma_done = [&]() {
        if (tid == 0) tc::commit(bar);
        const bool got = mbar_wait_bounded(bar, phase, nullptr);
        phase ^= 1u;
        if (!got && tid == 0) atomicOr(A.status, GDN_DEV_TIMEOUT);
        ok = __syncthreads_and(got) != 0;
        tc::fence_after_sync();
    };

    // the sequence's incoming state into TMEM: thread = d_v row
    for (int c0 = 0; c0 < D; c0 += 32) {
        float v[32];
        const float* row = Sg + (size_t)tid * D + c0;
#pragma unroll
        for (int e = 0; e < 32; e += 8) load8(row + e, v + e);
        tc::st32(tc::taddr(tm, warp, TM_S + c0), v);
    }
    tc::wait_st();
    sync_all();

    const int nchunks = (L + CH - 1) / CH;
    for (int c = 0; c < nchunks && ok; ++c) {
        const int tc0 = t0 + c * CH;
        const int n = min(CH, L - c * CH);

        // (a) operand tiles of the chunk: [K; Q], K^T, V^T; gates
        for (int idx = tid; idx < 128 * 16; idx += NT) {
            const int r = idx >> 4, c16 = idx & 15, i = r & 63;
            float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (i < n) load8((r < 64 ? A.ws.kh : A.ws.qh) + (size_t)(tc0 + i) * Dq + hk * D + c16 * 8, v);
            tc::st_chunk<Op>(sm + OFF_A1 + (c16 >> 3) * 16384, r, c16 & 7, v);
            if (r < 64) {
#pragma unroll
                for (int e = 0; e < 8; ++e) tc::st_elem<Op>(sm + OFF_KT, c16 * 8 + e, i, v[e]);
            }
        }
        for (int idx = tid; idx < 64 * 16; idx += NT) {
            const int i = idx >> 4, c16 = idx & 15;
            float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (i < n) load8(A.ws.vc + (size_t)(tc0 + i) * Dv + h * D + c16 * 8, v);
#pragma unroll
            for (int e = 0; e < 8; ++e) tc::st_elem<Op>(sm + OFF_VT, c16 * 8 + e, i, v[e]);
        }
        if (tid < 64) {
            const bool in = tid < n;
            sGraw[tid] = in ? A.ws.g[(size_t)(tc0 + tid) * A.hv + h] : 0.f;
            sB[tid] = in ? A.ws.beta[(size_t)(tc0 + tid) * A.hv + h] : 0.f;
        }
        tc::fence_proxy_async();
        sync_all();
        if (tid < 64) {
            float acc = 0.f;
            for (int t = 0; t <= tid; ++t) acc += sGraw[t];
            sG[tid] = acc;
            sEG[tid] = expf(acc);
        }
        __syncthreads();
        if (tid < 64) {
            const float gl = sG[n - 1];
            sGam[tid] = tid < n ? expf(gl - sG[tid]) : 0.f;
            if (tid == 0) sMisc[0] = expf(gl);
        }

        // (b) MMA1: [K; Q] x K^T -> K K^T (rows 0-63), Q K^T (rows 64-127), 64 columns
        if (tid == 0)
            tc::mma_k(tm + TM_D1, smem_addr(sm + OFF_A1), 128, smem_addr(sm + OFF_A1), 128, D,
                           tc::idesc_f16(128, 64), 0);
        mma_done();
        if (!ok) break;

        // (c) A (fp32, rows 0-63) and P (fp16 tile, rows 64-127 -> both halves of [P; P])
        {
            const int i = tid & 63;
            const float Gi = sG[i];
            float* FA = reinterpret_cast<float*>(sm + OFF_FA);
            for (int c0 = 0; c0 < 64; c0 += 32) {
                float v[32];
                tc::ld32(tc::taddr(tm, warp, TM_D1 + c0), v);
                tc::wait_ld();
                if (tid < 64) {
                    const float bi = sB[i];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int j = c0 + e;
                        FA[i * 64 + j] = (j < i && i < n) ? bi * expf(Gi - sG[j]) * v[e] : 0.f;
                    }
                } else {
                    float p[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int j = c0 + e;
                        p[e] = (j <= i && i < n) ? expf(Gi - sG[j]) * v[e] : 0.f;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        tc::st_chunk<Op>(sm + OFF_AP, i, c0 / 8 + q, p + 8 * q);
                        tc::st_chunk<Op>(sm + OFF_AP, 64 + i, c0 / 8 + q, p + 8 * q);
                    }
                }
            }
        }
        sync_all();

        // (d) T = (I + A)^-1 by forward substitution, one column per thread; then [T2; T1]
        if (tid < 64) {
            const int j = tid;
            const float* FA = reinterpret_cast<const float*>(sm + OFF_FA);
            float* FT = reinterpret_cast<float*>(sm + OFF_FT);
            for (int i = 0; i < 64; ++i) {
                float acc0 = (i == j) ? 1.f : 0.f, acc1 = 0.f;
                int k = j;
                for (; k + 1 < i; k += 2) {
                    acc0 -= FA[i * 64 + k] * FT[k * 64 + j];
                    acc1 -= FA[i * 64 + k + 1] * FT[(k + 1) * 64 + j];
                }
                if (k < i) acc0 -= FA[i * 64 + k] * FT[k * 64 + j];
                FT[i * 64 + j] = (i < j) ? 0.f : acc0 + acc1;
            }
            const float bj = sB[j], bej = sB[j] * sEG[j];
            for (int i = 0; i < 64; ++i) {
                const float t = FT[i * 64 + j];
                tc::st_elem<Op>(sm + OFF_AT, i, j, t * bj);
                tc::st_elem<Op>(sm + OFF_AT, 64 + i, j, t * bej);
            }
        }
        tc::fence_proxy_async();
        sync_all();

        // (e) MMA3: [T2; T1] x [K^T; V^T] -> U (rows 0-63, cols 256-383), W (rows 64-127, cols 128-255)
        if (tid == 0)
            tc::mma_k(tm + TM_D3, smem_addr(sm + OFF_AT), 128, smem_addr(sm + OFF_KT), 256, CH,
                           tc::idesc_f16(128, 256), 0);
        mma_done();
        if (!ok) break;

        // (f) W -> [W; .] rows 0-63 and W^T (rows 0-127 of [W^T; U^T]); U -> U^T (rows 128-255)
        {
            const int i = tid & 63;
            for (int c0 = 0; c0 < D; c0 += 32) {
                float v[32];
                tc::ld32(tc::taddr(tm, warp, (tid < 64 ? TM_U : TM_D3) + c0), v);
                tc::wait_ld();
                if (tid >= 64) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) tc::st_chunk<Op>(sm + OFF_A1 + (c0 >> 6) * 16384, i, (c0 & 63) / 8 + q, v + 8 * q);
#pragma unroll
                    for (int e = 0; e < 32; ++e) tc::st_elem<Op>(sm + OFF_BWU, c0 + e, i, v[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) tc::st_elem<Op>(sm + OFF_BWU, 128 + c0 + e, i, v[e]);
                }
            }
        }
        tc::fence_proxy_async();
        sync_all();

        // (g) MMA5: [P; P] x W^T -> P W (cols 128-255); [P; P] x U^T -> P U (cols 384-511)
        if (tid == 0) {
            tc::mma_k(tm + TM_PW, smem_addr(sm + OFF_AP), 128, smem_addr(sm + OFF_BWU), 256, CH,
                           tc::idesc_f16(128, 128), 0);
            tc::mma_k(tm + TM_PU, smem_addr(sm + OFF_AP), 128, smem_addr(sm + OFF_BWU) + 128 * 128, 256, CH,
                           tc::idesc_f16(128, 128), 0);
        }
        mma_done();
        if (!ok) break;

        // (h) Q' = e^G Q - P W -> rows 64-127 of [W; Q'] (Q from the fp32 workspace)
        if (tid >= 64) {
            const int i = tid - 64;
            const float eg = sEG[i];
            const float* qrow = A.ws.qh + (size_t)(tc0 + i) * Dq + hk * D;
            for (int c0 = 0; c0 < D; c0 += 32) {
                float v[32];
                tc::ld32(tc::taddr(tm, warp, TM_PW + c0), v);
                tc::wait_ld();
                float qv[32];
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    if (i < n) load8(qrow + c0 + e, qv + e);
                    else {
#pragma unroll
                        for (int x = 0; x < 8; ++x) qv[e + x] = 0.f;
                    }
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = eg * qv[e] - v[e];
#pragma unroll
                for (int q = 0; q < 4; ++q) tc::st_chunk<Op>(sm + OFF_A1 + (c0 >> 6) * 16384, 64 + i, (c0 & 63) / 8 + q, v + 8 * q);
            }
        }

        // (i) S0 (fp16) for MMA4; S <- e^{G_last} S in TMEM for MMA6
        {
            const float egl = sMisc[0];
            for (int c0 = 0; c0 < D; c0 += 32) {
                float v[32];
                tc::ld32(tc::taddr(tm, warp, TM_S + c0), v);
                tc::wait_ld();
#pragma unroll
                for (int q = 0; q < 4; ++q) tc::st_chunk<Op>(sm + OFF_B4 + (c0 >> 6) * 16384, tid, (c0 & 63) / 8 + q, v + 8 * q);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] *= egl;
                tc::st32(tc::taddr(tm, warp, TM_S + c0), v);
            }
            tc::wait_st();
        }
        tc::fence_proxy_async();
        sync_all();

        // (j) MMA4: [W; Q'] x S0^T -> W S0^T (rows 0-63), Q' S0^T (rows 64-127)
        if (tid == 0)
            tc::mma_k(tm + TM_D4, smem_addr(sm + OFF_A1), 128, smem_addr(sm + OFF_B4), 128, D,
                           tc::idesc_f16(128, 128), 0);
        mma_done();
        if (!ok) break;

        // (k) rows 0-63: Delta = U - W S0^T -> Delta~^T = (gamma_j Delta_j)^T;  rows 64-127: O = Q' S0^T + P U,
        //     gated RMSNorm, output
        if (tid < 64) {
            const int i = tid;
            const float gm = sGam[i];
            for (int c0 = 0; c0 < D; c0 += 32) {
                float ws_[32], u[32];
                tc::ld32(tc::taddr(tm, warp, TM_D4 + c0), ws_);
                tc::ld32(tc::taddr(tm, warp, TM_U + c0), u);
                tc::wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) tc::st_elem<Op>(sm + OFF_AP, c0 + e, i, gm * (u[e] - ws_[e]));
            }
        } else {
            const int i = tid - 64;
            float ss = 0.f;
            for (int c0 = 0; c0 < D; c0 += 32) {
                float a_[32], b_[32];
                tc::ld32(tc::taddr(tm, warp, TM_D4 + c0), a_);
                tc::ld32(tc::taddr(tm, warp, TM_PU + c0), b_);
                tc::wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float o = a_[e] + b_[e];
                    ss = fmaf(o, o, ss);
                }
            }
            // tcgen05.ld is warp-collective: every lane loads, only rows of real tokens are stored
            const float rs = rms_scale(ss, A.norm_eps, D);
            const size_t obase = (size_t)(tc0 + (i < n ? i : 0)) * Dv + (size_t)h * D;
            for (int c0 = 0; c0 < D; c0 += 32) {
                float a_[32], b_[32];
                tc::ld32(tc::taddr(tm, warp, TM_D4 + c0), a_);
                tc::ld32(tc::taddr(tm, warp, TM_PU + c0), b_);
                tc::wait_ld();
                if (i < n) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int dv = c0 + e;
                        const float y = (a_[e] + b_[e]) * rs * A.norm_w[dv] * silu_f(to_f(zin[obase + dv]));
                        out[obase + dv] = from_f<TOut>(y);
                    }
                }
            }
        }
        tc::fence_proxy_async();
        sync_all();

        // (l) MMA6: S += Delta~^T x K (accumulate onto the pre-scaled state)
        if (tid == 0)
            tc::mma_k(tm + TM_S, smem_addr(sm + OFF_AP), 128, smem_addr(sm + OFF_KT), 128, CH,
                           tc::idesc_f16(128, 128), 1);
        mma_done();
    }

    // the final state back to the slot
    if (ok) {
        for (int c0 = 0; c0 < D; c0 += 32) {
            float v[32];
            tc::ld32(tc::taddr(tm, warp, TM_S + c0), v);
            tc::wait_ld();
            float* row = Sg + (size_t)tid * D + c0;
#pragma unroll
            for (int e = 0; e < 32; e += 4) *reinterpret_cast<float4*>(row + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
    }
    sync_all();
    if (warp == 0) tc::dealloc(tm, 512);
}

}  // namespace

template <typename TIn, typename TOut>
cudaError_t launch_chunk(const PrefillArgs& A, cudaStream_t st)
{
    auto kern = chunk_kernel<TIn, TOut>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<A.n * A.hv, NT, SMEM_BYTES, st>>>(A);
    return cudaGetLastError();
}

template cudaError_t launch_chunk<float, float>(const PrefillArgs&, cudaStream_t);
template cudaError_t launch_chunk<float, __nv_bfloat16>(const PrefillArgs&, cudaStream_t);
template cudaError_t launch_chunk<__nv_bfloat16, float>(const PrefillArgs&, cudaStream_t);
template cudaError_t launch_chunk<__nv_bfloat16, __nv_bfloat16>(const PrefillArgs&, cudaStream_t);

}  // namespace gdn
