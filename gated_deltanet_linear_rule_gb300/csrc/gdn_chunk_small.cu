// gdn_chunk_small.cu -- chunked (WY / UT-transform) gated delta rule for the varlen prefill at
// d_k = d_v = d < 128, in fp32 on the CUDA cores.
//
// The same chunk form as the tensor-core path (gdn_chunk.cu), for the head sizes too small to
// fill tcgen05 tiles: within a chunk of n <= C tokens, with G_i = g_0 + ... + g_i,
//     A_ij  = beta_i e^{G_i - G_j} (k_i . k_j)  (i > j),   T = (I + A)^-1
//     W     = T diag(beta e^G) K,   U = T diag(beta) V,   Delta = U - W S0^T
//     P_ij  = e^{G_i - G_j} (q_i . k_j)  (i >= j),   O = diag(e^G) Q S0^T + P Delta
//     S_end = e^{G_last} S0 + Delta^T diag(e^{G_last - G_j}) K
// (the prefill branch of the System Design page's "GDN Kernel Dispatch Detail": a chunked
// gated delta rule over the prompt with the sequence's state).  Everything is fp32, so the
// result equals the recurrent definition to fp32 rounding.
//
// One CTA per (sequence, v-head) keeps the head's state S [d_v][d_k] in shared memory for the
// whole sequence and takes its chunks in order.  Its inputs are the prep kernel's per-token
// rows (conv + SiLU, normalised q and k, log decays, write strengths); it writes the pre-norm
// output o, which the epilogue kernel turns into rmsnorm(o) silu(z) w_n, and the final state.
// Every product of a chunk is a small GEMM in the "NT" form out[r][c] = sum_k X[r][k] Y[c][k]
// over shared-memory rows with k contiguous, each thread computing 2 x 2 outputs from float4
// loads; the operands that appear transposed (K, V, Delta) are kept in both orientations.
#include <algorithm>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int SNT = 256;  // threads per CTA

// out(r, c) = sum_k X[r][k] Y[c][k] for the M x N outputs (M, N even; K a multiple of 4; row
// pitches multiples of 4 floats), 2 x 2 per thread; epi(r, c, value) consumes each output.
template <typename Epi>
__device__ __forceinline__ void gemm_nt(int M, int N, int K, const float* X, int ldx, const float* Y, int ldy, Epi&& epi)
{
    const int tn = N >> 1, tiles = (M >> 1) * tn;
    for (int ti = threadIdx.x; ti < tiles; ti += SNT) {
        const int r = (ti / tn) * 2, c = (ti % tn) * 2;
        const float* x0 = X + (size_t)r * ldx;
        const float* x1 = x0 + ldx;
        const float* y0 = Y + (size_t)c * ldy;
        const float* y1 = y0 + ldy;
        float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
        for (int k = 0; k < K; k += 4) {
            const float4 p = *reinterpret_cast<const float4*>(x0 + k), q = *reinterpret_cast<const float4*>(x1 + k);
            const float4 u = *reinterpret_cast<const float4*>(y0 + k), v = *reinterpret_cast<const float4*>(y1 + k);
            a00 = fmaf(p.x, u.x, fmaf(p.y, u.y, fmaf(p.z, u.z, fmaf(p.w, u.w, a00))));
            a01 = fmaf(p.x, v.x, fmaf(p.y, v.y, fmaf(p.z, v.z, fmaf(p.w, v.w, a01))));
            a10 = fmaf(q.x, u.x, fmaf(q.y, u.y, fmaf(q.z, u.z, fmaf(q.w, u.w, a10))));
            a11 = fmaf(q.x, v.x, fmaf(q.y, v.y, fmaf(q.z, v.z, fmaf(q.w, v.w, a11))));
        }
        epi(r, c, a00);
        epi(r, c + 1, a01);
        epi(r + 1, c, a10);
        epi(r + 1, c + 1, a11);
    }
}

// shared-memory layout of one CTA, in floats (row pitches d + 4 / C + 4 keep float4 rows
// aligned and spread a warp's rows over the banks)
template <int D, int C>
struct SmallLayout {
    static constexpr int PD = D + 4, PC = C + 4;
    static constexpr int K = 0;                // [C][PD]  k_hat rows
    static constexpr int KT = K + C * PD;      // [D][PC]  k_hat^T
    static constexpr int Q = KT + D * PC;      // [C][PD]  q_hat rows
    static constexpr int VT = Q + C * PD;      // [D][PC]  v^T, then gamma K^T for the state update
    static constexpr int A = VT + D * PC;      // [C][PC]  A, then T diag(beta e^G)
    static constexpr int T = A + C * PC;       // [C][PC]  T = (I + A)^-1, then T diag(beta)
    static constexpr int P = T + C * PC;       // [C][PC]  P
    static constexpr int W = P + C * PC;       // [C][PD]  W
    static constexpr int U = W + C * PD;       // [C][PD]  U, then Delta
    static constexpr int DT = U + C * PD;      // [D][PC]  Delta^T
    static constexpr int S = DT + D * PC;      // [D][PD]  the state, S[i][j]: i = d_v, j = d_k
    static constexpr int G = S + D * PD;       // [C] G, [C] beta, [C] e^G, [C] beta e^G, [C] gamma, [4] e^{G_last}
    static constexpr int TOTAL = G + 5 * C + 4;
    static constexpr size_t BYTES = (size_t)TOTAL * sizeof(float);
};

template <int D, int C>
__global__ void __launch_bounds__(SNT) chunk_small_kernel(PrefillArgs A)
{
    using Ly = SmallLayout<D, C>;
    constexpr int PD = Ly::PD, PC = Ly::PC;
    extern __shared__ __align__(16) float smf[];
    float* sK = smf + Ly::K;
    float* sKT = smf + Ly::KT;
    float* sQ = smf + Ly::Q;
    float* sVT = smf + Ly::VT;
    float* sA = smf + Ly::A;
    float* sT = smf + Ly::T;
    float* sP = smf + Ly::P;
    float* sW = smf + Ly::W;
    float* sU = smf + Ly::U;
    float* sDT = smf + Ly::DT;
    float* sS = smf + Ly::S;
    float* sG = smf + Ly::G;
    float* sB = sG + C;
    float* sEG = sB + C;
    float* sBEG = sEG + C;
    float* sGam = sBEG + C;
    float* sEGL = sGam + C;

    if (!*A.ws.valid) return;
    const int s = blockIdx.x, h = blockIdx.y;
    const int t0 = A.cu[s], L = A.cu[s + 1] - t0;
    if (L <= 0) return;
    const int tid = threadIdx.x, hk = h / A.r, Dq = A.hqk * D, Dv = A.hv * D;
    float* Sg = reinterpret_cast<float*>(A.base + ((uint64_t)A.ids[s] * A.num_layers + A.layer) * A.slot_bytes) +
                (size_t)h * D * D;
    // a checked build tests the computed global ranges before the accesses
    const bool sok = chk(within(Sg, (size_t)D * D * sizeof(float), A.base,
                                (size_t)A.num_slots * A.num_layers * A.slot_bytes) && t0 >= 0 && t0 + L <= A.T,
                         A.status);
    if (!sok) return;
    for (int idx = tid; idx < D * D; idx += SNT) sS[(idx / D) * PD + idx % D] = Sg[idx];

    for (int c0 = 0; c0 < L; c0 += C) {
        const int n = min(C, L - c0), tb = t0 + c0;
        // the chunk's rows (zero past its end) in both orientations where a product needs them
        for (int idx = tid; idx < C * D; idx += SNT) {
            const int t = idx / D, j = idx % D;
            const bool in = t < n;
            const float kv = in ? A.ws.kh[(size_t)(tb + t) * Dq + hk * D + j] : 0.f;
            const float qv = in ? A.ws.qh[(size_t)(tb + t) * Dq + hk * D + j] : 0.f;
            const float vv = in ? A.ws.vc[(size_t)(tb + t) * Dv + h * D + j] : 0.f;
            sK[t * PD + j] = kv;
            sKT[j * PC + t] = kv;
            sQ[t * PD + j] = qv;
            sVT[j * PC + t] = vv;
        }
        // the decay prefix G (log decays below -40 are taken as -40, as on the tensor-core path:
        // alpha = e^-40 is zero against fp32 rounding, and the bound keeps G_i - G_j precise)
        if (tid == 0) {
            float acc = 0.f;
            for (int t = 0; t < C; ++t) {
                const bool in = t < n;
                acc += in ? fmaxf(A.ws.g[(size_t)(tb + t) * A.hv + h], -40.f) : 0.f;
                sG[t] = acc;
                sB[t] = in ? A.ws.beta[(size_t)(tb + t) * A.hv + h] : 0.f;
            }
            sEGL[0] = expf(sG[n - 1]);
        }
        __syncthreads();
        for (int t = tid; t < C; t += SNT) {
            const float eg = expf(sG[t]);
            sEG[t] = eg;
            sBEG[t] = sB[t] * eg;
            sGam[t] = t < n ? expf(sG[n - 1] - sG[t]) : 0.f;
        }
        __syncthreads();
        // A (strictly lower) and P (lower with the diagonal)
        gemm_nt(C, C, D, sK, PD, sK, PD, [&](int i, int j, float v) {
            sA[i * PC + j] = i > j ? sB[i] * expf(sG[i] - sG[j]) * v : 0.f;
        });
        gemm_nt(C, C, D, sQ, PD, sK, PD, [&](int i, int j, float v) {
            sP[i * PC + j] = i >= j ? expf(sG[i] - sG[j]) * v : 0.f;
        });
        __syncthreads();
        // T = (I + A)^-1 by forward substitution, row after row: T_ij = -sum_{j <= k < i} A_ik T_kj
        for (int i = 0; i < C; ++i) {
            for (int j = tid; j < C; j += SNT) {
                float acc = 0.f;
                for (int k = j; k < i; ++k) acc = fmaf(sA[i * PC + k], sT[k * PC + j], acc);
                sT[i * PC + j] = j < i ? -acc : (j == i ? 1.f : 0.f);
            }
            __syncthreads();
        }
        // T diag(beta e^G) into A's space, T diag(beta) in place
        for (int idx = tid; idx < C * C; idx += SNT) {
            const int i = idx / C, j = idx % C;
            const float t = sT[i * PC + j];
            sA[i * PC + j] = t * sBEG[j];
            sT[i * PC + j] = t * sB[j];
        }
        __syncthreads();
        // W = T diag(beta e^G) K,  U = T diag(beta) V
        gemm_nt(C, D, C, sA, PC, sKT, PC, [&](int t, int i, float v) { sW[t * PD + i] = v; });
        gemm_nt(C, D, C, sT, PC, sVT, PC, [&](int t, int i, float v) { sU[t * PD + i] = v; });
        __syncthreads();
        // Delta = U - W S0^T (in U's place and transposed), and e^G Q S0^T into the output rows
        gemm_nt(C, D, D, sW, PD, sS, PD, [&](int t, int i, float v) {
            const float d = sU[t * PD + i] - v;
            sU[t * PD + i] = d;
            sDT[i * PC + t] = d;
        });
        gemm_nt(C, D, D, sQ, PD, sS, PD, [&](int t, int i, float v) {
            if (t < n) A.ws.o[(size_t)(tb + t) * Dv + h * D + i] = sEG[t] * v;
        });
        __syncthreads();
        // O += P Delta (the thread that wrote an output element above adds to it: same tiling);
        // gamma K^T over v^T's space for the state update
        gemm_nt(C, D, C, sP, PC, sDT, PC, [&](int t, int i, float v) {
            if (t < n) A.ws.o[(size_t)(tb + t) * Dv + h * D + i] += v;
        });
        for (int idx = tid; idx < D * C; idx += SNT) {
            const int j = idx / C, t = idx % C;
            sVT[j * PC + t] = sGam[t] * sKT[j * PC + t];
        }
        __syncthreads();
        // S <- e^{G_last} S + Delta^T diag(gamma) K
        const float egl = sEGL[0];
        gemm_nt(D, D, C, sDT, PC, sVT, PC, [&](int i, int j, float v) { sS[i * PD + j] = fmaf(egl, sS[i * PD + j], v); });
        __syncthreads();
    }
    for (int idx = tid; idx < D * D; idx += SNT) Sg[idx] = sS[(idx / D) * PD + idx % D];
}

template <int D, int C>
cudaError_t launch_small(const PrefillArgs& A, cudaStream_t st)
{
    auto kern = chunk_small_kernel<D, C>;
    const size_t smem = SmallLayout<D, C>::BYTES;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kern<<<dim3(A.n, A.hv), SNT, smem, st>>>(A);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_small_c(const PrefillArgs& A, int chunk, cudaStream_t st)
{
    switch (chunk) {
        case 8: return launch_small<D, 8>(A, st);
        case 16: return launch_small<D, 16>(A, st);
        case 32: return launch_small<D, 32>(A, st);
        case 64: return launch_small<D, 64>(A, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_chunk_small(const PrefillArgs& A, int chunk, cudaStream_t st)
{
    switch (A.D) {
        case 16: return launch_small_c<16>(A, chunk, st);
        case 32: return launch_small_c<32>(A, chunk, st);
        case 64: return launch_small_c<64>(A, chunk, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
