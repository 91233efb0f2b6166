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
//     Delta  = U - W S0^T,             O  = diag(e^G) Q S0^T + P Delta
//     S_end  = e^{G_last} S0 + Delta^T diag(e^{G_last - G_j}) K
// (O is the chunk form of o_t = S_t q_t: S_t = e^{G_t} S0 + sum_{j<=t} e^{G_t - G_j} delta_j
// k_j^T with delta_j = Delta_j.)  Everything above the line "Delta = ..." is independent of
// the incoming state, so it runs in a fully parallel pre-pass over all chunks of all
// sequences at once; only the last two lines form the serial chain, run by one CTA per
// (sequence, v-head, d_v half) that keeps S in fp32 tensor memory across its chunks.
//
// Pre-pass (chunk_prep_kernel, 2 CTAs per SM):
//     MMA1  [K; Q]  x K^T          -> K K^T (rows 0-63), Q K^T (rows 64-127)     128 x 64  x 128
//     blocked triangular inverse of I + A on the CUDA cores (16-wide diagonal blocks, then
//     16 -> 32 -> 64 by  T_21 = -T_22 A_21 T_11)
//     MMA3  [T2; 0] x V + [0; T1] x K   -> U (rows 0-63), W (rows 64-127)       128 x 128 x 128
//   and writes per (chunk, v-head) a record: the W, U, P and output-gate images and the
//   chunk's scalars (decay factors, scale exponents); per (chunk, q/k head) the [K; Q] tile.
// State pass (chunk_state_kernel, double-buffered bulk copies of the records):
//     MMA4  [W; Q] x S0^T    -> W S0^T (rows 0-63), Q S0^T (rows 64-127)          128 x 64 x 128
//     Delta
//     MMA6  X = K^T x Delta~   (Delta~ = diag(gamma) Delta)                         128 x 64 x 64
//     MMA7  [0; P] x Delta  -> P Delta (rows 64-127), off the chain                128 x 64 x 64
//     S <- e^{G_last} S + X in fp32;  O = diag(e^G) (Q S0^T) + P Delta with the gated RMSNorm
// Operands are fp16 (11-bit significand; bf16's 8 bits put the chunked result at ~5e-3 of
// the recurrent definition) with fp32 accumulation.  fp16 spans 2^-24 .. 65504, far less
// than the layer's inputs may: every fp16 operand whose size follows the data carries a
// power-of-two scale of its own, chosen per chunk from measured maxima (V, U, W from the
// pre-pass's reductions; S0^T and Delta from the state's measured maximum and bounds on
// its growth), and the products are taken back to true units in fp32.  Power-of-two scales
// are exact, so they change no rounding but that of values that would otherwise overflow
// or fall below fp16's normal range.  The decay factors e^{G_i} multiply the output rows in
// fp32, after MMA4, for the same reason; the output gates silu(z) w_n are stored in fp16
// with a power-of-two scale per token.  Transposed operands (K, V, W, U as the N side;
// Delta~ as the M side) are read MN-major straight from row-wise tiles.
// Every tcgen05.ld / st is executed by whole warps (they are warp-collective); per-token
// conditions only guard stores.
//
// Records are numbered chunk-index-major (every sequence's chunk 0 in length order, then every
// chunk 1, ...: chunk c of the sequence of rank p is record coff[c] + p).  A call whose records
// exceed the workspace runs as segments, windows [seg_lo, seg_hi) of record numbers: the
// pre-pass of a segment writes its records at positions gc - seg_lo, and the segment's state
// pass takes, for each sequence with records in the window, the run of its chunks there,
// starting from the state the slot holds; only the segment holding a sequence's last chunk
// advances its conv buffer.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cstring>
#include <mutex>

#include "gdn_internal.cuh"
#include "gdn_tcgen05.cuh"

namespace gdn {
namespace {

constexpr int D = 128, CH = 64, NT = 256;
using Op = __half;

// record of one (chunk, v-head), written by the pre-pass, read by the state pass
constexpr uint32_t REC_W = 0;        // W' image [token][dk]: two 64-wide halves 8 KiB apart (W = W' 2^ew)
constexpr uint32_t REC_U = 16384;    // U' image [token][dv], same layout (U = U' 2^eu)
constexpr uint32_t REC_P = 32768;    // P image [i][j], 64 x 64
constexpr uint32_t REC_GZ = 40960;   // output gates silu(z) w_n 2^-ez(token), fp16 [token][dv], W' layout
constexpr uint32_t REC_SC = 57344;   // the chunk's scalars, SC_* below
constexpr uint32_t REC_BYTES = 58368;
// per (chunk, q/k head): the [K; Q] tile, two 64-wide d_k halves of 128 rows (64 K rows, then
// 64 Q rows), 16 KiB apart
constexpr uint32_t QK_BYTES = 32768;
// scalars of a record, in 4-byte words
constexpr int SC_GAM = 0;    // [64] gamma_j = e^{G_last - G_j} (0 past the end)
constexpr int SC_EG = 64;    // [64] e^{G_i}
constexpr int SC_EGL = 128;  // e^{G_last}
constexpr int SC_EU = 129;   // eu (int): U = U' 2^eu
constexpr int SC_EW = 130;   // ew (int): W = W' 2^ew
constexpr int SC_MU = 131;   // max |U'|
constexpr int SC_MW = 132;   // max |W'|
constexpr int SC_EZ = 136;   // [64] ez (int): token i's gates are stored times 2^-ez
constexpr uint32_t SC_BYTES = 800;

// pre-pass shared memory (offsets from a 1024-aligned base)
constexpr uint32_t P_A1 = 0;          // [K; Q] (MMA1 and MMA3; leaves as the (chunk, q/k head) [K; Q] tile)
// Five 8 KiB blocks T2 | Z | P | Z | T1 (64 rows of 64 fp16, swizzled; Z zero) hold the
// 128-row left operands of the block-diagonal products: [T2; Z] at P_T2, [Z; P] at P_Z0,
// [P; Z] at P_P and [Z; T1] at P_Z1.
constexpr uint32_t P_T2 = 32768;      // T diag(beta) 2^-eb
constexpr uint32_t P_Z0 = 40960;
constexpr uint32_t P_P = 49152;       // P
constexpr uint32_t P_Z1 = 57344;
constexpr uint32_t P_T1 = 65536;      // inverse scratch, then T diag(beta e^G) 2^-eg
constexpr uint32_t P_R4 = 73728;      // A (fp32, stride 68), then the V' image, then the U' image
constexpr uint32_t P_R5 = 91136;      // T (fp32, stride 68), then the W' image
constexpr uint32_t P_RAW = P_T2;      // first: raw bf16 k, q, v rows of the chunk (3 x (64 + WM - 1) x 256 B)
constexpr uint32_t P_SMALL = 108544;
constexpr size_t P_SMEM = P_SMALL + 3072 + 1024;  // small area (2.8 KB) + alignment slack
constexpr int FS = 68;                // fp32 matrix row stride: 16-B aligned rows, 4-wide row loads and stores

// state-pass shared memory (one CTA per (sequence, v-head, d_v half))
// One record buffer: the [W'; Q] operand (2 K-tiles of 128 rows) | K image | U' half | gates
// half | scalars.  P goes to a slot of its own (two of them, by chunk parity), each after an
// 8 KiB zero block: MMA7 reads [0; P] as its 128-row operand.
constexpr uint32_t B_A = 0, B_K = 32768, B_U = 49152, B_GZ = 57344, B_SC = 65536;
constexpr uint32_t S_TX = 32768 + 16384 + 8192 + 8192 + SC_BYTES;  // bytes fetched into one record buffer
constexpr uint32_t S_BUF = 66560;
constexpr uint32_t S_S0 = 2 * S_BUF;     // S0^T(:, half) 2^-Es in fp16, MN-major: 128 rows (d_k) of 64 d_v
constexpr uint32_t S_A6 = S_S0 + 16384;  // Delta~(:, half) 2^-Ed [token][64 d_v]
constexpr uint32_t S_DL = S_A6 + 8192;   // [2] Delta(:, half) 2^-Ed [token][64 d_v], by chunk parity
constexpr uint32_t S_PZ = S_DL + 16384;  // [2] zero block | P [i][j], by chunk parity
constexpr uint32_t S_SMALL = S_PZ + 32768;
constexpr uint32_t S_POS = S_SMALL + 2048;  // [kPrefillMaxRecords] workspace positions of the segment's chunks
constexpr size_t S_SMEM = S_POS + 4 * kPrefillMaxRecords + 1024;  // small area (barriers, sums, maxima) + slack

// state-pass tensor memory (512 columns): S^T(:, half) in true units, X = K^T Delta~ of the
// last chunk, MMA4's and MMA7's results by chunk parity
constexpr uint32_t TS = 0, TX = 64, TM4 = 128, TM7 = 256;

// 2^k for an integer k (0 below 2^-126, 2^127 above)
__device__ __forceinline__ float pow2f(int k) { return k < -126 ? 0.f : __int_as_float((min(k, 127) + 127) << 23); }
// floor(log2 m) of a finite m > 0 in fp32's normal range
__device__ __forceinline__ int ilog2f(float m) { return ((__float_as_int(m) >> 23) & 255) - 127; }
// the power-of-two scale exponent e that brings magnitudes up to m below 2^(b+1): m 2^-e < 2^(b+1)
// (0 for m = 0; clamped to [-100, 100], far outside any finite input the layer takes in fp32)
__device__ __forceinline__ int scale_exp(float m, int b) { return m > 0.f ? max(-100, min(100, ilog2f(m) - b)) : 0; }

__device__ __forceinline__ void sync_all()
{
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
}

// arrive on named barrier `id` (of `threads` threads) without waiting for it
__device__ __forceinline__ void named_bar_arrive(int id, int threads)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// 8 fp16 values of a 16-B chunk -> float
__device__ __forceinline__ void unpack8(uint4 w, float* v)
{
    const __half2* h = reinterpret_cast<const __half2*>(&w);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(h[q]);
        v[2 * q] = f.x;
        v[2 * q + 1] = f.y;
    }
}

// 8 consecutive outputs as one 16-B (bf16) or two 16-B (fp32) stores
template <typename T> __device__ __forceinline__ void store8(T* p, const float* y);
template <> __device__ __forceinline__ void store8<float>(float* p, const float* y)
{
    reinterpret_cast<float4*>(p)[0] = make_float4(y[0], y[1], y[2], y[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(y[4], y[5], y[6], y[7]);
}
template <> __device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* p, const float* y)
{
    uint4 w;
    w.x = tc::pack2<__nv_bfloat16>(y[0], y[1]);
    w.y = tc::pack2<__nv_bfloat16>(y[2], y[3]);
    w.z = tc::pack2<__nv_bfloat16>(y[4], y[5]);
    w.w = tc::pack2<__nv_bfloat16>(y[6], y[7]);
    *reinterpret_cast<uint4*>(p) = w;
}

__device__ __forceinline__ unsigned char* align1024(unsigned char* p)
{
    return p + ((1024 - (smem_addr(p) & 1023)) & 1023);
}

// 8 raw input values of one row (one 16-B word in bf16, two in fp32), read through the
// read-only path
template <typename TIn> struct Raw8 {
    uint4 w[sizeof(TIn) / 2];
};
template <typename TIn> __device__ __forceinline__ void ld_raw8(Raw8<TIn>& r, const TIn* p)
{
#pragma unroll
    for (int w = 0; w < (int)(sizeof(TIn) / 2); ++w) r.w[w] = __ldg(reinterpret_cast<const uint4*>(p) + w);
}
template <typename TIn> __device__ __forceinline__ void zero_raw8(Raw8<TIn>& r)
{
#pragma unroll
    for (int w = 0; w < (int)(sizeof(TIn) / 2); ++w) r.w[w] = make_uint4(0u, 0u, 0u, 0u);
}
template <typename TIn> __device__ __forceinline__ float raw_at(const Raw8<TIn>& r, int e)
{
    return to_f(reinterpret_cast<const TIn*>(r.w)[e]);
}

// Tensor maps of the raw bf16 q, k and v rows ([T][width], 2-D, box 128 channels x (64 + WM - 1)
// rows, no swizzle, zero fill outside the tensor), encoded on the host per call.
struct PrepMaps {
    CUtensorMap q, k, v;
};

// 2-D tiled bulk tensor copy global -> shared (the TMA engine), completing on an mbarrier.
// x (the channel coordinate) must be a multiple of 8 bf16 (16 B); y may be negative.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// One tensor (q, k or v) of a chunk, as a thread of the pre-pass sees it: 8 channels
// (column col of the input rows of width `width`, channel ch of the conv's C channels) over
// the output rows r0 .. r0 + 3.  The causal conv of width W <= WM is evaluated as a
// WM-tap conv whose leading WM - W taps are zero, over the input rows r0 - WM + 1 .. r0 + 3.
template <typename TIn, int WM>
struct ConvRows {
    static constexpr int NR = WM + 3;
    Raw8<TIn> x[NR];

    // rows before the sequence's first token come from the slot's conv buffer (its row W-1+p
    // holds position p < 0); rows before that, and rows at or past the chunk's end, are zero
    __device__ __forceinline__ void load(const TIn* src, int width, int col, const TIn* cbuf, int C, int ch, int W,
                                         int tc0, int p0, int r0, int n)
    {
#pragma unroll
        for (int j = 0; j < NR; ++j) {
            const int r = r0 - (WM - 1) + j, p = p0 + r;
            if (r < n && p >= 0) ld_raw8(x[j], src + (size_t)(tc0 + r) * width + col);
            else if (r < n && p >= -(W - 1)) ld_raw8(x[j], cbuf + (size_t)(W - 1 + p) * C + ch);
            else zero_raw8(x[j]);
        }
    }

    // conv taps of the 8 channels, right-aligned in WM slots
    __device__ __forceinline__ static void taps(float (&w)[8][WM], const float* conv_w, int ch, int W)
    {
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
            for (int j = 0; j < WM; ++j)
                w[e][j] = j >= WM - W ? __ldg(conv_w + (size_t)(ch + e) * W + (j - (WM - W))) : 0.f;
    }

    // SiLU(conv) of output row r0 + o
    __device__ __forceinline__ void row(const float (&w)[8][WM], int o, float (&y)[8]) const
    {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < WM; ++j) acc = fmaf(w[e][j], raw_at(x[o + j], e), acc);
            y[e] = silu_f(acc);
        }
    }
};

// ===================================================================== pre-pass ====
// One CTA per (chunk, q/k head): the q / k conv, norms, the K image and [K; Q] x K^T are
// shared by the r = Hv / Hqk v-heads of the q/k head, which the CTA then takes one after the
// other.  8 warps: warp w reads TMEM lane quarter w % 4 and works on column half w / 4.

// The sequences with chunk records in a segment [seg_lo, seg_hi) of a call run in segments, for
// the segment's state pass: chunk c of the sequence of rank p is record coff[c] + p, and the ranks
// with a chunk c are 0 .. K_c - 1 (K_c = coff[c+1] - coff[c], non-increasing in c), so they are
// the ranks [0, n1) and [p_lo, p_lo + n2).  Written by one thread of the pre-pass into the slot of
// the segment's parity (the next segment's pre-pass may run beside this segment's state pass).
__device__ __forceinline__ int* window_slot(const PrefillArgs& A)
{
    return A.ws.valid + 8 + 4 * ((A.seg_lo / (A.seg_hi - A.seg_lo)) & 1);
}

__device__ void window_plan(const PrefillArgs& A)
{
    const int* coff = A.ws.coff;
    const int nc = A.ws.valid[1], R = coff[nc];
    const int lo = A.seg_lo, hi = min(A.seg_hi, R);
    int n1 = 0, p_lo = 0, n2 = 0;
    if (lo < hi) {
        auto chunk_of = [&](int r) {  // the largest c < nc with coff[c] <= r
            int a = 0, b = nc;
            while (b - a > 1) {
                const int m = (a + b) >> 1;
                if (coff[m] <= r) a = m;
                else b = m;
            }
            return a;
        };
        const int ca = chunk_of(lo), cb = chunk_of(hi - 1), ka = coff[ca + 1] - coff[ca];
        p_lo = lo - coff[ca];
        if (ca == cb) {
            n2 = hi - lo;  // ranks p_lo .. of chunk ca only
        } else {
            // chunk ca: ranks [p_lo, ka); the later chunks: ranks [0, x)
            const int x = cb > ca + 1 ? coff[ca + 2] - coff[ca + 1] : hi - coff[cb];
            if (x >= p_lo) {
                n1 = ka;
                p_lo = 0;
            } else {
                n1 = x;
                n2 = ka - p_lo;
            }
        }
    }
    int* win = window_slot(A);
    win[0] = n1;
    win[1] = p_lo;
    win[2] = n2;
}

template <typename TIn, int WM>
__global__ void __launch_bounds__(NT, 2) chunk_prep_kernel(const __grid_constant__ PrefillArgs A,
                                                           const __grid_constant__ PrepMaps M)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = align1024(smem_raw);
    // two sets (by head parity) of per-token gate arrays, 5 x 64 floats each: beta e^G, G,
    // beta, e^G, gamma = e^{G_last - G}; then per set e^{G_last} and the two scanning warps'
    // maxima of beta and of beta e^G (bit patterns of non-negative floats)
    float* sSet = reinterpret_cast<float*>(sm + P_SMALL);
    float* sMisc2 = sSet + 640;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sSet + 656);
    uint64_t* sbar = bar + 1;  // raw rows staged (one phase per batch of tensor copies)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbar + 1);
    // per v-head of the CTA (at most 8): max |V| over the chunk (true units), max |U'|, max |W'|,
    // as bit patterns of non-negative floats, combined by atomicMax
    unsigned int* s_vmax = reinterpret_cast<unsigned int*>(sSet + 664);
    unsigned int* s_umax = s_vmax + 8;
    unsigned int* s_wmax = s_vmax + 16;
    int* sEZ = reinterpret_cast<int*>(sSet + 688);  // [64] the current head's gate scale exponents per token
    float* FA = reinterpret_cast<float*>(sm + P_R4);
    float* FT = reinterpret_cast<float*>(sm + P_R5);
    float* X = reinterpret_cast<float*>(sm + P_T1);

    if (!*A.ws.valid) return;
    if (A.seg_hi != INT_MAX && blockIdx.x == 0 && threadIdx.x == 0) window_plan(A);
    const int gc = A.seg_lo + (int)(blockIdx.x / A.hqk), hk = blockIdx.x % A.hqk;  // record, q/k head
    if (gc >= A.seg_hi || gc >= A.ws.coff[A.ws.valid[1]]) return;
    const int slot_rec = gc - A.seg_lo;  // the record's position in this segment's workspace
    const int2 cp = A.ws.rec_cp[gc];     // chunk index, rank of the sequence
    const int s = A.ws.order[cp.y], c = cp.x;
    const int tc0 = A.cu[s] + c * CH;
    const int n = min(CH, A.cu[s + 1] - tc0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, hf = warp >> 2;
    const int h0 = hk * A.r, Dq = A.hqk * D, Dv = A.hv * D;
    unsigned char* qkimg = A.ws.kimg + ((size_t)slot_rec * A.hqk + hk) * QK_BYTES;
    const TIn* cbuf = reinterpret_cast<const TIn*>(A.base + ((uint64_t)A.ids[s] * A.num_layers + A.layer) *
                                                                A.slot_bytes + A.state_bytes);

    constexpr int NRT = CH + WM - 1;  // raw rows of a tensor: r = -(WM-1) .. 63 (row slot r + WM - 1)
    const int rb = tid >> 4, cg = tid & 15, r0 = 4 * rb, p0 = c * CH;
    // the regions a checked build tests this kernel's computed accesses against
    const size_t sm_bytes = (size_t)(smem_raw + P_SMEM - sm);
    const size_t rec_region = (size_t)A.ws.chunk_cap * A.hv * REC_BYTES;
    const size_t qk_region = (size_t)A.ws.chunk_cap * A.hqk * QK_BYTES;
    const size_t slots_region = (size_t)A.num_slots * A.num_layers * A.slot_bytes;
    const size_t rowsv = (size_t)A.T * A.hv * D * sizeof(TIn);
    auto sm_ok = [&](const void* p, size_t b) { return chk(within(p, b, sm, sm_bytes), A.status); };
    auto tile_ok = [&](const void* p, size_t b, uint32_t off, uint32_t region) {
        return chk(within(p, b, sm + off, region), A.status);
    };
    auto rec_ok = [&](const void* p, size_t b) { return chk(within(p, b, A.ws.rec, rec_region), A.status); };
    const TIn* qin = static_cast<const TIn*>(A.q);
    const TIn* kin = static_cast<const TIn*>(A.k);
    const TIn* vin = static_cast<const TIn*>(A.v);
    const int ch_q = hk * D + 8 * cg, ch_k = Dq + hk * D + 8 * cg;

    // Per-head inputs nothing waits for yet are loaded one head ahead: the gate inputs a, b of
    // token tid and the head's A_log, dt_bias (warps 0 and 1), the chunk's z rows, and (bf16)
    // the head's v conv taps.
    TIn ga = TIn(0.f), gb = TIn(0.f);
    float a_log = 0.f, dt_b = 0.f;
    constexpr int ZW = sizeof(TIn) / 2;  // 16-B words per 8 values
    uint4 zpark[4][ZW];
    constexpr int KV = D * WM / NT;  // v taps per thread
    float tvv[KV];
    // gate inputs of head h for the threads of warp pair `pair` (token tid % 64)
    auto load_gate_inputs = [&](int h, int pair) {
        if ((tid >> 6) == pair) {
            const int t = tid & 63;
            a_log = __ldg(A.A_log + h);
            dt_b = __ldg(A.dt_bias + h);
            const size_t gi = (size_t)(tc0 + t) * A.hv + h;
            if (t < n && chk(within(static_cast<const TIn*>(A.a) + gi, sizeof(TIn), A.a, (size_t)A.T * A.hv * sizeof(TIn)),
                             A.status)) {
                ga = static_cast<const TIn*>(A.a)[gi];
                gb = static_cast<const TIn*>(A.b)[gi];
            }
        }
    };
    auto prefetch_head = [&](int h) {
        const TIn* zin = static_cast<const TIn*>(A.z);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int idx = tid + q * NT, i = idx >> 4, c8 = (idx & 15) * 8;
#pragma unroll
            for (int wd = 0; wd < ZW; ++wd) {
                const uint4* zp = reinterpret_cast<const uint4*>(zin + (size_t)(tc0 + i) * Dv + (size_t)h * D + c8) + wd;
                zpark[q][wd] = i < n && chk(within(zp, 16, A.z, rowsv), A.status) ? __ldg(zp) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if constexpr (sizeof(TIn) == 2) {
#pragma unroll
            for (int k = 0; k < KV; ++k) {
                const int idx = tid + k * NT, chl = idx / WM, j = idx - chl * WM;
                tvv[k] = j >= WM - A.W ? __ldg(A.conv_w + (size_t)(2 * Dq + h * D + chl) * A.W + (j - (WM - A.W))) : 0.f;
            }
        }
    };
    prefetch_head(h0);
    load_gate_inputs(h0, 0);
    if (A.r > 1) load_gate_inputs(h0 + 1, 1);
    constexpr int KT = 2 * D * WM / NT;  // q / k conv taps per thread (bf16)
    float tv[KT];
    if constexpr (sizeof(TIn) == 2) {
#pragma unroll
        for (int k = 0; k < KT; ++k) {
            const int idx = tid + k * NT;
            const int t = idx / (D * WM), rem = idx - t * (D * WM), chl = rem / WM, j = rem - chl * WM;
            const int ch = (t == 0 ? Dq + hk * D : hk * D) + chl;
            tv[k] = j >= WM - A.W ? __ldg(A.conv_w + (size_t)ch * A.W + (j - (WM - A.W))) : 0.f;
        }
    }
    const int y0 = tc0 - (WM - 1);
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(sbar, 1);
        fence_mbar_init();
        if constexpr (sizeof(TIn) == 2) {
            // raw bf16 k, q and the first head's v rows of the chunk by three tensor copies; rows
            // past the tensor are zero, rows of a neighbouring sequence are replaced or never used
            mbar_arrive_expect_tx(sbar, 3 * NRT * 256);
            if (sm_ok(sm + P_RAW, 3 * NRT * 256)) {
                tma_load_2d(sm + P_RAW, &M.k, hk * D, y0, sbar);
                tma_load_2d(sm + P_RAW + NRT * 256, &M.q, hk * D, y0, sbar);
                tma_load_2d(sm + P_RAW + 2 * NRT * 256, &M.v, h0 * D, y0, sbar);
            }
        }
    }
    if (tid < 24) s_vmax[tid] = 0u;
    if (warp == 0) tc::alloc(tmem_slot, 256);
    sync_all();
    const uint32_t tm = *tmem_slot;  // columns [0, 128): MMA3 of a head; [128, 192): MMA1
    uint32_t phase = 0;
    bool ok = true;
    auto mma_done = [&]() {
        if (tid == 0) tc::commit(bar);
        const bool got = mbar_wait_bounded(bar, phase, nullptr);
        phase ^= 1u;
        if (!got && tid == 0) atomicOr(A.status, GDN_DEV_TIMEOUT);
        ok = __syncthreads_and(got) != 0;
        tc::fence_after_sync();
    };

    // gates of a head and the decay prefix G_i = g_0 + ... + g_i into set k, by the 64 threads of
    // warp pair `pair` (which hold the head's gate inputs): a shuffle scan per warp, then the
    // second warp adds the first's total.  Heads 0 and 1 are scanned at the start by pairs 0
    // and 1; a head after that by pair 0 when its turn comes.
    // A log decay below kMinLogDecay is taken as kMinLogDecay: alpha = e^-40 = 4e-18 is already
    // zero against fp32's 6e-8 relative rounding of everything it is added to, and the bound
    // keeps |G| <= 64 * 40 within a chunk, so that G_i - G_j (a difference of two prefix sums)
    // keeps an absolute error near 2^-12.
    auto scan_set = [&](int k, int pair) {
        if ((tid >> 6) == pair) {
            constexpr float kMinLogDecay = -40.f;
            const int t = tid & 63;
            float* G = sSet + k * 320 + 64;
            float* B = G + 64;
            float* EG = B + 64;
            float* GAM = EG + 64;
            float* BEG = G - 64;
            const bool in = t < n;
            float x = in ? fmaxf(log_decay(a_log, to_f(ga), dt_b), kMinLogDecay) : 0.f;
            B[t] = in ? sigmoid_f(to_f(gb)) : 0.f;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            G[t] = x;
            named_bar_sync(1 + pair, 64);
            if (t >= 32) G[t] += G[31];
            named_bar_sync(1 + pair, 64);
            const float gl = G[n - 1];
            EG[t] = expf(G[t]);
            BEG[t] = B[t] * EG[t];
            GAM[t] = t < n ? expf(gl - G[t]) : 0.f;
            if (t == 0) sMisc2[k * 8] = expf(gl);
            // the column scales of T diag(beta) and T diag(beta e^G): their maxima (zero past the end)
            const unsigned ub = __reduce_max_sync(0xffffffffu, __float_as_uint(B[t]));
            const unsigned ug = __reduce_max_sync(0xffffffffu, __float_as_uint(BEG[t]));
            if (lane == 0) {
                sMisc2[k * 8 + 2 + (t >> 5)] = __uint_as_float(ub);
                sMisc2[k * 8 + 4 + (t >> 5)] = __uint_as_float(ug);
            }
        }
    };

    scan_set(0, 0);
    if (A.r > 1) scan_set(1, 1);

    // (a) conv1d + SiLU of the chunk's q, k rows and the first head's v rows from the raw inputs
    //     (the W-1 rows before a sequence's first token from its slot's conv buffer), L2 norms of
    //     q and k (q also scaled by dk^-1/2), fp16 rounding.  Thread (rb, cg) = (tid / 16,
    //     tid % 16) owns rows 4 rb .. 4 rb + 3 and channels 8 cg .. 8 cg + 7 of each tensor; a
    //     row's 16 threads are one half-warp, which sums the squares of two rows at a time by
    //     shuffles.  q, k go to the [K; Q] tile; v is parked in registers until the inverse has
    //     freed its shared-memory space.  bf16 rows are staged in shared memory by tensor
    //     copies; fp32 rows pass through registers, one tensor at a time.
    float w[8][WM];
    // q or k rows r0 .. r0 + 3 from their conv outputs: normalise, round, store.  The four rows'
    // sums of squares over the row's 16 threads take five dependent shuffles: across lane bit 3
    // each lane keeps one pair of rows and hands over the other pair, across bit 2 one row of
    // the pair, and a butterfly over bits 1..0 completes each row's sum (bitwise equal in the
    // four lanes that hold it); four independent shuffles then bring every row's scale.
    auto qk_rows4 = [&](const float (&y)[4][8], bool is_q) {
        float sq[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 8; e += 2) a2 = fma2(make_float2(y[r][e], y[r][e + 1]), make_float2(y[r][e], y[r][e + 1]), a2);
            sq[r] = a2.x + a2.y;
        }
        const bool b3 = (lane & 8) != 0, b2 = (lane & 4) != 0;
        const float k0 = b3 ? sq[2] : sq[0], k1 = b3 ? sq[3] : sq[1];
        const float t0 = k0 + __shfl_xor_sync(0xffffffffu, b3 ? sq[0] : sq[2], 8);
        const float t1 = k1 + __shfl_xor_sync(0xffffffffu, b3 ? sq[1] : sq[3], 8);
        float u = (b2 ? t1 : t0) + __shfl_xor_sync(0xffffffffu, b2 ? t0 : t1, 4);
        u += __shfl_xor_sync(0xffffffffu, u, 2);
        u += __shfl_xor_sync(0xffffffffu, u, 1);
        // this lane now holds row 2 b3 + b2
        const float mine = is_q ? rsqrtf(u + A.l2_eps) * rsqrtf((float)D) : rsqrtf(u + A.l2_eps);
        float sc[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int src = (lane & ~12) | ((r >> 1) << 3) | ((r & 1) << 2);
            const float v = __shfl_sync(0xffffffffu, mine, src);
            sc[r] = r0 + r < n ? v : 0.f;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float2 sc2 = make_float2(sc[r], sc[r]);
            float2 z2[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) z2[e] = mul2(make_float2(y[r][2 * e], y[r][2 * e + 1]), sc2);
            uint4 pk;
            pk.x = pack_half2(z2[0].x, z2[0].y);
            pk.y = pack_half2(z2[1].x, z2[1].y);
            pk.z = pack_half2(z2[2].x, z2[2].y);
            pk.w = pack_half2(z2[3].x, z2[3].y);
            const int i = r0 + r;
            const uint32_t off = (cg >> 3) * 16384 + tc::sw128_chunk(is_q ? 64 + i : i, cg & 7);
            if (tile_ok(sm + P_A1 + off, 16, P_A1, 32768)) *reinterpret_cast<uint4*>(sm + P_A1 + off) = pk;
        }
    };
    // v row r0 + o times the power of two sc, rounded to fp16 (zero past the chunk's end)
    auto v_row = [&](int o, const float (&y)[8], float sc) {
        const bool in = r0 + o < n;
        const float2 s2 = make_float2(sc, sc);
        uint4 pk;
        float2 p2 = mul2(make_float2(y[0], y[1]), s2);
        pk.x = in ? pack_half2(p2.x, p2.y) : 0u;
        p2 = mul2(make_float2(y[2], y[3]), s2);
        pk.y = in ? pack_half2(p2.x, p2.y) : 0u;
        p2 = mul2(make_float2(y[4], y[5]), s2);
        pk.z = in ? pack_half2(p2.x, p2.y) : 0u;
        p2 = mul2(make_float2(y[6], y[7]), s2);
        pk.w = in ? pack_half2(p2.x, p2.y) : 0u;
        return pk;
    };
    uint4 vpark[4];  // v rows r0 .. r0 + 3, channels 8 cg .. 8 cg + 7, times 2^-vexp, fp16
    int vexp = 0;    // the scale exponent of this thread's parked rows
    int vhead = 0;   // the CTA's v-head (0 .. r-1) whose rows are being parked
    // bf16: taps of channel pairs (8 cg + 2 p, 8 cg + 2 p + 1) from a [tap][channel] table
    float2 w2[4][WM];
    auto load_taps = [&](const float* table) {
#pragma unroll
        for (int j = 0; j < WM; ++j) {
            const float* base = table + j * D + 8 * cg;
            const float4 a4 = *reinterpret_cast<const float4*>(base);
            const float4 b4 = *reinterpret_cast<const float4*>(base + 4);
            w2[0][j] = make_float2(a4.x, a4.y);
            w2[1][j] = make_float2(a4.z, a4.w);
            w2[2][j] = make_float2(b4.x, b4.y);
            w2[3][j] = make_float2(b4.z, b4.w);
        }
    };
    // bf16: SiLU(conv) of output rows r0 .. r0 + 3 from a staged tile (row slot r + WM - 1 holds
    // row r); each input row is read and widened once and slides through the window
    auto conv_rows = [&](const unsigned char* tile_base, auto&& emit) {
        const unsigned char* tile = tile_base + (uint32_t)r0 * 256 + cg * 16;
        float2 x2[WM + 3][4];
#pragma unroll
        for (int j = 0; j < WM + 3; ++j) {
            const uint4 u = *reinterpret_cast<const uint4*>(tile + j * 256);
            const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
            for (int pr = 0; pr < 4; ++pr) x2[j][pr] = __bfloat1622float2(hb[pr]);
        }
        float y[4][8];
#pragma unroll
        for (int o = 0; o < 4; ++o)
#pragma unroll
            for (int pr = 0; pr < 4; ++pr) {
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < WM; ++j) acc = fma2(w2[pr][j], x2[o + j][pr], acc);
                const float2 yy = silu2(acc);
                y[o][2 * pr] = yy.x;
                y[o][2 * pr + 1] = yy.y;
            }
        emit(y);
    };
    // park v rows r0 .. r0 + 3 under this thread's own scale (2^-vexp brings its largest value
    // below 64), and bring the rows' maximum to the head's chunk maximum; the rows are brought
    // to the chunk's common scale when the V' image is written
    auto v_emit = [&](const float (&y)[4][8]) {
        float m = 0.f;
#pragma unroll
        for (int o = 0; o < 4; ++o)
#pragma unroll
            for (int e = 0; e < 8; ++e) m = r0 + o < n ? fmaxf(m, fabsf(y[o][e])) : m;
        vexp = scale_exp(m, 5);
        const float sc = pow2f(-vexp);
#pragma unroll
        for (int o = 0; o < 4; ++o) vpark[o] = v_row(o, y[o], sc);
        const unsigned mb = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
        if (lane == 0) atomicMax(s_vmax + vhead, mb);
    };
    // a sequence's first chunk: rows r < 0 of a staged tile from the slot's conv buffer (zero
    // before it); channel base ch0 of the conv's C channels
    auto halo = [&](unsigned char* tile_base, int ch0, int idx) {
        const int j = idx >> 4, c16 = idx & 15, p = j - (WM - 1);
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        const TIn* src = cbuf + (size_t)(A.W - 1 + p) * A.C + ch0 + 8 * c16;
        if (p >= -(A.W - 1) && chk(within(src, 16, A.base, slots_region), A.status))
            x = *reinterpret_cast<const uint4*>(src);
        unsigned char* dst = tile_base + (uint32_t)j * 256 + c16 * 16;
        if (sm_ok(dst, 16)) *reinterpret_cast<uint4*>(dst) = x;
    };
    // bf16: the v taps of a head (prefetched) into a [tap][channel] table
    auto store_vtaps = [&](float* table) {
#pragma unroll
        for (int k = 0; k < KV; ++k) {
            const int idx = tid + k * NT, chl = idx / WM, j = idx - chl * WM;
            table[j * D + chl] = tvv[k];
        }
    };
    if constexpr (sizeof(TIn) == 2) {
        // q, k and the first head's v rows arrive by the copies issued above; meanwhile the
        // taps go to shared memory, right-aligned in WM slots ([tensor][tap][channel], so that
        // a thread's 8 channels of a tap are two conflict-free 16-B reads)
        float* s_taps = reinterpret_cast<float*>(sm + P_RAW + 3 * NRT * 256);
#pragma unroll
        for (int k = 0; k < KT; ++k) {
            const int idx = tid + k * NT;
            const int t = idx / (D * WM), rem = idx - t * (D * WM), chl = rem / WM, j = rem - chl * WM;
            s_taps[(t * WM + j) * D + chl] = tv[k];
        }
        store_vtaps(s_taps + 2 * WM * D);
        const bool staged = mbar_wait_bounded(sbar, 0, nullptr);
        if (!staged && tid == 0) atomicOr(A.status, GDN_DEV_TIMEOUT);
        for (int idx = tid; p0 == 0 && idx < 3 * (WM - 1) * 16; idx += NT) {
            const int t = idx / ((WM - 1) * 16);
            halo(sm + P_RAW + t * NRT * 256, t == 0 ? Dq + hk * D : t == 1 ? hk * D : 2 * Dq + h0 * D,
                 idx - t * ((WM - 1) * 16));
        }
        ok = __syncthreads_and(staged) != 0;
        load_taps(s_taps);
        conv_rows(sm + P_RAW, [&](const float (&y)[4][8]) { qk_rows4(y, false); });
        load_taps(s_taps + WM * D);
        conv_rows(sm + P_RAW + NRT * 256, [&](const float (&y)[4][8]) { qk_rows4(y, true); });
        load_taps(s_taps + 2 * WM * D);
        conv_rows(sm + P_RAW + 2 * NRT * 256, v_emit);
    } else {
        // fp32: the rows through registers, one tensor at a time
        ConvRows<TIn, WM> x;
        x.load(kin, Dq, hk * D + 8 * cg, cbuf, A.C, ch_k, A.W, tc0, p0, r0, n);
        ConvRows<TIn, WM>::taps(w, A.conv_w, ch_k, A.W);
        {
            float y[4][8];
#pragma unroll
            for (int o = 0; o < 4; ++o) x.row(w, o, y[o]);
            qk_rows4(y, false);
        }
        x.load(qin, Dq, hk * D + 8 * cg, cbuf, A.C, ch_q, A.W, tc0, p0, r0, n);
        ConvRows<TIn, WM>::taps(w, A.conv_w, ch_q, A.W);
        {
            float y[4][8];
#pragma unroll
            for (int o = 0; o < 4; ++o) x.row(w, o, y[o]);
            qk_rows4(y, true);
        }
    }
    // fp32: v rows of head h through registers
    auto conv_v_f32 = [&](int h) {
        if constexpr (sizeof(TIn) != 2) {
            ConvRows<TIn, WM> x;
            x.load(vin, Dv, h * D + 8 * cg, cbuf, A.C, 2 * Dq + h * D + 8 * cg, A.W, tc0, p0, r0, n);
            ConvRows<TIn, WM>::taps(w, A.conv_w, 2 * Dq + h * D + 8 * cg, A.W);
            float y[4][8];
#pragma unroll
            for (int o = 0; o < 4; ++o) x.row(w, o, y[o]);
            v_emit(y);
        }
    };
    conv_v_f32(h0);
    tc::fence_proxy_async();
    sync_all();
    if (tid == 0 && chk(within(qkimg, QK_BYTES, A.ws.kimg, qk_region), A.status)) {
        // the [K; Q] tile is the (chunk, q/k head) part of the record
        bulk_s2g(qkimg, sm + P_A1, QK_BYTES);
        bulk_commit();
    }

    // the output gates silu(z) w_n of the head into the W area, from where one bulk copy takes
    // them to the record.  A token's gates are stored times 2^-ez, ez chosen from the token's
    // largest gate by the 16 threads that hold its 128 channels (a half-warp), so that any z
    // keeps fp16's relative precision; ez goes to the record with the chunk's scalars.
    auto gates = [&]() {
        float2 nw[4];  // the norm weights of this thread's 8 channels (the same for every q)
#pragma unroll
        for (int e = 0; e < 4; ++e) nw[e] = make_float2(__ldg(A.norm_w + 8 * cg + 2 * e), __ldg(A.norm_w + 8 * cg + 2 * e + 1));
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int idx = tid + q * NT, i = idx >> 4, c8 = (idx & 15) * 8;
            const TIn* zv = reinterpret_cast<const TIn*>(zpark[q]);
            float2 g2[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) g2[e] = mul2(silu2(make_float2(to_f(zv[2 * e]), to_f(zv[2 * e + 1]))), nw[e]);
            float m = fmaxf(fmaxf(fmaxf(fabsf(g2[0].x), fabsf(g2[0].y)), fmaxf(fabsf(g2[1].x), fabsf(g2[1].y))),
                            fmaxf(fmaxf(fabsf(g2[2].x), fabsf(g2[2].y)), fmaxf(fabsf(g2[3].x), fabsf(g2[3].y))));
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            const int ez = scale_exp(m, 14);
            const float2 f2 = make_float2(pow2f(-ez), pow2f(-ez));
#pragma unroll
            for (int e = 0; e < 4; ++e) g2[e] = mul2(g2[e], f2);
            uint4 wv;
            wv.x = i < n ? pack_half2(g2[0].x, g2[0].y) : 0u;
            wv.y = i < n ? pack_half2(g2[1].x, g2[1].y) : 0u;
            wv.z = i < n ? pack_half2(g2[2].x, g2[2].y) : 0u;
            wv.w = i < n ? pack_half2(g2[3].x, g2[3].y) : 0u;
            unsigned char* dst = sm + P_R5 + (c8 >> 6) * 8192 + tc::sw128_chunk(i, (c8 & 63) >> 3);
            if (tile_ok(dst, 16, P_R5, 16384)) *reinterpret_cast<uint4*>(dst) = wv;
            if ((idx & 15) == 0 && chk(i < 64, A.status)) sEZ[i] = ez;
        }
        tc::fence_proxy_async();
    };
    auto zero_block = [&](uint32_t off) {
#pragma unroll
        for (int q = 0; q < 2; ++q) *reinterpret_cast<uint4*>(sm + off + (tid + q * NT) * 16) = make_uint4(0u, 0u, 0u, 0u);
    };

    // (b) MMA1: [K; Q] x K^T into columns [128, 192); meanwhile the two zero blocks are cleared
    //     (the staging area they lie in is dead)
    if (tid == 0)
        tc::mma_k(tm + 128, smem_addr(sm + P_A1), 128, smem_addr(sm + P_A1), 128, D, tc::idesc_f16(128, 64), 0);
    zero_block(P_Z0);
    zero_block(P_Z1);
    gates();
    mma_done();

    for (int jh = 0; jh < A.r && ok; ++jh) {
        const int h = h0 + jh;
        unsigned char* rec = A.ws.rec + ((size_t)slot_rec * A.hv + h) * REC_BYTES;
        const int cs = jh & 1;  // this head's gate arrays
        float* sBEG = sSet + cs * 320;
        float* sG = sBEG + 64;
        float* sB = sG + 64;
        float* sEG = sB + 64;
        float* sGam = sEG + 64;
        const float* sMisc = sMisc2 + cs * 8;
        if (jh > 0) {
            // the head's v rows were staged at P_T2 by a copy issued once the previous head's MMA3
            // was done (bf16); its taps follow the tile.  The staging overlaps the Z0 block, which
            // is cleared again once the rows are consumed.
            if (jh > 1) scan_set(cs, 0);
            vhead = jh;
            if constexpr (sizeof(TIn) == 2) {
                float* vt = reinterpret_cast<float*>(sm + P_T2 + NRT * 256);
                store_vtaps(vt);
                const bool staged = mbar_wait_bounded(sbar, (uint32_t)(jh & 1), nullptr);
                if (!staged && tid == 0) atomicOr(A.status, GDN_DEV_TIMEOUT);
                for (int idx = tid; p0 == 0 && idx < (WM - 1) * 16; idx += NT) halo(sm + P_T2, 2 * Dq + h * D, idx);
                ok = __syncthreads_and(staged) != 0;
                if (!ok) break;
                load_taps(vt);
                conv_rows(sm + P_T2, v_emit);
                __syncthreads();
            } else {
                conv_v_f32(h);
            }
            if constexpr (sizeof(TIn) == 2) zero_block(P_Z0);  // it held these v rows
            gates();
            sync_all();
        }
        if (tid == 0 && rec_ok(rec + REC_GZ, 16384)) {
            bulk_s2g(rec + REC_GZ, sm + P_R5, 16384);
            bulk_commit();
        }
        if (jh + 1 < A.r) {
            prefetch_head(h + 1);
            if (jh + 1 > 1) load_gate_inputs(h + 1, 0);
        }

        // (c) A (fp32) from rows 0-63, P from rows 64-127 of [K; Q] x K^T; columns 32*hf ..
        //     The entries of A on and above the diagonal are never read (only strictly lower
        //     blocks enter the inverse), so A is written unmasked; rows past the chunk's end are
        //     zero through beta = 0 (A) and q = 0 (P).
        {
            const int row = qd * 32 + lane, i = row & 63, c0 = 32 * hf;
            const float Gi = sG[i];
            float v[32];
            tc::ld32(tc::taddr(tm, warp, 128 + c0), v);
            tc::wait_ld();
            if (row < 64) {
                const float bi = sB[i];
#pragma unroll
                for (int e4 = 0; e4 < 32; e4 += 4) {
                    const float4 g = *reinterpret_cast<const float4*>(sG + c0 + e4);
                    float4 a;
                    a.x = bi * __expf(Gi - g.x) * v[e4];
                    a.y = bi * __expf(Gi - g.y) * v[e4 + 1];
                    a.z = bi * __expf(Gi - g.z) * v[e4 + 2];
                    a.w = bi * __expf(Gi - g.w) * v[e4 + 3];
                    if (tile_ok(FA + i * FS + c0 + e4, 16, P_R4, 64 * FS * 4))
                        *reinterpret_cast<float4*>(FA + i * FS + c0 + e4) = a;
                }
            } else {
                float p[32];
#pragma unroll
                for (int e4 = 0; e4 < 32; e4 += 4) {
                    const float4 g = *reinterpret_cast<const float4*>(sG + c0 + e4);
                    const float gg[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        p[e4 + e] = (c0 + e4 + e <= i) ? __expf(Gi - gg[e]) * v[e4 + e] : 0.f;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (tile_ok(sm + P_P + tc::sw128_chunk(i, c0 / 8 + q), 16, P_P, 8192))
                        tc::st_chunk<Op>(sm + P_P, i, c0 / 8 + q, p + 8 * q);
            }
        }
        tc::fence_proxy_async();  // P leaves for the record by a bulk copy
        if (tid == 0) bulk_wait_read_all();  // the gates' copy has read the W area
        __syncthreads();
        if (tid == 0 && rec_ok(rec + REC_P, 8192)) {
            bulk_s2g(rec + REC_P, sm + P_P, 8192);
            bulk_commit();
        }
        // (d) T = (I + A)^-1, blocked.  16-wide diagonal blocks by forward substitution
        //     (one column per thread; zero above the diagonal and in the upper blocks) ...
        //     Rows of A and T are read 4 entries at a time; T's zeros above the diagonal are
        //     exact, so the merge sums below run over whole blocks.
        if (tid < 64) {
            const int b = tid >> 4, j = tid & 15, o = 16 * b;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float acc = (i == j) ? 1.f : 0.f;
#pragma unroll
                for (int k4 = 0; k4 < i; k4 += 4) {
                    const float4 a4 = *reinterpret_cast<const float4*>(FA + (o + i) * FS + o + k4);
                    const float aa[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                    for (int k = k4; k < k4 + 4 && k < i; ++k) acc -= aa[k - k4] * x[k];
                }
                x[i] = acc;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) FT[(o + i) * FS + o + j] = x[i];
        }
        for (int idx = tid; idx < 6 * 256; idx += NT) {  // the six 16x16 blocks above the diagonal
            const int blk = idx >> 8, e = idx & 255;
            const int bi = blk < 3 ? 0 : blk < 5 ? 1 : 2;
            const int bj = blk < 3 ? blk + 1 : blk < 5 ? blk - 1 : 3;
            FT[(16 * bi + (e >> 4)) * FS + 16 * bj + (e & 15)] = 0.f;
        }
        __syncthreads();
        //     ... then 16 -> 32: T_10 = -T_11 (A_10 T_00) for the block pairs (0,1), (2,3), both
        //     pairs' element (i, j) by one thread with two accumulators ...
        {
            const int i = (tid >> 4) & 15, j = tid & 15;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int k4 = 0; k4 < 16; k4 += 4) {
                const float4 f0 = *reinterpret_cast<const float4*>(FA + (16 + i) * FS + k4);
                const float4 f1 = *reinterpret_cast<const float4*>(FA + (48 + i) * FS + 32 + k4);
                const float g0[4] = {f0.x, f0.y, f0.z, f0.w}, g1[4] = {f1.x, f1.y, f1.z, f1.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    a0 = fmaf(g0[k], FT[(k4 + k) * FS + j], a0);
                    a1 = fmaf(g1[k], FT[(32 + k4 + k) * FS + 32 + j], a1);
                }
            }
            X[i * 17 + j] = a0;
            X[(16 + i) * 17 + j] = a1;
        }
        __syncthreads();
        {
            const int i = (tid >> 4) & 15, j = tid & 15;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int k4 = 0; k4 < 16; k4 += 4) {
                const float4 f0 = *reinterpret_cast<const float4*>(FT + (16 + i) * FS + 16 + k4);
                const float4 f1 = *reinterpret_cast<const float4*>(FT + (48 + i) * FS + 48 + k4);
                const float g0[4] = {f0.x, f0.y, f0.z, f0.w}, g1[4] = {f1.x, f1.y, f1.z, f1.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    a0 = fmaf(g0[k], X[(k4 + k) * 17 + j], a0);
                    a1 = fmaf(g1[k], X[(16 + k4 + k) * 17 + j], a1);
                }
            }
            FT[(16 + i) * FS + j] = -a0;
            FT[(48 + i) * FS + 32 + j] = -a1;
        }
        __syncthreads();
        //     ... then 32 -> 64: T_BA = -T_BB (A_BA T_AA), rows i0 + 8q (q < 4) of column j per thread
        {
            const int i0 = tid >> 5, j = tid & 31;
            float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
            for (int k4 = 0; k4 < 32; k4 += 4) {
                float t[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) t[k] = FT[(k4 + k) * FS + j];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 f = *reinterpret_cast<const float4*>(FA + (32 + i0 + 8 * q) * FS + k4);
                    a[q] = fmaf(f.x, t[0], a[q]);
                    a[q] = fmaf(f.y, t[1], a[q]);
                    a[q] = fmaf(f.z, t[2], a[q]);
                    a[q] = fmaf(f.w, t[3], a[q]);
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) X[(i0 + 8 * q) * 33 + j] = a[q];
        }
        __syncthreads();
        {
            const int i0 = tid >> 5, j = tid & 31;
            float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
            for (int k4 = 0; k4 < 32; k4 += 4) {
                float x[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) x[k] = X[(k4 + k) * 33 + j];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 f = *reinterpret_cast<const float4*>(FT + (32 + i0 + 8 * q) * FS + 32 + k4);
                    a[q] = fmaf(f.x, x[0], a[q]);
                    a[q] = fmaf(f.y, x[1], a[q]);
                    a[q] = fmaf(f.z, x[2], a[q]);
                    a[q] = fmaf(f.w, x[3], a[q]);
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) FT[(32 + i0 + 8 * q) * FS + j] = -a[q];
        }
        __syncthreads();
        //     T2 = T diag(beta) 2^-eb, T1 = T diag(beta e^G) 2^-eg, with the powers of two that
        //     bring the largest beta and beta e^G of the chunk into [1, 2) (a chunk of tiny write
        //     strengths or strong decay keeps its relative precision), one 8-column chunk per
        //     item; a warp takes 32 consecutive rows of one chunk column (conflict-free row reads)
        const int eb = scale_exp(fmaxf(sMisc[2], sMisc[3]), 0), eg = scale_exp(fmaxf(sMisc[4], sMisc[5]), 0);
        const float fb = pow2f(-eb), fg = pow2f(-eg);
        for (int idx = tid; idx < 128 * 8; idx += NT) {
            const int r = idx & 127, c8 = idx >> 7, i = r & 63;
            const float* sc = (r < 64 ? sB : sBEG) + c8 * 8;
            const float f = r < 64 ? fb : fg;
            const float4 t0 = *reinterpret_cast<const float4*>(FT + i * FS + c8 * 8);
            const float4 t1 = *reinterpret_cast<const float4*>(FT + i * FS + c8 * 8 + 4);
            const float4 s0 = *reinterpret_cast<const float4*>(sc), s1 = *reinterpret_cast<const float4*>(sc + 4);
            float v[8] = {t0.x * (s0.x * f), t0.y * (s0.y * f), t0.z * (s0.z * f), t0.w * (s0.w * f),
                          t1.x * (s1.x * f), t1.y * (s1.y * f), t1.z * (s1.z * f), t1.w * (s1.w * f)};
            const uint32_t toff = r < 64 ? P_T2 : P_T1;
            if (tile_ok(sm + toff + tc::sw128_chunk(i, c8), 16, toff, 8192)) tc::st_chunk<Op>(sm + toff, i, c8, v);
        }
        __syncthreads();  // A (fp32) is dead from here: its space takes the V image
        // (d') V' image [token][dv] = V 2^-ev for MMA3's second product, from the rows parked in
        //     registers, where each thread's rows sit at a scale of their own
        const int ev = scale_exp(__uint_as_float(s_vmax[jh]), 5);
        if (ev != vexp) {
            const float2 f2 = make_float2(pow2f(vexp - ev), pow2f(vexp - ev));
#pragma unroll
            for (int o = 0; o < 4; ++o) {
                uint32_t* wv = reinterpret_cast<uint32_t*>(&vpark[o]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 x = mul2(__half22float2(*reinterpret_cast<const __half2*>(&wv[q])), f2);
                    wv[q] = pack_half2(x.x, x.y);
                }
            }
        }
#pragma unroll
        for (int o = 0; o < 4; ++o) {
            unsigned char* dst = sm + P_R4 + (cg >> 3) * 8192 + tc::sw128_chunk(r0 + o, cg & 7);
            if (tile_ok(dst, 16, P_R4, 16384)) *reinterpret_cast<uint4*>(dst) = vpark[o];
        }
        tc::fence_proxy_async();
        sync_all();

        // (e) MMA3, block diagonal: [T2; Z] x V' + [Z; T1] x K (V' and K read MN-major; K from
        //     the [K; Q] tile) -> U' = U 2^-(eb+ev) in rows 0-63, W' = W 2^-eg in rows 64-127
        if (tid == 0) {
            tc::mma_k_mixed(tm, smem_addr(sm + P_T2), 128, 0, 0, smem_addr(sm + P_R4), 0, 1, 8192, CH,
                            tc::idesc_f16(128, 128, 0, 1), 0);
            tc::mma_k_mixed(tm, smem_addr(sm + P_Z1), 128, 0, 0, smem_addr(sm + P_A1), 0, 1, 16384, CH,
                            tc::idesc_f16(128, 128, 0, 1), 1);
        }
        mma_done();
        if (!ok) break;
        if constexpr (sizeof(TIn) == 2) {
            // the next head's v rows go to P_T2 (over T2, Z0 and the start of P: MMA3 is done
            // and P has been copied out), so that they arrive while this head finishes
            if (tid == 0 && jh + 1 < A.r) {
                bulk_wait_read_all();
                mbar_arrive_expect_tx(sbar, NRT * 256);
                if (sm_ok(sm + P_T2, NRT * 256)) tma_load_2d(sm + P_T2, &M.v, (h + 1) * D, y0, sbar);
            }
        }

        // (f) U' (rows 0-63) -> the U' image (over the dead V' image); W' (rows 64-127) -> the
        //     W' image, with their maxima; both go to the record with the chunk's scalars
        {
            const int row = qd * 32 + lane, i = row & 63;
            float mx = 0.f;
            for (int c0 = 64 * hf; c0 < 64 * hf + 64; c0 += 32) {
                float v[32];
                tc::ld32(tc::taddr(tm, warp, c0), v);
                tc::wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) mx = fmaxf(mx, fabsf(v[e]));
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int ch = (c0 & 63) / 8 + q;
                    const uint32_t toff = row >= 64 ? P_R5 : P_R4;
                    if (tile_ok(sm + toff + (c0 >> 6) * 8192 + tc::sw128_chunk(i, ch), 16, toff, 16384))
                        tc::st_chunk<Op>(sm + toff + (c0 >> 6) * 8192, i, ch, v + 8 * q);
                }
            }
            const unsigned mb = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
            if (lane == 0) atomicMax((row >= 64 ? s_wmax : s_umax) + jh, mb);
        }
        tc::fence_proxy_async();
        sync_all();
        if (tid == 0 && rec_ok(rec + REC_W, 16384) && rec_ok(rec + REC_U, 16384)) {
            bulk_s2g(rec + REC_W, sm + P_R5, 16384);
            bulk_s2g(rec + REC_U, sm + P_R4, 16384);
            bulk_commit();
        }
        float* scr = reinterpret_cast<float*>(rec + REC_SC);
        if (!rec_ok(scr, SC_BYTES)) break;
        if (tid < 64) {
            scr[SC_GAM + tid] = sGam[tid];
            scr[SC_EG + tid] = sEG[tid];
            reinterpret_cast<int*>(scr)[SC_EZ + tid] = sEZ[tid];
        }
        if (tid == 0) {
            scr[SC_EGL] = sMisc[0];
            reinterpret_cast<int*>(scr)[SC_EU] = eb + ev;
            reinterpret_cast<int*>(scr)[SC_EW] = eg;
            scr[SC_MU] = __uint_as_float(s_umax[jh]);
            scr[SC_MW] = __uint_as_float(s_wmax[jh]);
        }
        if (tid == 0) bulk_wait_read_all();  // the next head reuses every area
        sync_all();
    }
    if (tid == 0) bulk_wait_read_all();  // shared memory outlives every copy reading it
    sync_all();
    if (warp == 0) tc::dealloc(tm, 256);
}

// ================================================================== state pass ====
// One CTA per (sequence, v-head, d_v half); the two halves of a (sequence, v-head) form a
// cluster of two.  A CTA keeps S^T restricted to its half, [d_k][64 d_v], in fp32 TMEM
// columns TS .. TS + 63 (lane = d_k) in true units, so the products have M = 128 and N = 64:
//     MMA4  [W'; Q] x S0^T(:, half) 2^-Es  -> rows 0-63: W' S0^T, rows 64-127: Q S0^T
//     MMA6  X = K^T x Delta~(:, half) 2^-Ed   (Delta~ = diag(gamma) Delta; both MN-major)
//     MMA7  [0; P] x Delta(:, half) 2^-Ed  -> rows 64-127: P Delta
// and the next chunk starts from S <- e^{G_last} S + 2^Ed X, formed in fp32 while that
// chunk's S0^T is rounded.  MMA4 of chunk c writes TMEM columns TM4 + 64 (c % 2), MMA7
// TM7 + 64 (c % 2).  MMA7 of chunk c is issued right after its MMA6 and runs while the next
// S0^T is formed; the output warps read both results one chunk later:
//     O_i = e^{G_i} 2^Es (Q S0^T)_i + 2^Ed (P Delta)_i.
// Only S0^T -> MMA4 -> Delta -> MMA6 is serial from chunk to chunk.
// The scales: 2^-Es brings a bound on max |S0| below 2^13 -- the measured maximum for the
// first chunk; after that e^{G_last} times the last chunk's measured maximum plus 64 times
// the last chunk's Delta bound (|K^T Delta~| <= 64 max |Delta~| for unit keys) -- and 2^-Ed
// brings the bound max |U| + 128 max |W| max |S0| on |Delta| below 2^13.  The measured
// maximum of S0 comes from per-warp maxima of the values being rounded, read after the
// barrier that opens the chunk (no barrier of their own).
// The gated RMSNorm of an output row needs its sum of squares over all of d_v, so each CTA
// sends its half's 64 per-token sums into the other CTA's shared memory and arrives on that
// CTA's mbarrier (distributed shared memory).  Warps w with w % 4 < 2 hold rows 0-63 (Delta);
// the others hold rows 64-127 and read the output one chunk behind the chain, finishing its
// rows one more behind (once the other CTA's sums are in); thread PF of warp 2 fetches the
// records, thread 0 issues the products.  8 warps: warp w reads TMEM lane quarter w % 4 and works on columns
// 32 (w / 4) .. + 31.

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(NT, 1) chunk_state_kernel(PrefillArgs A)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = align1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + S_SMALL);  // [2] record buffers
    uint64_t* bar4 = full + 2;                                   // MMA4 completion (one phase per chunk)
    uint64_t* peer_bar = bar4 + 1;                               // [2] the other half's sums, by chunk parity
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(peer_bar + 2);
    uint64_t* bar6 = peer_bar + 3;                               // MMA6 completion (one phase per chunk)
    uint64_t* full_p = peer_bar + 5;                             // [2] P slots
    uint64_t* const bar7e = peer_bar + 4;                        // MMA7 completion, even chunks
    uint64_t* const bar7o = peer_bar + 7;                        // MMA7 completion, odd chunks
    float* s_ss = reinterpret_cast<float*>(sm + S_SMALL + 128);  // [2][2][64] sums of O^2: chunk parity, column half
    float* peer_ss = s_ss + 256;                                 // [2][64] the other CTA's sums, by chunk parity
    // [2][8] per-warp max |S0| by chunk parity, then [16] the incoming state's maximum (bit
    // patterns of non-negative floats)
    unsigned int* s_smax = reinterpret_cast<unsigned int*>(peer_ss + 128);

    // both CTAs of a cluster take these exits together (they depend on the sequence only)
    if (!*A.ws.valid) return;
    const int half = blockIdx.x & 1, pair = blockIdx.x >> 1, h = pair % A.hv;
    int rank = pair / A.hv;  // of the sequence in length order
    if (A.seg_hi != INT_MAX) {  // a segment: the i-th of the sequences with records in it
        const int* win = window_slot(A);
        const int i = rank;
        rank = i < win[0] ? i : i - win[0] < win[2] ? win[1] + (i - win[0]) : -1;
        if (rank < 0) return;
    }
    const int s = A.ws.order[rank];
    const int t0s = A.cu[s], Ls = A.cu[s + 1] - t0s;  // the whole sequence
    if (Ls <= 0) return;
    // This launch takes the sequence's chunks whose records (chunk c: coff[c] + rank) lie in the
    // segment [seg_lo, seg_hi): chunks cb .. ce-1, a contiguous run as the record numbers grow
    // with c, starting from the state the slot holds (the sequence's initial state, or the state
    // the previous segment's launch left there).
    const int nchs = (Ls + CH - 1) / CH;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int cb = 0, ce = nchs;
    if (A.seg_hi != INT_MAX) {
        // cb, ce = the numbers of chunks c whose record coff[c] + rank lies below seg_lo, seg_hi
        // (it grows with c): counted by all threads at once, one load per thread and step
        int nlo = 0, nhi = 0;
        for (int c = tid; c < nchs; c += NT) {
            const int r = A.ws.coff[c] + rank;
            nlo += r < A.seg_lo;
            nhi += r < A.seg_hi;
        }
        int* cnt = reinterpret_cast<int*>(sm + S_POS);
        if (tid == 0) cnt[0] = cnt[1] = 0;
        __syncthreads();
        if (nlo) atomicAdd(&cnt[0], nlo);
        if (nhi) atomicAdd(&cnt[1], nhi);
        __syncthreads();
        cb = cnt[0];
        ce = cnt[1];
        __syncthreads();
    }
    if (cb >= ce) return;
    const bool seq_end = ce == nchs;  // the sequence's last chunk is in this segment
    const int t0 = t0s + cb * CH, L = min(Ls - cb * CH, (ce - cb) * CH);  // this segment's tokens
    const int qd = warp & 3, hf = warp >> 2, row = qd * 32 + lane;
    const int hk = h / A.r, Dv = A.hv * D;
    const int nch = ce - cb;  // chunks here (at most kPrefillMaxRecords: one record each)
    if (nch > kPrefillMaxRecords) {  // cannot happen (segments hold at most that many records); both CTAs leave
        if (threadIdx.x == 0) atomicOr(A.status, GDN_DEV_BOUNDS);
        return;
    }
    // workspace positions of this segment's chunks
    int* s_pos = reinterpret_cast<int*>(sm + S_POS);
    for (int i = tid; i < nch; i += NT) s_pos[i] = A.ws.coff[cb + i] + rank - A.seg_lo;
    const uint32_t peer = cluster_ctarank() ^ 1u;
    float* Sg = reinterpret_cast<float*>(A.base + ((uint64_t)A.ids[s] * A.num_layers + A.layer) * A.slot_bytes) +
                (size_t)h * D * D;
    TOut* out = static_cast<TOut*>(A.out);
    // the regions a checked build tests this kernel's computed accesses against
    const size_t sm_bytes = (size_t)(smem_raw + S_SMEM - sm);
    const size_t rec_region = (size_t)A.ws.chunk_cap * A.hv * REC_BYTES;
    const size_t qk_region = (size_t)A.ws.chunk_cap * A.hqk * QK_BYTES;
    const size_t slots_region = (size_t)A.num_slots * A.num_layers * A.slot_bytes;
    auto sm_ok = [&](const void* p, size_t b) { return chk(within(p, b, sm, sm_bytes), A.status); };
    auto slot_ok = [&](const void* p, size_t b) { return chk(within(p, b, A.base, slots_region), A.status); };
    auto g2s = [&](void* dst, const void* src, uint32_t b, uint64_t* bar, const void* lo, size_t region) {
        if (sm_ok(dst, b) && chk(within(src, b, lo, region), A.status)) bulk_g2s(dst, src, b, bar);
    };

    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&full_p[0], 1);
        mbar_init(&full_p[1], 1);
        mbar_init(bar4, 1);
        mbar_init(bar6, 1);
        mbar_init(bar7e, 1);
        mbar_init(bar7o, 1);
        mbar_init(&peer_bar[0], 1);
        mbar_init(&peer_bar[1], 1);
        fence_mbar_init();
        s_smax[16] = 0u;
    }
    if (warp == 0) tc::alloc(tmem_slot, 512);
    sync_all();
    cluster_sync_all();  // the other CTA's barriers exist before anything arrives on them
    const uint32_t tm = *tmem_slot;
    bool ok = true;
    constexpr int PF = 64;  // the thread that fetches the records (warp 2 works on output rows)
    int main_issued = 0, p_issued = 0;  // fetches so far (thread PF)
    int mma7_issued = 0;    // MMA7s so far (thread 0)
    auto record = [&](int c) { return A.ws.rec + ((size_t)s_pos[c] * A.hv + h) * REC_BYTES; };
    // the record's [W'; Q] operand (the W' image and the Q rows of the [K; Q] tile, per 64-wide
    // d_k half), the K rows of the tile, the U' half, the gates half and the scalars.  (Issuing a
    // bulk copy costs its thread tens of nanoseconds; spreading these over three Delta-warp
    // threads measured slower: every warp of the chunk is on its critical path.)
    auto fetch_main = [&](int c) {
        unsigned char* dst = sm + (c & 1) * S_BUF;
        const unsigned char* rec = record(c);
        const unsigned char* qk = A.ws.kimg + ((size_t)s_pos[c] * A.hqk + hk) * QK_BYTES;
        uint64_t* fb = &full[c & 1];
        mbar_arrive_expect_tx(fb, S_TX);
        g2s(dst + B_A, rec + REC_W, 8192, fb, A.ws.rec, rec_region);
        g2s(dst + B_A + 16384, rec + REC_W + 8192, 8192, fb, A.ws.rec, rec_region);
        g2s(dst + B_A + 8192, qk + 8192, 8192, fb, A.ws.kimg, qk_region);
        g2s(dst + B_A + 16384 + 8192, qk + 16384 + 8192, 8192, fb, A.ws.kimg, qk_region);
        g2s(dst + B_K, qk, 8192, fb, A.ws.kimg, qk_region);
        g2s(dst + B_K + 8192, qk + 16384, 8192, fb, A.ws.kimg, qk_region);
        g2s(dst + B_U, rec + REC_U + half * 8192, 8192, fb, A.ws.rec, rec_region);
        g2s(dst + B_GZ, rec + REC_GZ + half * 8192, 8192, fb, A.ws.rec, rec_region);
        g2s(dst + B_SC, rec + REC_SC, SC_BYTES, fb, A.ws.rec, rec_region);
        main_issued = c + 1;
    };
    auto fetch_p = [&](int c) {
        mbar_arrive_expect_tx(&full_p[c & 1], 8192);
        g2s(sm + S_PZ + (c & 1) * 16384 + 8192, record(c) + REC_P, 8192, &full_p[c & 1], A.ws.rec, rec_region);
        p_issued = c + 1;
    };
    const int first_fetched = A.stall_fetch ? 1 : 0;  // the test hook leaves chunk 0's record unfetched
    if (tid == PF) {
        if (!A.stall_fetch) fetch_main(0);
        fetch_p(0);
        if (nch > 1) {
            fetch_main(1);
            fetch_p(1);
        }
    }
    // While the first records arrive (in the segment that holds the sequence's last chunk): the
    // slot's conv buffer becomes the sequence's last W-1 raw inputs (older buffer rows where the
    // sequence is shorter).  The pre-pass, which read the old rows, is complete, and this pass
    // never reads them.  This CTA's channels: its d_v half of the v-head's channels, and when h is
    // the q/k head's first v-head its half of the q/k head's q and k channels -- disjoint across
    // the CTAs of the call.
    if (seq_end) {
        TIn* cbuf = reinterpret_cast<TIn*>(A.base + ((uint64_t)A.ids[s] * A.num_layers + A.layer) * A.slot_bytes +
                                           A.state_bytes);
        const int Dq = A.hqk * D, W = A.W, C = A.C;
        if (tid < (h % A.r == 0 ? 192 : 64)) {
            const int ch = tid < 64    ? 2 * Dq + h * D + half * 64 + tid           // v
                           : tid < 128 ? hk * D + half * 64 + (tid - 64)            // q
                                       : Dq + hk * D + half * 64 + (tid - 128);     // k
            TIn old[7];
#pragma unroll
            for (int j = 0; j < 7; ++j)
                if (j < W - 1 && slot_ok(cbuf + (size_t)j * C + ch, sizeof(TIn)))
                    old[j] = static_cast<const TIn*>(static_cast<const void*>(cbuf))[(size_t)j * C + ch];
#pragma unroll
            for (int i = 0; i < 7; ++i) {
                if (i >= W - 1) break;
                const int pp = Ls - (W - 1) + i;
                TIn x = old[0];
                if (pp >= 0) {
                    const size_t t = (size_t)(t0s + pp);
                    const bool in = chk(t < (size_t)A.T, A.status);
                    x = !in           ? x
                        : ch < Dq     ? static_cast<const TIn*>(A.q)[t * Dq + ch]
                        : ch < 2 * Dq ? static_cast<const TIn*>(A.k)[t * Dq + (ch - Dq)]
                                      : static_cast<const TIn*>(A.v)[t * (size_t)(A.hv * D) + (ch - 2 * Dq)];
                } else {
#pragma unroll
                    for (int j = 0; j < 7; ++j)
                        if (j == W - 1 + pp) x = old[j];
                }
                if (slot_ok(cbuf + (size_t)i * C + ch, sizeof(TIn))) cbuf[(size_t)i * C + ch] = x;
            }
        }
    }
    // MMA7 of chunk pc (thread 0, right after the chunk's MMA6; issued from a second thread it
    // measured slower: the two threads' products do not issue in parallel, and that thread's warp
    // then reaches the next chunk's barrier late): [0; P] x Delta into chunk pc's MMA7 columns;
    // completes on the barrier of pc's parity; the commit is issued even when the product is not,
    // so that every wait has its phase
    auto issue_mma7 = [&](int pc, bool go) {
        const bool gotp = mbar_wait_bounded(&full_p[pc & 1], (uint32_t)((pc >> 1) & 1), nullptr);
        if (!gotp) atomicOr(A.status, GDN_DEV_TIMEOUT);
        if (go && gotp)
            tc::mma_k_mixed(tm + TM7 + 64 * (pc & 1), smem_addr(sm + S_PZ + (pc & 1) * 16384), 128, 0, 0,
                            smem_addr(sm + S_DL + (pc & 1) * 8192), 0, 1, 8192, CH, tc::idesc_f16(128, 64, 0, 1), 0);
        tc::commit((pc & 1) ? bar7o : bar7e);
        mma7_issued = pc + 1;
    };
    // the zero halves of MMA7's operands
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int idx = tid + NT * k;  // 16-B chunk of the two 8 KiB zero blocks
        *reinterpret_cast<uint4*>(sm + S_PZ + (idx >> 9) * 16384 + (idx & 511) * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    tc::fence_proxy_async();

    // incoming state: S^T(:, half) into TMEM columns TS .. TS + 63 (lane = d_k, column j = d_v
    // 64 half + j), true units; its maximum sets the first chunk's scale
    {
        float v[32];
        float m = 0.f;
        const int dv0 = half * 64 + 32 * hf;
        const bool sok = slot_ok(Sg + (size_t)dv0 * D, (size_t)32 * D * sizeof(float));
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            v[e] = sok ? Sg[(size_t)(dv0 + e) * D + row] : 0.f;
            m = fmaxf(m, fabsf(v[e]));
        }
        tc::st32(tc::taddr(tm, warp, TS + 32 * hf), v);
        tc::wait_st();
        const unsigned mb = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
        if (lane == 0) atomicMax(s_smax + 16, mb);
    }

    // output rows (rows >= 64 only, this thread's 32 columns): o holds O_i of the chunk waiting
    // for the other CTA's sums, gzr / ezr its gates and their scale exponent; gzn / ezn and eg_n
    // the gates, exponent and e^{G_i} of the chunk just computed
    float o[32];
    uint4 gzn[4], gzr[4];
    int ezn = 0, ezr = 0;
    float eg_n = 0.f;
    const int orow = row - 64, col0 = half * 64 + 32 * hf;
    auto finish_rows = [&](int pc) -> bool {  // false when the sums never came
        const bool gotp = mbar_wait_cluster_bounded(&peer_bar[pc & 1], (uint32_t)((pc >> 1) & 1));
        const int pn = min(CH, L - pc * CH);
        if (gotp && orow < pn) {
            const float rs =
                rms_scale(s_ss[(pc & 1) * 128 + orow] + s_ss[(pc & 1) * 128 + 64 + orow] + peer_ss[(pc & 1) * 64 + orow],
                          A.norm_eps, D) *
                pow2f(ezr);
            TOut* dst = out + (size_t)(t0 + pc * CH + orow) * Dv + (size_t)h * D + col0;
            const bool ook = chk(within(dst, 32 * sizeof(TOut), out, (size_t)A.T * Dv * sizeof(TOut)), A.status);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float gz[8], y[8];
                unpack8(gzr[q], gz);
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = o[8 * q + e] * rs * gz[e];
                if (ook) store8<TOut>(dst + 8 * q, y);
            }
        }
        return gotp;
    };
    // O of chunk pc from MMA4's rows 64-127 (scale 2^es) and MMA7 (scale 2^ed), its sums of squares
    auto complete_rows = [&](int pc, int es_c, int ed_c) -> bool {
        const bool got7 = mbar_wait_bounded((pc & 1) ? bar7o : bar7e, (uint32_t)((pc >> 1) & 1), nullptr);
        tc::fence_after_sync();
        float zz[32];
        tc::ld32(tc::taddr(tm, warp, TM4 + 64 * (pc & 1) + 32 * hf), o);
        tc::ld32(tc::taddr(tm, warp, TM7 + 64 * (pc & 1) + 32 * hf), zz);
        tc::wait_ld();
        const float fy = eg_n * pow2f(es_c), fz = pow2f(ed_c);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            o[e] = fmaf(fz, zz[e], fy * o[e]);
            ss = fmaf(o[e], o[e], ss);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) gzr[q] = gzn[q];
        ezr = ezn;
        s_ss[(pc & 1) * 128 + hf * 64 + orow] = ss;
        return got7;
    };
    // this half's per-token sums of squares of chunk pc -> the other CTA, by asynchronous
    // stores that complete on its barrier for that chunk (16 threads of warp 2)
    auto send_sums = [&](int pc) {
        if (tid >= PF && tid < PF + 16) {
            const int j = tid - PF;
            const float* mine = s_ss + (pc & 1) * 128;
            const float4 a = reinterpret_cast<const float4*>(mine)[j];
            const float4 b = reinterpret_cast<const float4*>(mine + 64)[j];
            st_async_cluster_v4(map_to_rank(smem_addr(peer_ss + (pc & 1) * 64 + 4 * j), peer),
                                make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w),
                                map_to_rank(smem_addr(&peer_bar[pc & 1]), peer));
        }
    };

    // The barrier for the other CTA's 64 sums of chunk c is armed (for 256 bytes) before the
    // loop for chunks 0 and 1, and for chunk c >= 2 by thread PF in chunk c once it has seen
    // the sums of chunk c - 2 arrive (never after a failed wait).  The other CTA sends its
    // sums of chunk c only after it has received this CTA's sums of chunk c - 1, which are
    // sent after that point, so a phase is never armed or completed twice and a sums slot is
    // never overwritten before it is read.
    if (tid == 0) {
        mbar_arrive_expect_tx(&peer_bar[0], 256);
        if (nch > 1) mbar_arrive_expect_tx(&peer_bar[1], 256);
    }
    sync_all();
    // Scale state carried from chunk to chunk, the same in every thread: the last chunk's
    // e^{G_last}, measured max |S0|, Delta bound and the exponents of its S0^T and Delta.
    float egl_p = 1.f, smax_p = __uint_as_float(s_smax[16]), dbound_p = 0.f;
    int es_p = 0, ed_p = 0;
    // MMA4 and MMA6 complete on barriers of their own, one phase per chunk; MMA7 on one barrier
    // per chunk parity (its result is read a chunk later), one phase per two chunks.  No
    // waiter can fall two phases behind one of them.  Per-thread verdicts of the bounded
    // waits become uniform at the barrier opening the next chunk, the only full barrier of
    // the loop (so the loop runs on c alone).
    for (int c = 0; c < nch; ++c) {
        unsigned char* buf = sm + (c & 1) * S_BUF;
        const bool got = mbar_wait_bounded(&full[c & 1], (uint32_t)((c >> 1) & 1), nullptr);
        if (!got && tid == 0) atomicOr(A.status, GDN_DEV_TIMEOUT);
        // the chunk's scalars (read before this buffer is refetched)
        const float* sc = reinterpret_cast<const float*>(buf + B_SC);
        const float egl = sc[SC_EGL], mu = sc[SC_MU], mw = sc[SC_MW];
        const int eu = __float_as_int(sc[SC_EU]), ew = __float_as_int(sc[SC_EW]);

        // S0 of this chunk (from the last chunk: e^{G_last} S + 2^Ed X, back to TMEM) and S0^T
        // 2^-Es in fp16 (MN-major: row = d_k) for MMA4, with this thread's share of max |S0|
        const int es = scale_exp(c == 0 ? smax_p : fmaf(egl_p, smax_p, 64.f * dbound_p), 12);
        {
            float v[32];
            tc::wait_st();  // the last chunk's store of S (long complete by now)
            tc::ld32(tc::taddr(tm, warp, TS + 32 * hf), v);
            if (c > 0) {
                float x[32];
                tc::ld32(tc::taddr(tm, warp, TX + 32 * hf), x);
                tc::wait_ld();
                const float fx = pow2f(ed_p);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = fmaf(fx, x[e], egl_p * v[e]);
                tc::st32(tc::taddr(tm, warp, TS + 32 * hf), v);
            } else {
                tc::wait_ld();
            }
            float mx[8];  // max |v| as a tree (independent partial maxima)
#pragma unroll
            for (int e = 0; e < 8; ++e) mx[e] = fmaxf(fmaxf(fabsf(v[e]), fabsf(v[e + 8])), fmaxf(fabsf(v[e + 16]), fabsf(v[e + 24])));
            const float m = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            const float f = pow2f(-es);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float t8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) t8[e] = v[8 * q + e] * f;
                tc::st_chunk<Op>(sm + S_S0, row, 4 * hf + q, t8);
            }
            const unsigned mb = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
            if (lane == 0) s_smax[(c & 1) * 8 + warp] = mb;
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        ok = __syncthreads_and(got && ok) != 0;
        tc::fence_after_sync();
        if (!ok) break;

        // MMA4: [W'; Q] x S0^T(:, half) 2^-Es -> columns TM4 + 64 (c % 2)
        if (tid == 0) {
            tc::mma_k_mixed(tm + TM4 + 64 * (c & 1), smem_addr(buf + B_A), 128, 0, 0, smem_addr(sm + S_S0), 0, 1,
                            8192, D, tc::idesc_f16(128, 64, 0, 1), 0);
            tc::commit(bar4);
        }
        // this chunk's measured max |S0|, the bound on |Delta| and its scale
        float smax;
        {
            const uint4 a = *reinterpret_cast<const uint4*>(s_smax + (c & 1) * 8);
            const uint4 b = *reinterpret_cast<const uint4*>(s_smax + (c & 1) * 8 + 4);
            smax = __uint_as_float(max(max(max(a.x, a.y), max(a.z, a.w)), max(max(b.x, b.y), max(b.z, b.w))));
        }
        const float dbound = fmaf(128.f * mw * pow2f(ew), smax, mu * pow2f(eu));
        const int ed = scale_exp(dbound, 12);
        if (row < 64) {
            // Delta_i 2^-Ed = U'_i 2^(eu-Ed) - (W' S0^T 2^-Es)_i 2^(ew+Es-Ed) and Delta~_i = gamma_i
            // Delta_i -> row i of this chunk's Delta image and of the Delta~ image, then MMA6
            float u[32];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                unpack8(*reinterpret_cast<const uint4*>(buf + B_U + tc::sw128_chunk(row, 4 * hf + q)), u + 8 * q);
            const float gm = sc[SC_GAM + row];
            const float fu = pow2f(eu - ed), fd = pow2f(ew + es - ed);
            const bool got4 = mbar_wait_bounded(bar4, (uint32_t)(c & 1), nullptr);
            if (!got4 && lane == 0) atomicOr(A.status, GDN_DEV_TIMEOUT);
            ok = got4;
            tc::fence_after_sync();
            float d[32];
            tc::ld32(tc::taddr(tm, warp, TM4 + 64 * (c & 1) + 32 * hf), d);
            tc::wait_ld();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float dl[8], dg[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    dl[e] = fmaf(u[8 * q + e], fu, -(d[8 * q + e] * fd));
                    dg[e] = gm * dl[e];
                }
                tc::st_chunk<Op>(sm + S_A6, row, 4 * hf + q, dg);
                tc::st_chunk<Op>(sm + S_DL + (c & 1) * 8192, row, 4 * hf + q, dl);
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            named_bar_sync(1, NT);  // the output warps only arrive
            // MMA6: X = K^T x Delta~ 2^-Ed, then this chunk's MMA7; the commits are issued even
            // when the products are not, so that every wait has its phase
            if (tid == 0) {
                tc::fence_after_sync();
                if (ok)
                    tc::mma_k_mixed(tm + TX, smem_addr(buf + B_K), 0, 1, 8192, smem_addr(sm + S_A6), 0, 1, 8192, CH,
                                    tc::idesc_f16(128, 64, 1, 1), 0);
                tc::commit(bar6);
                issue_mma7(c, ok);
            }
        } else {
            tc::fence_before_sync();
            named_bar_arrive(1, NT);
            // the chunk before last: finished rows out; the next sums barrier phase armed
            bool gotp = true;
            if (c >= 2) {
                gotp = finish_rows(c - 2);
                if (tid == PF && gotp) mbar_arrive_expect_tx(&peer_bar[c & 1], 256);
            }
            // the chunk before: its output rows (its MMA7, issued after its MMA6, is done with its
            // P slot, which PF refills; the next chunk's MMA4 and MMA7 overwrite these columns
            // only after the next full barrier)
            bool got7 = true;
            if (c >= 1) {
                got7 = complete_rows(c - 1, es_p, ed_p);
                if (tid == PF && got7 && c + 1 < nch) fetch_p(c + 1);
            }
            if ((!gotp || !got7) && lane == 0) atomicOr(A.status, GDN_DEV_TIMEOUT);
            ok = gotp && got7;
            // this chunk's gates, their exponent and e^{G_i} of the thread's row, read before this
            // buffer is refetched
#pragma unroll
            for (int q = 0; q < 4; ++q)
                gzn[q] = *reinterpret_cast<const uint4*>(buf + B_GZ + tc::sw128_chunk(orow, 4 * hf + q));
            ezn = __float_as_int(sc[SC_EZ + orow]);
            eg_n = sc[SC_EG + orow];
            named_bar_sync(2, NT / 2);  // the four output warps: sums of chunk c - 1 written, buffer read
            if (c >= 1) send_sums(c - 1);
        }
        const bool got6 = mbar_wait_bounded(bar6, (uint32_t)(c & 1), nullptr);
        if (!got6 && lane == 0) atomicOr(A.status, GDN_DEV_TIMEOUT);
        ok = ok && got6;
        tc::fence_after_sync();
        // this buffer is free (MMA4 and MMA6 are done, its rows were read before barriers 1
        // and 2): fetch the record two chunks ahead into it
        if (tid == PF && ok && c + 2 < nch) fetch_main(c + 2);
        egl_p = egl;
        smax_p = smax;
        dbound_p = dbound;
        es_p = es;
        ed_p = ed;
    }
    ok = __syncthreads_and(ok) != 0;
    if (ok) {
        // the last two chunks' output rows
        bool gotp = true, got7 = true;
        if (row >= 64) {
            if (nch >= 2) gotp = finish_rows(nch - 2);
            got7 = complete_rows(nch - 1, es_p, ed_p);
            named_bar_sync(2, NT / 2);
            send_sums(nch - 1);
            gotp = finish_rows(nch - 1) && gotp;
        }
        if ((!gotp || !got7) && lane == 0) atomicOr(A.status, GDN_DEV_TIMEOUT);
        ok = __syncthreads_and(gotp && got7) != 0;
    }

    if (ok) {
        // the final state S <- e^{G_last} S + 2^Ed X of the last chunk, in true units
        float v[32], x[32];
        tc::wait_st();
        tc::ld32(tc::taddr(tm, warp, TS + 32 * hf), v);
        tc::ld32(tc::taddr(tm, warp, TX + 32 * hf), x);
        tc::wait_ld();
        const float fx = pow2f(ed_p);
        const int dv0 = half * 64 + 32 * hf;
        if (slot_ok(Sg + (size_t)dv0 * D, (size_t)32 * D * sizeof(float))) {
#pragma unroll
            for (int e = 0; e < 32; ++e) Sg[(size_t)(dv0 + e) * D + row] = fmaf(fx, x[e], egl_p * v[e]);
        }
    }
    // every fetched copy must land, and the last MMA7 be done, before the CTA's shared and
    // tensor memory go away
    if (tid == 0 && mma7_issued > 0)
        mbar_wait_bounded(((mma7_issued - 1) & 1) ? bar7o : bar7e, (uint32_t)(((mma7_issued - 1) >> 1) & 1), nullptr);
    if (tid == PF) {
        for (int c = max(main_issued - 2, first_fetched); c < main_issued; ++c)
            mbar_wait_bounded(&full[c & 1], (uint32_t)((c >> 1) & 1), nullptr);
        for (int c = (p_issued > 2 ? p_issued - 2 : 0); c < p_issued; ++c)
            mbar_wait_bounded(&full_p[c & 1], (uint32_t)((c >> 1) & 1), nullptr);
    }
    tc::wait_st();
    sync_all();
    if (warp == 0) tc::dealloc(tm, 512);
    // Neither CTA leaves while the other may still write into its shared memory.  Both reach
    // this barrier: every wait above is bounded and a failed wait ends the loop in both CTAs.
    cluster_sync_all();
}

}  // namespace

size_t chunk_record_bytes(int hv, int hqk) { return (size_t)hv * REC_BYTES + (size_t)hqk * QK_BYTES; }

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
std::once_flag g_encode_once;

// [rows][width] bf16 rows at base, read as boxes of 128 channels x box_rows rows
cudaError_t encode_rows_map(CUtensorMap* m, const void* base, int width, int rows, int box_rows)
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode_tiled) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)width * 2};
    const cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)box_rows};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = g_encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                                      box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

template <typename TIn>
cudaError_t launch_chunk_prep(const PrefillArgs& A, cudaStream_t st)
{
    const int WM = A.W <= 4 ? 4 : 8;
    auto prep = WM == 4 ? chunk_prep_kernel<TIn, 4> : chunk_prep_kernel<TIn, 8>;
    cudaError_t e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P_SMEM);
    if (e != cudaSuccess) return e;
    PrepMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (sizeof(TIn) == 2) {  // bf16 rows come in by tensor copies
        const int Dq = A.hqk * D, Dv = A.hv * D;
        if ((e = encode_rows_map(&maps.q, A.q, Dq, A.T, CH + WM - 1)) != cudaSuccess) return e;
        if ((e = encode_rows_map(&maps.k, A.k, Dq, A.T, CH + WM - 1)) != cudaSuccess) return e;
        if ((e = encode_rows_map(&maps.v, A.v, Dv, A.T, CH + WM - 1)) != cudaSuccess) return e;
    }
    // the segment's records that this call can have (a bound: the exact count is on the device)
    const int recs = std::min(A.seg_hi, prefill_call_chunks(A.T, A.n)) - A.seg_lo;
    if (recs <= 0) return cudaSuccess;
    prep<<<recs * A.hqk, NT, P_SMEM, st>>>(A, maps);
    return cudaGetLastError();
}

template <typename TIn, typename TOut>
cudaError_t launch_chunk_state(const PrefillArgs& A, cudaStream_t st)
{
    auto state = chunk_state_kernel<TIn, TOut>;
    cudaError_t e = cudaFuncSetAttribute(state, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S_SMEM);
    if (e != cudaSuccess) return e;
    // one CTA per (sequence, v-head, d_v half); the two halves form a cluster
    // one segment of several: at most one sequence per record of the segment has records in it
    const int seqs = A.seg_hi == INT_MAX ? A.n : std::min(A.n, A.seg_hi - A.seg_lo);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(seqs * A.hv * 2));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = S_SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, state, A);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template cudaError_t launch_chunk_prep<float>(const PrefillArgs&, cudaStream_t);
template cudaError_t launch_chunk_prep<__nv_bfloat16>(const PrefillArgs&, cudaStream_t);
template cudaError_t launch_chunk_state<float, float>(const PrefillArgs&, cudaStream_t);
template cudaError_t launch_chunk_state<float, __nv_bfloat16>(const PrefillArgs&, cudaStream_t);
template cudaError_t launch_chunk_state<__nv_bfloat16, float>(const PrefillArgs&, cudaStream_t);
template cudaError_t launch_chunk_state<__nv_bfloat16, __nv_bfloat16>(const PrefillArgs&, cudaStream_t);

}  // namespace gdn
