// gdn_prefill.cu -- varlen prefill of one GDN layer into the slot pool.
//
// The prefill branch of the System Design page's "GDN Kernel Dispatch Detail": conv1d,
// L2norm, the gated delta rule over the prompt starting from the sequence's state, then
// "Update temporal_state" (the final S and conv buffer land in the slot, where the
// decode kernel reads them) and the gated RMSNorm.
//
// Kernels (all on the caller's stream, no host synchronisation):
//   1. validate   one CTA: cu_seqlens 0-based, non-decreasing, ending at total_tokens;
//                 slot ids allocated and distinct.  The verdict gates every later kernel.
// d_k = d_v = 128 (the chunked tensor-core path, gdn_chunk.cu):
//   2. chunk pre-pass  conv, norms, gates and the chunk-local products, one CTA per
//                 (chunk, q/k head) taking the q/k head's v-heads in turn; it reads the
//                 slots' old conv buffers
//   3. chunk state pass  one CTA per (sequence, v-head, d_v half), the two halves a
//                 cluster: output, final state, and the slot's conv buffer advanced to the
//                 last W-1 raw inputs (the pre-pass has read the old rows by then)
// d < 128:
//   2. prep       one CTA per token: conv + SiLU over all C channels (the left context
//                 before a sequence's first token comes from its slot's conv buffer),
//                 L2 scales of q and k, k.q per q/k head, gates per v-head.
//   3. conv_tail  as above
//   4. with a chunk length set in the shape (8, 16, 32 or 64): chunk_small_kernel
//                 (gdn_chunk_small.cu), the chunked form in fp32, one CTA per (sequence,
//                 v-head); with chunk = 0: recurrent, one CTA per (sequence, v-head, row
//                 tile of S), the tile of S in registers across the whole sequence, token
//                 after token (measured faster at these head sizes).
//   5. epilogue   gated RMSNorm per (token, v-head).
// The recurrent kernel and kernels 2 and 5 use the decode kernel's arithmetic in the same
// order, so with chunk = 0 a prefill of L tokens equals L decode steps bit for bit.
#include <algorithm>
#include <climits>

#include "gdn_internal.cuh"

namespace gdn {

namespace {

// In-place exclusive prefix sum of a[0 .. n) by one CTA of 256 threads (every thread calls it).
__device__ void block_exclusive_scan(int* a, int n)
{
    __shared__ int part[256];
    const int per = (n + 255) / 256, lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += a[i];
    part[threadIdx.x] = sum;
    __syncthreads();
    for (int off = 1; off < 256; off <<= 1) {  // inclusive scan of the 256 partial sums
        const int v = threadIdx.x >= (unsigned)off ? part[threadIdx.x - off] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    int run = threadIdx.x ? part[threadIdx.x - 1] : 0;
    for (int i = lo; i < hi; ++i) {
        const int v = a[i];
        a[i] = run;
        run += v;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(256) validate_kernel(PrefillArgs A)
{
    __shared__ int bad;
    if (A.gate && *A.gate) {  // a mixed step whose parts overlap: nothing runs
        if (threadIdx.x == 0) *A.ws.valid = 0;
        return;
    }
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    if (threadIdx.x == 0 && (A.cu[0] != 0 || A.cu[A.n] != A.T)) atomicOr(&bad, 1);
    // Up to kPairwiseSeqs sequences the ids are compared pairwise and ranked by counting; more take
    // a mark per slot (mark[id], zero between calls) and a histogram of the lengths, in O(n + T).
    const bool many = A.n > kPairwiseSeqs;
    for (int s = threadIdx.x; s < A.n; s += blockDim.x) {
        if (A.cu[s + 1] < A.cu[s]) atomicOr(&bad, 1);
        const int id = A.ids[s];
        bool ok = id >= 0 && id < A.num_slots && A.live[id];
        if (!many) {
            for (int j = 0; ok && j < s; ++j) ok = A.ids[j] != id;
        } else if (ok && atomicExch(A.mark + id, 1) != 0) {
            ok = false;  // a second sequence on this slot
        }
        if (!ok) atomicOr(&bad, 2);
    }
    __syncthreads();
    if (many)
        for (int s = threadIdx.x; s < A.n; s += blockDim.x) {
            const int id = A.ids[s];
            if (id >= 0 && id < A.num_slots) A.mark[id] = 0;
        }
    if (bad == 0) {
        // rank by length, longest first: long sequences start in the first wave
        if (!many) {
            for (int s = threadIdx.x; s < A.n; s += blockDim.x) {  // ties by index
                const int len = A.cu[s + 1] - A.cu[s];
                int rank = 0;
                for (int j = 0; j < A.n; ++j) {
                    const int lj = A.cu[j + 1] - A.cu[j];
                    rank += (lj > len) || (lj == len && j < s);
                }
                A.ws.order[rank] = s;
            }
        } else {
            // ties in arrival order: which of two equal lengths comes first changes no result
            int* cnt = A.ws.lcnt;  // [T + 2]: sequences of each length, then of shorter lengths
            int* tie = A.ws.ltie;  // [T + 2]
            for (int l = threadIdx.x; l < A.T + 2; l += blockDim.x) {
                cnt[l] = 0;
                tie[l] = 0;
            }
            __syncthreads();
            for (int s = threadIdx.x; s < A.n; s += blockDim.x) atomicAdd(cnt + (A.cu[s + 1] - A.cu[s]), 1);
            __syncthreads();
            block_exclusive_scan(cnt, A.T + 2);
            for (int s = threadIdx.x; s < A.n; s += blockDim.x) {
                const int len = A.cu[s + 1] - A.cu[s];
                A.ws.order[A.n - cnt[len + 1] + atomicAdd(tie + len, 1)] = s;  // longer ones first
            }
        }
        if (A.D == 128) {  // the chunked path's record numbering (chunk-index-major)
            __syncthreads();
            const int nc = (A.cu[A.ws.order[0] + 1] - A.cu[A.ws.order[0]] + 63) / 64;  // longest sequence
            int* cnt = A.ws.ctmp;  // [nc + 1]: sequences with exactly v chunks, then the prefix sums
            for (int v = threadIdx.x; v <= nc; v += blockDim.x) cnt[v] = 0;
            __syncthreads();
            for (int s = threadIdx.x; s < A.n; s += blockDim.x) atomicAdd(&cnt[(A.cu[s + 1] - A.cu[s] + 63) / 64], 1);
            __syncthreads();
            block_exclusive_scan(cnt, nc + 1);  // cnt[v] = sequences with fewer than v chunks
            // sequences with more than c chunks, then the records of chunk index < c
            for (int c = threadIdx.x; c <= nc; c += blockDim.x) A.ws.coff[c] = c < nc ? A.n - cnt[c + 1] : 0;
            __syncthreads();
            block_exclusive_scan(A.ws.coff, nc + 1);
            const int total = A.ws.coff[nc];
            for (int r = threadIdx.x; r < total; r += blockDim.x) {
                int lo = 0, hi = nc;  // the largest c with coff[c] <= r
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (A.ws.coff[mid] <= r) lo = mid;
                    else hi = mid;
                }
                A.ws.rec_cp[r] = make_int2(lo, r - A.ws.coff[lo]);
            }
            if (threadIdx.x == 0) A.ws.valid[1] = nc;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        *A.ws.valid = bad == 0;
        if (bad & 1) atomicOr(A.status, GDN_DEV_BAD_SEQLENS);
        if (bad & 2) atomicOr(A.status, GDN_DEV_BAD_SLOT_ID);
    }
}

// sequence owning packed token t: the largest s with cu[s] <= t
__device__ __forceinline__ int seq_of(const int* cu, int n, int t)
{
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= t) lo = mid;
        else hi = mid;
    }
    return lo;
}

template <typename TIn>
__device__ __forceinline__ TIn channel_input(const PrefillArgs& A, int t, int c)
{
    const int Dq = A.hqk * A.D;
    if (c < Dq) return static_cast<const TIn*>(A.q)[(size_t)t * Dq + c];
    if (c < 2 * Dq) return static_cast<const TIn*>(A.k)[(size_t)t * Dq + (c - Dq)];
    return static_cast<const TIn*>(A.v)[(size_t)t * (A.hv * A.D) + (c - 2 * Dq)];
}

template <typename TIn>
__global__ void __launch_bounds__(256) prep_kernel(PrefillArgs A)
{
    extern __shared__ float y[];  // [C] conv + SiLU of this token, then [3*Hqk] scales and dots
    if (!*A.ws.valid) return;
    const int t = blockIdx.x;
    const int s = seq_of(A.cu, A.n, t);
    const int pos = t - A.cu[s];
    const TIn* cbuf =
        reinterpret_cast<const TIn*>(A.base + ((uint64_t)A.ids[s] * A.num_layers + A.layer) * A.slot_bytes + A.state_bytes);
    const int W = A.W, C = A.C, D = A.D;
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
        const float* w = A.conv_w + (size_t)c * W;
        float acc = 0.0f;
        for (int j = 0; j < W; ++j) {
            const int pp = pos - (W - 1) + j;
            const TIn x = pp >= 0 ? channel_input<TIn>(A, t - (W - 1) + j, c) : cbuf[(size_t)(W - 1 + pp) * C + c];
            acc = fmaf(w[j], to_f(x), acc);
        }
        y[c] = silu_f(acc);
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    const int Dq = A.hqk * D;
    float* scale = y + C;            // [2*Hqk] q scales, then k scales
    float* dots = scale + 2 * A.hqk;  // [Hqk] q.k before scaling
    for (int hh = warp; hh < 3 * A.hqk; hh += nwarps) {
        if (hh < 2 * A.hqk) {  // q heads then k heads: contiguous channel blocks
            const float ss = warp_dot(y + hh * D, y + hh * D, D, lane);
            if (lane == 0) scale[hh] = hh < A.hqk ? q_scale(ss, A.l2_eps, D) : k_scale(ss, A.l2_eps);
        } else {
            const int hk = hh - 2 * A.hqk;
            const float d = warp_dot(y + hk * D, y + Dq + hk * D, D, lane);
            if (lane == 0) dots[hk] = d;
        }
    }
    for (int h = threadIdx.x; h < A.hv; h += blockDim.x) {
        const TIn* ain = static_cast<const TIn*>(A.a);
        const TIn* bin = static_cast<const TIn*>(A.b);
        A.ws.g[(size_t)t * A.hv + h] = log_decay(A.A_log[h], to_f(ain[(size_t)t * A.hv + h]), A.dt_bias[h]);
        A.ws.beta[(size_t)t * A.hv + h] = sigmoid_f(to_f(bin[(size_t)t * A.hv + h]));
    }
    __syncthreads();
    for (int hk = threadIdx.x; hk < A.hqk; hk += blockDim.x)
        A.kq[(size_t)t * A.hqk + hk] = dots[hk] * scale[hk] * scale[A.hqk + hk];
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
        if (c < Dq) A.ws.qh[(size_t)t * Dq + c] = y[c] * scale[c / D];
        else if (c < 2 * Dq) A.ws.kh[(size_t)t * Dq + (c - Dq)] = y[c] * scale[c / D];
        else A.ws.vc[(size_t)t * (A.hv * D) + (c - 2 * Dq)] = y[c];
    }
}

template <typename TIn>
__global__ void __launch_bounds__(256) conv_tail_kernel(PrefillArgs A)
{
    if (!*A.ws.valid) return;
    const int s = blockIdx.x;
    const int t0 = A.cu[s], L = A.cu[s + 1] - t0;
    if (L == 0) return;
    TIn* cbuf = reinterpret_cast<TIn*>(A.base + ((uint64_t)A.ids[s] * A.num_layers + A.layer) * A.slot_bytes +
                                       A.state_bytes);
    const int W = A.W, C = A.C;
    for (int c = blockIdx.y * blockDim.x + threadIdx.x; c < C; c += gridDim.y * blockDim.x) {
        TIn old[8];
        for (int j = 0; j < W - 1; ++j) old[j] = cbuf[(size_t)j * C + c];
        for (int i = 0; i < W - 1; ++i) {
            const int pp = L - (W - 1) + i;
            cbuf[(size_t)i * C + c] = pp >= 0 ? channel_input<TIn>(A, t0 + pp, c) : old[W - 1 + pp];
        }
    }
}

// S row tile of one (sequence, v-head): 8 warps x RPW rows, LPR lanes per row.
template <int D>
__global__ void __launch_bounds__(256) recurrent_kernel(PrefillArgs A)
{
    constexpr int LPR = D / 16, RPW = 32 / LPR, ROWS = 8 * RPW < D ? 8 * RPW : D;
    if (!*A.ws.valid) return;
    const int s = blockIdx.x, h = blockIdx.y, tile = blockIdx.z;
    const int t0 = A.cu[s], t1 = A.cu[s + 1];
    if (t0 == t1) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rsub = lane / LPR, cl = lane % LPR;
    const int lr = warp * RPW + rsub;
    const int i = tile * ROWS + lr;
    const bool rv = lr < ROWS;
    const int hk = h / A.r, Dq = A.hqk * D, Dv = A.hv * D;
    float* S = reinterpret_cast<float*>(A.base + ((uint64_t)A.ids[s] * A.num_layers + A.layer) * A.slot_bytes) +
               (size_t)h * D * D;

    float sv[16];
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
        float4 x = rv ? *reinterpret_cast<const float4*>(S + (size_t)i * D + row_col<LPR>(j, cl))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        sv[j] = x.x;
        sv[j + 1] = x.y;
        sv[j + 2] = x.z;
        sv[j + 3] = x.w;
    }
    // software pipeline: the next token's operands are loaded while this token is processed
    float kr[16], qr[16], nk[16], nq[16];
    float v_i, g, be, kq, nv = 0.f, ng = 0.f, nb = 0.f, nkq = 0.f;
    auto load = [&](int t, float (&kk)[16], float (&qq)[16], float& vv, float& gg, float& bb, float& dot) {
        const float* kp = A.ws.kh + (size_t)t * Dq + hk * D;
        const float* qp = A.ws.qh + (size_t)t * Dq + hk * D;
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
            const float4 a4 = *reinterpret_cast<const float4*>(kp + row_col<LPR>(j, cl));
            const float4 b4 = *reinterpret_cast<const float4*>(qp + row_col<LPR>(j, cl));
            kk[j] = a4.x; kk[j + 1] = a4.y; kk[j + 2] = a4.z; kk[j + 3] = a4.w;
            qq[j] = b4.x; qq[j + 1] = b4.y; qq[j + 2] = b4.z; qq[j + 3] = b4.w;
        }
        vv = rv ? A.ws.vc[(size_t)t * Dv + (size_t)h * D + i] : 0.f;
        gg = A.ws.g[(size_t)t * A.hv + h];
        bb = A.ws.beta[(size_t)t * A.hv + h];
        dot = A.kq[(size_t)t * A.hqk + hk];
    };
    load(t0, kr, qr, v_i, g, be, kq);
    for (int t = t0; t < t1; ++t) {
        if (t + 1 < t1) load(t + 1, nk, nq, nv, ng, nb, nkq);
        const float o = row_update<LPR>(sv, kr, qr, expf(g), be, v_i, kq);
        if (rv && cl == 0) A.ws.o[(size_t)t * Dv + (size_t)h * D + i] = o;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            kr[j] = nk[j];
            qr[j] = nq[j];
        }
        v_i = nv;
        g = ng;
        be = nb;
        kq = nkq;
    }
    if (rv) {
#pragma unroll
        for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4*>(S + (size_t)i * D + row_col<LPR>(j, cl)) =
                make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
    }
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(256) epilogue_kernel(PrefillArgs A)
{
    if (!*A.ws.valid) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = blockIdx.x * 8 + warp;  // (token, v-head)
    if (pair >= A.T * A.hv) return;
    const int t = pair / A.hv, h = pair % A.hv, D = A.D;
    const size_t base = (size_t)t * A.hv * D + (size_t)h * D;
    const float* o = A.ws.o + base;
    const float rs = rms_scale(warp_dot(o, o, D, lane), A.norm_eps, D);
    const TIn* zin = static_cast<const TIn*>(A.z);
    TOut* out = static_cast<TOut*>(A.out);
    for (int i = lane; i < D; i += 32)
        out[base + i] = from_f<TOut>(o[i] * rs * A.norm_w[i] * silu_f(to_f(zin[base + i])));
}

// The chunked path (d = 128) as one pre-pass / state-pass pair per segment of records (one pair
// unless the call has more chunks than the workspace holds); a segment's state pass continues from
// the states the previous one left in the slots.  With the pool's segment stream, the workspace is
// split in two halves: the state pass of segment g runs on that stream while the caller's stream
// runs the pre-pass of segment g + 1 into the other half (its records are independent of every
// state; the conv buffers it reads belong to sequences that start in it, which no earlier state
// pass touches), so one long prompt's state chain no longer leaves the other SMs idle.
template <typename TIn, typename TOut>
cudaError_t run_chunked(const PrefillArgs& A, cudaStream_t st, const SegStreams* ss, cudaEvent_t prep_done,
                        bool* split)
{
    const int cap = std::min(A.ws.chunk_cap, kPrefillMaxRecords);
    const bool two = ss && ss->side && cap >= 2 && prefill_segments(A.T, A.n, cap) > 1;
    const int seg = two ? cap / 2 : cap;
    const int nseg = prefill_segments(A.T, A.n, seg);
    PrefillArgs S = A;
    cudaError_t e = cudaSuccess;
    if (prep_done && ss && ss->side && nseg == 1) {  // a mixed step's prefill: the state pass on the side
        S.seg_lo = 0;
        S.seg_hi = INT_MAX;
        e = launch_chunk_prep<TIn>(S, st);
        if (e == cudaSuccess) e = cudaEventRecord(prep_done, st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->side, prep_done, 0);
        if (e == cudaSuccess) e = launch_chunk_state<TIn, TOut>(S, ss->side);
        if (e == cudaSuccess) e = cudaEventRecord(ss->state[0], ss->side);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ss->state[0], 0);
        if (split) *split = e == cudaSuccess;
        return e;
    }
    for (int g = 0; g < nseg && e == cudaSuccess; ++g) {
        S.seg_lo = g * seg;
        S.seg_hi = nseg == 1 ? INT_MAX : S.seg_lo + seg;  // INT_MAX: every record of the call
        if (!two) {
            e = launch_chunk_prep<TIn>(S, st);  // reads the conv buffers ...
            if (e == cudaSuccess) e = launch_chunk_state<TIn, TOut>(S, st);  // ... which the state pass advances
            continue;
        }
        const int half = g & 1;
        S.ws.chunk_cap = seg;
        S.ws.rec = A.ws.rec + (size_t)half * seg * chunk_record_bytes(A.hv, 0);
        S.ws.kimg = A.ws.kimg + (size_t)half * seg * chunk_record_bytes(0, A.hqk);
        if (g >= 2) e = cudaStreamWaitEvent(st, ss->state[half], 0);  // segment g - 2 has read this half
        if (e == cudaSuccess) e = launch_chunk_prep<TIn>(S, st);
        if (e == cudaSuccess) e = cudaEventRecord(ss->prep[half], st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->side, ss->prep[half], 0);
        if (e == cudaSuccess) e = launch_chunk_state<TIn, TOut>(S, ss->side);
        if (e == cudaSuccess) e = cudaEventRecord(ss->state[half], ss->side);
    }
    // join: the caller's stream continues after the last state pass
    if (two && e == cudaSuccess) e = cudaStreamWaitEvent(st, ss->state[(nseg - 1) & 1], 0);
    return e;
}

template <typename TIn, typename TOut>
cudaError_t run(const PrefillArgs& A, cudaStream_t st, const SegStreams* ss, cudaEvent_t prep_done = nullptr,
                bool* split = nullptr)
{
    validate_kernel<<<1, 256, 0, st>>>(A);
    if (A.T > 0 && A.D == 128) return run_chunked<TIn, TOut>(A, st, ss, prep_done, split);
    if (A.T > 0) {
        const size_t smem = (size_t)(A.C + 3 * A.hqk) * sizeof(float);
        if (smem > 48 * 1024) {
            cudaError_t e =
                cudaFuncSetAttribute(prep_kernel<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        prep_kernel<TIn><<<A.T, 256, smem, st>>>(A);
    }
    conv_tail_kernel<TIn><<<dim3(A.n, (A.C + 255) / 256), 256, 0, st>>>(A);
    if (A.T > 0) {
        if (A.chunk > 0) {  // the chunked form, with the chunk length the caller asked for
            cudaError_t e = launch_chunk_small(A, A.chunk, st);
            if (e != cudaSuccess) return e;
        } else {  // the token-recurrent kernel (faster at these head sizes)
            const int rows = std::min(A.D, 8 * (32 / (A.D / 16)));
            dim3 grid(A.n, A.hv, A.D / rows);
            switch (A.D) {
                case 16: recurrent_kernel<16><<<grid, 256, 0, st>>>(A); break;
                case 32: recurrent_kernel<32><<<grid, 256, 0, st>>>(A); break;
                case 64: recurrent_kernel<64><<<grid, 256, 0, st>>>(A); break;
                default: return cudaErrorInvalidValue;
            }
        }
        const int pairs = A.T * A.hv;
        epilogue_kernel<TIn, TOut><<<(pairs + 7) / 8, 256, 0, st>>>(A);
    }
    return cudaGetLastError();
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

size_t prefill_workspace_bytes(const gdn_shape& s, int T, int chunk_cap)
{
    const size_t Dq = (size_t)s.hqk * s.dk, Dv = (size_t)s.hv * s.dv;
    size_t b = 0;
    if (!prefill_chunked(s)) {
        b += align256((size_t)T * Dq * 4) * 2;        // qh, kh
        b += align256((size_t)T * Dv * 4) * 2;        // vc, o
        b += align256((size_t)T * s.hqk * 4);         // k.q
        b += align256((size_t)T * s.hv * 4) * 2;      // g, beta
    }
    b += align256((size_t)prefill_max_seqs(T) * 4);   // length order
    b += align256((size_t)(T + 2) * 4) * 2;             // length histogram, ties (many sequences)
    if (prefill_chunked(s)) {
        b += align256((size_t)((T + 63) / 64 + 2) * 4) * 2;  // coff, ctmp
        b += align256((size_t)prefill_call_chunks(T, prefill_max_seqs(T)) * 8);  // rec_cp
    }
    b += (size_t)chunk_cap * chunk_record_bytes(s.hv, s.hqk);  // chunk records (multiple of 256)
    b += 256;                                         // valid flag
    return b;
}

bool prefill_workspace_carve(PrefillWorkspace& ws, const gdn_shape& s, int T, int chunk_cap)
{
    const size_t Dq = (size_t)s.hqk * s.dk, Dv = (size_t)s.hv * s.dv;
    char* p = static_cast<char*>(ws.base);
    auto take = [&](size_t bytes) {
        char* r = p;
        p += align256(bytes);
        return r;
    };
    if (!prefill_chunked(s)) {
        ws.qh = reinterpret_cast<float*>(take((size_t)T * Dq * 4));
        ws.kh = reinterpret_cast<float*>(take((size_t)T * Dq * 4));
        ws.vc = reinterpret_cast<float*>(take((size_t)T * Dv * 4));
        ws.o = reinterpret_cast<float*>(take((size_t)T * Dv * 4));
        ws.kq = reinterpret_cast<float*>(take((size_t)T * s.hqk * 4));
        ws.g = reinterpret_cast<float*>(take((size_t)T * s.hv * 4));
        ws.beta = reinterpret_cast<float*>(take((size_t)T * s.hv * 4));
    }
    ws.order = reinterpret_cast<int*>(take((size_t)prefill_max_seqs(T) * 4));
    ws.lcnt = reinterpret_cast<int*>(take((size_t)(T + 2) * 4));
    ws.ltie = reinterpret_cast<int*>(take((size_t)(T + 2) * 4));
    if (prefill_chunked(s)) {
        ws.coff = reinterpret_cast<int*>(take((size_t)((T + 63) / 64 + 2) * 4));
        ws.ctmp = reinterpret_cast<int*>(take((size_t)((T + 63) / 64 + 2) * 4));
        ws.rec_cp = reinterpret_cast<int2*>(take((size_t)prefill_call_chunks(T, prefill_max_seqs(T)) * 8));
    }
    ws.rec = reinterpret_cast<unsigned char*>(take((size_t)chunk_cap * chunk_record_bytes(s.hv, 0)));
    ws.kimg = reinterpret_cast<unsigned char*>(take((size_t)chunk_cap * chunk_record_bytes(0, s.hqk)));
    ws.chunk_cap = chunk_cap;
    ws.valid = reinterpret_cast<int*>(take(256));
    // the parts must fit the bytes prefill_workspace_bytes sized
    return (size_t)(p - static_cast<char*>(ws.base)) <= ws.bytes;
}

cudaError_t launch_prefill(const Pool& P, int layer, const int* cu_seqlens, const int* slot_ids, int n_seqs,
                           int total_tokens, const void* q, const void* k, const void* v, const void* a,
                           const void* b, const void* z, void* out, cudaStream_t st, const int* gate,
                           cudaEvent_t prep_done, bool* split)
{
    if (split) *split = false;
    const LayerParams& L = P.params[(size_t)layer];
    PrefillArgs A;
    A.cu = cu_seqlens;
    A.ids = slot_ids;
    A.n = n_seqs;
    A.T = total_tokens;
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
    A.base = P.base;
    A.slot_bytes = P.slot_bytes;
    A.state_bytes = (uint32_t)P.state_bytes;
    A.num_layers = P.num_layers;
    A.layer = layer;
    A.num_slots = P.num_slots;
    A.live = P.live_dev;
    A.mark = P.mark_dev;
    A.status = P.status_dev;
    A.hqk = P.shape.hqk;
    A.hv = P.shape.hv;
    A.r = P.r;
    A.D = P.shape.dk;
    A.W = P.shape.conv_w;
    A.C = P.C;
    A.l2_eps = P.shape.l2_eps;
    A.norm_eps = P.shape.norm_eps;
    A.ws = P.ws;
    A.kq = P.ws.kq;
    A.gate = gate;
    A.chunk = P.shape.chunk;
    A.stall_fetch = (P.debug_flags >> 1) & 1;
    const bool in_bf16 = P.shape.io_dtype == 1, out_bf16 = P.shape.out_dtype == 1;
    if (in_bf16 && out_bf16) return run<__nv_bfloat16, __nv_bfloat16>(A, st, &P.seg, prep_done, split);
    if (in_bf16) return run<__nv_bfloat16, float>(A, st, &P.seg, prep_done, split);
    if (out_bf16) return run<float, __nv_bfloat16>(A, st, &P.seg, prep_done, split);
    return run<float, float>(A, st, &P.seg, prep_done, split);
}

cudaError_t create_seg_streams(SegStreams* ss)
{
    int least = 0, greatest = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&ss->side, cudaStreamNonBlocking, greatest);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&ss->prep[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss->state[i], cudaEventDisableTiming);
    }
    return e;
}

void destroy_seg_streams(SegStreams* ss)
{
    for (int i = 0; i < 2; ++i) {
        if (ss->prep[i]) cudaEventDestroy(ss->prep[i]);
        if (ss->state[i]) cudaEventDestroy(ss->state[i]);
        ss->prep[i] = ss->state[i] = nullptr;
    }
    if (ss->side) cudaStreamDestroy(ss->side);
    ss->side = nullptr;
}

}  // namespace gdn

// ---------------------------------------------------------------------------------------
// Allocation-free varlen prefill.
//
// For callers that cannot call cudaMalloc (for example code running where the device heap
// belongs to someone else, or inside a region that must not allocate), this entry point
// runs the same prefill kernels as gdn_prefill_varlen, but takes the scratch it needs
// from one fixed static device array instead of a pool's workspace, and takes the state
// slots from memory the caller already owns.  It allocates nothing.
namespace gdn {
namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB, held by every GPU that loads libgdn

// Host code must not use this name as a device address: the address comes from
// cudaGetSymbolAddress, once per device (see static_scratch_address).
static __device__ __align__(256) unsigned char g_prefill_scratch[kStaticScratchBytes];

__global__ void fill_ones_kernel(unsigned char* p, int n)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = 1;
}

std::mutex g_scratch_mu;
constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_prefill_scratch on the current device, looked up on the first call per device.
cudaError_t static_scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_prefill_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

}  // namespace gdn

extern "C" int gdn_prefill_varlen_noalloc(const gdn_shape* shape, const float* conv_w, const float* A_log,
                                          const float* dt_bias, const float* norm_w, void* states_dev, int num_slots,
                                          const int* cu_seqlens_dev, const int* slot_ids_dev, int n_seqs,
                                          int total_tokens, const void* q, const void* k, const void* v,
                                          const void* a, const void* b, const void* z, void* out,
                                          unsigned int* status_dev, void* stream)
{
    using namespace gdn;
    if (!shape || !conv_w || !A_log || !dt_bias || !norm_w || !states_dev || num_slots <= 0) return GDN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(states_dev) % 256 != 0) return GDN_ERR_INVALID_ARG;
    if (n_seqs < 0 || total_tokens < 0) return GDN_ERR_INVALID_ARG;
    if (n_seqs == 0) return total_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (!cu_seqlens_dev || !slot_ids_dev) return GDN_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !a || !b || !z || !out)) return GDN_ERR_INVALID_ARG;
    if (total_tokens > 0 && !rows_aligned16(q, k, v, z, out)) return GDN_ERR_INVALID_ARG;
    const gdn_shape& s = *shape;
    if (s.hqk <= 0 || s.hv <= 0 || s.hv % s.hqk != 0 || s.conv_w < 1 || s.conv_w > 8) return GDN_ERR_INVALID_ARG;
    if (s.io_dtype < 0 || s.io_dtype > 1 || s.out_dtype < 0 || s.out_dtype > 1) return GDN_ERR_INVALID_ARG;
    if (!(s.l2_eps >= 0.0f) || !(s.norm_eps >= 0.0f)) return GDN_ERR_INVALID_ARG;
    if (s.dk != s.dv || (s.dk != 16 && s.dk != 32 && s.dk != 64 && s.dk != 128)) return GDN_ERR_UNSUPPORTED_SHAPE;

    if (n_seqs > prefill_max_seqs(total_tokens)) return GDN_ERR_UNSUPPORTED_SHAPE;
    // everything the call needs must fit in the static scratch: workspace, live flags, id marks,
    // status word
    const int chunk_cap = prefill_chunked(s) ? prefill_call_chunks(total_tokens, n_seqs) : 0;
    const size_t ws_bytes = prefill_workspace_bytes(s, total_tokens, chunk_cap);
    const size_t live_bytes = align256((size_t)num_slots);
    const size_t mark_bytes = align256((size_t)num_slots * sizeof(int));
    if (ws_bytes + live_bytes + mark_bytes + 256 > kStaticScratchBytes) return GDN_ERR_UNSUPPORTED_SHAPE;

    void* scratch = nullptr;
    if (static_scratch_address(&scratch) != cudaSuccess) return GDN_ERR_CUDA;
    PrefillWorkspace ws;
    ws.base = scratch;
    ws.bytes = ws_bytes;
    if (!prefill_workspace_carve(ws, s, total_tokens, chunk_cap)) return GDN_ERR_CUDA;
    unsigned char* live = static_cast<unsigned char*>(scratch) + ws_bytes;
    int* mark = reinterpret_cast<int*>(live + live_bytes);
    unsigned int* status = status_dev ? status_dev : reinterpret_cast<unsigned int*>(live + live_bytes + mark_bytes);

    const int C = 2 * s.hqk * s.dk + s.hv * s.dv;
    const int io_size = s.io_dtype == 1 ? 2 : 4;
    const size_t state_bytes = (size_t)s.hv * s.dv * s.dk * sizeof(float);
    const size_t slot_bytes = (state_bytes + (size_t)(s.conv_w - 1) * C * io_size + 255) / 256 * 256;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    fill_ones_kernel<<<(num_slots + 255) / 256, 256, 0, st>>>(live, num_slots);
    // the marks must start at zero, and this call's carve may put them where other data was
    if (cudaMemsetAsync(mark, 0, (size_t)num_slots * sizeof(int), st) != cudaSuccess) return GDN_ERR_CUDA;

    PrefillArgs A;
    A.cu = cu_seqlens_dev;
    A.ids = slot_ids_dev;
    A.n = n_seqs;
    A.T = total_tokens;
    A.q = q;
    A.k = k;
    A.v = v;
    A.a = a;
    A.b = b;
    A.z = z;
    A.out = out;
    A.conv_w = conv_w;
    A.A_log = A_log;
    A.dt_bias = dt_bias;
    A.norm_w = norm_w;
    A.base = static_cast<char*>(states_dev);
    A.slot_bytes = slot_bytes;
    A.state_bytes = (uint32_t)state_bytes;
    A.num_layers = 1;
    A.layer = 0;
    A.num_slots = num_slots;
    A.live = live;
    A.mark = mark;
    A.status = status;
    A.hqk = s.hqk;
    A.hv = s.hv;
    A.r = s.hv / s.hqk;
    A.D = s.dk;
    A.W = s.conv_w;
    A.C = C;
    A.l2_eps = s.l2_eps;
    A.norm_eps = s.norm_eps;
    A.ws = ws;
    A.kq = ws.kq;
    A.gate = nullptr;
    A.chunk = s.chunk;
    cudaError_t e;
    const bool in_bf16 = s.io_dtype == 1, out_bf16 = s.out_dtype == 1;
    if (in_bf16 && out_bf16) e = run<__nv_bfloat16, __nv_bfloat16>(A, st, nullptr);
    else if (in_bf16) e = run<__nv_bfloat16, float>(A, st, nullptr);
    else if (out_bf16) e = run<float, __nv_bfloat16>(A, st, nullptr);
    else e = run<float, float>(A, st, nullptr);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

