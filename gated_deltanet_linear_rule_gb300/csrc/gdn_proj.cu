// gdn_proj.cu -- the projections around a GDN layer on tcgen05 tensor cores: the fused input
// projection X -> [q | k | v | z | a | b] and the output projection O -> Y.
//
// The pages' layer tree ("qwen3_5.py: Qwen3_5ForCausalLM.forward()", the GatedDeltaNet layer)
// opens the layer with the projections in_proj_qkv, in_proj_z, in_proj_b, in_proj_a and closes
// it with out_proj.  Here the four input projections are one GEMM whose weight rows are the
// concatenation [W_q; W_k; W_v; W_z; W_a; W_b] (each [out][hidden], row-major), and the epilogue
// writes every output column straight into the buffer and layout the layer's calls read (q, k,
// v, z, a, b, each [T][width] row-major), so no split or copy follows.  out_proj is the same
// kernel with one output segment.
//
// C[M][N] = A[M][K] . B[N][K]^T, bf16 operands, fp32 accumulation in tensor memory, bf16 out.
// All kernels are warp-specialised: warp 0 streams 64-wide K slices of A and B by 2-D tensor
// copies with the 128-byte swizzle (which lays them out as the MMA's K-major operand tiles) into
// a stage ring; warp 1 issues the MMAs (K = 16 per instruction) into TMEM, releasing each stage
// by a commit; warps 2-5 read the accumulator (one TMEM lane quarter each, warp w -> lanes
// 32 (w % 4) ..), round to bf16 and store 16 B at a time.  The persistent kernels take tiles
// t = block (or pair) index, + grid size, ..., N tiles fastest, with two 256-column
// accumulators so that a tile's epilogue overlaps the next tile's products:
//  - proj_kernel: one CTA per 128 x 256 tile (cta_group::1, 4 stages of 48 KiB).
//  - proj_pair_kernel<BNP>: clusters of two CTAs share 256 x BNP tiles (cta_group::2, M = 256;
//    BNP = 256, or 192 when that puts more SMs to work in a single round): each CTA holds 128
//    rows of A and BNP / 2 rows of B per K slice (6 stages) and receives its 128 rows of the
//    result, so an SM streams about half the operand bytes per output.
//  - proj_splitk_kernel<KS, BNS> (few tiles): a cluster of KS CTAs splits one 128 x BNS tile's
//    K range and reduce-scatters the partial accumulators through distributed shared memory
//    (BNS = 256, or 128 where that puts more CTAs to work).
// Rows past M and columns past N are zero-filled by the copies and skipped by the stores.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "gdn_internal.cuh"
#include "gdn_tcgen05.cuh"

namespace gdn {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;  // 16 KiB
constexpr uint32_t B_BYTES = BN * BK * 2;  // 32 KiB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t BAR_OFF = STAGES * STAGE_BYTES;
constexpr size_t PROJ_SMEM = BAR_OFF + 256 + 1024;  // ring + barriers + alignment slack
constexpr int PT = 192;                             // 6 warps

constexpr int MAX_SEG = 6;
struct Seg {
    int n0, n1;  // output columns [n0, n1) of C ...
    void* dst;   // ... go to dst[row * ld + (n - n0)] (bf16)
    int ld;
};
struct ProjArgs {
    int M, N, K;
    Seg seg[MAX_SEG];
    int nseg;
    unsigned int* status;
};
struct ProjMaps {
    CUtensorMap a, b;
};

__device__ __forceinline__ void tma_load(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// the 32 output columns n .. n + 31 of row m (in registers) to their segments' buffers
__device__ __forceinline__ void store_cols(const ProjArgs& P, int m, int n, const float (&v)[32])
{
    if (!chk(m >= 0 && m < P.M && n >= 0 && n < P.N, P.status)) return;
    // the segment holding column n (constant indices: the segment table stays in registers)
    Seg sg = P.seg[0];
#pragma unroll
    for (int i = 1; i < MAX_SEG; ++i)
        if (i < P.nseg && n >= P.seg[i].n0) sg = P.seg[i];
    if (n + 32 <= sg.n1 && ((n - sg.n0) & 7) == 0 && (sg.ld & 7) == 0) {
        // the 32 columns lie in one segment, 16-B aligned: four 16-B stores
        __nv_bfloat16* d = static_cast<__nv_bfloat16*>(sg.dst) + (size_t)m * sg.ld + (n - sg.n0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = tc::pack2<__nv_bfloat16>(v[8 * q + 0], v[8 * q + 1]);
            w.y = tc::pack2<__nv_bfloat16>(v[8 * q + 2], v[8 * q + 3]);
            w.z = tc::pack2<__nv_bfloat16>(v[8 * q + 4], v[8 * q + 5]);
            w.w = tc::pack2<__nv_bfloat16>(v[8 * q + 6], v[8 * q + 7]);
            *reinterpret_cast<uint4*>(d + 8 * q) = w;
        }
    } else {  // narrow segments (small shapes): one column at a time
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int ne = n + e;
            if (ne >= P.N) continue;
            Seg g = P.seg[0];
#pragma unroll
            for (int i = 1; i < MAX_SEG; ++i)
                if (i < P.nseg && ne >= P.seg[i].n0) g = P.seg[i];
            static_cast<__nv_bfloat16*>(g.dst)[(size_t)m * g.ld + (ne - g.n0)] = __float2bfloat16_rn(v[e]);
        }
    }
}

__global__ void __launch_bounds__(PT, 1) proj_kernel(const __grid_constant__ ProjArgs P,
                                                       const __grid_constant__ ProjMaps T)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + BAR_OFF);  // [STAGES] slice landed
    uint64_t* empty = full + STAGES;                             // [STAGES] slice consumed by the MMAs
    uint64_t* accf = empty + STAGES;                             // [2] accumulator complete
    uint64_t* acce = accf + 2;                                   // [2] accumulator read out (4 warps)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int KT = P.K / BK;
    const int tiles_n = (P.N + BN - 1) / BN, tiles = tiles_n * ((P.M + BM - 1) / BM);

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 4);
        }
        fence_mbar_init();
    }
    if (warp == 1) tc::alloc(tmem_slot, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = *tmem_slot;

    // tiles of this CTA: blockIdx.x, + gridDim.x, ...; N-tiles vary fastest (the CTAs running at
    // once share a few A row blocks and stream B through L2)
    if (warp == 0) {
        // producer: K slices of A and B, STAGES ahead of the MMAs, across tiles
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                const int n0 = (t % tiles_n) * BN, m0 = (t / tiles_n) * BM;
                for (int kt = 0; kt < KT; ++kt, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (uint32_t)((it / STAGES) & 1);
                    if (!mbar_wait_bounded(&empty[s], ph ^ 1u, nullptr)) {
                        atomicOr(P.status, GDN_DEV_TIMEOUT);
                        ok = false;
                        break;
                    }
                    unsigned char* st = sm + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                    tma_load(st, &T.a, kt * BK, m0, &full[s]);
                    tma_load(st + A_BYTES, &T.b, kt * BK, n0, &full[s]);
                }
            }
        }
    } else if (warp == 1) {
        // MMA issuer: tile i accumulates into TMEM columns 256 (i % 2) ..; the commits release the
        // slices and hand the accumulator to the epilogue.  A failed wait still commits, so that
        // every other wait ends.
        if (lane == 0) {
            int it = 0, i = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
                const int ab = i & 1;
                if (ok && !mbar_wait_bounded(&acce[ab], (uint32_t)(((i >> 1) & 1) ^ 1), nullptr)) {
                    atomicOr(P.status, GDN_DEV_TIMEOUT);
                    ok = false;
                }
                tc::fence_after_sync();
                for (int kt = 0; kt < KT; ++kt, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (uint32_t)((it / STAGES) & 1);
                    if (ok && !mbar_wait_bounded(&full[s], ph, nullptr)) {
                        atomicOr(P.status, GDN_DEV_TIMEOUT);
                        ok = false;
                    }
                    tc::fence_after_sync();
                    unsigned char* st = sm + s * STAGE_BYTES;
                    if (ok)
                        tc::mma_k(tm + 256 * ab, smem_addr(st), BM, smem_addr(st + A_BYTES), BN, BK,
                                  tc::idesc_bf16(BM, BN), kt > 0);
                    tc::commit(&empty[s]);
                }
                tc::commit(&accf[ab]);
            }
        }
    } else {
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 = rows of the tile
        int i = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
            const int ab = i & 1;
            const int n0 = (t % tiles_n) * BN, m0 = (t / tiles_n) * BM;
            const bool got = mbar_wait_bounded(&accf[ab], (uint32_t)((i >> 1) & 1), nullptr);
            if (!got && lane == 0) atomicOr(P.status, GDN_DEV_TIMEOUT);
            tc::fence_after_sync();
            const int row = (warp & 3) * 32 + lane, m = m0 + row;
            for (int c0 = 0; c0 < BN; c0 += 32) {
                float v[32];
                tc::ld32(tc::taddr(tm + 256 * ab, warp, c0), v);  // whole warp
                tc::wait_ld();
                const int n = n0 + c0;
                if (!got || m >= P.M || n >= P.N) continue;
                store_cols(P, m, n, v);
            }
            // this warp has read its quarter of the accumulator: the MMAs may reuse it
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[ab]);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) tc::dealloc(tm, 512);
}

// ---- CTA-pair kernel: 256 x BNP tiles, one MMA (M = 256) over the two CTAs of a cluster ----
// CTA r of a pair holds rows 128 r .. of the tile's A rows and B rows BNP/2 r .. in its own stage
// ring (16 KiB of A and BNP/2 rows of B per 64-wide K slice; 6 stages), and receives D rows
// 128 r .. over all BNP columns in its own TMEM.  Per output element each SM thus streams about
// half the operand bytes of the single-CTA kernel.  The even CTA's warp 1 issues the MMAs; the
// odd CTA's copies complete on the even CTA's full barriers, and the MMA commits arrive on the
// stage and accumulator barriers of both.  The tile width BNP is 256, or 192 where that puts
// more SMs to work (each CTA then holds 128 or 96 rows of B).
constexpr int STAGES2 = 6;
constexpr uint32_t A2_BYTES = 128 * BK * 2;  // this CTA's 128 A rows of a 64-wide K slice
template <int BNP> struct PairCfg {
    static constexpr uint32_t B_BYTES = (BNP / 2) * BK * 2;  // this CTA's B rows
    static constexpr uint32_t STAGE = A2_BYTES + B_BYTES;     // a multiple of 1024
    static constexpr uint32_t BAR_OFF = STAGES2 * STAGE;
    static constexpr size_t SMEM = BAR_OFF + 256 + 1024;
};

// 2-D tile copy whose completion may be counted on the mbarrier of the other CTA of the pair
// (bar is a shared::cluster address)
__device__ __forceinline__ void tma_load_pair(void* dst, const CUtensorMap* map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cbar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}

template <int BNP>
__global__ void __launch_bounds__(PT, 1) proj_pair_kernel(const __grid_constant__ ProjArgs P,
                                                            const __grid_constant__ ProjMaps T)
{
    using C = PairCfg<BNP>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);  // [STAGES2] both CTAs' slices landed (even CTA)
    uint64_t* empty = full + STAGES2;                             // [STAGES2] slice consumed by the MMAs
    uint64_t* accf = empty + STAGES2;                             // [2] accumulator complete
    uint64_t* acce = accf + 2;                                    // [2] accumulator read out, 8 warps (even CTA)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
    const int KT = P.K / BK;
    const int tiles_n = (P.N + BNP - 1) / BNP, tiles = tiles_n * ((P.M + 255) / 256);

    if (tid == 0) {
        for (int s = 0; s < STAGES2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 8);
        }
        fence_mbar_init();
    }
    if (warp == 1) tc::alloc_pair(tmem_slot, 512);
    tc::fence_before_sync();
    cluster_sync_all();  // both CTAs' barriers and TMEM exist before either side touches them
    tc::fence_after_sync();
    const uint32_t tm = *tmem_slot;

    if (warp == 0) {
        // producer: this CTA's 128 A rows and 128 B rows of each K slice
        if (lane == 0) {
            const uint32_t full0 = map_to_rank(smem_addr(&full[0]), 0);
            int it = 0;
            bool ok = true;
            for (int t = pair; t < tiles && ok; t += npairs) {
                const int n0 = (t % tiles_n) * BNP + (BNP / 2) * (int)rank, m0 = (t / tiles_n) * 256 + 128 * (int)rank;
                for (int kt = 0; kt < KT; ++kt, ++it) {
                    const int s = it % STAGES2;
                    const uint32_t ph = (uint32_t)((it / STAGES2) & 1);
                    if (!mbar_wait_bounded(&empty[s], ph ^ 1u, nullptr)) {
                        atomicOr(P.status, GDN_DEV_TIMEOUT);
                        ok = false;
                        break;
                    }
                    unsigned char* st = sm + s * C::STAGE;
                    if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * C::STAGE);
                    const uint32_t fb = full0 + (uint32_t)(s * 8);
                    tma_load_pair(st, &T.a, kt * BK, m0, fb);
                    tma_load_pair(st + A2_BYTES, &T.b, kt * BK, n0, fb);
                }
            }
        }
    } else if (warp == 1) {
        // MMA issuer (even CTA): tile i into TMEM columns 256 (i % 2) .. of both CTAs.  A failed wait
        // still commits, so that every other wait ends.
        if (lane == 0 && rank == 0) {
            int it = 0, i = 0;
            bool ok = true;
            for (int t = pair; t < tiles; t += npairs, ++i) {
                const int ab = i & 1;
                if (ok && !mbar_wait_cluster_bounded(&acce[ab], (uint32_t)(((i >> 1) & 1) ^ 1))) {
                    atomicOr(P.status, GDN_DEV_TIMEOUT);
                    ok = false;
                }
                tc::fence_after_sync();
                for (int kt = 0; kt < KT; ++kt, ++it) {
                    const int s = it % STAGES2;
                    const uint32_t ph = (uint32_t)((it / STAGES2) & 1);
                    if (ok && !mbar_wait_bounded(&full[s], ph, nullptr)) {
                        atomicOr(P.status, GDN_DEV_TIMEOUT);
                        ok = false;
                    }
                    tc::fence_after_sync();
                    unsigned char* st = sm + s * C::STAGE;
                    if (ok)
                        tc::mma_pair_k64(tm + 256 * ab, smem_addr(st), smem_addr(st + A2_BYTES),
                                         tc::idesc_bf16(256, BNP), kt > 0);
                    tc::commit_pair_mc(&empty[s], 0x3);
                }
                tc::commit_pair_mc(&accf[ab], 0x3);
            }
        }
    } else {
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 = rows 128 rank + .. of the tile
        const uint32_t acce0 = map_to_rank(smem_addr(&acce[0]), 0);
        int i = 0;
        for (int t = pair; t < tiles; t += npairs, ++i) {
            const int ab = i & 1;
            const int n0 = (t % tiles_n) * BNP, m0 = (t / tiles_n) * 256 + 128 * (int)rank;
            const bool got = mbar_wait_cluster_bounded(&accf[ab], (uint32_t)((i >> 1) & 1));
            if (!got && lane == 0) atomicOr(P.status, GDN_DEV_TIMEOUT);
            tc::fence_after_sync();
            const int m = m0 + (warp & 3) * 32 + lane;
            for (int c0 = 0; c0 < BNP; c0 += 32) {
                float v[32];
                tc::ld32(tc::taddr(tm + 256 * ab, warp, c0), v);  // whole warp
                tc::wait_ld();
                const int n = n0 + c0;
                if (!got || m >= P.M || n >= P.N) continue;
                store_cols(P, m, n, v);
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acce0 + (uint32_t)(ab * 8));
        }
    }
    tc::fence_before_sync();
    cluster_sync_all();  // neither CTA leaves while the other may still arrive on its barriers
    if (warp == 1) tc::dealloc_pair(tm, 512);
}

// ---- split-K kernel: few tiles (small T), each tile's K range shared by a cluster of KS CTAs ----
// CTA r of a cluster accumulates K slices r * KT/KS .. into its own 256 TMEM columns (a
// single-CTA 128 x 256 tile, as proj_kernel).  The partial sums are then reduce-scattered
// through distributed shared memory: CTA g owns the output columns g * 256/KS .. of the tile.
// Each CTA writes the other groups of its partial into its (by then free) stage ring and sends
// each to its owner with one bulk copy; the owner adds the KS partials in rank order and
// stores its columns.  A group is [128 rows][GW floats] with the 16-B chunks of row i at
// chunk position c ^ (i % 8), so that both the row-wise writes and reads are conflict-free.
// bulk copy of `bytes` from this CTA's shared memory to another CTA's (dst and its mbarrier as
// shared::cluster addresses), completing on that mbarrier; 16-B aligned, a multiple of 16 bytes
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "r"(smem_addr(src)), "r"(bytes), "r"(bar)
        : "memory");
}

template <int KS, int BNS>
__global__ void __launch_bounds__(PT, 1) proj_splitk_kernel(const __grid_constant__ ProjArgs P,
                                                              const __grid_constant__ ProjMaps T)
{
    static_assert(BNS == 128 || BNS == 256, "tile width");
    constexpr int GW = BNS / KS;               // columns of the group a CTA owns
    constexpr uint32_t GROUP = 128u * GW * 4u;  // bytes of one group of a partial
    static_assert(2 * (KS - 1) * GROUP <= BAR_OFF, "sent and received groups fit the stage ring");
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + BAR_OFF);  // [STAGES]
    uint64_t* empty = full + STAGES;                             // [STAGES]
    uint64_t* accf = empty + STAGES;                             // accumulator complete
    uint64_t* red = accf + 1;                                    // the other CTAs' groups landed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red + 1);
    unsigned char* recv = sm;                                    // [KS - 1] groups received, by sender
    unsigned char* sendb = sm + (KS - 1) * GROUP;                // [KS - 1] groups to send, by owner

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)cluster_ctarank(), tile = (int)blockIdx.x / KS;
    const int tiles_n = (P.N + BNS - 1) / BNS;
    const int n0 = (tile % tiles_n) * BNS, m0 = (tile / tiles_n) * BM;
    const int kper = (P.K / BK) / KS, kt0 = rank * kper;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accf, 1);
        mbar_init(red, 1);
        mbar_arrive_expect_tx(red, (uint32_t)(KS - 1) * GROUP);
        fence_mbar_init();
    }
    if (warp == 1) tc::alloc(tmem_slot, 256);
    tc::fence_before_sync();
    cluster_sync_all();  // every CTA's barriers exist before any group is sent
    tc::fence_after_sync();
    const uint32_t tm = *tmem_slot;

    bool got = true;
    if (warp == 0) {
        if (lane == 0) {
            for (int i = 0; i < kper; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (uint32_t)((i / STAGES) & 1);
                if (!mbar_wait_bounded(&empty[s], ph ^ 1u, nullptr)) {
                    atomicOr(P.status, GDN_DEV_TIMEOUT);
                    break;
                }
                unsigned char* st = sm + s * STAGE_BYTES;  // B takes BNS of the stage's BN rows
                mbar_arrive_expect_tx(&full[s], A_BYTES + (uint32_t)BNS * BK * 2);
                tma_load(st, &T.a, (kt0 + i) * BK, m0, &full[s]);
                tma_load(st + A_BYTES, &T.b, (kt0 + i) * BK, n0, &full[s]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = true;
            for (int i = 0; i < kper; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (uint32_t)((i / STAGES) & 1);
                if (ok && !mbar_wait_bounded(&full[s], ph, nullptr)) {
                    atomicOr(P.status, GDN_DEV_TIMEOUT);
                    ok = false;
                }
                tc::fence_after_sync();
                unsigned char* st = sm + s * STAGE_BYTES;
                if (ok)
                    tc::mma_k(tm, smem_addr(st), BM, smem_addr(st + A_BYTES), BNS, BK, tc::idesc_bf16(BM, BNS), i > 0);
                tc::commit(&empty[s]);
            }
            tc::commit(accf);
        }
    } else {
        got = mbar_wait_bounded(accf, 0, nullptr);
        if (!got && lane == 0) atomicOr(P.status, GDN_DEV_TIMEOUT);
    }
    // every CTA's products are done (its stage ring is free for the groups)
    tc::fence_before_sync();
    cluster_sync_all();
    tc::fence_after_sync();
    if (warp >= 2) {
        const int row = (warp & 3) * 32 + lane, m = m0 + row;
        // this CTA's partial of every other group -> the send area, swizzled rows
        for (int g = 0; g < KS; ++g) {
            if (g == rank) continue;
            unsigned char* dst = sendb + (g < rank ? g : g - 1) * GROUP + (size_t)row * GW * 4;
#pragma unroll
            for (int c0 = 0; c0 < GW; c0 += 32) {
                float v[32];
                tc::ld32(tc::taddr(tm, warp, g * GW + c0), v);  // whole warp
                tc::wait_ld();
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int c = c0 / 4 + q;  // 16-B chunk of the row
                    *reinterpret_cast<float4*>(dst + ((c ^ (row & 7)) << 4)) =
                        make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
            }
        }
        tc::fence_proxy_async();  // the rows are read by the bulk copies
        named_bar_sync(1, 128);   // the four epilogue warps
        if (tid == 64)
            for (int g = 0; g < KS; ++g) {
                if (g == rank) continue;
                const uint32_t slot = (uint32_t)(rank < g ? rank : rank - 1);
                bulk_s2cluster(map_to_rank(smem_addr(recv) + slot * GROUP, (uint32_t)g),
                               sendb + (g < rank ? g : g - 1) * GROUP, GROUP, map_to_rank(smem_addr(red), (uint32_t)g));
            }
        // the others' partials of this CTA's group: add all KS in rank order, store
        const bool gotr = mbar_wait_cluster_bounded(red, 0);
        if (!gotr && lane == 0) atomicOr(P.status, GDN_DEV_TIMEOUT);
#pragma unroll
        for (int c0 = 0; c0 < GW; c0 += 32) {
            float own[32], v[32];
            tc::ld32(tc::taddr(tm, warp, rank * GW + c0), own);  // whole warp
            tc::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0.f;
            for (int k = 0; k < KS; ++k) {
                if (k == rank) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] += own[e];
                } else {
                    const unsigned char* src = recv + (k < rank ? k : k - 1) * GROUP + (size_t)row * GW * 4;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int c = c0 / 4 + q;
                        const float4 t = *reinterpret_cast<const float4*>(src + ((c ^ (row & 7)) << 4));
                        v[4 * q] += t.x;
                        v[4 * q + 1] += t.y;
                        v[4 * q + 2] += t.z;
                        v[4 * q + 3] += t.w;
                    }
                }
            }
            const int n = n0 + rank * GW + c0;
            if (got && gotr && m < P.M && n < P.N) store_cols(P, m, n, v);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) tc::dealloc(tm, 256);
    cluster_sync_all();  // no CTA leaves while its groups may still be read by the copies to the others
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// [rows][k] bf16 row-major at base, read as 64-wide K slices of box_rows rows, 128-byte swizzle
cudaError_t encode_kmajor(CUtensorMap* m, const void* base, int k, int rows, int box_rows)
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)k * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                                elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

__device__ unsigned int g_proj_status;  // status word of calls that pass none

using ProjKernel = void (*)(ProjArgs, ProjMaps);

// launch configuration: `grid` CTAs of PT threads in clusters of `cluster` along x (grid a
// multiple of it), `smem` bytes of dynamic shared memory each
cudaLaunchConfig_t cluster_config(cudaLaunchAttribute* attr, unsigned grid, unsigned cluster, size_t smem,
                                  cudaStream_t st)
{
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(PT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// clusters of `cluster` CTAs of `kern` that can be resident at once (0 when the query fails)
int resident_clusters(ProjKernel kern, unsigned cluster, size_t smem)
{
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = cluster_config(attr, cluster * 16, cluster, smem, nullptr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_clusters(ProjKernel kern, unsigned grid, unsigned cluster, size_t smem, cudaStream_t st,
                            const ProjArgs& P, const ProjMaps& T)
{
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = cluster_config(attr, grid, cluster, smem, st);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, P, T);
    return e != cudaSuccess ? e : cudaGetLastError();
}

constexpr int kMaxDevices = 64;  // per-device caches below (kernel attributes are per device)

// the split-K kernel for c CTAs per tile (2 or 4) and tiles bn wide (128 or 256)
ProjKernel splitk_kernel(int c, int bn)
{
    if (bn == 128) return c == 4 ? proj_splitk_kernel<4, 128> : proj_splitk_kernel<2, 128>;
    return c == 4 ? proj_splitk_kernel<4, 256> : proj_splitk_kernel<2, 256>;
}

// clusters of c split-K CTAs (tiles bn wide) resident at once on device dev (cached; 0 when the
// query fails)
int split_clusters(int dev, int c, int bn)
{
    static std::mutex mu;
    static int cached[kMaxDevices][2][5];
    static bool init[kMaxDevices] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (!init[dev]) {
        for (auto& w : cached[dev])
            for (int& x : w) x = -1;
        init[dev] = true;
    }
    int& slot = cached[dev][bn == 128 ? 0 : 1][c];
    if (slot < 0) {
        const ProjKernel kern = splitk_kernel(c, bn);
        slot = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PROJ_SMEM) == cudaSuccess
                   ? resident_clusters(kern, (unsigned)c, PROJ_SMEM)
                   : 0;
        (void)cudaGetLastError();
    }
    return slot;
}

cudaError_t launch_proj(int M, int N, int K, const void* a, const void* b, const Seg* seg, int nseg,
                        unsigned int* status, cudaStream_t st)
{
    if (M <= 0 || N <= 0) return cudaSuccess;
    ProjArgs P;
    memset(&P, 0, sizeof(P));
    P.M = M;
    P.N = N;
    P.K = K;
    P.nseg = nseg;
    P.status = status;
    int dev = 0;
    {
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    }
    if (!P.status) {  // the library's own word on this device (address looked up once per device)
        static std::mutex mu;
        static unsigned int* addr[kMaxDevices] = {};
        cudaError_t e = cudaSuccess;
        std::lock_guard<std::mutex> lock(mu);
        if (!addr[dev]) {
            void* a_ = nullptr;
            e = cudaGetSymbolAddress(&a_, g_proj_status);
            if (e != cudaSuccess) return e;
            addr[dev] = static_cast<unsigned int*>(a_);
        }
        P.status = addr[dev];
    }
    for (int i = 0; i < nseg; ++i) P.seg[i] = seg[i];
    cudaError_t e = cudaSuccess;
    // resident CTAs / CTA pairs of the device (cached per device; calls from several host threads
    // are serialised here)
    static std::mutex mu;
    static int cached_sms[kMaxDevices] = {}, cached_pairs[kMaxDevices] = {};
    int num_sms = 0, num_pairs = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (cached_sms[dev] == 0) {
            int sms = 0, pairs = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PROJ_SMEM);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(proj_pair_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)PairCfg<256>::SMEM);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(proj_pair_kernel<192>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)PairCfg<192>::SMEM);
            if (e == cudaSuccess) pairs = resident_clusters(proj_pair_kernel<256>, 2, PairCfg<256>::SMEM);
            if (e != cudaSuccess) return e;
            cached_sms[dev] = sms;
            cached_pairs[dev] = pairs;
        }
        num_sms = cached_sms[dev];
        num_pairs = cached_pairs[dev];
    }
    // Few tiles (small T): split each tile's K range over a cluster of KS CTAs when at least
    // two CTAs per tile fit on the GPU at once (KS dividing the K slices, every cluster resident),
    // with 128 x 256 tiles, or 128 x 128 tiles where those put more CTAs to work (each then
    // streams half the B rows: the weights are the bytes that bound a small batch).
    {
        const int KT = K / BK;
        int ks = 0, bns = 0;
        long best = 0;
        for (int bn : {256, 128}) {
            const long tiles = (long)((N + bn - 1) / bn) * ((M + BM - 1) / BM);
            for (int c : {4, 2}) {
                if (tiles * c > num_sms || KT % c != 0 || tiles * c <= best) continue;
                if (split_clusters(dev, c, bn) < tiles) continue;
                ks = c;
                bns = bn;
                best = tiles * c;
                break;
            }
        }
        if (ks) {
            ProjMaps T;
            memset(&T, 0, sizeof(T));
            e = encode_kmajor(&T.a, a, K, M, BM);
            if (e == cudaSuccess) e = encode_kmajor(&T.b, b, K, N, bns);
            if (e != cudaSuccess) return e;
            const long tiles = (long)((N + bns - 1) / bns) * ((M + BM - 1) / BM);
            return launch_clusters(splitk_kernel(ks, bns), (unsigned)(tiles * ks), (unsigned)ks, PROJ_SMEM, st, P,
                                   T);
        }
    }
    // persistent grids: tiles are taken in turn by num_sms CTAs (128 x 256 tiles) or by num_pairs
    // CTA pairs (256 x 256 tiles, half the operand traffic per SM); the pairs are used unless they
    // need more rounds over the tiles than single CTAs do (a few rows past a multiple of 256).
    // When the pairs' tiles take a single round, 256 x 192 tiles put more SMs to work, each on
    // three quarters of the products, if they still take a single round.
    const long tiles1 = (long)((N + BN - 1) / BN) * ((M + BM - 1) / BM);
    const long tiles2 = (long)((N + 255) / 256) * ((M + 255) / 256);
    const long tiles3 = (long)((N + 191) / 192) * ((M + 255) / 256);
    const long rounds1 = (tiles1 + num_sms - 1) / num_sms;
    const long rounds2 = num_pairs > 0 ? (tiles2 + num_pairs - 1) / num_pairs : rounds1 + 1;
    const int bnp = rounds2 > rounds1 ? 0 : (rounds2 == 1 && tiles3 <= num_pairs && tiles3 > tiles2) ? 192 : 256;
    // A is read 128 rows at a time on every path; B 256 rows per CTA, or bnp / 2 per CTA of a pair
    ProjMaps T;
    memset(&T, 0, sizeof(T));
    e = encode_kmajor(&T.a, a, K, M, 128);
    if (e == cudaSuccess) e = encode_kmajor(&T.b, b, K, N, bnp ? bnp / 2 : BN);
    if (e != cudaSuccess) return e;
    if (bnp) {
        const unsigned pairs = (unsigned)std::min<long>(bnp == 256 ? tiles2 : tiles3, num_pairs);
        return bnp == 256 ? launch_clusters(proj_pair_kernel<256>, 2 * pairs, 2, PairCfg<256>::SMEM, st, P, T)
                          : launch_clusters(proj_pair_kernel<192>, 2 * pairs, 2, PairCfg<192>::SMEM, st, P, T);
    }
    proj_kernel<<<(unsigned)std::min<long>(tiles1, num_sms), PT, PROJ_SMEM, st>>>(P, T);
    return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// the shape facts both projections need; false when the shape is unusable here
bool proj_shape_ok(const gdn_shape* s, int hidden)
{
    return s && s->hqk > 0 && s->hv > 0 && s->dk > 0 && s->dv > 0 && s->hv % s->hqk == 0 && s->io_dtype == 1 &&
           hidden > 0 && hidden % BK == 0 && s->dk % 8 == 0 && s->dv % 8 == 0;
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_in_proj(const gdn_shape* shape, int hidden, int T, const void* x, const void* w_in, void* q,
                           void* k, void* v, void* z, void* a, void* b, unsigned int* status_dev, void* stream)
{
    using namespace gdn;
    if (!proj_shape_ok(shape, hidden) || T < 0) return GDN_ERR_INVALID_ARG;
    if (T == 0) return GDN_OK;
    if (!x || !w_in || !q || !k || !v || !z || !a || !b) return GDN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_in) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(z) ||
        !aligned16(a) || !aligned16(b))
        return GDN_ERR_INVALID_ARG;
    const int Dq = shape->hqk * shape->dk, Dv = shape->hv * shape->dv, Hv = shape->hv;
    const int N = 2 * Dq + 2 * Dv + 2 * Hv;
    const Seg seg[6] = {{0, Dq, q, Dq},
                        {Dq, 2 * Dq, k, Dq},
                        {2 * Dq, 2 * Dq + Dv, v, Dv},
                        {2 * Dq + Dv, 2 * Dq + 2 * Dv, z, Dv},
                        {2 * Dq + 2 * Dv, 2 * Dq + 2 * Dv + Hv, a, Hv},
                        {2 * Dq + 2 * Dv + Hv, N, b, Hv}};
    const cudaError_t e = launch_proj(T, N, hidden, x, w_in, seg, 6, status_dev, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" int gdn_out_proj(const gdn_shape* shape, int hidden, int T, const void* o, const void* w_out, void* y,
                            unsigned int* status_dev, void* stream)
{
    using namespace gdn;
    if (!proj_shape_ok(shape, hidden) || T < 0) return GDN_ERR_INVALID_ARG;
    const int Dv = shape->hv * shape->dv;
    if (Dv % BK != 0 || shape->out_dtype != 1) return GDN_ERR_INVALID_ARG;
    if (T == 0) return GDN_OK;
    if (!o || !w_out || !y || !aligned16(o) || !aligned16(w_out) || !aligned16(y)) return GDN_ERR_INVALID_ARG;
    const Seg seg[1] = {{0, hidden, y, hidden}};
    const cudaError_t e = launch_proj(T, hidden, Dv, o, w_out, seg, 1, status_dev, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
