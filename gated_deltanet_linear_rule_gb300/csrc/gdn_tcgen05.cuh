// gdn_tcgen05.cuh -- 5th-generation tensor-core (tcgen05 / TMEM) helpers, written from the PTX ISA.
//
// Operand tiles are 16-bit (fp16 or bf16; one MMA uses one type for both), K-major, in the
// 128-byte swizzle layout: a tile holds R rows
// (the M or N index) of 64 K-elements (128 B per row); rows are grouped by 8 into 1024-B
// atoms, and inside an atom the 16-B chunk c of row r sits at chunk position c ^ (r % 8).
// A K extent of 128 is two such tiles side by side in memory (k 0..63, then 64..127).
// Tile bases are 1024-B aligned.  Accumulators are fp32 in tensor memory: for M = 128
// (cta_group::1) row i of D is TMEM lane i and column j is TMEM column j.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "gdn_internal.cuh"

namespace gdn {
namespace tc {

// byte offset of element (r, k), k < 64, inside a swizzled K-major tile
__device__ __forceinline__ uint32_t sw128(int r, int k)
{
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((k >> 3) ^ r) & 7) << 4) + (k & 7) * 2);
}

// byte offset of the 16-B chunk holding elements (r, 8c .. 8c+7)
__device__ __forceinline__ uint32_t sw128_chunk(int r, int c)
{
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + (((c ^ r) & 7) << 4));
}

// Shared-memory matrix descriptor of a swizzled K-major tile starting at shared address saddr
// (saddr may be advanced by 32 B steps inside an atom to select K = 16 slices).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address, 16-B units
    d |= (uint64_t)(1024u >> 4) << 32;         // stride byte offset: 8-row groups 1024 B apart
    d |= (uint64_t)1 << 46;                    // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                    // 128-byte swizzle
    return d;
}

// MN-major operand tiles (the MMA reads the operand transposed) use the same swizzled rows,
// but a row is one K index holding 64 consecutive M (or N) elements: element (mn, k) sits at
// (mn / 64) * lbo + sw128(k, mn % 64).  8-row groups along K are 1024 B apart; the two 64-wide
// halves of a 128-wide M or N extent are lbo bytes apart.
__device__ __forceinline__ uint64_t sdesc_mn(uint32_t saddr, uint32_t lbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;  // leading byte offset: next 64-wide M/N block
    d |= (uint64_t)(1024u >> 4) << 32;             // stride byte offset: next 8 K rows
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor: kind::f16, fp32 accumulator, A and B of the 16-bit type given
// (format code 0 = fp16, 1 = bf16); a_mn / b_mn mark MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_kind_f16(int M, int N, uint32_t ab_format, uint32_t a_mn = 0,
                                                      uint32_t b_mn = 0)
{
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | (a_mn << 15) | (b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) { return idesc_kind_f16(M, N, 1u); }
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, uint32_t a_mn = 0, uint32_t b_mn = 0)
{
    return idesc_kind_f16(M, N, 0u, a_mn, b_mn);
}

// D[tmem] (+)= A[smem] * B[smem]^T for one K = 16 slice; issued by one thread.
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// K = 16 * ksteps GEMM slice loop over operands of K extent 64 * ktiles (each K tile is
// R rows * 128 B; a_rows / b_rows give the tile pitch of A and B in rows).
// (The start-address field holds address / 16 in its low 14 bits; shared addresses stay below
// 256 KiB, so a K slice's descriptor is the base descriptor plus its byte offset / 16.)
__device__ __forceinline__ void mma_k(uint32_t d_tmem, uint32_t a_saddr, int a_rows, uint32_t b_saddr,
                                           int b_rows, int kdim, uint32_t idesc, uint32_t accumulate)
{
    const uint64_t a0 = sdesc(a_saddr), b0 = sdesc(b_saddr);
#pragma unroll 8
    for (int k16 = 0; k16 < kdim / 16; ++k16) {
        const int kt = k16 >> 2, kin = (k16 & 3) * 32;
        const uint64_t a = a0 + (uint64_t)((kt * a_rows * 128 + kin) >> 4);
        const uint64_t b = b0 + (uint64_t)((kt * b_rows * 128 + kin) >> 4);
        mma(d_tmem, a, b, idesc, (k16 > 0 || accumulate) ? 1u : 0u);
    }
}

// Same loop where either operand may be MN-major: for a K-major operand the tile pitch in rows
// is given (as above); for an MN-major operand (mn != 0) the K slices advance by 16 rows
// (2048 B) and lbo is the distance between its 64-wide M/N halves.
__device__ __forceinline__ void mma_k_mixed(uint32_t d_tmem, uint32_t a_saddr, int a_rows, uint32_t a_mn,
                                            uint32_t a_lbo, uint32_t b_saddr, int b_rows, uint32_t b_mn,
                                            uint32_t b_lbo, int kdim, uint32_t idesc, uint32_t accumulate)
{
    const uint64_t a0 = a_mn ? sdesc_mn(a_saddr, a_lbo) : sdesc(a_saddr);
    const uint64_t b0 = b_mn ? sdesc_mn(b_saddr, b_lbo) : sdesc(b_saddr);
#pragma unroll 8
    for (int k16 = 0; k16 < kdim / 16; ++k16) {
        const int kt = k16 >> 2, kin = (k16 & 3) * 32;
        const uint64_t a = a0 + (uint64_t)((a_mn ? k16 * 2048 : kt * a_rows * 128 + kin) >> 4);
        const uint64_t b = b0 + (uint64_t)((b_mn ? k16 * 2048 : kt * b_rows * 128 + kin) >> 4);
        mma(d_tmem, a, b, idesc, (k16 > 0 || accumulate) ? 1u : 0u);
    }
}

// Arrive on an mbarrier once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// One full warp: allocate ncols (power of two >= 32) TMEM columns; the base address lands in *dst.
__device__ __forceinline__ void alloc(uint32_t* dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ---- CTA pairs (cta_group::2): one MMA spans the two CTAs of a cluster pair ----
// A kernel uses one cta_group throughout.  With M = 256 the even CTA of the pair issues the MMA;
// each CTA holds 128 rows of A and N/2 rows of B at the same shared-memory offsets, and its TMEM
// receives its own 128 rows of D (lane i = row i of its half) over all N columns.

// D[tmem, both CTAs] (+)= A[smem, both] * B[smem, both]^T for one K = 16 slice
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// K = 64 slice of K-major swizzled tiles (one 64-wide K tile each): four K = 16 MMAs
__device__ __forceinline__ void mma_pair_k64(uint32_t d_tmem, uint32_t a_saddr, uint32_t b_saddr, uint32_t idesc,
                                             uint32_t accumulate)
{
    const uint64_t a0 = sdesc(a_saddr), b0 = sdesc(b_saddr);
#pragma unroll
    for (int k16 = 0; k16 < 4; ++k16)
        mma_pair(d_tmem, a0 + (uint64_t)(k16 * 2), b0 + (uint64_t)(k16 * 2), idesc, (k16 > 0 || accumulate) ? 1u : 0u);
}

// Arrive once on the mbarrier at this shared offset in every CTA of cta_mask when every
// tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void commit_pair_mc(uint64_t* bar, uint16_t cta_mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_addr(bar)),
        "h"(cta_mask)
        : "memory");
}

// One full warp in EACH CTA of the pair: ncols TMEM columns in both CTAs, base address in *dst.
__device__ __forceinline__ void alloc_pair(uint32_t* dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// generic-proxy shared-memory writes -> visible to the tensor cores (async proxy)
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes 32*(w%4) .. +31).
__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void st32(uint32_t taddr, const float (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

// TMEM address of (lane quarter of this warp, column col) relative to the allocation base
__device__ __forceinline__ uint32_t taddr(uint32_t base, int warp, int col)
{
    return base + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)col;
}

// pack two floats into a 16-bit pair (round to nearest even), low half = first
template <typename T> __device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi)
{
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi)
{
    __half2 p = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}

template <typename T> __device__ __forceinline__ T to16(float v);
template <> __device__ __forceinline__ __nv_bfloat16 to16<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }
template <> __device__ __forceinline__ __half to16<__half>(float v) { return __float2half_rn(v); }

// store 8 values (row r, elements 8c .. 8c+7) of a swizzled tile as one 16-B chunk
template <typename T>
__device__ __forceinline__ void st_chunk(unsigned char* tile, int r, int c, const float* v8)
{
    uint4 w;
    w.x = pack2<T>(v8[0], v8[1]);
    w.y = pack2<T>(v8[2], v8[3]);
    w.z = pack2<T>(v8[4], v8[5]);
    w.w = pack2<T>(v8[6], v8[7]);
    *reinterpret_cast<uint4*>(tile + sw128_chunk(r, c)) = w;
}

// store one element (r, k) of a swizzled tile
template <typename T>
__device__ __forceinline__ void st_elem(unsigned char* tile, int r, int k, float v)
{
    *reinterpret_cast<T*>(tile + sw128(r, k)) = to16<T>(v);
}

}  // namespace tc
}  // namespace gdn
