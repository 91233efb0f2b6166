// umma_probe.cu -- test-only GEMM through the library's tcgen05 helpers (gdn_tcgen05.cuh).
//
// D[128 x N] = A[128 x K] * B[N x K]^T with bf16 or fp16 inputs (row-major, K contiguous) and an fp32
// result, computed by one CTA: operands staged into swizzled K-major shared-memory tiles,
// K/16 tcgen05.mma issues, commit to an mbarrier, tcgen05.ld of the accumulator.  The GPU test
// compares the result with a plain fp32 matmul: it checks the descriptor and instruction
// encodings that the prefill kernel relies on.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_tcgen05.cuh"

using namespace gdn;

__global__ void __launch_bounds__(128) umma_probe_kernel(const uint16_t* A, const uint16_t* B, float* D, int N,
                                                         int K, uint32_t ncols, uint32_t idesc, int a_mn, int b_mn,
                                                         unsigned int* status)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    const int ktiles = K / 64;
    unsigned char* a_tiles = smem;                          // ktiles x [128 rows x 128 B]
    unsigned char* b_tiles = a_tiles + ktiles * 128 * 128;  // ktiles x [N rows x 128 B]
    uint64_t* bar = reinterpret_cast<uint64_t*>(b_tiles + ktiles * N * 128);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    const int kc = K / 8;  // 16-B chunks per row
    if (!a_mn) {
        for (int i = tid; i < 128 * kc; i += 128) {
            const int r = i / kc, c = i % kc;
            const uint4 v = *reinterpret_cast<const uint4*>(A + (size_t)r * K + c * 8);
            *reinterpret_cast<uint4*>(a_tiles + (c / 8) * 128 * 128 + tc::sw128_chunk(r, c % 8)) = v;
        }
    } else {  // [K rows][M] with 64-wide M halves K * 128 B apart
        for (int i = tid; i < 128 * K; i += 128) {
            const int m = i / K, k = i % K;
            *reinterpret_cast<uint16_t*>(a_tiles + (m / 64) * K * 128 + tc::sw128(k, m % 64)) = A[(size_t)m * K + k];
        }
    }
    if (!b_mn) {
        for (int i = tid; i < N * kc; i += 128) {
            const int r = i / kc, c = i % kc;
            const uint4 v = *reinterpret_cast<const uint4*>(B + (size_t)r * K + c * 8);
            *reinterpret_cast<uint4*>(b_tiles + (c / 8) * N * 128 + tc::sw128_chunk(r, c % 8)) = v;
        }
    } else {
        for (int i = tid; i < N * K; i += 128) {
            const int n = i / K, k = i % K;
            *reinterpret_cast<uint16_t*>(b_tiles + (n / 64) * K * 128 + tc::sw128(k, n % 64)) = B[(size_t)n * K + k];
        }
    }
    tc::fence_proxy_async();
    if (warp == 0) tc::alloc(tmem_slot, ncols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t base = *tmem_slot;
    if (tid == 0) {
        tc::mma_k_mixed(base, smem_addr(a_tiles), 128, (uint32_t)a_mn, (uint32_t)(K * 128), smem_addr(b_tiles), N,
                        (uint32_t)b_mn, (uint32_t)(K * 128), K, idesc, 0);
        tc::commit(bar);
    }
    if (!mbar_wait_bounded(bar, 0, nullptr)) {
        if (tid == 0) atomicOr(status, 1u);
    } else {
        tc::fence_after_sync();
        for (int col = 0; col < N; col += 32) {
            float v[32];
            tc::ld32(tc::taddr(base, warp, col), v);
            tc::wait_ld();
            const int row = warp * 32 + lane;
            for (int j = 0; j < 32; ++j) D[(size_t)row * N + col + j] = v[j];
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::dealloc(base, ncols);
}

// half_inputs: 0 = bf16 operands, 1 = fp16 operands; a_mn / b_mn: stage that operand MN-major
extern "C" int umma_probe_gemm(const void* A, const void* B, void* D, int N, int K, int half_inputs, int a_mn,
                               int b_mn, unsigned int* status, void* stream)
{
    if ((N != 64 && N != 128 && N != 256) || (K != 64 && K != 128)) return -1;
    if ((a_mn || b_mn) && N > 128) return -1;  // MN-major operands here span at most two 64-wide halves
    const uint32_t ncols = N < 32 ? 32 : (uint32_t)N;
    // the operands need at most 1024 + 2 * 384 * 128 + 64 bytes; the CTA takes 220 KB so that
    // every tile address the descriptors can form stays inside its own shared memory
    const size_t smem = 220 * 1024;
    cudaError_t e = cudaFuncSetAttribute(umma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return -4;
    umma_probe_kernel<<<1, 128, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(A), static_cast<const uint16_t*>(B), static_cast<float*>(D), N, K, ncols,
        tc::idesc_kind_f16(128, N, half_inputs ? 0u : 1u, (uint32_t)a_mn, (uint32_t)b_mn), a_mn, b_mn, status);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
