// gdn_pool.cu -- the slot pool (host free list + device state memory) and the C ABI entry points.
//
// The pool is the fixed-size per-sequence state store of the qLLM README ("What this
// is": StateManager, a recurrent-state / conv-buffer slot pool whose size does not grow
// with context) and of the System Design page ("Architecture": mamba_cache.py).  Its
// calls follow the engine trait of issue #5279 (phase P0: add slot, recycle slot,
// cleanup, reset) and phase P5's device array of u64 per-layer state pointers.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_map>

#include "gdn_internal.cuh"

using gdn::Pool;

struct gdn_pool : public Pool {};

namespace {

constexpr int kVersion = 10000;  // 1.0.0

__global__ void zero_kernel(uint4* p, size_t n16)
{
    size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    size_t stride = (size_t)gridDim.x * blockDim.x;
    for (; i < n16; i += stride) p[i] = make_uint4(0u, 0u, 0u, 0u);
}

__global__ void slot_ptrs_kernel(const int* ids, int m, uint64_t base, uint64_t slot_bytes, int num_layers,
                                 int num_slots, int layer, const unsigned char* live, uint64_t* out,
                                 unsigned int* status)
{
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= m) return;
    int id = ids[i];
    bool ok = id >= 0 && id < num_slots && live[id];
    // a repeated id would make two rows of one launch update the same state
    for (int j = 0; ok && j < i; ++j) ok = ids[j] != id;
    if (!ok) {
        atomicOr(status, GDN_DEV_BAD_SLOT_ID);
        out[i] = 0;
        return;
    }
    out[i] = base + ((uint64_t)id * num_layers + layer) * slot_bytes;
}

// A mixed step's overlap check (one CTA): does a decode row's slot pointer equal the address of
// (a prefill sequence's slot, layer)?  Writes the verdict to *gate (read by both parts' kernels,
// which then do nothing) and sets GDN_DEV_SLOT_OVERLAP.  Ids the prefill's own validation will
// reject are skipped here (they name no slot).
__global__ void mixed_overlap_kernel(const uint64_t* ptrs, int m, const int* ids, int n, uint64_t base,
                                     uint64_t slot_bytes, int num_layers, int num_slots, int layer, int* gate,
                                     unsigned int* status)
{
    __shared__ int hit;
    if (threadIdx.x == 0) hit = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < m; i += blockDim.x) {
        const uint64_t p = ptrs[i];
        for (int j = 0; j < n; ++j) {
            const int id = ids[j];
            if (id >= 0 && id < num_slots && p == base + ((uint64_t)id * num_layers + layer) * slot_bytes) hit = 1;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        *gate = hit;
        if (hit) atomicOr(status, GDN_DEV_SLOT_OVERLAP);
    }
}

cudaError_t enqueue_zero(void* p, size_t bytes, cudaStream_t st, int num_sms)
{
    // every region zeroed here is 256-B aligned and a multiple of 256 B long
    size_t n16 = bytes / 16;
    if (n16 == 0) return cudaSuccess;
    size_t want = (n16 + 255) / 256;
    int blocks = (int)std::min<size_t>(want, (size_t)num_sms * 8);
    zero_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<uint4*>(p), n16);
    return cudaGetLastError();
}

bool shape_ok(const gdn_shape& s)
{
    if (s.hqk <= 0 || s.hv <= 0 || s.hv % s.hqk != 0) return false;
    if (s.dk <= 0 || s.dv <= 0 || s.conv_w < 1 || s.conv_w > 8) return false;
    if (s.io_dtype < 0 || s.io_dtype > 1 || s.out_dtype < 0 || s.out_dtype > 1) return false;
    if (!(s.l2_eps >= 0.0f) || !(s.norm_eps >= 0.0f)) return false;
    if (s.chunk < 0 || s.max_prefill_tokens < 0) return false;
    return true;
}

bool shape_built(const gdn_shape& s)
{
    if (s.dk != s.dv) return false;
    if (s.dk != 16 && s.dk != 32 && s.dk != 64 && s.dk != 128) return false;
    if ((s.hv / s.hqk) * s.dv > 1024) return false;  // per-item vectors of the decode kernel
    if (s.chunk != 0 && s.chunk != 8 && s.chunk != 16 && s.chunk != 32 && s.chunk != 64) return false;
    return true;
}

}  // namespace

extern "C" {

int gdn_version(void) { return kVersion; }

const char* gdn_status_string(int status)
{
    switch (status) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID_ARG: return "invalid argument";
        case GDN_ERR_POOL_FULL: return "pool full";
        case GDN_ERR_BAD_SLOT: return "bad slot";
        case GDN_ERR_CUDA: return "CUDA error";
        case GDN_ERR_TIMEOUT: return "device wait timed out";
        case GDN_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case GDN_ERR_NO_PARAMS: return "layer parameters not registered";
        case GDN_ERR_DEVICE: return "device reported skipped work";
        default: return "unknown status";
    }
}

int gdn_pool_create(const gdn_shape* shape, int num_slots, int num_layers, gdn_pool** out)
{
    if (!shape || !out || num_slots <= 0 || num_layers <= 0) return GDN_ERR_INVALID_ARG;
    *out = nullptr;
    if (!shape_ok(*shape)) return GDN_ERR_INVALID_ARG;
    if (!shape_built(*shape)) return GDN_ERR_UNSUPPORTED_SHAPE;

    gdn_pool* P = new (std::nothrow) gdn_pool();
    if (!P) return GDN_ERR_INVALID_ARG;
    P->shape = *shape;
    P->num_slots = num_slots;
    P->num_layers = num_layers;
    P->C = 2 * shape->hqk * shape->dk + shape->hv * shape->dv;
    P->r = shape->hv / shape->hqk;
    P->io_size = shape->io_dtype == 1 ? 2 : 4;
    P->state_bytes = (size_t)shape->hv * shape->dv * shape->dk * sizeof(float);
    P->conv_bytes = (size_t)(shape->conv_w - 1) * P->C * P->io_size;
    P->slot_bytes = (P->state_bytes + P->conv_bytes + 255) / 256 * 256;
    P->total_bytes = P->slot_bytes * (size_t)num_slots * num_layers;

    int rc = GDN_OK;
    if (cudaGetDevice(&P->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&P->num_sms, cudaDevAttrMultiProcessorCount, P->device) != cudaSuccess) {
        rc = GDN_ERR_CUDA;
    }
    if (rc == GDN_OK && cudaMalloc(&P->base, P->total_bytes) != cudaSuccess) rc = GDN_ERR_CUDA;
    if (rc == GDN_OK && cudaMalloc(&P->live_dev, (size_t)num_slots) != cudaSuccess) rc = GDN_ERR_CUDA;
    if (rc == GDN_OK && cudaMalloc(&P->mark_dev, (size_t)num_slots * sizeof(int)) != cudaSuccess) rc = GDN_ERR_CUDA;
    // the status word and, beside it, the mixed step's overlap gate
    if (rc == GDN_OK && cudaMalloc(&P->status_dev, 2 * sizeof(unsigned int)) != cudaSuccess) rc = GDN_ERR_CUDA;
    if (rc == GDN_OK) P->gate_dev = reinterpret_cast<int*>(P->status_dev + 1);
    if (rc == GDN_OK && P->shape.max_prefill_tokens > 0) {
        const int cap = gdn::prefill_pool_chunk_cap(P->shape, P->shape.max_prefill_tokens);
        P->ws.bytes = gdn::prefill_workspace_bytes(P->shape, P->shape.max_prefill_tokens, cap);
        if (cudaMalloc(&P->ws.base, P->ws.bytes) != cudaSuccess) rc = GDN_ERR_CUDA;
        else if (!gdn::prefill_workspace_carve(P->ws, P->shape, P->shape.max_prefill_tokens, cap)) rc = GDN_ERR_CUDA;
        if (rc == GDN_OK && gdn::prefill_chunked(P->shape) && gdn::create_seg_streams(&P->seg) != cudaSuccess)
            rc = GDN_ERR_CUDA;
    }
    if (rc == GDN_OK) {
        if (enqueue_zero(P->base, P->total_bytes, 0, P->num_sms) != cudaSuccess) rc = GDN_ERR_CUDA;
        if (cudaMemset(P->live_dev, 0, (size_t)num_slots) != cudaSuccess) rc = GDN_ERR_CUDA;
        if (cudaMemset(P->mark_dev, 0, (size_t)num_slots * sizeof(int)) != cudaSuccess) rc = GDN_ERR_CUDA;
        if (cudaMemset(P->status_dev, 0, 2 * sizeof(unsigned int)) != cudaSuccess) rc = GDN_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) rc = GDN_ERR_CUDA;
    }
    if (rc != GDN_OK) {
        gdn::destroy_seg_streams(&P->seg);
        cudaFree(P->base);
        cudaFree(P->live_dev);
        cudaFree(P->mark_dev);
        cudaFree(P->status_dev);
        cudaFree(P->ws.base);
        delete P;
        // a failed allocation is not a sticky error: clear it, so that later launches, which
        // read the runtime's last error, do not report it as their own
        (void)cudaGetLastError();
        return rc;
    }
    P->live.assign((size_t)num_slots, 0);
    P->free_list.resize((size_t)num_slots);
    for (int i = 0; i < num_slots; ++i) P->free_list[(size_t)i] = num_slots - 1 - i;
    P->params.resize((size_t)num_layers);
    if (const char* dbg = std::getenv("GDN_DEBUG_FLAGS")) P->debug_flags = std::atoi(dbg);
    *out = P;
    return GDN_OK;
}

namespace {
void release_mixed_streams(const gdn_pool* P);  // the internal stream of gdn_mixed_step, below
}

int gdn_pool_destroy(gdn_pool* P)
{
    if (!P) return GDN_ERR_INVALID_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    release_mixed_streams(P);
    gdn::destroy_seg_streams(&P->seg);
    cudaFree(P->base);
    cudaFree(P->live_dev);
    cudaFree(P->mark_dev);
    cudaFree(P->status_dev);
    cudaFree(P->ws.base);
    delete P;
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_pool_reset(gdn_pool* P, void* stream)
{
    if (!P) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // on the stream, after the work already queued there that still reads the live flags
    if (cudaMemsetAsync(P->live_dev, 0, (size_t)P->num_slots, st) != cudaSuccess) return GDN_ERR_CUDA;
    if (enqueue_zero(P->base, P->total_bytes, st, P->num_sms) != cudaSuccess) return GDN_ERR_CUDA;
    std::fill(P->live.begin(), P->live.end(), 0);
    P->free_list.resize((size_t)P->num_slots);
    for (int i = 0; i < P->num_slots; ++i) P->free_list[(size_t)i] = P->num_slots - 1 - i;
    return GDN_OK;
}

int gdn_slot_alloc(gdn_pool* P, int* slot_id)
{
    if (!P || !slot_id) return GDN_ERR_INVALID_ARG;
    if (P->free_list.empty()) return GDN_ERR_POOL_FULL;
    int id = P->free_list.back();
    unsigned char one = 1;
    if (cudaMemcpy(P->live_dev + id, &one, 1, cudaMemcpyHostToDevice) != cudaSuccess) return GDN_ERR_CUDA;
    P->free_list.pop_back();
    P->live[(size_t)id] = 1;
    *slot_id = id;
    return GDN_OK;
}

int gdn_slot_recycle(gdn_pool* P, int slot_id, void* stream)
{
    if (!P) return GDN_ERR_INVALID_ARG;
    if (slot_id < 0 || slot_id >= P->num_slots || !P->live[(size_t)slot_id]) return GDN_ERR_BAD_SLOT;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the device live flag is cleared on the stream, so that a prefill or slot_ptrs call queued
    // there earlier still sees the slot allocated
    if (cudaMemsetAsync(P->live_dev + slot_id, 0, 1, st) != cudaSuccess) return GDN_ERR_CUDA;
    // the slot's layers are contiguous: one region of num_layers * slot_bytes
    char* p = P->base + (size_t)slot_id * P->num_layers * P->slot_bytes;
    if (enqueue_zero(p, P->slot_bytes * P->num_layers, st, P->num_sms) != cudaSuccess) return GDN_ERR_CUDA;
    P->live[(size_t)slot_id] = 0;
    // keep the free list ordered so that the lowest free id is handed out first
    auto it = std::upper_bound(P->free_list.begin(), P->free_list.end(), slot_id, std::greater<int>());
    P->free_list.insert(it, slot_id);
    return GDN_OK;
}

int gdn_slot_addr(gdn_pool* P, int layer, int slot_id, uint64_t* addr)
{
    if (!P || !addr || layer < 0 || layer >= P->num_layers) return GDN_ERR_INVALID_ARG;
    if (slot_id < 0 || slot_id >= P->num_slots) return GDN_ERR_BAD_SLOT;
    *addr = reinterpret_cast<uint64_t>(P->base) + ((uint64_t)slot_id * P->num_layers + layer) * P->slot_bytes;
    return GDN_OK;
}

int gdn_slot_snapshot(gdn_pool* P, int slot_id, void* dst, void* stream)
{
    if (!P || !dst) return GDN_ERR_INVALID_ARG;
    if (slot_id < 0 || slot_id >= P->num_slots || !P->live[(size_t)slot_id]) return GDN_ERR_BAD_SLOT;
    const size_t bytes = P->slot_bytes * P->num_layers;
    const char* src = P->base + (size_t)slot_id * bytes;
    cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_slot_restore(gdn_pool* P, int slot_id, const void* src, void* stream)
{
    if (!P || !src) return GDN_ERR_INVALID_ARG;
    if (slot_id < 0 || slot_id >= P->num_slots || !P->live[(size_t)slot_id]) return GDN_ERR_BAD_SLOT;
    const size_t bytes = P->slot_bytes * P->num_layers;
    char* dst = P->base + (size_t)slot_id * bytes;
    cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_slot_ptrs(gdn_pool* P, int layer, const int* slot_ids_dev, int m, uint64_t* out_dev, void* stream)
{
    if (!P || layer < 0 || layer >= P->num_layers || m < 0) return GDN_ERR_INVALID_ARG;
    if (m == 0) return GDN_OK;
    if (!slot_ids_dev || !out_dev) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    slot_ptrs_kernel<<<(m + 127) / 128, 128, 0, st>>>(slot_ids_dev, m, reinterpret_cast<uint64_t>(P->base),
                                                       P->slot_bytes, P->num_layers, P->num_slots, layer,
                                                       P->live_dev, out_dev, P->status_dev);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_layer_params(gdn_pool* P, int layer, const float* conv_w, const float* A_log, const float* dt_bias,
                     const float* norm_w)
{
    if (!P || layer < 0 || layer >= P->num_layers) return GDN_ERR_INVALID_ARG;
    if (!conv_w || !A_log || !dt_bias || !norm_w) return GDN_ERR_INVALID_ARG;
    P->params[(size_t)layer] = gdn::LayerParams{conv_w, A_log, dt_bias, norm_w};
    return GDN_OK;
}

namespace {

// the argument checks of gdn_decode_step (GDN_OK: enqueue; m == 0 passes and enqueues nothing)
int check_decode(gdn_pool* P, int layer, const uint64_t* slot_ptrs_dev, int m, const void* q, const void* k,
                 const void* v, const void* a, const void* b, const void* z, void* out)
{
    if (!P || layer < 0 || layer >= P->num_layers || m < 0) return GDN_ERR_INVALID_ARG;
    if (m == 0) return GDN_OK;
    if (!slot_ptrs_dev || !q || !k || !v || !a || !b || !z || !out) return GDN_ERR_INVALID_ARG;
    if (!P->params[(size_t)layer].set()) return GDN_ERR_NO_PARAMS;
    return GDN_OK;
}

// the argument checks of gdn_prefill_varlen (n_seqs == 0 with no tokens passes and enqueues nothing)
int check_prefill(gdn_pool* P, int layer, const int* cu_seqlens_dev, const int* slot_ids_dev, int n_seqs,
                  int total_tokens, const void* q, const void* k, const void* v, const void* a, const void* b,
                  const void* z, void* out)
{
    if (!P || layer < 0 || layer >= P->num_layers || n_seqs < 0 || total_tokens < 0) return GDN_ERR_INVALID_ARG;
    if (n_seqs == 0) return total_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (!cu_seqlens_dev || !slot_ids_dev) return GDN_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !a || !b || !z || !out)) return GDN_ERR_INVALID_ARG;
    if (total_tokens > 0 && !gdn::rows_aligned16(q, k, v, z, out)) return GDN_ERR_INVALID_ARG;
    if (!P->params[(size_t)layer].set()) return GDN_ERR_NO_PARAMS;
    if (total_tokens > P->shape.max_prefill_tokens) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (n_seqs > gdn::prefill_max_seqs(P->shape.max_prefill_tokens)) return GDN_ERR_UNSUPPORTED_SHAPE;
    return GDN_OK;
}

// per pool: the internal stream a mixed step runs its decode on, and the fork / join events
struct MixedStreams {
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, prep = nullptr;
};
std::mutex g_mixed_mu;
std::unordered_map<const gdn_pool*, MixedStreams> g_mixed;

cudaError_t mixed_streams(const gdn_pool* P, MixedStreams* out)
{
    std::lock_guard<std::mutex> lk(g_mixed_mu);
    auto it = g_mixed.find(P);
    if (it != g_mixed.end()) {
        *out = it->second;
        return cudaSuccess;
    }
    MixedStreams m;
    cudaError_t e = cudaStreamCreateWithFlags(&m.side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m.join, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m.prep, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        if (m.prep) cudaEventDestroy(m.prep);
        if (m.join) cudaEventDestroy(m.join);
        if (m.fork) cudaEventDestroy(m.fork);
        if (m.side) cudaStreamDestroy(m.side);
        return e;
    }
    g_mixed[P] = m;
    *out = m;
    return cudaSuccess;
}

void release_mixed_streams(const gdn_pool* P)
{
    std::lock_guard<std::mutex> lk(g_mixed_mu);
    auto it = g_mixed.find(P);
    if (it == g_mixed.end()) return;
    cudaEventDestroy(it->second.prep);
    cudaEventDestroy(it->second.join);
    cudaEventDestroy(it->second.fork);
    cudaStreamDestroy(it->second.side);
    g_mixed.erase(it);
}

}  // namespace

int gdn_decode_step(gdn_pool* P, int layer, const uint64_t* slot_ptrs_dev, int m, const void* q, const void* k,
                    const void* v, const void* a, const void* b, const void* z, void* out, void* stream)
{
    const int rc = check_decode(P, layer, slot_ptrs_dev, m, q, k, v, a, b, z, out);
    if (rc != GDN_OK || m == 0) return rc;
    cudaError_t e = gdn::launch_decode(*P, layer, slot_ptrs_dev, m, q, k, v, a, b, z, out,
                                       reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_prefill_varlen(gdn_pool* P, int layer, const int* cu_seqlens_dev, const int* slot_ids_dev, int n_seqs,
                       int total_tokens, const void* q, const void* k, const void* v, const void* a, const void* b,
                       const void* z, void* out, void* stream)
{
    const int rc = check_prefill(P, layer, cu_seqlens_dev, slot_ids_dev, n_seqs, total_tokens, q, k, v, a, b, z, out);
    if (rc != GDN_OK || n_seqs == 0) return rc;
    cudaError_t e = gdn::launch_prefill(*P, layer, cu_seqlens_dev, slot_ids_dev, n_seqs, total_tokens, q, k, v, a,
                                        b, z, out, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_mixed_step(gdn_pool* P, int layer, const uint64_t* slot_ptrs_dev, int m, const void* dq, const void* dk,
                   const void* dv, const void* da, const void* db, const void* dz, void* dout,
                   const int* cu_seqlens_dev, const int* slot_ids_dev, int n_seqs, int total_tokens, const void* pq,
                   const void* pk, const void* pv, const void* pa, const void* pb, const void* pz, void* pout,
                   void* stream)
{
    int rc = check_decode(P, layer, slot_ptrs_dev, m, dq, dk, dv, da, db, dz, dout);
    if (rc != GDN_OK) return rc;
    rc = check_prefill(P, layer, cu_seqlens_dev, slot_ids_dev, n_seqs, total_tokens, pq, pk, pv, pa, pb, pz, pout);
    if (rc != GDN_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (m == 0 || n_seqs == 0) {  // one part only: nothing to overlap
        cudaError_t e = cudaSuccess;
        if (m > 0) e = gdn::launch_decode(*P, layer, slot_ptrs_dev, m, dq, dk, dv, da, db, dz, dout, st);
        if (n_seqs > 0)
            e = gdn::launch_prefill(*P, layer, cu_seqlens_dev, slot_ids_dev, n_seqs, total_tokens, pq, pk, pv, pa, pb,
                                    pz, pout, st);
        return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    MixedStreams ms;
    if (mixed_streams(P, &ms) != cudaSuccess) return GDN_ERR_CUDA;
    // the two parts must name different slots: checked on the device first, both parts gated on it
    mixed_overlap_kernel<<<1, 256, 0, st>>>(slot_ptrs_dev, m, slot_ids_dev, n_seqs, reinterpret_cast<uint64_t>(P->base),
                                            P->slot_bytes, P->num_layers, P->num_slots, layer, P->gate_dev,
                                            P->status_dev);
    cudaError_t e = cudaGetLastError();
    // fork point: everything enqueued on `stream` so far (the overlap check among it)
    if (e == cudaSuccess) e = cudaEventRecord(ms.fork, st);
    // The chunked prefill's state pass takes one SM per CTA, two CTAs per (sequence, v-head); when
    // that leaves SMs idle, the state pass runs on the pool's high-priority segment stream once the
    // pre-pass is done and the decode, sized for the idle SMs, beside it (dispatched after it).
    // Otherwise the decode runs beside the whole prefill from the fork point.
    const int idle = P->num_sms - n_seqs * P->shape.hv * 2;
    const bool beside_state = gdn::prefill_chunked(P->shape) && P->seg.side && idle >= 16;
    bool split = false;
    if (e == cudaSuccess)
        e = gdn::launch_prefill(*P, layer, cu_seqlens_dev, slot_ids_dev, n_seqs, total_tokens, pq, pk, pv, pa, pb, pz,
                                pout, st, P->gate_dev, beside_state ? ms.prep : nullptr, &split);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ms.side, split ? ms.prep : ms.fork, 0);
    if (e == cudaSuccess)
        e = gdn::launch_decode(*P, layer, slot_ptrs_dev, m, dq, dk, dv, da, db, dz, dout, ms.side, P->gate_dev,
                               split ? idle : 0);
    // join: `stream` continues after the decode too
    if (e == cudaSuccess) e = cudaEventRecord(ms.join, ms.side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ms.join, 0);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_last_device_status(gdn_pool* P, void* stream)
{
    if (!P) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return GDN_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpy(&word, P->status_dev, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaMemset(P->status_dev, 0, sizeof(unsigned int)) != cudaSuccess) return GDN_ERR_CUDA;
    return (int)(word & 0x7fffffffu);
}

int gdn_pool_get_info(gdn_pool* P, gdn_pool_info* info)
{
    if (!P || !info) return GDN_ERR_INVALID_ARG;
    info->base = reinterpret_cast<uint64_t>(P->base);
    info->total_bytes = P->total_bytes;
    info->slot_bytes = P->slot_bytes;
    info->state_bytes = P->state_bytes;
    info->conv_bytes = P->conv_bytes;
    info->num_slots = P->num_slots;
    info->num_layers = P->num_layers;
    info->free_slots = (int)P->free_list.size();
    info->workspace_bytes = P->ws.bytes;
    return GDN_OK;
}

}  // extern "C"
