/*
 * gdn.h -- C ABI of libgdn, a GB300 (sm_103a) library that runs the Gated
 * Delta Rule (GDN) linear-attention layer of Qwen3.5-style hybrid models over
 * many sequences at once, each sequence owning a fixed-size slot of a state pool.
 *
 * Where the calls come from:
 *   - The slot pool is the fixed-size recurrent-state / conv-buffer pool that
 *     the qLLM README ("What this is": StateManager) wires in next to the KV
 *     block manager, and that the System Design page lists as the GDN state
 *     cache manager (mamba_cache.py, "Architecture").
 *   - The call set follows the seven-method engine trait of issue #5279
 *     ("serve: Qwen3.5 on CUDA never batches ...", phase plan P0: setup+prefill,
 *     decode step, add slot, recycle slot, cleanup, reset) and its phase P5
 *     (the GDN conv1d and delta rule gain a slot dimension: one launch over m
 *     slots through a device array of u64 per-layer state pointers).
 *   - The arithmetic is the GatedDeltaNet layer of the System Design page
 *     ("Runtime Data Flow" and "GDN Kernel Dispatch Detail"): depthwise causal
 *     conv1d + SiLU over the q/k/v channels, L2 normalisation of q and k, gates
 *     g = -exp(A_log) softplus(a + dt_bias), alpha = exp(g), beta = sigmoid(b),
 *     the state update S <- alpha S; u = S k; S <- S + beta (v - u) k^T, the
 *     read-out o = S q d_k^-1/2, and the gated RMSNorm rmsnorm(o) * silu(z).
 *
 * Conventions for every call:
 *   - Return value: GDN_OK (0) or a negative gdn_status code.  Calls validate
 *     their host-side arguments before enqueuing any GPU work; a call that
 *     returns an error has enqueued nothing.
 *   - Pointers named *_dev are device pointers; everything else is host memory.
 *   - `stream` is a cudaStream_t passed as an opaque pointer (NULL = the legacy
 *     default stream).  GPU work is enqueued on it; the hot calls
 *     (gdn_slot_ptrs, gdn_decode_step, gdn_prefill_varlen) neither allocate nor
 *     synchronise the host.
 *   - Ownership: the pool owns its state memory and its prefill workspace.
 *     Activation buffers, parameter arrays and streams belong to the caller
 *     and are only borrowed for the duration of the call (parameter arrays:
 *     for as long as they are registered with gdn_layer_params).
 *   - Layouts are row-major and contiguous; a token's heads are contiguous:
 *       q, k    [rows][Hqk * dk]     v, z, out  [rows][Hv * dv]     a, b [rows][Hv]
 *     in the pool's io dtype (out in its out dtype).  v-head h reads q/k head
 *     h / (Hv / Hqk).
 *   - Device-side faults in the arguments (a slot pointer outside the layer's
 *     slots, a freed or repeated slot id, a non-monotone cu_seqlens) are not
 *     turned into memory faults: the affected work is skipped and a bit is set
 *     in the pool's device status word, read by gdn_last_device_status.
 *   - Work on one slot is ordered by the stream; calls on different streams
 *     that touch the same slot must be ordered by the caller.
 *   - Input range: any finite inputs whose conv outputs, states and per-row sums of
 *     squares of the outputs stay within fp32 range (|v|, |z| and |S| up to about 1e18).
 *     The chunked prefill's 16-bit tensor-core operands carry per-chunk power-of-two
 *     scales, so its range is fp32's, not fp16's.
 *   - Not thread-safe: one host thread per pool at a time.
 *   - Test hooks: GDN_DEBUG_FLAGS in the environment when a pool is created, a bit mask.
 *     Bit 0 (value 1): that pool's decode kernel fills none of its pipeline stages, so every
 *     consumer wait runs out after its 1 s limit: the launch returns with GDN_DEV_TIMEOUT set
 *     and the outputs unwritten, and the CUDA context stays usable.  Bit 1 (value 2): its
 *     chunked prefill's state pass never fetches a sequence's first chunk record, with the
 *     same outcome for the prefill (no output row, no state written; the conv buffers are
 *     advanced already).
 */
#ifndef GDN_H
#define GDN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = -1,       /* NULL or out-of-range host argument */
    GDN_ERR_POOL_FULL = -2,         /* no free slot */
    GDN_ERR_BAD_SLOT = -3,          /* slot id out of range, or not in the state the call needs */
    GDN_ERR_CUDA = -4,              /* a CUDA runtime call failed (allocation, launch, copy) */
    GDN_ERR_TIMEOUT = -5,           /* a kernel's bounded wait ran out (device status bit) */
    GDN_ERR_UNSUPPORTED_SHAPE = -6, /* the shape is valid but not built into this library */
    GDN_ERR_NO_PARAMS = -7,         /* the layer's parameters were never registered */
    GDN_ERR_DEVICE = -8             /* the device status word reports skipped work */
} gdn_status;

/* Bits of the device status word (see gdn_last_device_status). */
#define GDN_DEV_BAD_SLOT_PTR 0x1u  /* a slot pointer was not a slot of the call's layer: item skipped */
#define GDN_DEV_BAD_SLOT_ID 0x2u   /* gdn_slot_ptrs / prefill got a freed, repeated or out-of-range id */
#define GDN_DEV_BAD_SEQLENS 0x4u   /* prefill cu_seqlens not 0-based, non-decreasing, ending at total */
#define GDN_DEV_TIMEOUT 0x8u       /* a pipeline wait gave up (the kernel returned early) */
#define GDN_DEV_SLOT_OVERLAP 0x10u /* gdn_mixed_step: a decode row and a prefill sequence named the same
                                      slot; the whole step was skipped */
#define GDN_DEV_BOUNDS 0x20u       /* checked builds only (libgdn_checked.so): a kernel computed an address
                                      outside the region it belongs to; that access was skipped */

typedef struct {
    int hqk;        /* q/k heads */
    int hv;         /* v heads; a multiple of hqk (GQA ratio r = hv / hqk) */
    int dk, dv;     /* head dims; this build supports dk == dv in {16, 32, 64, 128} */
    int conv_w;     /* causal conv taps W, 1..8 */
    int chunk;      /* prefill chunk length: 0 = the library's choice, or 8, 16, 32, 64.  At d = 128
                       the tensor-core path always takes chunks of 64.  At d < 128, 0 runs the
                       token-recurrent kernel and 8..64 the chunked form with that chunk length
                       (both fp32; the result depends on it only through rounding). */
    int io_dtype;   /* q, k, v, z, a, b and the conv buffer: 0 = fp32, 1 = bf16 */
    int out_dtype;  /* out: 0 = fp32, 1 = bf16 */
    float l2_eps;   /* q, k L2 norm: x * rsqrt(sum x^2 + l2_eps) */
    float norm_eps; /* gated RMSNorm: o * rsqrt(mean o^2 + norm_eps) */
    int max_prefill_tokens; /* the most tokens one prefill call may carry (0 = no prefill).  At
                               d = 128 the workspace holds the chunk records of at most 512 chunks of
                               64 tokens (2.4 MB each at Hqk 16, Hv 32); a call with more chunks runs
                               in segments of that many, one after the other. */
} gdn_shape;

typedef struct gdn_pool gdn_pool;

/* Sizes and addresses of a pool (host-side facts, no GPU work). */
typedef struct {
    uint64_t base;        /* device address of slot 0, layer 0 */
    uint64_t total_bytes; /* bytes of state memory */
    uint64_t slot_bytes;  /* bytes of one (slot, layer): state then conv buffer, 256-B aligned */
    uint64_t state_bytes; /* Hv * dv * dk * 4: fp32 S, head-major, rows indexed by dv */
    uint64_t conv_bytes;  /* (W - 1) * C * io size, C = 2 Hqk dk + Hv dv, channels [q | k | v] */
    int num_slots, num_layers, free_slots;
    uint64_t workspace_bytes; /* prefill workspace owned by the pool */
} gdn_pool_info;

/* Create a pool of num_slots slots for num_layers GDN layers on the current
 * CUDA device.  (slot, layer) lives at base + (slot * num_layers + layer) *
 * slot_bytes and holds [S: Hv x dv x dk fp32 | conv buffer: (W-1) x C io].
 * All slots start zeroed and free.  Allocates the state memory and the
 * prefill workspace (cudaMalloc) and, for the chunked prefill (d = 128 with
 * max_prefill_tokens > 0), a second stream (the device's highest priority) and four
 * events that a prefill running in several segments uses internally; *out receives the pool.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, CUDA (allocation failed). */
int gdn_pool_create(const gdn_shape* shape, int num_slots, int num_layers, gdn_pool** out);

/* Free the pool and everything it owns ("cleanup").  Waits for the device. */
int gdn_pool_destroy(gdn_pool* pool);

/* Mark every slot free and enqueue, on `stream`, the clearing of the device-side allocation
 * flags and the zeroing of all state memory ("reset"): work queued on `stream` before the call
 * still sees its slots allocated. */
int gdn_pool_reset(gdn_pool* pool, void* stream);

/* Take a free slot ("add slot").  The slot is zero (S and conv buffer of every
 * layer) once work already enqueued by recycle/reset on their streams has run.
 * Errors: INVALID_ARG, POOL_FULL. */
int gdn_slot_alloc(gdn_pool* pool, int* slot_id);

/* Return a slot to the free list ("recycle slot") after enqueuing, on
 * `stream`, the clearing of its device-side allocation flag and the zeroing of
 * its S and conv buffer in every layer, so that a later owner starts from a
 * clean state (the slot-reuse contamination checks of the qLLM README,
 * "Results").  Work queued on `stream` before the call still sees the slot
 * allocated.  Errors: INVALID_ARG, BAD_SLOT (free or out of range). */
int gdn_slot_recycle(gdn_pool* pool, int slot_id, void* stream);

/* Device address of (slot, layer) (host computation, no GPU work). */
int gdn_slot_addr(gdn_pool* pool, int layer, int slot_id, uint64_t* addr);

/* Snapshot / restore of one slot, for per-slot prefix reuse and checkpoints (issue #5279,
 * "What done needs" item 6 and phase P7: per-slot prefix reuse with longest-prefix
 * admission; the qLLM README, "What's still open": prefix caching is off because a
 * recurrent state cannot be rebuilt from a cached KV prefix -- a snapshot of the state is
 * what can be reused).  A snapshot is num_layers * slot_bytes bytes (gdn_pool_get_info):
 * every layer's S and conv buffer in the pool's own layout.
 * gdn_slot_snapshot copies the slot's layers to dst; gdn_slot_restore overwrites an
 * allocated slot's layers with src.  dst / src may be device or host memory (pinned host
 * memory keeps the copy asynchronous); the copy is enqueued on `stream`.
 * Errors: INVALID_ARG, BAD_SLOT (free or out of range), CUDA. */
int gdn_slot_snapshot(gdn_pool* pool, int slot_id, void* dst, void* stream);
int gdn_slot_restore(gdn_pool* pool, int slot_id, const void* src, void* stream);

/* Enqueue on `stream` the gather out_dev[i] = address of (slot_ids_dev[i], layer),
 * for i < m: the device u64 slot-pointer array of issue #5279 phase P5.  An id
 * that is out of range or not allocated gives 0 and sets GDN_DEV_BAD_SLOT_ID.
 * Errors: INVALID_ARG. */
int gdn_slot_ptrs(gdn_pool* pool, int layer, const int* slot_ids_dev, int m, uint64_t* out_dev, void* stream);

/* Register the parameters of one layer (device fp32 arrays, borrowed until
 * replaced or the pool is destroyed): conv_w [C][W] (tap W-1 multiplies the
 * current token), A_log [Hv], dt_bias [Hv], norm_w [dv] (shared by all heads).
 * Errors: INVALID_ARG. */
int gdn_layer_params(gdn_pool* pool, int layer, const float* conv_w, const float* A_log, const float* dt_bias,
                     const float* norm_w);

/* One decode step of `layer` for m sequences ("decode step"): row i of
 * q_dev..z_dev is the current token of the sequence whose (slot, layer) state
 * is at slot_ptrs_dev[i].  For each row: conv + SiLU against the slot's conv
 * buffer (which then shifts by one token), L2 norms, gates, the delta-rule
 * update of every v-head's S in place, the gated RMSNorm; out_dev[i] receives
 * the result.  The slot pointers must be distinct.  Each row's result depends
 * only on that row's inputs and state, never on m or the other rows.  The call only
 * enqueues one kernel, so a sequence of decode steps can be captured into a CUDA graph
 * keyed by the slot-pointer array (issue #5279 phase P8); the first call for a given
 * shape and dtypes also sets the kernel's attributes, so make one call before capturing.
 * Errors: INVALID_ARG, NO_PARAMS, CUDA (launch). */
int gdn_decode_step(gdn_pool* pool, int layer, const uint64_t* slot_ptrs_dev, int m, const void* q_dev,
                    const void* k_dev, const void* v_dev, const void* a_dev, const void* b_dev, const void* z_dev,
                    void* out_dev, void* stream);

/* Varlen prefill of `layer` ("setup+prefill"): n_seqs sequences packed along
 * the token axis, sequence s owning rows [cu_seqlens_dev[s], cu_seqlens_dev[s+1])
 * and slot slot_ids_dev[s].  Each sequence continues from its slot's current S
 * and conv buffer (zero after alloc/recycle), so a prompt may be split across
 * calls, and leaves its final S and conv buffer in the slot where
 * gdn_decode_step reads them (the System Design page, "GDN Kernel Dispatch
 * Detail": prefill, then "Update temporal_state").  total_tokens must equal
 * cu_seqlens_dev[n_seqs] and not exceed the pool's max_prefill_tokens; slot
 * ids must be allocated and distinct; n_seqs may be up to max_prefill_tokens + 64.
 * At d = 128 a call whose 64-token chunks (counted per sequence) exceed the pool's chunk
 * records runs as several pre-pass / state-pass segments, each continuing from the states
 * the one before left in the slots; their state passes run on the pool's second stream,
 * forked from `stream` and joined back by events (stream-capture safe), so that one
 * segment's state pass overlaps the next one's pre-pass.  The call's work is ordered after
 * earlier work on `stream` and later work on `stream` after all of it.  q, k, v, z and out are row-major
 * [total_tokens][width] device buffers whose base addresses are 16-B aligned
 * (they are moved in 16-B pieces and, at d = 128 in bf16, by tensor copies).
 * Uses the pool's workspace: calls on one pool must not overlap on the GPU.
 * Errors: INVALID_ARG (incl. a misaligned row buffer), NO_PARAMS,
 * UNSUPPORTED_SHAPE (too many tokens or sequences), CUDA. */
int gdn_prefill_varlen(gdn_pool* pool, int layer, const int* cu_seqlens_dev, const int* slot_ids_dev, int n_seqs,
                       int total_tokens, const void* q_dev, const void* k_dev, const void* v_dev, const void* a_dev,
                       const void* b_dev, const void* z_dev, void* out_dev, void* stream);

/* One continuous-batching step of `layer` over a mixed batch (issue #5279's serving loop):
 * m decode rows exactly as gdn_decode_step (d* arguments) and n_seqs prefill
 * sequences exactly as gdn_prefill_varlen (p* arguments), in one call.  The result equals
 * gdn_decode_step(...) followed by gdn_prefill_varlen(...) on `stream`, bit for bit.  The
 * decode kernel runs on an internal stream of the pool, forked from `stream` by an event and
 * joined back before the call's work ends.  When the prefill's state pass (one SM per CTA,
 * two CTAs per sequence and v-head) leaves at least 16 SMs idle, the state pass runs on the
 * pool's second stream after the pre-pass and the decode, sized for the idle SMs, beside it;
 * otherwise the decode overlaps the whole prefill.  The work of the call is ordered after
 * earlier work on `stream`, and later work on `stream` is ordered after all of it.  The fork and join are stream-capture safe; the first call creates
 * the internal stream and events on the current device, so make one call before capturing.
 * The decode rows' slots and the prefill sequences' slots must be different slots (each
 * call's own rules apply within its part): a kernel on `stream` compares them first, and if
 * any slot is named by both parts it sets GDN_DEV_SLOT_OVERLAP and neither part runs (no
 * output, state or conv buffer is written).  m = 0 or n_seqs = 0 leaves that part out.  Calls
 * on one pool from several host threads at once are not supported.
 * Errors: those of the two calls; every argument is checked before anything is enqueued. */
int gdn_mixed_step(gdn_pool* pool, int layer, const uint64_t* slot_ptrs_dev, int m, const void* dq_dev,
                   const void* dk_dev, const void* dv_dev, const void* da_dev, const void* db_dev, const void* dz_dev,
                   void* dout_dev, const int* cu_seqlens_dev, const int* slot_ids_dev, int n_seqs, int total_tokens,
                   const void* pq_dev, const void* pk_dev, const void* pv_dev, const void* pa_dev, const void* pb_dev,
                   const void* pz_dev, void* pout_dev, void* stream);

/* Allocation-free varlen prefill.  The pages have no counterpart of this call; it
 * exists for callers that cannot call cudaMalloc -- code that runs where device memory
 * is owned and budgeted by someone else, or in a phase that must not allocate -- and so
 * cannot create a pool or its workspace.  It runs the same kernels as
 * gdn_prefill_varlen and allocates nothing: its scratch is one static device array of
 * 64 MiB inside libgdn (held by every GPU that loads the library until the process
 * exits), and the state slots are memory the caller owns.
 *   shape         as for gdn_pool_create (max_prefill_tokens is ignored).
 *   conv_w, A_log, dt_bias, norm_w   the layer's device parameters (as gdn_layer_params).
 *   states_dev    num_slots slots laid out like one layer of a pool: slot i at
 *                 states_dev + i * slot_bytes, slot_bytes = the 256-rounded sum of
 *                 Hv*dv*dk*4 (fp32 S) and (W-1)*C*io_size (conv buffer); 256-B aligned.
 *   cu_seqlens_dev, slot_ids_dev, n_seqs, total_tokens, q..z, out   as for gdn_prefill_varlen
 *                 (every slot id below num_slots counts as allocated).
 *   status_dev    a device word receiving GDN_DEV_* bits (OR-ed in), or NULL to drop them.
 * The scratch is shared by every call and keeps the last call's contents; every value the
 * kernels read from it is written earlier in the same call, so nothing needs clearing, but
 * calls that overlap on the GPU (on different streams, or from different host threads)
 * race on it.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it for the life of the process; make that first call
 * before any stream capture, and do not call this entry point again after a
 * cudaDeviceReset in the same process (the kept address does not survive it).
 * Errors: INVALID_ARG; UNSUPPORTED_SHAPE when the shape is not built or the call needs more
 * than the 64 MiB of scratch (at Hqk 16, Hv 32, d 128 about 37 KB per token plus 2.4 MB per
 * sequence, i.e. up to 1 728 tokens of one sequence per call: split longer prompts into
 * several calls, which continue from the slots' state); CUDA. */
int gdn_prefill_varlen_noalloc(const gdn_shape* shape, const float* conv_w, const float* A_log, const float* dt_bias,
                               const float* norm_w, void* states_dev, int num_slots, const int* cu_seqlens_dev,
                               const int* slot_ids_dev, int n_seqs, int total_tokens, const void* q_dev,
                               const void* k_dev, const void* v_dev, const void* a_dev, const void* b_dev,
                               const void* z_dev, void* out_dev, unsigned int* status_dev, void* stream);

/* The projections around the layer (the layer tree's in_proj_qkv / in_proj_z / in_proj_b /
 * in_proj_a and out_proj), bf16 on the tensor cores with fp32 accumulation.
 *
 * gdn_in_proj: the four input projections as one GEMM.  x_dev [T][hidden] holds the hidden
 * states; w_in_dev [N][hidden] is the concatenation of the weight rows of q (Hqk*dk rows), k
 * (Hqk*dk), v (Hv*dv), z (Hv*dv), a (Hv) and b (Hv), N their total, each row one output
 * feature.  Row t of q_dev [T][Hqk*dk], k_dev, v_dev [T][Hv*dv], z_dev, a_dev [T][Hv] and b_dev
 * receives x_t times the matching weight rows, rounded to bf16: the buffers and layouts that
 * gdn_decode_step and gdn_prefill_varlen read.
 * gdn_out_proj: y_dev [T][hidden] = o_dev [T][Hv*dv] times w_out_dev^T, w_out_dev [hidden][Hv*dv].
 * shape: io_dtype (and, for gdn_out_proj, out_dtype) must be bf16; hidden a positive multiple of
 * 64 (and Hv*dv, the out_proj reduction, too); dk, dv multiples of 8.  Every buffer is
 * row-major, contiguous, 16-B aligned, caller-owned.  status_dev: a device word receiving
 * GDN_DEV_TIMEOUT if a bounded wait of the kernel ran out, or NULL (a library word is used).
 * One launch on `stream`; no allocation, no host sync.
 * Errors: INVALID_ARG (shape, sizes, NULL or misaligned buffer); CUDA. */
int gdn_in_proj(const gdn_shape* shape, int hidden, int T, const void* x_dev, const void* w_in_dev, void* q_dev,
                void* k_dev, void* v_dev, void* z_dev, void* a_dev, void* b_dev, unsigned int* status_dev,
                void* stream);
int gdn_out_proj(const gdn_shape* shape, int hidden, int T, const void* o_dev, const void* w_out_dev, void* y_dev,
                 unsigned int* status_dev, void* stream);

/* Synchronise `stream`, then read and clear the pool's device status word.
 * Returns the GDN_DEV_* bits (>= 0), or CUDA / INVALID_ARG. */
int gdn_last_device_status(gdn_pool* pool, void* stream);

/* Host-side facts about the pool. */
int gdn_pool_get_info(gdn_pool* pool, gdn_pool_info* info);

/* Static text for a gdn_status code. */
const char* gdn_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
