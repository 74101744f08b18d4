/*
 * moe.h — C ABI of the B300 routed Mixture-of-Experts layer with an LRU expert
 * cache fed from pinned host memory.
 *
 * The operation (what one moe_layer_forward call computes), following
 * "FreeToken量子化：MoE推論のセットアップガイド" (freetoken.wiki, architecture
 * page: two-tier expert memory, decode LRU cache, prefill whole-layer double
 * buffering) and the bhrtaym-blog post on FreeToken (section on the four MoE
 * backends, `offload`: experts live in host RAM, the GPU holds LRU slots,
 * misses stream over PCIe):
 *
 *   logits[t,e] = sum_h hidden[t,h] * router_w[e,h]      (one fixed fp32 order)
 *   p[t,:]      = softmax(logits[t,:])
 *   idx[t,0..k) = the k largest logits (ties: lower expert index), descending
 *   gate[t,j]   = p[t,idx[t,j]] / sum_j' p[t,idx[t,j']]
 *   out[t]      = sum_j gate[t,j] * FFN_{idx[t,j]}(hidden[t]) + sum_s SHARED_s(hidden[t])
 *   FFN_e(x)    = W_down,e ( silu(W_gate,e x) * (W_up,e x) )
 *
 * Every routed expert of every layer lives in a library-owned pinned host
 * bank; the GPU holds one pool of S expert slots shared by all layers. Each
 * call looks its experts up in a device-side LRU table. Misses of prefill calls
 * (T > 8) are copied into the pool with cudaMemcpyAsync on side streams, and
 * with MOE_CACHE_PREFETCH_NEXT_LAYER all experts of layer+1 also stream into
 * the pool while this layer computes, when the pool has room for both. Decode
 * calls (T <= 8) with FP4 or FP8 weights run as one kernel that copies its own misses
 * from the mapped banks (or, with MOE_CACHE_HOST_MISSES, waits for the host's
 * cudaMemcpyAsync copies).
 *
 * Calls are asynchronous: moe_layer_forward enqueues the call's kernels and
 * returns. A service thread owned by the handle reads each call's cache result
 * from mapped host memory; for host-copied misses it issues the copies and
 * then releases the call's expert kernels, which wait for that release on the
 * device (bounded). A call whose experts all hit releases itself on the
 * device. Errors that the device side of a call finds (capacity, bounded-wait
 * timeouts) are reported by the next moe_layer_forward or moe_sync.
 *
 * Conventions
 *  - Every call returns MOE_OK (0) or a negative moe_status. Nothing throws and
 *    nothing aborts. moe_last_error() gives a human-readable reason.
 *  - Device pointers: hidden, router_w, out (caller-owned, caller keeps them
 *    alive until the work on `stream` has completed).
 *  - Host pointers: everything in moe_model_desc / moe_expert_host / result
 *    buffers; the library copies what it keeps before returning.
 *  - One handle is used by one host thread at a time (moe_load_expert excepted:
 *    see there), and all forward calls on a handle are issued on one CUDA
 *    stream (the cache's slot reuse is ordered by it).
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID = -1,   /* bad argument or unsupported shape */
    MOE_ERR_OOM = -2,       /* host (pinned) or device allocation failed */
    MOE_ERR_CUDA = -3,      /* a CUDA runtime call failed */
    MOE_ERR_CAPACITY = -4,  /* the experts one call needs do not fit in the pool */
    MOE_ERR_TIMEOUT = -5,   /* a bounded device wait gave up */
    MOE_ERR_STATE = -6      /* call out of order (e.g. forward before moe_cache_config) */
} moe_status;

typedef enum moe_weight_fmt {
    MOE_FMT_FP32 = 0,   /* float32 rows */
    MOE_FMT_BF16 = 1,   /* bfloat16 rows */
    MOE_FMT_NVFP4 = 2,  /* E2M1 codes, E4M3 scale per 16 elements, fp32 scale per tensor */
    MOE_FMT_MXFP4 = 3,  /* E2M1 codes, E8M0 scale per 32 elements */
    MOE_FMT_FP8 = 4     /* E4M3 codes, fp32 scale per tensor */
} moe_weight_fmt;

typedef enum moe_act_dtype { MOE_ACT_FP32 = 0, MOE_ACT_BF16 = 1 } moe_act_dtype;

/* MOE_MODE_LINEAR_TEST replaces silu by the identity; it exists so that tests
 * can check the layer against closed forms. */
typedef enum moe_act_mode { MOE_MODE_SWIGLU = 0, MOE_MODE_LINEAR_TEST = 1 } moe_act_mode;

#define MOE_DECODE_MAX_T 8                /* T <= 8: decode path; T > 8: prefill path */
#define MOE_CACHE_PREFETCH_NEXT_LAYER 1u  /* prefill: stream layer+1 behind layer */
#define MOE_CACHE_LOG_EVENTS 2u           /* keep a per-expert hit/miss event log */
#define MOE_CACHE_SYNC_MISSES 4u          /* host-copied misses: service each call's misses
                                             before its expert kernels are launched (the
                                             calling thread waits for the routing kernel and
                                             the copies); for debugging and for tools that
                                             serialise launches */
#define MOE_CACHE_HOST_MISSES 8u          /* decode calls with FP4/FP8 weights: the host copies
                                             their misses with cudaMemcpyAsync on a side stream
                                             and the decode kernel waits (bounded) for its
                                             release; by default that kernel copies its misses
                                             itself, reading the mapped pinned banks */

typedef struct moe_model_desc {
    int32_t num_layers;   /* L >= 1 */
    int32_t num_experts;  /* E routed experts per layer, 1..1024 */
    int32_t num_shared;   /* always-on shared experts per layer, 0..1 */
    int32_t top_k;        /* k, 1..min(E, 32) */
    int32_t hidden;       /* H; multiple of 128 (FP32 weights: multiple of 8) */
    int32_t inter;        /* I; multiple of 128 (FP32 weights: any >= 1) */
    int32_t weight_fmt;   /* moe_weight_fmt */
    int32_t act_dtype;    /* moe_act_dtype of hidden, router_w and out */
    int32_t act_mode;     /* moe_act_mode */
    int32_t max_tokens;   /* largest T a forward call may pass (0 = 4096) */
    int32_t device;       /* CUDA device ordinal */
} moe_model_desc;

/* One weight tensor in the canonical host layout: row-major [N, K] with K the
 * input dimension (gate, up: [I, H]; down: [H, I]).
 *  FP32 / BF16: data = N*K elements; scales unused.
 *  NVFP4: data = N*K/2 bytes, element 2i in the low nibble of byte i;
 *         scales = N*K/16 E4M3 bytes (row-major [N, K/16]); global_scale used.
 *  MXFP4: data as NVFP4; scales = N*K/32 E8M0 bytes ([N, K/32]).
 *  FP8:   data = N*K E4M3 (FN) bytes, one per element; scales unused;
 *         global_scale used (weight = code * global_scale). The bhrtaym-blog
 *         post names FP8 among the supported formats (section on supported
 *         models and quantisation formats) without a layout; this is the
 *         per-tensor-scaled E4M3 reading, the same per-tensor scale NVFP4
 *         carries. */
typedef struct moe_tensor_host {
    const void* data;
    const uint8_t* scales;
    float global_scale;
} moe_tensor_host;

typedef struct moe_expert_host {
    moe_tensor_host gate, up, down;
} moe_expert_host;

typedef struct moe_stats_t {
    uint64_t calls, decode_calls, prefill_calls;
    uint64_t hits, misses;                    /* demand accesses of routed experts */
    uint64_t prefetch_hits, prefetch_misses;  /* next-layer prefetch batches */
    uint64_t evictions;
    uint64_t copies_h2d, bytes_h2d;           /* expert copies issued */
    uint64_t device_errors;
    uint64_t kernel_launches;                 /* CUDA kernels this library launched */
} moe_stats_t;

/* Per-kernel device time and algorithmic bytes, measured with CUDA events
 * recorded around the library's own launches on the launching stream (and
 * around each call's copies on the copy stream) while timing is enabled.
 * Algorithmic bytes count what each step must move at least once: the active
 * experts' weights and block scales, the activations read and the results
 * written. */
typedef struct moe_timing_t {
    uint64_t calls;
    double route_ms;      /* routing kernel: router, top-k, permutation, cache lookup (all calls) */
    double gate_up_ms;    /* gate/up projection + SwiGLU (decode with FP4/FP8 weights: the whole
                             expert kernel, gate/up and down+combine) */
    double down_ms;       /* down projection (+ combine, decode) */
    double combine_ms;    /* prefill combine */
    double copy_ms;       /* expert copies (misses and prefetch) on the copy stream (all calls) */
    uint64_t gate_up_bytes, down_bytes, combine_bytes, copy_bytes;
    uint64_t resident_calls;  /* calls whose expert kernels did not wait for copies (no demand
                                 misses, no prefetch of an earlier call outstanding):
                                 gate_up/down/combine ms and bytes cover only these */
} moe_timing_t;

typedef struct moe_event {
    int32_t layer, expert, hit, slot, evicted_key, prefetch;
} moe_event;

typedef struct moe_handle moe_handle;

/* Creates a handle for one MoE layer stack (the layer whose experts the pages
 * keep in host RAM with the GPU as their cache: freetoken.wiki architecture
 * page, two-tier expert memory paragraph). Validates the shape, picks the
 * device, creates the copy streams and events, and allocates the per-call
 * device scratch (sized for max_tokens). Host banks are allocated lazily per
 * layer by moe_load_expert. Returns MOE_ERR_INVALID for an unsupported shape,
 * MOE_ERR_OOM/CUDA on allocation failure (nothing is leaked). */
int moe_init(const moe_model_desc* desc, moe_handle** out);

/* Bytes of one expert in the library's device layout: the unit the cache
 * stores and copies (one expert is the unit of the pages' expert cache,
 * freetoken.wiki architecture page, two-tier expert memory paragraph). */
int moe_expert_bytes(const moe_model_desc* desc, size_t* bytes);

/* Writes one expert, given in the canonical host layout, into `blob` (host
 * memory of blob_bytes >= moe_expert_bytes) in the library's device layout:
 * the bytes moe_load_expert keeps in its pinned bank and a cache slot holds.
 * Host-only (no device is touched); for tools that prepare or inspect blobs.
 * MOE_ERR_INVALID for a bad shape, NULL pointers or a short buffer. The
 * formats are those the bhrtaym-blog post lists (section on supported models
 * and quantisation formats: MXFP4, NVFP4, FP8, BF16). */
int moe_repack_expert(const moe_model_desc* desc, const moe_expert_host* w, void* blob, size_t blob_bytes);

/* Copies one expert from the canonical host layout into the library's pinned
 * host bank (routed experts, expert < E) or into device-resident memory
 * (shared experts, E <= expert < E + num_shared), repacking it into the device
 * layout ("every routed expert lives in host RAM": freetoken.wiki architecture
 * page, two-tier expert memory paragraph). Banks are pinned and mapped into the
 * device's address space. The caller's buffers may be freed on return.
 * Synchronous. Unlike the other calls, which expect one host thread at a time
 * per handle, this one may run concurrently from several host threads (e.g.
 * one per layer), as long as no forward call is in progress; each (layer,
 * expert) is loaded by one thread. */
int moe_load_expert(moe_handle* h, int layer, int expert, const moe_expert_host* w);

/* A safe point that (re)builds the cache (freetoken.wiki architecture page:
 * the scheduler resizes and rebuilds the GPU expert cache at its safe points).
 * Waits until every enqueued call has finished, then makes a pool of
 * capacity_slots slots shared by all layers, empties the LRU table and the
 * event log, and clears errors of earlier calls (including a bounded-wait
 * timeout).
 *  flags: MOE_CACHE_PREFETCH_NEXT_LAYER, MOE_CACHE_LOG_EVENTS,
 *         MOE_CACHE_SYNC_MISSES, MOE_CACHE_HOST_MISSES; other bits give
 *         MOE_ERR_INVALID.
 *  pool_dev, pool_bytes: optional caller-owned device buffer for the pool
 *         (e.g. from the caller's framework allocator): 256-byte aligned, at
 *         least capacity_slots * moe_expert_bytes bytes, kept alive by the
 *         caller until the next moe_cache_config / moe_cache_resize with
 *         another buffer or moe_destroy; the library never frees it. NULL:
 *         the library allocates (and frees) the pool.
 * Every routed expert must have been loaded before the first forward call.
 * capacity_slots < top_k gives MOE_ERR_CAPACITY; a short or misaligned
 * pool_dev gives MOE_ERR_INVALID. */
int moe_cache_config(moe_handle* h, int capacity_slots, unsigned flags, void* pool_dev, size_t pool_bytes);

/* A safe point that resizes the cache and keeps what it holds (freetoken.wiki
 * architecture page: the cache is resized at the scheduler's safe points; the
 * bhrtaym-blog post's CLI table: `ft ctl cache --moe N` changes it without
 * stopping the server). Waits until every enqueued call has finished. The
 * min(capacity_slots, resident) most recently used experts stay cached with
 * their recency; a kept expert whose slot is below capacity_slots keeps its
 * slot, the other kept experts move, in ascending order of their old slot, to
 * the lowest slots left free; every other expert leaves the cache. Flags,
 * statistics, the event log and pending errors are unchanged.
 *  pool_dev, pool_bytes: as for moe_cache_config. The current pool buffer may
 *         be passed again (resizing in place: bytes of moved experts are copied
 *         within it); NULL: the library allocates a new pool (and frees the
 *         old one if it owned it).
 * MOE_ERR_STATE before moe_cache_config; capacity_slots < top_k gives
 * MOE_ERR_CAPACITY. */
int moe_cache_resize(moe_handle* h, int capacity_slots, void* pool_dev, size_t pool_bytes);

/* One call of MoE layer `layer_id` on T tokens (0 <= T <= max_tokens): the
 * routed MoE layer of the pages' offload backend (bhrtaym-blog post, section
 * on the four MoE backends, `offload`; freetoken.wiki architecture page:
 * decode runs hits on the GPU and copies misses into the cache over PCIe,
 * prefill streams the next layer's experts behind the current layer).
 *  hidden [T, H], router_w [E, H], out [T, H]: device memory in the handle's
 *         act_dtype, row-major, 16-byte aligned, owned by the caller (alive
 *         until `stream` has passed the call).
 *  stream: a cudaStream_t (NULL = the handle's own stream).
 * Returns without waiting for the device; the host blocks only when 16 calls
 * are already waiting for the service thread (with MOE_CACHE_SYNC_MISSES it
 * also blocks until the call's host-copied misses have landed). out is
 * complete once `stream` has passed the call. Decode (T <= 8) with FP4/FP8 weights
 * is one kernel that also copies the call's misses from the mapped banks
 * (unless MOE_CACHE_HOST_MISSES). A call whose experts exceed the pool leaves
 * the cache unchanged and out unwritten; the next moe_layer_forward or
 * moe_sync returns MOE_ERR_CAPACITY for it. Errors found for earlier calls are
 * returned before anything is enqueued. */
int moe_layer_forward(moe_handle* h, const void* hidden, const void* router_w, int layer_id,
                      int T, void* out, void* stream);

/* Waits until every call enqueued so far has been serviced and has finished on
 * the device (its stream and the copy streams), then returns the first error
 * found for any of them (MOE_ERR_CAPACITY once; MOE_ERR_TIMEOUT until the next
 * moe_cache_config), or MOE_OK. */
int moe_sync(moe_handle* h);

/* Cumulative cache counters since moe_init (or the last moe_stats_reset):
 * hits, misses, prefetches, evictions, bytes copied (the quantities the
 * pages' cache reasons about: freetoken.wiki architecture page, decode LRU
 * paragraph). Waits for the service thread. */
int moe_stats(moe_handle* h, moe_stats_t* s);
int moe_stats_reset(moe_handle* h);

/* enable != 0: start timing the following forward calls (accumulators reset);
 * enable == 0: stop. Measurement support (no counterpart on the pages). */
int moe_timing_enable(moe_handle* h, int enable);

/* Waits for all timed work to finish and returns the accumulated totals. */
int moe_timing(moe_handle* h, moe_timing_t* t);

/* Drains up to cap logged events (MOE_CACHE_LOG_EVENTS) into buf, in the order
 * the cache served them; *n receives the number written. One event per expert
 * access of the decode LRU and of the prefill prefetch batch (freetoken.wiki
 * architecture page, decode LRU and prefill double-buffering paragraphs). */
int moe_stats_events(moe_handle* h, moe_event* buf, int cap, int* n);

/* Host copies of the routing of the last forward call (any pointer may be
 * NULL): topk_idx [T*k], gates [T*k], perm [T*k], counts [E], uniq [E]
 * (ascending experts with at least one token; *n_uniq entries). Synchronous.
 * Test support (no counterpart on the pages). */
int moe_debug_routing(moe_handle* h, int32_t* topk_idx, float* gates, int32_t* perm,
                      int32_t* counts, int32_t* uniq, int32_t* n_uniq);

/* Host copy of the LRU table [L*E] (slot or -1) after the last call. Test
 * support (no counterpart on the pages). */
int moe_debug_lru_table(moe_handle* h, int32_t* table);

/* Router top-k that allocates nothing (the pages describe no counterpart: it
 * exists for callers that cannot call cudaMalloc, e.g. a plugin whose host
 * framework's memory pool owns all device memory, or a path that must not
 * allocate; moe_init allocates, so those callers cannot create a handle).
 * Computes, for T tokens, the router logits in the same fixed summation order
 * as moe_layer_forward, the softmax, the top-k experts (larger logit first,
 * ties to the lower index) and the renormalised gates.
 *  hidden [T, H], router_w [E, H]: device, act_dtype (MOE_ACT_*), 16-byte aligned
 *  topk_idx [T*k] int32, gates [T*k] float32: device outputs, written on stream
 *  stream: a cudaStream_t (NULL = legacy default stream), on the current device
 * Scratch: a file-scope device array of MOE_ROUTE_NOALLOC_MAX_LOGITS floats
 * (4 MiB, held by every GPU that loads the library until exit); T*E above it,
 * T above 8 * 65535 = 524280 (the token blocks of its logits grid), E > 1024,
 * k > min(E, 32), H not a positive multiple of 8 or too large for the
 * shared-memory tile give MOE_ERR_INVALID. A failed launch gives MOE_ERR_CUDA;
 * CUDA errors that other calls left pending are neither reported nor cleared.
 * Calls no allocator. The first call on a device, with that device current, looks the array's address up
 * (cudaGetSymbolAddress) and sets the kernel's shared-memory limit: make it
 * before any stream capture. All calls share the array and it keeps the last
 * call's contents; calls whose work overlaps on the GPU race on it. */
#define MOE_ROUTE_NOALLOC_MAX_LOGITS (1 << 20)
int moe_route_topk_noalloc(const void* hidden, const void* router_w, int T, int E, int H, int k, int act_dtype,
                           int32_t* topk_idx, float* gates, void* stream);

/* Human-readable reason of the handle's last failed call ("NULL handle" for NULL). */
const char* moe_last_error(const moe_handle* h);

/* Waits for the device, stops the service thread and frees everything the
 * library allocated (a caller-owned pool buffer is left alone). */
void moe_destroy(moe_handle* h);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
