// Internal definitions shared by the host runtime and the CUDA kernels of the
// routed MoE layer (not part of the public C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

constexpr int kDecodeMaxT = 8;     // T <= 8 takes the decode path
constexpr int kMaxExperts = 1024;  // E limit (router keeps E/32 logits per lane)
constexpr int kMaxTopK = 32;
constexpr int kGroupK = 128;       // K elements per device-order group
constexpr int kMaxSlots = 16384;   // pool slots (slot index fits 14 bits)
constexpr int kSortMax = 16384;    // bitonic sort size bound for victim selection

enum Fmt { FMT_FP32 = 0, FMT_BF16 = 1, FMT_NVFP4 = 2, FMT_MXFP4 = 3, FMT_FP8 = 4 };
enum Act { ACT_FP32 = 0, ACT_BF16 = 1 };

// Device layout of one expert ("blob"), identical in the pinned host bank and
// in a pool slot, so that a miss is one contiguous copy.
//
// Within every weight row, K is stored in "device order": each group of 128
// consecutive elements is reordered so that position 32q + 4s + i holds
// element 16s + 4q + i of the group (q < 4, s < 8, i < 4). A warp lane with
// quad index q then finds, in one contiguous 16-byte (FP4), 32-byte (FP8) or 64-byte (BF16)
// run, its operands for the eight m16n8k16 MMA steps s of the group, and step s
// covers exactly one 16-element NVFP4 scale block (half of an MXFP4 block).
// Activations fed to the same MMAs are stored in the same order.
//
// BF16 / FP32 blobs:
//   gu : gate/up rows [2I][H]. Rows come in blocks of 128: 64 gate rows then
//        the 64 up rows of the same intermediate units (FP32: plain [gate I][up I]).
//   d  : down rows [H][I].
// FP4 and FP8 blobs (NVFP4, MXFP4, FP8) are tiled for streaming: the gu region
// is I/8 tiles (tile u: rows 0-7 = gate units 8u..8u+7, rows 8-15 = their up
// units), the d region H/16 tiles (tile r: down rows 16r..16r+15); a tile is a
// run of chunks of up to 8 K-groups (1024 elements), and chunk c with ng groups
// is, for FP4,
//   codes  [16 rows][ng * 64 bytes]   (16-byte units of row r XOR-swizzled,
//                                      see fp4_code_off)
//   scales [16 rows][ng * sbpg bytes] (sbpg = 8 E4M3 (NVFP4) or 4 E8M0 (MXFP4)
//                                      bytes per group, canonical order)
// and for FP8 (one E4M3 byte per element, no block scales)
//   codes  [16 rows][ng * 128 bytes]  (see fp8_code_off)
// so that one 16-row x 1024-K slice of a projection is one contiguous run.
//   gsc: float[4] per-tensor scales (gate, up, down, 1) - NVFP4 and FP8; else 1.
struct BlobLayout {
    size_t gu, d, gsc, bytes;
    size_t gu_tile, d_tile;  // tiled formats: bytes of one tile of each region
    int sbpg;                // FP4: scale bytes per 128-element group (FP8: 0)
    int rowb;                // tiled formats: bytes of one tile row of one K group
};

constexpr int kTileRows = 16;
constexpr int kChunkGroups = 8;

// tiled formats: bytes of one tile row of one 128-element K group (codes and
// block scales)
__host__ __device__ constexpr int tiled_scale_bytes(int fmt) { return fmt == FMT_NVFP4 ? 8 : fmt == FMT_MXFP4 ? 4 : 0; }
__host__ __device__ constexpr int tiled_row_bytes(int fmt) { return fmt == FMT_FP8 ? 128 : 64 + tiled_scale_bytes(fmt); }

// tiled formats: offset of chunk c (all earlier chunks are full)
__host__ __device__ inline size_t tile_chunk_off(int c, int rowb) {
    return static_cast<size_t>(kTileRows) * kChunkGroups * c * rowb;
}
__host__ __device__ inline int fp4_chunk_groups(int G, int c) {
    return G - kChunkGroups * c < kChunkGroups ? G - kChunkGroups * c : kChunkGroups;
}
// offset, inside its chunk (ng groups), of the 16 code bytes of row r, group w,
// lane quad q. Rows of an even-ng chunk are 512-byte multiples apart, so the
// odd rows swap the two halves of each 128-byte bank window: the 8 lanes of a
// quarter-warp (rows 2m, 2m+1, quads 0-3) then hit 8 distinct 16-byte bank groups.
__host__ __device__ inline int fp4_code_off(int ng, int r, int w, int q) {
    const int x = ((r & 1) && !(ng & 1)) ? 4 : 0;
    return r * ng * 64 + (((w * 4 + q) ^ x) * 16);
}
__host__ __device__ inline int fp4_scale_off(int ng, int sbpg, int r, int w) {
    return kTileRows * ng * 64 + r * ng * sbpg + w * sbpg;
}
// FP8: offset, inside its chunk (ng groups), of half hf (MMA steps 4hf..4hf+3)
// of the 32 code bytes of row r, group w, lane quad q. A row of a group is one
// 128-byte bank window; odd rows swap the two halves of each quad's run, so the
// 8 lanes of a quarter-warp (rows 2m, 2m+1, quads 0-3) hit 8 distinct 16-byte
// bank groups.
__host__ __device__ inline int fp8_code_off(int ng, int r, int w, int q, int hf) {
    return (r * ng + w) * 128 + (((2 * q + hf) ^ (r & 1)) * 16);
}

// Written by the cache kernel into mapped host memory; read by the host after
// the cache kernel completes.
struct CallInfo {
    unsigned long long done;  // the call's sequence number, written last by the routing kernel
    int32_t status;          // 0 ok, else a negative moe_status
    int32_t n_uniq;
    int32_t n_hit, n_miss;   // demand batch
    int32_t n_pf, n_pf_hit, n_pf_miss;  // prefetch batch (n_pf = 0: none)
    int32_t n_events;
    int32_t dev_err;         // sticky device error word at the time of this call (0 = none)
    int32_t device_copied;   // 1: the call's misses were copied by its own kernel (decode)
    int32_t pad_;
    unsigned long long copy_ns;  // device-copied misses: first copy issued -> all landed (%globaltimer)
    // misses to copy: demand misses first, then prefetch misses
    int32_t miss_layer[2 * kMaxExperts];
    int32_t miss_expert[2 * kMaxExperts];
    int32_t miss_slot[2 * kMaxExperts];
    // event log of both batches in service order
    int32_t ev_layer[2 * kMaxExperts];
    int32_t ev_expert[2 * kMaxExperts];
    int32_t ev_hit[2 * kMaxExperts];
    int32_t ev_slot[2 * kMaxExperts];
    int32_t ev_evicted[2 * kMaxExperts];
    int32_t ev_prefetch[2 * kMaxExperts];
};

// Decode plan: what the decode expert kernel needs about each active expert,
// written by the routing kernel into one contiguous buffer (a 128-byte header
// with the number of active experts, then one 128-byte record per expert) so
// that the expert kernel fetches it with a single bulk copy.
struct DecExpert {
    const uint8_t* ptr;          // blob (pool slot or shared-expert area)
    int32_t row0, cnt;           // first h row, rows (tokens) of the expert
    int32_t tok[kDecodeMaxT];    // token of the expert's row n (n < cnt), else -1
    int32_t hrow[kDecodeMaxT];   // h row of token t, else -1
    float gate[kDecodeMaxT];     // routing gate of the expert's row n
    float gs[3];                 // per-tensor scales (filled by the expert kernel)
    int32_t pad;                 // decode kernel: 1 once gs holds the per-tensor scales
};
static_assert(sizeof(DecExpert) == 128, "decode plan record");
constexpr int kDecPlanHeader = 128;

// phase marks the decode kernel records per CTA when a trace buffer is given
// (MOE_TRACE): 0 start, 1 logits written, 2 barrier 1 passed, 3 plan done,
// 4 cache updated (CTA 0), 5 misses copied, 6 phase 1 done, 7 barrier 2
// passed, 8 phase 2 done, 9 end; 10 token and router rows staged, 11 logits
// computed, 12 top-k done, 13 first phase-1 stage landed, 14 last phase-1
// stage landed, 15 last phase-2 stage landed (all as the consumers saw them);
// producer: 16 first stage issued, 17 last phase-1 stage issued, 18 every
// stage issued, 19 last phase-1 stage landed, 20 producer set up
constexpr int kTracePoints = 24;
// calls whose entry / dependency-wait / exit times the trace buffer keeps
// after the per-CTA marks (4 words each: first entry, wait returned, last exit, unused)
constexpr int kTraceCalls = 64;

// Published by the CTA of the fused decode kernel that runs the cache lookup,
// for the kernel's other CTAs: the pool slots chosen for the call's misses (in
// the ascending order of the missed experts), valid once seq equals the call's
// sequence number.
struct DecPub {
    unsigned long long seq;
    int32_t slot[kMaxExperts];
};

struct CallArgs {
    // shape
    int T, E, k, H, I, n_shared, L, layer, S;
    int fmt, act, mode;
    int prefetch, log_events;
    // caller buffers (device)
    const void* hidden;    // [T][H] act
    const void* router_w;  // [E][H] act
    void* out;             // [T][H] act
    // scratch (device)
    void* xh;              // [T][H] f16 (FP4) or bf16 (BF16), device K-order
    float* logits;         // [T][E] (prefill with BF16 activations: the tensor cores' approximate logits)
    float* wnorm;          // [E] router row norms, rounded up (prefill tensor-core routing)
    int32_t tc_router;     // 1: this prefill call's logits come from the tensor cores
    unsigned long long* dlog;  // [kDecodeMaxT][E] decode logits: (call sequence << 32) | fp32 bits
    int32_t* topk;         // [T*k]
    float* gates;          // [T*k]
    int32_t* counts;       // [E]
    int32_t* offsets;      // [E+1]
    int32_t* perm;         // [T*k]
    int32_t* inv_perm;     // [T*k]
    int32_t* row_tok;      // [T*k + T*n_shared]
    float* row_gate;       // [T*k + T*n_shared]
    int32_t* act_expert;   // [E + n_shared]  active experts: routed (ascending), then shared
    int32_t* act_row0;     // [E + n_shared]  first h/Y row of the active expert
    int32_t* act_cnt;      // [E + n_shared]  rows (tokens) of the active expert
    const uint8_t** act_ptr;  // [E + n_shared] blob address
    int32_t* e2u;          // [E] active index of routed expert e, or -1
    int32_t* tok_row;      // [(E + n_shared) * 8] decode: h row of (active u, token t) or -1
    int32_t* act_slot;     // [E + n_shared]  pool slot of the active expert; shared: -(1 + layer*n_shared + s)
    void* xperm;           // [T*k + T*n_shared][H] gathered activations, device K-order (prefill): bf16,
                           // or f16 scaled per token row (NVFP4 / FP8 weights)
    float* xsc;            // [T] prefill, NVFP4 / FP8 weights: power of two of each token row in xperm
    float* xunr;           // [T*k + T*n_shared] its inverse, per gathered row
    int32_t* dev_err;      // [1] sticky device error word (bounded waits that gave up)
    int32_t* route_done;   // [1] routing CTAs finished in this call (0 between calls)
    // prefill permutation, computed in parts: each routing CTA b (8 tokens)
    // ranks its assignments among those of the same expert and adds its
    // per-expert counts; the permutation kernel sums each column over the
    // earlier CTAs to get every CTA's base row per expert
    int32_t* cacc;         // [E] per-expert assignment counts (0 between calls)
    int16_t* cntT;         // [E][nb] per-CTA counts of each expert (nb = ceil(max_tokens / 8))
    int16_t* lrank;        // [T*k] rank of assignment a among its CTA's assignments to the same expert
    int nb_max;            // column stride of cntT
    unsigned long long* bar_cnt;     // [3] arrival counters of the decode kernel's grid barriers
    unsigned long long dcall;        // decode kernel launches before this one since the counters were reset
    unsigned char* dplan;  // decode plan: header + (E + n_shared) records
    int32_t* n_uniq;       // [1]
    int32_t* n_active;     // [1]
    void* hbuf;            // [rows][I] intermediate (f16 / bf16 / f32)
    void* ybuf;            // [rows][H] bf16 down-projection rows (prefill)
    // cache (device)
    int32_t* table;        // [L*E] slot or -1
    int32_t* owner;        // [S] key or -1
    unsigned long long* stamp;  // [S] recency (0 = never filled)
    unsigned long long* clock;  // [1]
    const uint8_t* pool;   // S * blob bytes
    const uint8_t* shared_base;  // this layer's shared experts (n_shared blobs)
    BlobLayout lay;
    CallInfo* info;        // mapped host memory (device pointer): this call's record
    // miss pipeline: the expert kernels of call `seq` start once *ready >= seq.
    // The routing kernel releases the call itself when it has no demand misses
    // and self_release is set; otherwise the host writes seq after the copies.
    unsigned long long* ready;
    unsigned long long seq;
    int self_release;
    unsigned long long wait_ns;  // bound of every device-side wait
    // fused decode (FP4 weights, T <= 8)
    const uint8_t* const* banks;  // [L] device views of the mapped pinned host banks
    float* xmax;           // [8] max |x| of each token row (this call)
    unsigned int* hmax;    // [2][8] decode: per-token max |h| of a call (float bits), by call parity
    DecPub* pub;           // miss slots for the kernel's CTAs
    int device_misses;     // 1: the decode kernel copies its misses itself; 0: the host does
    unsigned long long* trace;  // optional [CTAs][kTracePoints] %globaltimer marks of the decode kernel
    int32_t trace_ctas;         // CTAs of the decode kernel (the trace's per-call ring follows their marks)
};

// Bounded wait of the expert kernels for their call's weights (one thread);
// false (and the device error word set) if the bound ran out.
__device__ __forceinline__ bool wait_ready(const CallArgs& a) {
    const volatile unsigned long long* r = a.ready;
    if (*r >= a.seq) {
        __threadfence();
        return true;
    }
    unsigned long long t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
        if (*r >= a.seq) {
            __threadfence();
            return true;
        }
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > a.wait_ns) {
            atomicExch(a.dev_err, 4);  // MOE_DEVERR_TIMEOUT_READY
            return false;
        }
        __nanosleep(64);
    }
}

// device error codes written to CallArgs::dev_err
enum DevErr {
    DEVERR_NONE = 0,
    MOE_DEVERR_TIMEOUT_PRODUCER = 1,
    MOE_DEVERR_TIMEOUT_MMA = 2,
    MOE_DEVERR_TIMEOUT_EPILOGUE = 3,
    MOE_DEVERR_TIMEOUT_READY = 4
};

// an opaque CUtensorMap (128 bytes, 64-byte aligned)
struct alignas(64) UmmaMap {
    unsigned char bytes[128];
};

// TMA descriptors of the prefill tensor-core path: the pool's gate/up and down
// regions (3-D: K, rows, slot), the resident shared experts (same), the gathered
// activations and the intermediate h (2-D: K, rows)
struct UmmaMaps {
    UmmaMap pool_gu, pool_d, shared_gu, shared_d, x, h;
    bool have_pool = false, have_io = false;
};

bool umma_map_2d(UmmaMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);
bool umma_map_3d(UmmaMap* m, const void* base, uint64_t slots, uint64_t slot_bytes, uint64_t rows, uint64_t cols,
                 uint32_t box_rows);
cudaError_t umma_set_attributes();
// gather + gate/up + down on the tensor cores (prefill, BF16 weights); records
// ev_gu after the gate/up GEMM when non-null
// prefill routing with BF16 activations: router row norms and approximate
// logits on the tensor cores (the routing kernel makes the top-k exact)
bool router_tc_eligible(const CallArgs& a);
cudaError_t launch_router_tc(const CallArgs& a, cudaStream_t s);
cudaError_t launch_prefill_umma(const CallArgs& a, const UmmaMaps& maps, int num_sms, cudaStream_t s,
                                cudaEvent_t ev_gu, int* launches);

// launchers; all enqueue on `s` and return cudaGetLastError()
// routing + permutation + LRU cache lookup: one kernel
cudaError_t launch_route(const CallArgs& a, cudaStream_t s);
// launches the expert kernels; records ev_gu after the gate/up kernel and
// ev_down after the down-projection kernel when they are non-null; *launches
// receives the number of kernels launched. Prefill with BF16 weights takes the
// tensor-core path when `maps` holds valid descriptors.
cudaError_t launch_experts(const CallArgs& a, cudaStream_t s, cudaEvent_t ev_gu, cudaEvent_t ev_down,
                           const UmmaMaps* maps, int num_sms, int* launches);
// decode (T <= 8) with FP4 weights: the whole call (router, top-k,
// permutation, cache lookup, miss copies, gate/up, down, combine) in one
// cooperative kernel
inline bool decode_fused(int fmt, int T) { return fmt >= FMT_NVFP4 && T <= kDecodeMaxT; }
cudaError_t decode_set_attributes();
// smem_ok: false when the shape's cache-lookup scratch does not fit
cudaError_t launch_decode(const CallArgs& a, int num_sms, cudaStream_t s, bool pdl);
// loads every expert kernel (called once by moe_init)
cudaError_t experts_preload();
// true when a prefill call of this shape takes the tensor-core path
inline bool prefill_uses_umma(int fmt, int T) { return fmt != FMT_FP32 && T > kDecodeMaxT; }

}  // namespace moe
