// Host runtime of the routed MoE layer: the C ABI declared in include/moe.h.
//
// Two-tier expert memory as on "FreeToken量子化：MoE推論のセットアップガイド"
// (freetoken.wiki, architecture page): every routed expert lives in host RAM
// (here: library-owned pinned banks, one per layer), the GPU holds one expert
// cache shared by all MoE layers (a pool of S slots), misses are copied over
// PCIe, and prefill streams the next layer's experts while the current layer
// computes. Cache resizing happens at a safe point (moe_cache_config), as the
// same page describes for the scheduler's safe points.
//
// Miss pipeline. moe_layer_forward only enqueues work: the routing kernel (which
// also runs the cache lookup) and the expert kernels of call number `seq` go on
// the caller's stream back to back, and the expert kernels wait on the device
// until a "ready" word reaches seq. The routing kernel writes the call's record
// (hits, misses with their slots, events) into a ring of mapped host memory. A
// service thread per handle reads the records in call order; for a call with
// misses it issues one cudaMemcpyAsync per missed expert (pinned bank -> pool
// slot) on the copy stream and then writes `ready = seq` on the same stream, so
// the expert kernels start once the copies have landed. A call whose experts
// all hit releases itself from inside the routing kernel, and the host is not
// on its critical path at all. Prefill prefetch copies of layer+1 go on the
// copy stream after the call's own release, and the next call is then released
// by the service thread behind them.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <mutex>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace moe {
cudaError_t routing_set_attributes();
}

using moe::BlobLayout;
using moe::CallArgs;
using moe::CallInfo;

namespace {

constexpr int kRing = 16;  // calls in flight between the caller and the service thread
typedef CUresult (*WriteValue64Fn)(CUstream, CUdeviceptr, cuuint64_t, unsigned int);

}  // namespace

// CUDA events of one timed forward call
struct TimedCall {
    uint64_t seq = 0;
    cudaEvent_t r0 = nullptr, r1 = nullptr, f0 = nullptr, f1 = nullptr, f2 = nullptr, f3 = nullptr;
    cudaEvent_t c0 = nullptr, c1 = nullptr;
    bool has_copy = false, has_combine = false, had_miss = false;
    bool fused = false;         // one decode kernel (r0 -> r1) covers the whole call
    bool dev_copy = false;      // its misses were copied by the kernel: copy_ns from the call record
    uint64_t copy_ns = 0;
    uint64_t gu_bytes = 0, down_bytes = 0, combine_bytes = 0, copy_bytes = 0;
};

// one enqueued call, as the service thread sees it
struct PendingCall {
    uint64_t seq = 0;
    int layer = 0, T = 0;
    bool self_release = true;
    bool fused = false;
    TimedCall* tc = nullptr;
};

struct moe_handle {
    moe_model_desc d{};
    BlobLayout lay{};
    int max_tokens = 0;
    // host banks: per layer, E blobs (pinned); loaded flags
    std::vector<uint8_t*> bank;
    std::vector<uint8_t> loaded;
    std::vector<uint8_t> layer_complete;  // 1 once every expert of the layer has been seen loaded (it stays so)
    std::vector<const uint8_t*> bank_dev;  // device views of the mapped banks
    bool banks_dirty = false;             // bank_dev changed since the device table was written
    // shared experts: device resident [L][n_shared] blobs
    uint8_t* shared_dev = nullptr;
    // pool and LRU state
    uint8_t* pool = nullptr;
    bool pool_owned = false;  // false: the caller's buffer (moe_cache_config / moe_cache_resize)
    int S = 0;
    unsigned flags = 0;
    int32_t* table = nullptr;
    int32_t* owner = nullptr;
    unsigned long long* stamp = nullptr;
    unsigned long long* clock = nullptr;
    // scratch
    void* scratch = nullptr;
    // prefill tensor-core path: TMA descriptors, SM count
    moe::UmmaMaps maps{};
    int num_sms = 148;
    CallArgs base{};
    // call records (mapped ring) and the ready word
    CallInfo* info_h = nullptr;
    CallInfo* info_d = nullptr;
    unsigned long long* ready = nullptr;       // device
    unsigned long long* ready_vals = nullptr;  // pinned host [kRing] (used without cuStreamWriteValue64)
    WriteValue64Fn write64 = nullptr;
    unsigned long long wait_ns = 5000000000ull;
    // host-side fault injection (MOE_FAULT=drop_release): the service thread
    // skips the release of the first call that has misses, so that its expert
    // kernels run into their bounded wait
    bool fault_drop_release = false;
    bool log = false;  // MOE_LOG: one stderr line per serviced call
    unsigned long long* trace = nullptr;  // MOE_TRACE: the decode kernel's per-CTA phase marks
    bool last_fused = false;
    unsigned long long dcalls = 0;  // decode kernel launches since the barrier counters were reset
    // streams / events
    // miss copies alternate between two copy streams (the copy engines overlap
    // one copy's setup with another's transfer); `copy` joins `copy2` before
    // every release, so a release always follows all of its call's copies
    cudaStream_t stream = nullptr, copy = nullptr, copy2 = nullptr;
    cudaEvent_t ev_join = nullptr;
    cudaEvent_t ev_pf = nullptr;  // a decode call's stream waits on it for earlier prefetch copies
    // enqueue side (caller's thread)
    uint64_t submitted = 0;
    bool prefetch_may_be_pending = false;
    int last_T = 0;
    cudaStream_t last_stream = nullptr;
    // service thread
    std::thread svc;
    std::mutex mu;
    std::condition_variable cv, done_cv;
    std::deque<PendingCall> queue;
    std::atomic<uint64_t> serviced{0};
    bool stop = false;
    // errors found while servicing, reported by the next call (mu)
    int pending_err = MOE_OK;
    std::string pending_msg;
    bool sticky_timeout = false;
    // timing
    bool timing = false;
    moe_timing_t tm{};
    std::deque<TimedCall*> pending;
    std::vector<TimedCall*> spare;
    // stats (mu)
    moe_stats_t st{};
    std::vector<moe_event> events;
    // message of the last failed call (err_mu: loaders may fail concurrently)
    std::mutex err_mu;
    std::string err;
    // host banks are allocated by whichever loader thread first needs them
    std::mutex load_mu;
};

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int fail(moe_handle* h, int code, const std::string& msg) {
    if (h) {
        std::lock_guard<std::mutex> lk(h->err_mu);
        h->err = msg;
    }
    return code;
}

int cuda_fail(moe_handle* h, cudaError_t e, const char* what) {
    return fail(h, MOE_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define CK(h, x)                                          \
    do {                                                  \
        cudaError_t e_ = (x);                             \
        if (e_ != cudaSuccess) return cuda_fail(h, e_, #x); \
    } while (0)

int validate_desc(const moe_model_desc* d, std::string* why) {
    auto bad = [&](const char* m) { *why = m; return MOE_ERR_INVALID; };
    if (!d) return bad("desc is NULL");
    if (d->num_layers < 1) return bad("num_layers must be >= 1");
    if (d->num_experts < 1 || d->num_experts > moe::kMaxExperts) return bad("num_experts must be in 1..1024");
    if (d->num_shared < 0 || d->num_shared > 1) return bad("num_shared must be 0 or 1");
    if (d->top_k < 1 || d->top_k > moe::kMaxTopK || d->top_k > d->num_experts) return bad("top_k must be in 1..min(E, 32)");
    if (d->weight_fmt < 0 || d->weight_fmt > 4) return bad("unknown weight_fmt");
    if (d->act_dtype < 0 || d->act_dtype > 1) return bad("unknown act_dtype");
    if (d->act_mode < 0 || d->act_mode > 1) return bad("unknown act_mode");
    if (d->max_tokens < 0) return bad("max_tokens must be >= 0");
    if (d->weight_fmt == moe::FMT_FP32) {
        if (d->hidden < 8 || d->hidden % 8) return bad("hidden must be a positive multiple of 8");
        if (d->inter < 1) return bad("inter must be >= 1");
    } else {
        if (d->hidden < 128 || d->hidden % 128) return bad("hidden must be a positive multiple of 128");
        if (d->inter < 128 || d->inter % 128) return bad("inter must be a positive multiple of 128");
    }
    const size_t xbytes = static_cast<size_t>(8) * d->hidden * (d->act_dtype == moe::ACT_BF16 ? 2 : 4);
    if (xbytes > 192 * 1024) return bad("hidden too large for the router's shared-memory tile");
    return MOE_OK;
}

BlobLayout layout_for(const moe_model_desc& d) {
    BlobLayout L{};
    const size_t H = d.hidden, I = d.inter;
    size_t o = 0;
    switch (d.weight_fmt) {
        case moe::FMT_FP32:
            L.gu = 0; o = 2 * I * H * 4;
            L.d = align_up(o, 256); o = L.d + H * I * 4;
            L.gsc = align_up(o, 256); o = L.gsc + 16;
            break;
        case moe::FMT_BF16:
            L.gu = 0; o = 2 * I * H * 2;
            L.d = align_up(o, 256); o = L.d + H * I * 2;
            L.gsc = align_up(o, 256); o = L.gsc + 16;
            break;
        default: {
            L.sbpg = moe::tiled_scale_bytes(d.weight_fmt);
            L.rowb = moe::tiled_row_bytes(d.weight_fmt);
            L.gu_tile = static_cast<size_t>(moe::kTileRows) * (H / moe::kGroupK) * L.rowb;
            L.d_tile = static_cast<size_t>(moe::kTileRows) * (I / moe::kGroupK) * L.rowb;
            L.gu = 0; o = (I / 8) * L.gu_tile;
            L.d = align_up(o, 256); o = L.d + (H / moe::kTileRows) * L.d_tile;
            L.gsc = align_up(o, 256); o = L.gsc + 16;
        }
    }
    L.bytes = align_up(o, 1024);
    return L;
}

// device gu row of canonical gate (which = 0) / up (which = 1) row i
inline size_t gu_row(int i, int which) { return static_cast<size_t>(i / 64) * 128 + 64 * which + (i % 64); }

// one canonical row of K elements -> device K-order
void reorder_row_fp4(const uint8_t* src, uint8_t* dst, int K) {
    for (int j = 0; j < K / 128; ++j) {
        const uint8_t* s = src + 64 * j;
        uint8_t* d = dst + 64 * j;
        for (int q = 0; q < 4; ++q)
            for (int st = 0; st < 8; ++st) {
                d[16 * q + 2 * st] = s[8 * st + 2 * q];
                d[16 * q + 2 * st + 1] = s[8 * st + 2 * q + 1];
            }
    }
}

void reorder_row_fp8(const uint8_t* src, uint8_t* dst, int K) {
    for (int j = 0; j < K / 128; ++j) {
        const uint8_t* s = src + 128 * j;
        uint8_t* d = dst + 128 * j;
        for (int q = 0; q < 4; ++q)
            for (int st = 0; st < 8; ++st) std::memcpy(d + 32 * q + 4 * st, s + 16 * st + 4 * q, 4);
    }
}

void reorder_row_bf16(const uint16_t* src, uint16_t* dst, int K) {
    for (int j = 0; j < K / 128; ++j) {
        const uint16_t* s = src + 128 * j;
        uint16_t* d = dst + 128 * j;
        for (int q = 0; q < 4; ++q)
            for (int st = 0; st < 8; ++st) std::memcpy(d + 32 * q + 4 * st, s + 16 * st + 4 * q, 8);
    }
}

// canonical expert -> device blob (host memory)
int repack_expert(const moe_model_desc& d, const BlobLayout& L, const moe_expert_host* w, uint8_t* blob,
                  std::string* why) {
    const int H = d.hidden, I = d.inter;
    const moe_tensor_host* ts[3] = {&w->gate, &w->up, &w->down};
    for (int i = 0; i < 3; ++i) {
        if (!ts[i]->data) { *why = "expert tensor data is NULL"; return MOE_ERR_INVALID; }
        const bool scaled = d.weight_fmt == moe::FMT_NVFP4 || d.weight_fmt == moe::FMT_MXFP4;
        if (scaled && !ts[i]->scales) { *why = "expert scales are NULL"; return MOE_ERR_INVALID; }
    }
    std::memset(blob, 0, L.bytes);
    float* gsc = reinterpret_cast<float*>(blob + L.gsc);
    gsc[0] = gsc[1] = gsc[2] = gsc[3] = 1.0f;
    switch (d.weight_fmt) {
        case moe::FMT_FP32: {
            const size_t n = static_cast<size_t>(I) * H;
            std::memcpy(blob + L.gu, w->gate.data, n * 4);
            std::memcpy(blob + L.gu + n * 4, w->up.data, n * 4);
            std::memcpy(blob + L.d, w->down.data, n * 4);
            break;
        }
        case moe::FMT_BF16: {
            uint16_t* gu = reinterpret_cast<uint16_t*>(blob + L.gu);
            for (int which = 0; which < 2; ++which) {
                const uint16_t* src = static_cast<const uint16_t*>(ts[which]->data);
                for (int i = 0; i < I; ++i)
                    reorder_row_bf16(src + static_cast<size_t>(i) * H, gu + gu_row(i, which) * H, H);
            }
            const uint16_t* src = static_cast<const uint16_t*>(w->down.data);
            uint16_t* dd = reinterpret_cast<uint16_t*>(blob + L.d);
            for (int r = 0; r < H; ++r)
                reorder_row_bf16(src + static_cast<size_t>(r) * I, dd + static_cast<size_t>(r) * I, I);
            break;
        }
        case moe::FMT_FP8: {
            // device-order rows, scattered into 16-row tiles of 1024-element chunks
            std::vector<uint8_t> drow(std::max(H, I));
            auto put_row = [&](uint8_t* tile, int r, const uint8_t* codes, int K) {
                reorder_row_fp8(codes, drow.data(), K);
                const int G = K / moe::kGroupK;
                for (int c = 0; c * moe::kChunkGroups < G; ++c) {
                    const int ng = moe::fp4_chunk_groups(G, c);
                    uint8_t* chunk = tile + moe::tile_chunk_off(c, L.rowb);
                    for (int w = 0; w < ng; ++w) {
                        const int j = c * moe::kChunkGroups + w;
                        for (int q = 0; q < 4; ++q)
                            for (int hf = 0; hf < 2; ++hf)
                                std::memcpy(chunk + moe::fp8_code_off(ng, r, w, q, hf),
                                            drow.data() + j * 128 + 32 * q + 16 * hf, 16);
                    }
                }
            };
            for (int which = 0; which < 2; ++which) {
                const uint8_t* src = static_cast<const uint8_t*>(ts[which]->data);
                for (int i = 0; i < I; ++i)
                    put_row(blob + L.gu + static_cast<size_t>(i / 8) * L.gu_tile, 8 * which + i % 8,
                            src + static_cast<size_t>(i) * H, H);
            }
            const uint8_t* src = static_cast<const uint8_t*>(w->down.data);
            for (int r = 0; r < H; ++r)
                put_row(blob + L.d + static_cast<size_t>(r / moe::kTileRows) * L.d_tile, r % moe::kTileRows,
                        src + static_cast<size_t>(r) * I, I);
            gsc[0] = w->gate.global_scale;
            gsc[1] = w->up.global_scale;
            gsc[2] = w->down.global_scale;
            break;
        }
        default: {
            // device-order rows, scattered into 16-row tiles of 1024-element chunks
            const int blk = d.weight_fmt == moe::FMT_NVFP4 ? 16 : 32;
            const int sbpg = L.sbpg;
            std::vector<uint8_t> drow(std::max(H, I) / 2);
            auto put_row = [&](uint8_t* tile, int r, const uint8_t* codes, const uint8_t* scales, int K) {
                reorder_row_fp4(codes, drow.data(), K);
                const int G = K / moe::kGroupK;
                for (int c = 0; c * moe::kChunkGroups < G; ++c) {
                    const int ng = moe::fp4_chunk_groups(G, c);
                    uint8_t* chunk = tile + moe::tile_chunk_off(c, L.rowb);
                    for (int w = 0; w < ng; ++w) {
                        const int j = c * moe::kChunkGroups + w;
                        for (int q = 0; q < 4; ++q)
                            std::memcpy(chunk + moe::fp4_code_off(ng, r, w, q), drow.data() + j * 64 + 16 * q, 16);
                        std::memcpy(chunk + moe::fp4_scale_off(ng, sbpg, r, w), scales + static_cast<size_t>(j) * (128 / blk),
                                    128 / blk);
                    }
                }
            };
            for (int which = 0; which < 2; ++which) {
                const uint8_t* src = static_cast<const uint8_t*>(ts[which]->data);
                const uint8_t* sc = ts[which]->scales;
                for (int i = 0; i < I; ++i)
                    put_row(blob + L.gu + static_cast<size_t>(i / 8) * L.gu_tile, 8 * which + i % 8,
                            src + static_cast<size_t>(i) * H / 2, sc + static_cast<size_t>(i) * (H / blk), H);
            }
            const uint8_t* src = static_cast<const uint8_t*>(w->down.data);
            for (int r = 0; r < H; ++r)
                put_row(blob + L.d + static_cast<size_t>(r / moe::kTileRows) * L.d_tile, r % moe::kTileRows,
                        src + static_cast<size_t>(r) * I / 2, w->down.scales + static_cast<size_t>(r) * (I / blk), I);
            if (d.weight_fmt == moe::FMT_NVFP4) {
                gsc[0] = w->gate.global_scale;
                gsc[1] = w->up.global_scale;
                gsc[2] = w->down.global_scale;
            }
        }
    }
    return MOE_OK;
}

void free_pool(moe_handle* h) {
    if (h->pool_owned) cudaFree(h->pool);
    h->pool = nullptr;
    h->pool_owned = false;
    cudaFree(h->table); h->table = nullptr;
    cudaFree(h->owner); h->owner = nullptr;
    cudaFree(h->stamp); h->stamp = nullptr;
    cudaFree(h->clock); h->clock = nullptr;
    h->S = 0;
}

TimedCall* acquire_timed(moe_handle* h) {
    if (!h->spare.empty()) {
        TimedCall* t = h->spare.back();
        h->spare.pop_back();
        t->has_copy = t->has_combine = t->had_miss = t->fused = t->dev_copy = false;
        t->copy_ns = 0;
        t->gu_bytes = t->down_bytes = t->combine_bytes = t->copy_bytes = 0;
        return t;
    }
    TimedCall* t = new (std::nothrow) TimedCall();
    if (!t) return nullptr;
    cudaEvent_t* evs[8] = {&t->r0, &t->r1, &t->f0, &t->f1, &t->f2, &t->f3, &t->c0, &t->c1};
    for (auto* e : evs)
        if (cudaEventCreate(e) != cudaSuccess) return nullptr;
    return t;
}

float elapsed(cudaEvent_t a, cudaEvent_t b) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, a, b) != cudaSuccess) {
        cudaGetLastError();
        return 0.f;
    }
    return ms;
}

// folds finished (and serviced) timed calls into the totals; wait = block until all finished
void harvest(moe_handle* h, bool wait) {
    const uint64_t done = h->serviced.load(std::memory_order_acquire);
    while (!h->pending.empty()) {
        TimedCall* t = h->pending.front();
        if (t->seq > done) break;
        cudaEvent_t last = t->fused ? t->r1 : (t->has_combine ? t->f3 : t->f2);
        if (wait) {
            cudaEventSynchronize(last);
            if (t->has_copy) cudaEventSynchronize(t->c1);
        } else if (cudaEventQuery(last) != cudaSuccess || (t->has_copy && cudaEventQuery(t->c1) != cudaSuccess)) {
            cudaGetLastError();
            break;
        }
        h->tm.calls++;
        if (t->fused) {
            // the decode kernel does routing, cache lookup and the experts
            if (!t->had_miss) {
                h->tm.resident_calls++;
                h->tm.gate_up_ms += elapsed(t->r0, t->r1);
                h->tm.gate_up_bytes += t->gu_bytes;
                h->tm.down_bytes += t->down_bytes;
            }
            if (t->dev_copy) h->tm.copy_ms += static_cast<double>(t->copy_ns) * 1e-6;
            else if (t->has_copy) h->tm.copy_ms += elapsed(t->c0, t->c1);
            h->tm.copy_bytes += t->copy_bytes;
            h->pending.pop_front();
            h->spare.push_back(t);
            continue;
        }
        h->tm.route_ms += elapsed(t->r0, t->r1);
        if (!t->had_miss) {
            // expert kernels of calls without demand misses: pure kernel time
            h->tm.resident_calls++;
            h->tm.gate_up_ms += elapsed(t->f0, t->f1);
            h->tm.down_ms += elapsed(t->f1, t->f2);
            if (t->has_combine) h->tm.combine_ms += elapsed(t->f2, t->f3);
            h->tm.gate_up_bytes += t->gu_bytes;
            h->tm.down_bytes += t->down_bytes;
            h->tm.combine_bytes += t->combine_bytes;
        }
        if (t->has_copy) h->tm.copy_ms += elapsed(t->c0, t->c1);
        h->tm.copy_bytes += t->copy_bytes;
        h->pending.pop_front();
        h->spare.push_back(t);
    }
}

void free_timed(moe_handle* h) {
    auto kill = [](TimedCall* t) {
        cudaEvent_t evs[8] = {t->r0, t->r1, t->f0, t->f1, t->f2, t->f3, t->c0, t->c1};
        for (auto e : evs)
            if (e) cudaEventDestroy(e);
        delete t;
    };
    for (auto* t : h->pending) kill(t);
    for (auto* t : h->spare) kill(t);
    h->pending.clear();
    h->spare.clear();
}

inline void cpu_relax() {
#if defined(__x86_64__) || defined(__i386__)
    __builtin_ia32_pause();
#endif
}

void record_error(moe_handle* h, int code, const std::string& msg) {
    std::lock_guard<std::mutex> lk(h->mu);
    if (code == MOE_ERR_TIMEOUT) h->sticky_timeout = true;
    if (h->pending_err == MOE_OK || code == MOE_ERR_TIMEOUT) {
        h->pending_err = code;
        h->pending_msg = msg;
    }
}

// writes `ready = seq` on the copy stream, behind every copy issued before it
cudaError_t post_ready(moe_handle* h, uint64_t seq) {
    if (h->write64) {
        const CUresult r = h->write64(reinterpret_cast<CUstream>(h->copy), reinterpret_cast<CUdeviceptr>(h->ready),
                                      static_cast<cuuint64_t>(seq), 0);
        return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
    }
    unsigned long long* v = h->ready_vals + (seq % kRing);
    *v = seq;
    return cudaMemcpyAsync(h->ready, v, 8, cudaMemcpyHostToDevice, h->copy);
}

// the service thread's work for one call
void service_call(moe_handle* h, const PendingCall& pc) {
    volatile CallInfo* inf = h->info_h + (pc.seq % kRing);
    // wait for the call's routing kernel: spin while it is near, then back off
    const auto t0 = std::chrono::steady_clock::now();
    uint64_t spins = 0;
    while (inf->done != pc.seq) {
        if (++spins < 200000) {
            cpu_relax();
            continue;
        }
        std::this_thread::sleep_for(std::chrono::microseconds(20));
        if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(120)) {
            record_error(h, MOE_ERR_TIMEOUT, "the routing kernel of a call did not report back");
            return;
        }
    }
    std::atomic_thread_fence(std::memory_order_acquire);
    const int status = inf->status;
    const int nm = inf->n_miss, npm = inf->n_pf_miss, nu = inf->n_uniq;
    const bool dev_copied = inf->device_copied != 0;  // the decode kernel copied its own misses
    const bool kernel_released = dev_copied || (pc.self_release && nm == 0);
    if (status == MOE_ERR_CAPACITY)
        record_error(h, MOE_ERR_CAPACITY, "the layer's experts do not fit in the expert pool");
    else if (status != 0)
        record_error(h, MOE_ERR_CUDA, "the routing kernel reported an unknown status");
    if (inf->dev_err != 0)
        record_error(h, MOE_ERR_TIMEOUT, "a kernel gave up a bounded wait (device error " +
                                             std::to_string(inf->dev_err) + "); call moe_cache_config to reset");
    const size_t B = h->lay.bytes;
    TimedCall* tc = pc.tc;
    cudaError_t ce = cudaSuccess;
    if (tc && nm + npm > 0 && !dev_copied) {
        cudaEventRecord(tc->c0, h->copy);
        tc->has_copy = true;
    }
    auto copy_range = [&](int i0, int i1) -> cudaError_t {
        cudaError_t r = cudaSuccess;
        for (int i = i0; i < i1 && r == cudaSuccess; ++i) {
            const int l = inf->miss_layer[i], e = inf->miss_expert[i], sl = inf->miss_slot[i];
            r = cudaMemcpyAsync(h->pool + static_cast<size_t>(sl) * B, h->bank[l] + static_cast<size_t>(e) * B, B,
                                cudaMemcpyHostToDevice, ((i - i0) & 1) ? h->copy2 : h->copy);
        }
        if (r == cudaSuccess && i1 - i0 > 1) {
            r = cudaEventRecord(h->ev_join, h->copy2);
            if (r == cudaSuccess) r = cudaStreamWaitEvent(h->copy, h->ev_join, 0);
        }
        return r;
    };
    if (!dev_copied) ce = copy_range(0, nm);
    if (ce == cudaSuccess && !kernel_released) {
        if (h->fault_drop_release && nm > 0) h->fault_drop_release = false;
        else ce = post_ready(h, pc.seq);
    }
    if (ce == cudaSuccess) ce = copy_range(nm, nm + npm);
    if (tc && tc->has_copy) cudaEventRecord(tc->c1, h->copy);
    if (h->log)
        std::fprintf(stderr, "[moe] call %llu layer %d T %d status %d uniq %d miss %d pf_miss %d self_release %d "
                             "kernel_released %d copy_err %d dev_err %d\n",
                     static_cast<unsigned long long>(pc.seq), pc.layer, pc.T, status, nu, nm, npm,
                     pc.self_release ? 1 : 0, kernel_released ? 1 : 0, static_cast<int>(ce), inf->dev_err);
    if (ce != cudaSuccess) {
        record_error(h, MOE_ERR_CUDA, std::string("expert copy: ") + cudaGetErrorString(ce));
        cudaGetLastError();
    }
    if (tc) {
        // algorithmic bytes of this call
        const uint64_t H = h->d.hidden, I = h->d.inter, k = h->d.top_k, ns = h->d.num_shared, T = pc.T;
        const uint64_t na = static_cast<uint64_t>(nu) + ns;
        const uint64_t rows = T * (k + ns);
        const uint64_t ea = h->d.act_dtype == moe::ACT_BF16 ? 2 : 4;
        const uint64_t he = h->d.weight_fmt == moe::FMT_FP32 ? 4 : 2;
        uint64_t wgu, wd;
        switch (h->d.weight_fmt) {
            case moe::FMT_FP32: wgu = 2 * I * H * 4; wd = H * I * 4; break;
            case moe::FMT_BF16: wgu = 2 * I * H * 2; wd = H * I * 2; break;
            case moe::FMT_FP8: wgu = 2 * I * H; wd = H * I; break;
            default: {
                const uint64_t blk = h->d.weight_fmt == moe::FMT_NVFP4 ? 16 : 32;
                wgu = 2 * I * H / 2 + 2 * I * H / blk;
                wd = H * I / 2 + H * I / blk;
            }
        }
        tc->had_miss = nm > 0 || !pc.self_release;  // the kernels waited for copies
        tc->gu_bytes = na * wgu + T * H * ea + rows * I * he;
        tc->down_bytes = na * wd + rows * I * he + (tc->has_combine ? rows * H * 2 : T * H * ea);
        tc->combine_bytes = tc->has_combine ? rows * H * 2 + T * H * ea : 0;
        tc->copy_bytes = static_cast<uint64_t>(nm + npm) * B;
        if (pc.fused) {
            // the decode kernel also reads the router matrix [E][H] (and writes h as bf16)
            tc->had_miss = nm > 0;
            tc->gu_bytes += static_cast<uint64_t>(h->d.num_experts) * H * ea;
            tc->dev_copy = dev_copied;
            tc->copy_ns = inf->copy_ns;
        }
    }
    std::lock_guard<std::mutex> lk(h->mu);
    h->st.calls++;
    (pc.T <= moe::kDecodeMaxT ? h->st.decode_calls : h->st.prefill_calls)++;
    if (status == 0) {
        h->st.hits += inf->n_hit;
        h->st.misses += nm;
        h->st.prefetch_hits += inf->n_pf_hit;
        h->st.prefetch_misses += npm;
        h->st.copies_h2d += nm + npm;
        h->st.bytes_h2d += static_cast<uint64_t>(nm + npm) * B;
        const int nev = inf->n_events;
        for (int i = 0; i < nev; ++i) {
            if (inf->ev_evicted[i] >= 0) h->st.evictions++;
            if (h->flags & MOE_CACHE_LOG_EVENTS) {
                moe_event ev{inf->ev_layer[i], inf->ev_expert[i], inf->ev_hit[i], inf->ev_slot[i], inf->ev_evicted[i],
                             inf->ev_prefetch[i]};
                h->events.push_back(ev);
            }
        }
    } else {
        h->st.device_errors++;
    }
    if (inf->dev_err != 0) h->st.device_errors++;
}

void service_loop(moe_handle* h) {
    cudaSetDevice(h->d.device);
    for (;;) {
        PendingCall pc;
        {
            std::unique_lock<std::mutex> lk(h->mu);
            h->cv.wait(lk, [&] { return h->stop || !h->queue.empty(); });
            if (h->queue.empty()) return;  // stopping, and every call has been serviced
            pc = h->queue.front();
        }
        service_call(h, pc);
        {
            std::lock_guard<std::mutex> lk(h->mu);
            h->queue.pop_front();
            h->serviced.store(pc.seq, std::memory_order_release);
        }
        h->done_cv.notify_all();
    }
}

// MOE_TRACE buffer: per-CTA phase marks, then per-call entry / wait / exit times
size_t trace_words(const moe_handle* h) {
    return static_cast<size_t>(h->num_sms) * moe::kTracePoints + moe::kTraceCalls * 4;
}
void reset_trace(moe_handle* h) {
    std::vector<unsigned long long> t(trace_words(h), 0ull);
    for (int c = 0; c < moe::kTraceCalls; ++c) t[static_cast<size_t>(h->num_sms) * moe::kTracePoints + c * 4] = ~0ull;
    cudaMemcpy(h->trace, t.data(), t.size() * 8, cudaMemcpyHostToDevice);
}

// waits until the service thread has handled every enqueued call
void drain(moe_handle* h) {
    std::unique_lock<std::mutex> lk(h->mu);
    h->done_cv.wait(lk, [&] { return h->serviced.load(std::memory_order_acquire) >= h->submitted; });
}

// error found by the service thread for an earlier call; capacity errors are
// reported once, bounded-wait timeouts until moe_cache_config
int take_error(moe_handle* h) {
    std::lock_guard<std::mutex> lk(h->mu);
    if (h->pending_err == MOE_OK) return MOE_OK;
    const int e = h->pending_err;
    {
        std::lock_guard<std::mutex> lk2(h->err_mu);
        h->err = h->pending_msg;
    }
    if (!h->sticky_timeout) {
        h->pending_err = MOE_OK;
        h->pending_msg.clear();
    }
    return e;
}

void stop_service(moe_handle* h) {
    if (!h->svc.joinable()) return;
    {
        std::lock_guard<std::mutex> lk(h->mu);
        h->stop = true;
    }
    h->cv.notify_all();
    h->svc.join();
}

}  // namespace

extern "C" {

int moe_expert_bytes(const moe_model_desc* desc, size_t* bytes) {
    std::string why;
    const int v = validate_desc(desc, &why);
    if (v != MOE_OK) return v;
    if (!bytes) return MOE_ERR_INVALID;
    *bytes = layout_for(*desc).bytes;
    return MOE_OK;
}

int moe_repack_expert(const moe_model_desc* desc, const moe_expert_host* w, void* blob, size_t blob_bytes) {
    std::string why;
    const int v = validate_desc(desc, &why);
    if (v != MOE_OK) return v;
    if (!w || !blob) return MOE_ERR_INVALID;
    const BlobLayout L = layout_for(*desc);
    if (blob_bytes < L.bytes) return MOE_ERR_INVALID;
    return repack_expert(*desc, L, w, static_cast<uint8_t*>(blob), &why);
}

int moe_init(const moe_model_desc* desc, moe_handle** out) {
    if (!out) return MOE_ERR_INVALID;
    *out = nullptr;
    std::string why;
    int v = validate_desc(desc, &why);
    if (v != MOE_OK) return v;
    moe_handle* h = new (std::nothrow) moe_handle();
    if (!h) return MOE_ERR_OOM;
    h->d = *desc;
    h->max_tokens = desc->max_tokens > 0 ? desc->max_tokens : 4096;
    h->lay = layout_for(h->d);
    if (const char* f = std::getenv("MOE_FAULT")) h->fault_drop_release = std::strcmp(f, "drop_release") == 0;
    h->log = std::getenv("MOE_LOG") != nullptr;
    const bool want_trace = std::getenv("MOE_TRACE") != nullptr;
    if (const char* w = std::getenv("MOE_WAIT_MS")) {
        const long ms = std::strtol(w, nullptr, 10);
        if (ms > 0) h->wait_ns = static_cast<unsigned long long>(ms) * 1000000ull;
    }
    auto bail = [&](int code) { moe_destroy(h); return code; };
    cudaError_t e = cudaSetDevice(desc->device);
    if (e != cudaSuccess) return bail(MOE_ERR_CUDA);
    if (moe::routing_set_attributes() != cudaSuccess) return bail(MOE_ERR_CUDA);
    if (moe::umma_set_attributes() != cudaSuccess) return bail(MOE_ERR_CUDA);
    if (moe::decode_set_attributes() != cudaSuccess) return bail(MOE_ERR_CUDA);
    if (moe::experts_preload() != cudaSuccess) return bail(MOE_ERR_CUDA);
    if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, desc->device) != cudaSuccess)
        return bail(MOE_ERR_CUDA);
    {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue64", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            h->write64 = reinterpret_cast<WriteValue64Fn>(p);
        cudaGetLastError();
    }
    const int L = h->d.num_layers, E = h->d.num_experts, ns = h->d.num_shared, k = h->d.top_k;
    const size_t H = h->d.hidden, I = h->d.inter, Tm = h->max_tokens;
    h->bank.assign(L, nullptr);
    h->bank_dev.assign(L, nullptr);
    h->loaded.assign(static_cast<size_t>(L) * E, 0);
    h->layer_complete.assign(L, 0);
    if (ns > 0) {
        if (cudaMalloc(&h->shared_dev, static_cast<size_t>(L) * ns * h->lay.bytes) != cudaSuccess) return bail(MOE_ERR_OOM);
        cudaMemset(h->shared_dev, 0, static_cast<size_t>(L) * ns * h->lay.bytes);
    }
    // scratch carve-up
    const size_t rows = Tm * (k + ns);
    const size_t hes = h->d.weight_fmt == moe::FMT_FP32 ? 4 : 2;
    const size_t nb_max = align_up((Tm + 7) / 8, 16);  // routing CTAs of a prefill call, padded to 16
    const bool umma = moe::prefill_uses_umma(h->d.weight_fmt, static_cast<int>(Tm));
    struct Part { size_t bytes; void** dst; };
    CallArgs& a = h->base;
    std::vector<Part> parts = {
        {Tm * H * 2, &a.xh},
        {Tm * E * 4, reinterpret_cast<void**>(&a.logits)},
        {static_cast<size_t>(E) * 4, reinterpret_cast<void**>(&a.wnorm)},
        {Tm * k * 4, reinterpret_cast<void**>(&a.topk)},
        {Tm * k * 4, reinterpret_cast<void**>(&a.gates)},
        {static_cast<size_t>(E) * 4, reinterpret_cast<void**>(&a.counts)},
        {static_cast<size_t>(E + 1) * 4, reinterpret_cast<void**>(&a.offsets)},
        {Tm * k * 4, reinterpret_cast<void**>(&a.perm)},
        {Tm * k * 4, reinterpret_cast<void**>(&a.inv_perm)},
        {rows * 4, reinterpret_cast<void**>(&a.row_tok)},
        {rows * 4, reinterpret_cast<void**>(&a.row_gate)},
        {static_cast<size_t>(E + ns) * 4, reinterpret_cast<void**>(&a.act_expert)},
        {static_cast<size_t>(E + ns) * 4, reinterpret_cast<void**>(&a.act_row0)},
        {static_cast<size_t>(E + ns) * 4, reinterpret_cast<void**>(&a.act_cnt)},
        {static_cast<size_t>(E + ns) * 8, reinterpret_cast<void**>(&a.act_ptr)},
        {static_cast<size_t>(E) * 4, reinterpret_cast<void**>(&a.e2u)},
        {static_cast<size_t>(E + ns) * moe::kDecodeMaxT * 4, reinterpret_cast<void**>(&a.tok_row)},
        {static_cast<size_t>(E + ns) * 4, reinterpret_cast<void**>(&a.act_slot)},
        {umma ? rows * H * 2 : 16, &a.xperm},
        {umma ? Tm * 4 : 16, reinterpret_cast<void**>(&a.xsc)},
        {umma ? rows * 4 : 16, reinterpret_cast<void**>(&a.xunr)},
        {4, reinterpret_cast<void**>(&a.dev_err)},
        {4, reinterpret_cast<void**>(&a.route_done)},
        {static_cast<size_t>(E) * 4, reinterpret_cast<void**>(&a.cacc)},
        {static_cast<size_t>(E) * nb_max * 2, reinterpret_cast<void**>(&a.cntT)},
        {Tm * k * 2, reinterpret_cast<void**>(&a.lrank)},
        {3 * 8, reinterpret_cast<void**>(&a.bar_cnt)},
        {static_cast<size_t>(moe::kDecodeMaxT) * E * 8, reinterpret_cast<void**>(&a.dlog)},
        {moe::kDecodeMaxT * 4, reinterpret_cast<void**>(&a.xmax)},
        {2 * moe::kDecodeMaxT * 4, reinterpret_cast<void**>(&a.hmax)},
        {sizeof(moe::DecPub), reinterpret_cast<void**>(&a.pub)},
        {static_cast<size_t>(L) * 8, reinterpret_cast<void**>(const_cast<uint8_t***>(&a.banks))},
        {moe::kDecPlanHeader + static_cast<size_t>(E + ns) * sizeof(moe::DecExpert), reinterpret_cast<void**>(&a.dplan)},
        {8, reinterpret_cast<void**>(&a.ready)},
        {4, reinterpret_cast<void**>(&a.n_uniq)},
        {4, reinterpret_cast<void**>(&a.n_active)},
        {rows * I * hes, &a.hbuf},
        {h->d.weight_fmt == moe::FMT_FP32 || Tm <= moe::kDecodeMaxT ? 16 : rows * H * 2, &a.ybuf},
    };
    size_t total = 0;
    for (auto& p : parts) total += align_up(p.bytes, 256);
    if (cudaMalloc(&h->scratch, total) != cudaSuccess) return bail(MOE_ERR_OOM);
    cudaMemset(h->scratch, 0, total);
    size_t off = 0;
    for (auto& p : parts) {
        *p.dst = static_cast<uint8_t*>(h->scratch) + off;
        off += align_up(p.bytes, 256);
    }
    h->ready = a.ready;
    if (want_trace) {
        if (cudaMalloc(&h->trace, trace_words(h) * 8) != cudaSuccess) return bail(MOE_ERR_OOM);
        reset_trace(h);
        a.trace = h->trace;
        a.trace_ctas = h->num_sms;
    }
    if (umma) {
        // TMA descriptors over the gathered activations, h, and the resident shared experts
        bool ok = moe::umma_map_2d(&h->maps.x, a.xperm, rows, H, 128) && moe::umma_map_2d(&h->maps.h, a.hbuf, rows, I, 128);
        if (ok && ns > 0 && h->d.weight_fmt == moe::FMT_BF16) {
            ok = moe::umma_map_3d(&h->maps.shared_gu, h->shared_dev + h->lay.gu, static_cast<uint64_t>(L) * ns,
                                  h->lay.bytes, 2 * I, H, 64) &&
                 moe::umma_map_3d(&h->maps.shared_d, h->shared_dev + h->lay.d, static_cast<uint64_t>(L) * ns,
                                  h->lay.bytes, H, I, 128);
        }
        if (!ok) return bail(MOE_ERR_CUDA);
        h->maps.have_io = true;
    }
    if (cudaHostAlloc(reinterpret_cast<void**>(&h->info_h), sizeof(CallInfo) * kRing, cudaHostAllocMapped) !=
        cudaSuccess)
        return bail(MOE_ERR_OOM);
    std::memset(h->info_h, 0, sizeof(CallInfo) * kRing);
    if (cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->info_d), h->info_h, 0) != cudaSuccess)
        return bail(MOE_ERR_CUDA);
    if (cudaHostAlloc(reinterpret_cast<void**>(&h->ready_vals), 8 * kRing, cudaHostAllocDefault) != cudaSuccess)
        return bail(MOE_ERR_OOM);
    if (cudaStreamCreateWithFlags(&h->stream, cudaStreamNonBlocking) != cudaSuccess) return bail(MOE_ERR_CUDA);
    if (cudaStreamCreateWithFlags(&h->copy, cudaStreamNonBlocking) != cudaSuccess) return bail(MOE_ERR_CUDA);
    if (cudaStreamCreateWithFlags(&h->copy2, cudaStreamNonBlocking) != cudaSuccess) return bail(MOE_ERR_CUDA);
    if (cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess) return bail(MOE_ERR_CUDA);
    if (cudaEventCreateWithFlags(&h->ev_pf, cudaEventDisableTiming) != cudaSuccess) return bail(MOE_ERR_CUDA);
    if (cudaDeviceSynchronize() != cudaSuccess) return bail(MOE_ERR_CUDA);
    a.E = E; a.k = k; a.H = static_cast<int>(H); a.I = static_cast<int>(I); a.n_shared = ns; a.L = L;
    a.nb_max = static_cast<int>(nb_max);
    a.fmt = h->d.weight_fmt; a.act = h->d.act_dtype; a.mode = h->d.act_mode;
    a.lay = h->lay;
    a.wait_ns = h->wait_ns;
    try {
        h->svc = std::thread(service_loop, h);
    } catch (...) {
        return bail(MOE_ERR_OOM);
    }
    *out = h;
    return MOE_OK;
}

int moe_load_expert(moe_handle* h, int layer, int expert, const moe_expert_host* w) {
    if (!h || !w) return MOE_ERR_INVALID;
    const int L = h->d.num_layers, E = h->d.num_experts, ns = h->d.num_shared;
    if (layer < 0 || layer >= L) return fail(h, MOE_ERR_INVALID, "layer out of range");
    if (expert < 0 || expert >= E + ns) return fail(h, MOE_ERR_INVALID, "expert out of range");
    CK(h, cudaSetDevice(h->d.device));
    const size_t B = h->lay.bytes;
    std::string why;
    if (expert >= E) {
        std::vector<uint8_t> tmp(B);
        int r = repack_expert(h->d, h->lay, w, tmp.data(), &why);
        if (r != MOE_OK) return fail(h, r, why);
        CK(h, cudaMemcpy(h->shared_dev + (static_cast<size_t>(layer) * ns + (expert - E)) * B, tmp.data(), B,
                         cudaMemcpyHostToDevice));
        return MOE_OK;
    }
    uint8_t* bank;
    {
        std::lock_guard<std::mutex> lk(h->load_mu);
        if (!h->bank[layer]) {
            // mapped: the decode kernel reads missed experts straight from the bank
            void* p = nullptr;
            void* dp = nullptr;
            if (cudaHostAlloc(&p, static_cast<size_t>(E) * B, cudaHostAllocMapped | cudaHostAllocPortable) !=
                cudaSuccess) {
                cudaGetLastError();
                return fail(h, MOE_ERR_OOM, "pinned host bank allocation failed");
            }
            if (cudaHostGetDevicePointer(&dp, p, 0) != cudaSuccess) {
                cudaGetLastError();
                cudaFreeHost(p);
                return fail(h, MOE_ERR_CUDA, "no device view of the pinned host bank");
            }
            h->bank[layer] = static_cast<uint8_t*>(p);
            h->bank_dev[layer] = static_cast<const uint8_t*>(dp);
            h->banks_dirty = true;
        }
        bank = h->bank[layer];
    }
    int r = repack_expert(h->d, h->lay, w, bank + static_cast<size_t>(expert) * B, &why);
    if (r != MOE_OK) return fail(h, r, why);
    h->loaded[static_cast<size_t>(layer) * E + expert] = 1;
    return MOE_OK;
}

}  // extern "C"

namespace {

// a pool of S slots: the caller's buffer (checked) or a new allocation
int take_pool(moe_handle* h, size_t S, void* pool_dev, size_t pool_bytes, uint8_t** out, bool* owned) {
    const size_t need = S * h->lay.bytes;
    if (pool_dev) {
        if (reinterpret_cast<uintptr_t>(pool_dev) & 255u) return fail(h, MOE_ERR_INVALID, "pool buffer must be 256-byte aligned");
        if (pool_bytes < need) return fail(h, MOE_ERR_INVALID, "pool buffer smaller than capacity_slots expert blobs");
        *out = static_cast<uint8_t*>(pool_dev);
        *owned = false;
        return MOE_OK;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, need) != cudaSuccess) {
        cudaGetLastError();
        return fail(h, MOE_ERR_OOM, "device pool allocation failed");
    }
    *out = static_cast<uint8_t*>(p);
    *owned = true;
    return MOE_OK;
}

// TMA descriptors of the prefill GEMMs over the pool's weight regions
int build_pool_maps(moe_handle* h) {
    h->maps.have_pool = false;
    if (h->maps.have_io && h->d.weight_fmt != moe::FMT_BF16) {
        h->maps.have_pool = true;  // FP4 / FP8 prefill builds its weight tiles in shared memory: no pool maps
    } else if (h->maps.have_io) {
        const uint64_t H = h->d.hidden, I = h->d.inter, S = h->S;
        if (!moe::umma_map_3d(&h->maps.pool_gu, h->pool + h->lay.gu, S, h->lay.bytes, 2 * I, H, 64) ||
            !moe::umma_map_3d(&h->maps.pool_d, h->pool + h->lay.d, S, h->lay.bytes, H, I, 128))
            return fail(h, MOE_ERR_CUDA, "TMA descriptor encoding failed");
        if (h->d.num_shared == 0) {
            h->maps.shared_gu = h->maps.pool_gu;  // never selected: no shared experts
            h->maps.shared_d = h->maps.pool_d;
        }
        h->maps.have_pool = true;
    }
    return MOE_OK;
}

void bind_pool(moe_handle* h) {
    CallArgs& a = h->base;
    a.table = h->table; a.owner = h->owner; a.stamp = h->stamp; a.clock = h->clock;
    a.pool = h->pool; a.S = h->S;
}

}  // namespace

extern "C" {

int moe_cache_config(moe_handle* h, int capacity_slots, unsigned flags, void* pool_dev, size_t pool_bytes) {
    if (!h) return MOE_ERR_INVALID;
    if (capacity_slots < h->d.top_k) return fail(h, MOE_ERR_CAPACITY, "capacity below top_k");
    if (capacity_slots > moe::kMaxSlots) return fail(h, MOE_ERR_INVALID, "capacity above 16384 slots");
    if (flags & ~(MOE_CACHE_PREFETCH_NEXT_LAYER | MOE_CACHE_LOG_EVENTS | MOE_CACHE_SYNC_MISSES | MOE_CACHE_HOST_MISSES))
        return fail(h, MOE_ERR_INVALID, "unknown cache flag");
    CK(h, cudaSetDevice(h->d.device));
    drain(h);
    CK(h, cudaDeviceSynchronize());
    free_pool(h);
    const int L = h->d.num_layers, E = h->d.num_experts;
    const size_t S = capacity_slots;
    int r = take_pool(h, S, pool_dev, pool_bytes, &h->pool, &h->pool_owned);
    if (r != MOE_OK) return r;
    if (cudaMalloc(&h->table, static_cast<size_t>(L) * E * 4) != cudaSuccess ||
        cudaMalloc(&h->owner, S * 4) != cudaSuccess || cudaMalloc(&h->stamp, S * 8) != cudaSuccess ||
        cudaMalloc(&h->clock, 8) != cudaSuccess) {
        cudaGetLastError();
        free_pool(h);
        return fail(h, MOE_ERR_OOM, "LRU table allocation failed");
    }
    CK(h, cudaMemset(h->table, 0xFF, static_cast<size_t>(L) * E * 4));
    CK(h, cudaMemset(h->owner, 0xFF, S * 4));
    CK(h, cudaMemset(h->stamp, 0, S * 8));
    CK(h, cudaMemset(h->clock, 0, 8));
    CK(h, cudaMemset(h->base.dev_err, 0, 4));
    CK(h, cudaMemset(h->base.route_done, 0, 4));
    CK(h, cudaMemset(h->base.bar_cnt, 0, 3 * 8));
    CK(h, cudaMemset(h->base.dlog, 0, static_cast<size_t>(moe::kDecodeMaxT) * h->d.num_experts * 8));
    CK(h, cudaMemset(h->base.hmax, 0, 2 * moe::kDecodeMaxT * 4));
    h->dcalls = 0;

    // the ready word continues from the last serviced call
    const unsigned long long rv = h->submitted;
    CK(h, cudaMemcpy(h->ready, &rv, 8, cudaMemcpyHostToDevice));
    CK(h, cudaDeviceSynchronize());
    h->S = capacity_slots;
    if ((r = build_pool_maps(h)) != MOE_OK) {
        free_pool(h);
        return r;
    }
    {
        std::lock_guard<std::mutex> lk(h->mu);
        h->pending_err = MOE_OK;
        h->pending_msg.clear();
        h->sticky_timeout = false;
        h->events.clear();
    }
    h->flags = flags;
    h->prefetch_may_be_pending = false;
    bind_pool(h);
    CallArgs& a = h->base;
    a.device_misses = (flags & MOE_CACHE_HOST_MISSES) ? 0 : 1;
    a.prefetch = (flags & MOE_CACHE_PREFETCH_NEXT_LAYER) ? 1 : 0;
    a.log_events = (flags & MOE_CACHE_LOG_EVENTS) ? 1 : 0;
    return MOE_OK;
}

int moe_cache_resize(moe_handle* h, int capacity_slots, void* pool_dev, size_t pool_bytes) {
    if (!h) return MOE_ERR_INVALID;
    if (!h->pool) return fail(h, MOE_ERR_STATE, "moe_cache_config has not been called");
    if (capacity_slots < h->d.top_k) return fail(h, MOE_ERR_CAPACITY, "capacity below top_k");
    if (capacity_slots > moe::kMaxSlots) return fail(h, MOE_ERR_INVALID, "capacity above 16384 slots");
    CK(h, cudaSetDevice(h->d.device));
    drain(h);
    CK(h, cudaDeviceSynchronize());
    const int L = h->d.num_layers, E = h->d.num_experts;
    const int S0 = h->S, S1 = capacity_slots;
    const size_t B = h->lay.bytes;
    // the cache state, on the host
    std::vector<int32_t> table(static_cast<size_t>(L) * E), owner(S0);
    std::vector<unsigned long long> stamp(S0);
    CK(h, cudaMemcpy(table.data(), h->table, table.size() * 4, cudaMemcpyDeviceToHost));
    CK(h, cudaMemcpy(owner.data(), h->owner, owner.size() * 4, cudaMemcpyDeviceToHost));
    CK(h, cudaMemcpy(stamp.data(), h->stamp, stamp.size() * 8, cudaMemcpyDeviceToHost));
    // keep the S1 most recently used experts; those in slots below S1 stay put,
    // the others fill the free slots below S1 in ascending order of their old slot
    std::vector<int> resident;
    for (int s = 0; s < S0; ++s)
        if (owner[s] >= 0) resident.push_back(s);
    std::sort(resident.begin(), resident.end(), [&](int x, int y) {
        return stamp[x] != stamp[y] ? stamp[x] > stamp[y] : x < y;
    });
    std::vector<uint8_t> kept(S0, 0);
    for (size_t i = 0; i < resident.size() && i < static_cast<size_t>(S1); ++i) kept[resident[i]] = 1;
    std::vector<int> dest(S0, -1);
    std::vector<uint8_t> taken(S1, 0);
    for (int s = 0; s < S0 && s < S1; ++s)
        if (kept[s]) {
            dest[s] = s;
            taken[s] = 1;
        }
    int hole = 0;
    for (int s = S1; s < S0; ++s) {
        if (!kept[s]) continue;
        while (taken[hole]) ++hole;
        dest[s] = hole;
        taken[hole] = 1;
    }
    std::vector<int32_t> owner1(S1, -1);
    std::vector<unsigned long long> stamp1(S1, 0ull);
    for (int s = 0; s < S0; ++s) {
        if (owner[s] < 0) continue;
        if (dest[s] >= 0) {
            owner1[dest[s]] = owner[s];
            stamp1[dest[s]] = stamp[s];
            table[owner[s]] = dest[s];
        } else {
            table[owner[s]] = -1;
        }
    }
    // the new pool, and the kept experts' blobs in their new slots
    uint8_t* pool1 = nullptr;
    bool owned1 = false;
    const bool in_place = pool_dev != nullptr && pool_dev == h->pool;
    if (in_place) {
        if (pool_bytes < static_cast<size_t>(S1) * B) return fail(h, MOE_ERR_INVALID, "pool buffer smaller than capacity_slots expert blobs");
        pool1 = h->pool;
        owned1 = h->pool_owned;
    } else {
        const int r = take_pool(h, S1, pool_dev, pool_bytes, &pool1, &owned1);
        if (r != MOE_OK) return r;
    }
    for (int s = 0; s < S0; ++s)
        if (dest[s] >= 0 && (!in_place || dest[s] != s))
            CK(h, cudaMemcpy(pool1 + static_cast<size_t>(dest[s]) * B, h->pool + static_cast<size_t>(s) * B, B,
                             cudaMemcpyDeviceToDevice));
    int32_t* owner_d = nullptr;
    unsigned long long* stamp_d = nullptr;
    if (cudaMalloc(&owner_d, static_cast<size_t>(S1) * 4) != cudaSuccess ||
        cudaMalloc(&stamp_d, static_cast<size_t>(S1) * 8) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(owner_d);
        if (owned1 && !in_place) cudaFree(pool1);
        return fail(h, MOE_ERR_OOM, "LRU table allocation failed");
    }
    CK(h, cudaMemcpy(owner_d, owner1.data(), owner1.size() * 4, cudaMemcpyHostToDevice));
    CK(h, cudaMemcpy(stamp_d, stamp1.data(), stamp1.size() * 8, cudaMemcpyHostToDevice));
    CK(h, cudaMemcpy(h->table, table.data(), table.size() * 4, cudaMemcpyHostToDevice));
    CK(h, cudaDeviceSynchronize());
    if (!in_place && h->pool_owned) cudaFree(h->pool);
    cudaFree(h->owner);
    cudaFree(h->stamp);
    h->pool = pool1;
    h->pool_owned = owned1;
    h->owner = owner_d;
    h->stamp = stamp_d;
    h->S = S1;
    const int r = build_pool_maps(h);
    if (r != MOE_OK) return r;
    bind_pool(h);
    return MOE_OK;
}

int moe_layer_forward(moe_handle* h, const void* hidden, const void* router_w, int layer_id, int T, void* out,
                      void* stream) {
    if (!h) return MOE_ERR_INVALID;
    if (const int e = take_error(h)) return e;
    if (!h->pool) return fail(h, MOE_ERR_STATE, "moe_cache_config has not been called");
    const int L = h->d.num_layers, E = h->d.num_experts;
    if (layer_id < 0 || layer_id >= L) return fail(h, MOE_ERR_INVALID, "layer out of range");
    if (T < 0 || T > h->max_tokens) return fail(h, MOE_ERR_INVALID, "T out of range");
    if (T == 0) return MOE_OK;
    if (!hidden || !router_w || !out) return fail(h, MOE_ERR_INVALID, "NULL device buffer");
    if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(router_w) |
         reinterpret_cast<uintptr_t>(out)) & 15u)
        return fail(h, MOE_ERR_INVALID, "device buffers must be 16-byte aligned");
    // experts are never unloaded: a layer found complete once is complete for good
    auto complete = [&](int l) {
        if (h->layer_complete[l]) return true;
        for (int e = 0; e < E; ++e)
            if (!h->loaded[static_cast<size_t>(l) * E + e]) return false;
        h->layer_complete[l] = 1;
        return true;
    };
    if (!complete(layer_id)) return fail(h, MOE_ERR_STATE, "layer has unloaded experts");
    const bool decode = T <= moe::kDecodeMaxT;
    const bool want_pf = !decode && (h->flags & MOE_CACHE_PREFETCH_NEXT_LAYER) && layer_id + 1 < L;
    if (want_pf && !complete(layer_id + 1)) return fail(h, MOE_ERR_STATE, "next layer has unloaded experts");
    CK(h, cudaSetDevice(h->d.device));
    cudaStream_t s = stream ? static_cast<cudaStream_t>(stream) : h->stream;
    const uint64_t seq = h->submitted + 1;
    // the record slot of call seq - kRing must have been read
    if (seq > static_cast<uint64_t>(kRing) && h->serviced.load(std::memory_order_acquire) < seq - kRing) {
        std::unique_lock<std::mutex> lk(h->mu);
        h->done_cv.wait(lk, [&] { return h->serviced.load(std::memory_order_acquire) >= seq - kRing; });
    }
    CallInfo* rec = h->info_h + (seq % kRing);
    reinterpret_cast<volatile unsigned long long*>(&rec->done)[0] = 0;
    reinterpret_cast<volatile int32_t*>(&rec->device_copied)[0] = 0;
    CallArgs a = h->base;
    a.T = T;
    a.layer = layer_id;
    a.hidden = hidden;
    a.router_w = router_w;
    a.out = out;
    a.shared_base = h->shared_dev ? h->shared_dev + static_cast<size_t>(layer_id) * h->d.num_shared * h->lay.bytes
                                  : nullptr;
    a.info = h->info_d + (seq % kRing);
    a.seq = seq;
    a.self_release = h->prefetch_may_be_pending ? 0 : 1;
    TimedCall* tc = nullptr;
    if (h->timing) {
        harvest(h, false);
        tc = acquire_timed(h);
        if (!tc) return fail(h, MOE_ERR_OOM, "timing events");
        tc->seq = seq;
    }
    if (moe::decode_fused(h->d.weight_fmt, T)) {
        // decode with FP4 or FP8 weights: one kernel does the whole call, including the
        // copies of its misses (unless MOE_CACHE_HOST_MISSES); it never waits for
        // the host except in that mode
        if (h->banks_dirty) {
            CK(h, cudaMemcpy(const_cast<uint8_t**>(a.banks), h->bank_dev.data(), sizeof(void*) * L,
                             cudaMemcpyHostToDevice));
            h->banks_dirty = false;
        }
        if (h->prefetch_may_be_pending) {
            // a prefill call's prefetch copies of this layer may still be landing
            drain(h);
            CK(h, cudaEventRecord(h->ev_pf, h->copy));
            CK(h, cudaStreamWaitEvent(s, h->ev_pf, 0));
        }
        a.self_release = 1;
        a.dcall = h->dcalls;
        if (tc) CK(h, cudaEventRecord(tc->r0, s));
        const cudaError_t le = moe::launch_decode(a, h->num_sms, s, true);
        if (le != cudaSuccess) return cuda_fail(h, le, "decode kernel launch");
        h->dcalls++;
        if (tc) {
            CK(h, cudaEventRecord(tc->r1, s));
            tc->fused = true;
        }
        h->submitted = seq;
        h->prefetch_may_be_pending = false;
        h->last_fused = true;
        h->last_T = T;
        h->last_stream = s;
        {
            std::lock_guard<std::mutex> lk(h->mu);
            PendingCall pc;
            pc.seq = seq;
            pc.layer = layer_id;
            pc.T = T;
            pc.self_release = true;
            pc.fused = true;
            pc.tc = tc;
            h->queue.push_back(pc);
            if (tc) h->pending.push_back(tc);
            h->st.kernel_launches += 1;
        }
        h->cv.notify_one();
        return MOE_OK;
    }
    if (tc) CK(h, cudaEventRecord(tc->r0, s));
    CK(h, moe::launch_route(a, s));
    if (tc) {
        CK(h, cudaEventRecord(tc->r1, s));
        CK(h, cudaEventRecord(tc->f0, s));
        tc->has_combine = !decode && h->d.weight_fmt != moe::FMT_FP32;
    }
    // the call is enqueued from here on (the routing kernel is in flight): hand
    // it to the service thread even if the expert launch fails, so that its
    // record is consumed in order
    h->submitted = seq;
    h->prefetch_may_be_pending = want_pf;
    h->last_fused = false;
    h->last_T = T;
    h->last_stream = s;
    {
        std::lock_guard<std::mutex> lk(h->mu);
        PendingCall pc;
        pc.seq = seq;
        pc.layer = layer_id;
        pc.T = T;
        pc.self_release = a.self_release != 0;
        pc.tc = tc;
        h->queue.push_back(pc);
        if (tc) h->pending.push_back(tc);
    }
    h->cv.notify_one();
    if (h->flags & MOE_CACHE_SYNC_MISSES) {
        // the service thread reads the call's cache result, copies its misses and
        // posts its release; once those copies have run, the expert kernels below
        // find the release already there and never wait on the host
        {
            std::unique_lock<std::mutex> lk(h->mu);
            h->done_cv.wait(lk, [&] { return h->serviced.load(std::memory_order_acquire) >= seq; });
        }
        CK(h, cudaStreamSynchronize(h->copy));
        CK(h, cudaStreamSynchronize(h->copy2));
    }
    int nl = 0;
    const cudaError_t le =
        moe::launch_experts(a, s, tc ? tc->f1 : nullptr, tc ? tc->f2 : nullptr, &h->maps, h->num_sms, &nl);
    if (tc && tc->has_combine) CK(h, cudaEventRecord(tc->f3, s));
    {
        std::lock_guard<std::mutex> lk(h->mu);
        h->st.kernel_launches += (decode ? 1 : 2 + (moe::router_tc_eligible(a) ? 2 : 0)) + nl;
    }
    if (le != cudaSuccess) return cuda_fail(h, le, "expert kernel launch");
    return MOE_OK;
}

int moe_sync(moe_handle* h) {
    if (!h) return MOE_ERR_INVALID;
    CK(h, cudaSetDevice(h->d.device));
    drain(h);
    if (h->last_stream) CK(h, cudaStreamSynchronize(h->last_stream));
    CK(h, cudaStreamSynchronize(h->copy));
    CK(h, cudaStreamSynchronize(h->copy2));
    // a bounded wait that gave up after the call's routing kernel had reported
    int32_t dev_err = 0;
    CK(h, cudaMemcpy(&dev_err, h->base.dev_err, 4, cudaMemcpyDeviceToHost));
    if (h->log) {
        unsigned long long rv = 0;
        cudaMemcpy(&rv, h->ready, 8, cudaMemcpyDeviceToHost);
        std::fprintf(stderr, "[moe] sync: submitted %llu serviced %llu ready %llu dev_err %d write64 %d\n",
                     static_cast<unsigned long long>(h->submitted),
                     static_cast<unsigned long long>(h->serviced.load()), rv, dev_err, h->write64 ? 1 : 0);
    }
    if (dev_err != 0)
        record_error(h, MOE_ERR_TIMEOUT, "a kernel gave up a bounded wait (device error " + std::to_string(dev_err) +
                                             "); call moe_cache_config to reset");
    if (h->trace && !h->last_fused) {
        const size_t base = static_cast<size_t>(h->num_sms) * moe::kTracePoints + (moe::kTraceCalls - 1) * 4;
        unsigned long long r[4];
        CK(h, cudaMemcpy(r, h->trace + base, sizeof(r), cudaMemcpyDeviceToHost));
        if (r[0] != ~0ull && r[2] != 0)
            std::fprintf(stderr, "[moe] route: phase A %.2f us, phase B %.2f us\n", (r[1] - r[0]) * 1e-3, (r[2] - r[1]) * 1e-3);
        unsigned long long q[8];
        CK(h, cudaMemcpy(q, h->trace + base - 8, sizeof(q), cudaMemcpyDeviceToHost));
        if (q[0] && q[5] >= q[0])
            std::fprintf(stderr, "[moe] route, last CTA: staged %.2f, candidates %.2f, exact %.2f, top-k %.2f, end %.2f us; %llu candidates\n",
                         (q[1] - q[0]) * 1e-3, (q[2] - q[0]) * 1e-3, (q[3] - q[0]) * 1e-3, (q[4] - q[0]) * 1e-3,
                         (q[5] - q[0]) * 1e-3, q[7]);
        unsigned long long w0[4];
        CK(h, cudaMemcpy(w0, h->trace + base - 16, sizeof(w0), cudaMemcpyDeviceToHost));
        if (q[0] && w0[3] >= w0[0] && w0[0] >= q[0])
            std::fprintf(stderr, "[moe] route, last CTA, warp 0: norm %.2f, bounds %.2f, top-k of the bounds %.2f, candidates %.2f us\n",
                         (w0[0] - q[0]) * 1e-3, (w0[1] - q[0]) * 1e-3, (w0[2] - q[0]) * 1e-3, (w0[3] - q[0]) * 1e-3);
        unsigned long long b[8];
        CK(h, cudaMemcpy(b, h->trace + base - 24, sizeof(b), cudaMemcpyDeviceToHost));
        if (r[0] != ~0ull && r[2] != 0 && b[0] >= r[1] && b[6] >= b[0])
            std::fprintf(stderr,
                         "[moe] route phase B (us after its start): state loaded %.2f, offsets %.2f, permutation %.2f, "
                         "LRU batch %.2f, events %.2f, prefetch batch and shared rows %.2f, end %.2f\n",
                         (b[0] - r[1]) * 1e-3, (b[1] - r[1]) * 1e-3, (b[2] - r[1]) * 1e-3, (b[3] - r[1]) * 1e-3,
                         (b[4] - r[1]) * 1e-3, (b[5] - r[1]) * 1e-3, (b[6] - r[1]) * 1e-3);
        reset_trace(h);
    }
    if (h->trace && h->last_fused) {
        // the last decode call's phase marks: min / median / max over CTAs, in us after the first start
        const int G = h->num_sms, P = moe::kTracePoints;
        std::vector<unsigned long long> t(static_cast<size_t>(G) * P);
        CK(h, cudaMemcpy(t.data(), h->trace, t.size() * 8, cudaMemcpyDeviceToHost));
        unsigned long long t0 = ~0ull;
        for (int b = 0; b < G; ++b)
            if (t[static_cast<size_t>(b) * P]) t0 = std::min(t0, t[static_cast<size_t>(b) * P]);
        std::string line = "[moe] trace T=" + std::to_string(h->last_T);
        for (int p = 0; p < P; ++p) {
            std::vector<double> v;
            for (int b = 0; b < G; ++b) {
                const unsigned long long x = t[static_cast<size_t>(b) * P + p];
                if (x >= t0) v.push_back((x - t0) * 1e-3);
            }
            if (v.empty()) continue;
            std::sort(v.begin(), v.end());
            char buf[96];
            std::snprintf(buf, sizeof(buf), " p%d=%.2f/%.2f/%.2f", p, v.front(), v[v.size() / 2], v.back());
            line += buf;
        }
        std::fprintf(stderr, "%s\n", line.c_str());
        // the calls since the last report: entry, dependency wait, exit, and the gap to the previous exit
        const size_t base = static_cast<size_t>(G) * P;
        std::vector<unsigned long long> c(moe::kTraceCalls * 4);
        CK(h, cudaMemcpy(c.data(), h->trace + base, c.size() * 8, cudaMemcpyDeviceToHost));
        unsigned long long prev_exit = 0;
        const unsigned long long n = std::min<unsigned long long>(h->dcalls, moe::kTraceCalls);
        for (unsigned long long d = h->dcalls - n; d < h->dcalls; ++d) {
            const unsigned long long* e = c.data() + (d % moe::kTraceCalls) * 4;
            if (e[0] == ~0ull || e[2] == 0) continue;
            char buf[160];
            std::snprintf(buf, sizeof(buf), "[moe] call %llu entry->wait %.2f us, wait->exit %.2f us, gap after previous exit %.2f us",
                          d, (e[1] - e[0]) * 1e-3, (e[2] - e[1]) * 1e-3,
                          prev_exit ? (static_cast<double>(e[0]) - static_cast<double>(prev_exit)) * 1e-3 : 0.0);
            std::fprintf(stderr, "%s\n", buf);
            prev_exit = e[2];
        }
        reset_trace(h);
    }
    return take_error(h);
}

int moe_timing_enable(moe_handle* h, int enable) {
    if (!h) return MOE_ERR_INVALID;
    CK(h, cudaSetDevice(h->d.device));
    drain(h);
    harvest(h, true);
    h->tm = moe_timing_t{};
    h->timing = enable != 0;
    return MOE_OK;
}

int moe_timing(moe_handle* h, moe_timing_t* t) {
    if (!h || !t) return MOE_ERR_INVALID;
    CK(h, cudaSetDevice(h->d.device));
    drain(h);
    harvest(h, true);
    *t = h->tm;
    return MOE_OK;
}

int moe_stats(moe_handle* h, moe_stats_t* s) {
    if (!h || !s) return MOE_ERR_INVALID;
    drain(h);
    std::lock_guard<std::mutex> lk(h->mu);
    *s = h->st;
    return MOE_OK;
}

int moe_stats_reset(moe_handle* h) {
    if (!h) return MOE_ERR_INVALID;
    drain(h);
    std::lock_guard<std::mutex> lk(h->mu);
    h->st = moe_stats_t{};
    h->events.clear();
    return MOE_OK;
}

int moe_stats_events(moe_handle* h, moe_event* buf, int cap, int* n) {
    if (!h || !n || cap < 0 || (cap > 0 && !buf)) return MOE_ERR_INVALID;
    drain(h);
    std::lock_guard<std::mutex> lk(h->mu);
    const int m = std::min<int>(cap, static_cast<int>(h->events.size()));
    for (int i = 0; i < m; ++i) buf[i] = h->events[i];
    h->events.erase(h->events.begin(), h->events.begin() + m);
    *n = m;
    return MOE_OK;
}

int moe_debug_routing(moe_handle* h, int32_t* topk_idx, float* gates, int32_t* perm, int32_t* counts,
                      int32_t* uniq, int32_t* n_uniq) {
    if (!h) return MOE_ERR_INVALID;
    CK(h, cudaSetDevice(h->d.device));
    drain(h);
    if (h->last_stream) CK(h, cudaStreamSynchronize(h->last_stream));
    const size_t n = static_cast<size_t>(h->last_T) * h->d.top_k;
    const CallArgs& a = h->base;
    if (topk_idx) CK(h, cudaMemcpy(topk_idx, a.topk, n * 4, cudaMemcpyDeviceToHost));
    if (gates) CK(h, cudaMemcpy(gates, a.gates, n * 4, cudaMemcpyDeviceToHost));
    if (perm) CK(h, cudaMemcpy(perm, a.perm, n * 4, cudaMemcpyDeviceToHost));
    if (counts) CK(h, cudaMemcpy(counts, a.counts, static_cast<size_t>(h->d.num_experts) * 4, cudaMemcpyDeviceToHost));
    int32_t nu = 0;
    CK(h, cudaMemcpy(&nu, a.n_uniq, 4, cudaMemcpyDeviceToHost));
    if (uniq) CK(h, cudaMemcpy(uniq, a.act_expert, static_cast<size_t>(nu) * 4, cudaMemcpyDeviceToHost));
    if (n_uniq) *n_uniq = nu;
    return MOE_OK;
}

int moe_debug_lru_table(moe_handle* h, int32_t* table) {
    if (!h || !table) return MOE_ERR_INVALID;
    if (!h->table) return fail(h, MOE_ERR_STATE, "moe_cache_config has not been called");
    CK(h, cudaSetDevice(h->d.device));
    drain(h);
    if (h->last_stream) CK(h, cudaStreamSynchronize(h->last_stream));
    CK(h, cudaMemcpy(table, h->table, static_cast<size_t>(h->d.num_layers) * h->d.num_experts * 4,
                     cudaMemcpyDeviceToHost));
    return MOE_OK;
}

const char* moe_last_error(const moe_handle* h) { return h ? h->err.c_str() : "NULL handle"; }

void moe_destroy(moe_handle* h) {
    if (!h) return;
    cudaSetDevice(h->d.device);
    stop_service(h);
    cudaDeviceSynchronize();
    free_timed(h);
    free_pool(h);
    for (auto* b : h->bank)
        if (b) cudaFreeHost(b);
    cudaFree(h->shared_dev);
    cudaFree(h->scratch);
    cudaFree(h->trace);
    if (h->info_h) cudaFreeHost(h->info_h);
    if (h->ready_vals) cudaFreeHost(h->ready_vals);
    if (h->stream) cudaStreamDestroy(h->stream);
    if (h->copy) cudaStreamDestroy(h->copy);
    if (h->copy2) cudaStreamDestroy(h->copy2);
    if (h->ev_join) cudaEventDestroy(h->ev_join);
    if (h->ev_pf) cudaEventDestroy(h->ev_pf);
    delete h;
}

}  // extern "C"
