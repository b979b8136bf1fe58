// qknr_api.cu -- the C ABI (include/qknr.h): validation, work map, launch.
//
// Argument rules follow the tensor contract of the fused_inplace_qknorm_rope
// deep-dive §3 and the host checks of §4.7 (shape/stride/dtype checks before
// launch, int32 or int64 positions, grid sized from occupancy x SM count, the
// CUDA launch error checked), restated for this library's kernels.
//
// Two kernels compute the op, with the same bits: the register kernel
// qknr_fused_kernel (qknr_kernel.cuh), which loads straight into registers,
// and the ring kernel qknr_ring_kernel (qknr_ring_kernel.cuh), which
// double-buffers each warp's items in shared memory with asynchronous
// copies. The work map picks one per call by a measured rule (plan_register).
//
// Entry points beyond the op itself: the position-checked variants (one with
// no allocation), the unfused two-kernel baseline, the host-buffer variant
// (direct or staged) and the variant with separate q and k head strides.
#include "../../include/qknr.h"
#include "qknr_dispatch.h"
#include "qknr_kernel.cuh"
#include "qknr_ring_kernel.cuh"

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <initializer_list>
#include <mutex>
#include <array>
#include <set>
#include <string>
#include <unordered_map>
#include <vector>

namespace {

using qknr::Params;

constexpr int kMaxDevices = 64;
constexpr int kVersion = 10400;             // 1.4.0: the ring kernel
constexpr int kStatusWords = 2;             // {bad-token count, first bad token}
constexpr int kMaxHeads = 1 << 24;                // largest n_qo + n_kv accepted
constexpr long long kMaxExtentBytes = 1LL << 56;  // largest q or k extent accepted (far above any GPU's memory)

thread_local std::string t_last_error;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

int fail_cuda(cudaError_t e, const char *what) {
    return fail(QKNR_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

// ------------------------------------------------------------------ tuning
constexpr int kNumTuneKeys = 11;  // keys 1..6, 9 and 10 (QKNR_TUNE_*); the other slots are unused
// the value that means "automatic" for each key
constexpr int kTuneAuto[kNumTuneKeys] = {0, 0, 0, 0, 0, -1, 0, 0, 0, 0, 0};
std::atomic<int> g_tune[kNumTuneKeys] = {{0}, {0}, {0}, {0}, {0}, {-1}, {0}, {0}, {0}, {0}, {0}};
// items per warp prefetched into L2 before the wait (automatic): the register
// kernel's first loads all wait on DRAM, the ring kernel's first copies go out
// right after the wait and compete with more prefetches (measured on a
// 4608-token DiT call: one item 5802 GB/s, two 5725, four 5623)
constexpr int kAutoPrefetchItems = 4;
constexpr int kAutoPrefetchRing = 1;
constexpr int kMaxPrefetchItems = 4;
std::once_flag g_env_once;

int tune_check(int key, int value) {
    switch (key) {
        case QKNR_TUNE_KERNEL:
            return (value >= 0 && value <= QKNR_KERNEL_RING)
                       ? QKNR_OK
                       : fail(QKNR_ERR_INVALID_ARG, "kernel must be 0 (auto), 1 (register) or 2 (ring)");
        case QKNR_TUNE_RING_ORDER:
            return (value >= 0 && value <= 2)
                       ? QKNR_OK
                       : fail(QKNR_ERR_INVALID_ARG, "ring order must be 0 (auto), 1 (next after the wait) or 2 (two ahead)");
        case QKNR_TUNE_PASSES:
            return (value >= 0 && value <= qknr::kUnrollClass[qknr::kNumUnroll - 1])
                       ? QKNR_OK
                       : fail(QKNR_ERR_INVALID_ARG, "passes per item must be in [0, %d]",
                              qknr::kUnrollClass[qknr::kNumUnroll - 1]);
        case QKNR_TUNE_THREADS:
            return (value == 0 || value == 64 || value == 128 || value == 256 || value == 512)
                       ? QKNR_OK
                       : fail(QKNR_ERR_INVALID_ARG, "threads per CTA must be 0 or one of 64/128/256/512");
        case QKNR_TUNE_CTAS_PER_SM:
            return (value >= 0 && value <= 32) ? QKNR_OK
                                               : fail(QKNR_ERR_INVALID_ARG, "CTAs per SM must be in [0, 32]");
        case QKNR_TUNE_PDL:
            return (value >= -1 && value <= 1) ? QKNR_OK
                                                : fail(QKNR_ERR_INVALID_ARG, "use_pdl must be -1, 0 or 1");
        case QKNR_TUNE_ORDER:
            return (value >= 0 && value <= 2)
                       ? QKNR_OK
                       : fail(QKNR_ERR_INVALID_ARG, "order must be 0 (auto), 1 (contiguous) or 2 (interleaved)");
        case QKNR_TUNE_PREFETCH:
            return (value >= -1 && value <= kMaxPrefetchItems)
                       ? QKNR_OK
                       : fail(QKNR_ERR_INVALID_ARG, "prefetch must be -1 (none), 0 (auto) or 1..%d items",
                              kMaxPrefetchItems);
        default:
            return fail(QKNR_ERR_INVALID_ARG, "unknown tuning key %d", key);
    }
}

// QKNR_TUNE="kernel=2,ring_order=1,passes=4,threads=256,ctas=2,pdl=1,order=2,prefetch=1"
void read_env_tuning() {
    const char *s = std::getenv("QKNR_TUNE");
    if (!s) return;
    static const struct {
        const char *name;
        int key;
    } names[] = {{"kernel", QKNR_TUNE_KERNEL}, {"ring_order", QKNR_TUNE_RING_ORDER},
                 {"passes", QKNR_TUNE_PASSES}, {"threads", QKNR_TUNE_THREADS},
                 {"ctas", QKNR_TUNE_CTAS_PER_SM}, {"pdl", QKNR_TUNE_PDL},
                 {"order", QKNR_TUNE_ORDER},      {"prefetch", QKNR_TUNE_PREFETCH}};
    std::string spec(s);
    size_t pos = 0;
    while (pos < spec.size()) {
        size_t end = spec.find(',', pos);
        if (end == std::string::npos) end = spec.size();
        const std::string item = spec.substr(pos, end - pos);
        const size_t eq = item.find('=');
        if (eq != std::string::npos) {
            const std::string k = item.substr(0, eq);
            const int v = std::atoi(item.c_str() + eq + 1);
            for (const auto &n : names)
                if (k == n.name && tune_check(n.key, v) == QKNR_OK) g_tune[n.key] = v;
        }
        pos = end + 1;
    }
}

int tune(int key) {
    std::call_once(g_env_once, read_env_tuning);
    return g_tune[key].load(std::memory_order_relaxed);
}

// ------------------------------------------------------------------ devices
// A call shape and layout that qknr_tune measured, and the work map it chose.
struct ShapeKey {
    long long num_tokens, q_stride, k_stride, head_stride;
    int n_qo, n_kv, head_dim, rope_dim, is_neox, dtype;
    bool operator==(const ShapeKey &o) const {
        return num_tokens == o.num_tokens && q_stride == o.q_stride && k_stride == o.k_stride &&
               head_stride == o.head_stride && n_qo == o.n_qo && n_kv == o.n_kv && head_dim == o.head_dim &&
               rope_dim == o.rope_dim && is_neox == o.is_neox && dtype == o.dtype;
    }
};
struct ShapeHash {
    size_t operator()(const ShapeKey &k) const {
        size_t h = std::hash<long long>()(k.num_tokens);
        for (long long v : {k.q_stride, k.k_stride, k.head_stride, static_cast<long long>(k.n_qo),
                            static_cast<long long>(k.n_kv), static_cast<long long>(k.head_dim),
                            static_cast<long long>(k.rope_dim), static_cast<long long>(k.is_neox),
                            static_cast<long long>(k.dtype)})
            h = h * 1000003u ^ std::hash<long long>()(v);
        return h;
    }
};
// The knobs qknr_tune chooses: the kernel (and the ring kernel's issue order,
// 1 or 2 as QKNR_TUNE_RING_ORDER), warp passes per item and items per warp
// prefetched into L2 before the wait (-1: none). A 0 in any field leaves that
// knob to the fixed rule, so an all-zero map is the rule's own launch.
struct TunedMap {
    int kernel = QKNR_KERNEL_AUTO;
    int ring_order = 0;
    int passes = 0;
    int prefetch = 0;
};

struct DeviceState {
    std::atomic<bool> ready{false};
    int sm_count = 0;
    unsigned long long *status = nullptr;       // device: kStatusWords words
    unsigned long long *status_host = nullptr;  // pinned host copy (qknr_init) or nullptr
    std::mutex checked_mu;                      // serialises status read-backs on this device
    // resident CTAs per SM for the register kernel, by (early, dtype, pos64, d_idx, mode, u_idx,
    // rope_dim class, threads class)
    std::atomic<int> occupancy[2][2][2][qknr::kNumHeadDim][2][qknr::kNumUnroll][qknr::kNumRope][4];
    // the same for the ring kernel, by (early, dtype, pos64, d_idx, mode, rope_dim class, threads class)
    std::atomic<int> ring_occ[2][2][2][qknr::kNumHeadDim][2][qknr::kNumRope][4];
    // resident CTAs per SM of the unfused-baseline kernels, by (dtype, op-1, pos64, d_idx, mode)
    std::atomic<int> unfused_occ[2][2][2][qknr::kNumHeadDim][2];
    // host-buffer pipeline (qknr_apply_host): a host-to-device and a
    // device-to-host copy stream and the events that order them against the
    // caller's stream; made by the first such call on this device
    std::mutex host_mu;
    bool host_ready = false;
    cudaStream_t host_in = nullptr, host_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_in = nullptr, ev_kernel = nullptr, ev_out = nullptr;
    // work maps chosen by qknr_tune, by call shape; kept until qknr_shutdown
    std::mutex tuned_mu;
    std::unordered_map<ShapeKey, TunedMap, ShapeHash> tuned;
    std::atomic<bool> has_tuned{false};
};

DeviceState g_dev[kMaxDevices];
std::mutex g_init_mu;

int head_dim_index(int d) {
    for (int i = 0; i < qknr::kNumHeadDim; ++i)
        if (qknr::kHeadDims[i] == d) return i;
    return -1;
}

int threads_index(int threads) {
    switch (threads) {
        case 64: return 0;
        case 128: return 1;
        case 256: return 2;
        case 512: return 3;
        default: return -1;
    }
}

// Accepted set (qknr_can_use).
bool shape_ok(int head_dim, int rope_dim, int is_neox) {
    if (head_dim_index(head_dim) < 0) return false;
    if (rope_dim <= 0 || rope_dim > head_dim || (rope_dim & 1)) return false;
    if (is_neox) return (rope_dim % 16) == 0 || rope_dim <= 8;
    return true;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Heads one warp pass covers: a head's lane group is head_dim/16 lanes rounded
// up to a power of two (the kernels' padding for head_dim 80, 96 and 192).
int heads_per_pass(int head_dim) {
    int lph = 1;
    while (lph < head_dim / 16) lph *= 2;
    return qknr::kWarp / lph;
}

// ------------------------------------------------------------------ one call
struct Call {
    void *q = nullptr, *k = nullptr;
    const void *q_w = nullptr, *k_w = nullptr;
    const float *cache = nullptr;
    const void *positions = nullptr;
    long long cache_len = 0;  // > 0: checked
    long long num_tokens = 0;
    int n_qo = 0, n_kv = 0, head_dim = 0, rope_dim = 0, is_neox = 0;
    long long q_stride = 0, k_stride = 0, head_stride = 0;  // elements
    long long k_head_stride = -1;  // elements; < 0: k's heads are head_stride apart too
    float eps = 0.f;
    int dtype = 0;
};

struct WorkMap {
    int kind = QKNR_KERNEL_REGISTER;
    int grid = 0, threads = 0, ctas_per_sm = 0, pdl = 1;
    long long items = 0;  // warp items: (token, chunk of warp passes)
    int chunks_per_token = 0;
    int passes_per_token = 0, max_passes = 0, u_idx = 0;
    int r_idx = 0;        // rope_dim class of the instantiation (qknr::kRope*)
    int interleave = 0;   // item order
    int prefetch_items = 0;  // items per warp prefetched into L2 before the wait
    int smem = 0;            // dynamic shared memory per CTA (ring kernel)
    int ring_ahead = 0;      // ring kernel's issue order (Params::ring_ahead)
    const void *kernel = nullptr;
};

// Resident CTAs per SM of `kernel` at `threads` threads and `smem` bytes of
// dynamic shared memory: asked of the occupancy API once, then cached in
// `slot`. A kernel with dynamic shared memory first gets its limit raised to
// what the largest CTA (512 threads) would need, once per kernel; that limit
// is an attribute of the kernel, not of a launch.
int cached_occupancy(std::atomic<int> &slot, const void *kernel, int threads, const char *what, int *out,
                     int smem = 0) {
    int v = slot.load(std::memory_order_relaxed);
    if (v == 0) {
        cudaError_t e = cudaSuccess;
        if (smem > 0)
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, qknr::ring_smem_bytes(512));
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kernel, threads, smem);
        if (e != cudaSuccess) return fail_cuda(e, what);
        if (v <= 0) return fail(QKNR_ERR_CUDA, "%s: the kernel cannot be resident with %d threads", what, threads);
        slot.store(v, std::memory_order_relaxed);
    }
    *out = v;
    return QKNR_OK;
}

// A persistent grid: CTAs for every warp item, at most one wave of resident CTAs.
int persistent_grid(long long items, int threads, int ctas_per_sm, int sm_count) {
    const long long warps_per_cta = threads / qknr::kWarp;
    const long long needed = (items + warps_per_cta - 1) / warps_per_cta;
    return static_cast<int>(std::max(1LL, std::min(needed, static_cast<long long>(ctas_per_sm) * sm_count)));
}

int resident_ctas(DeviceState &st, int dt, int pos64, int d_idx, int mode, int u_idx, int r_idx, int threads,
                  int early, const void *kernel, int *out) {
    return cached_occupancy(st.occupancy[early][dt][pos64][d_idx][mode][u_idx][r_idx][threads_index(threads)],
                            kernel, threads, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(register)", out);
}

const void *ring_kernel(int dt, int early, int pos64, int d_idx, int mode, int r_idx) {
    return early ? (dt ? qknr::ring_kernel_fp16_early(pos64, d_idx, mode, r_idx)
                       : qknr::ring_kernel_bf16_early(pos64, d_idx, mode, r_idx))
                 : (dt ? qknr::ring_kernel_fp16(pos64, d_idx, mode, r_idx)
                       : qknr::ring_kernel_bf16(pos64, d_idx, mode, r_idx));
}

const void *register_kernel(int dt, int early, int pos64, int d_idx, int mode, int u_idx, int r_idx) {
    return early ? (dt ? qknr::kernel_fp16_early(pos64, d_idx, mode, u_idx, r_idx)
                       : qknr::kernel_bf16_early(pos64, d_idx, mode, u_idx, r_idx))
                 : (dt ? qknr::kernel_fp16(pos64, d_idx, mode, u_idx, r_idx)
                       : qknr::kernel_bf16(pos64, d_idx, mode, u_idx, r_idx));
}

ShapeKey shape_key(const Call &c) {
    ShapeKey k;
    k.num_tokens = c.num_tokens;
    k.q_stride = c.q_stride;
    k.k_stride = c.k_stride;
    k.head_stride = c.head_stride;
    k.n_qo = c.n_qo;
    k.n_kv = c.n_kv;
    k.head_dim = c.head_dim;
    k.rope_dim = c.rope_dim;
    k.is_neox = c.is_neox;
    k.dtype = c.dtype;
    return k;
}

// The work map qknr_tune chose for this call's shape, if any.
bool tuned_for(DeviceState &st, const Call &c, TunedMap *out) {
    if (!st.has_tuned.load(std::memory_order_acquire) || c.k_head_stride >= 0) return false;
    std::lock_guard<std::mutex> lock(st.tuned_mu);
    auto it = st.tuned.find(shape_key(c));
    if (it == st.tuned.end()) return false;
    *out = it->second;
    return true;
}

// The measured rule (GB300, same-box sweeps of both kernels and both ring
// orders over call shapes and sizes): the ring kernel for every call whose
// items have three or four passes (+4% to +14% over the register kernel at
// the benchmark's sizes), the register kernel for decode-sized calls.
//
// The ring's issue order: order 2 (two items ahead, Params::ring_ahead = 1)
// starts slower than order 1 and then sustains more bandwidth, but only where
// an item's arithmetic is light for its bytes: interleaved pairing, bf16, and
// a head_dim whose lane groups have no idle lanes (64, 128, 256). There it
// pays from about 6.5 rounds of items per warp up (a 4608-token DiT call runs
// 5.7 and keeps order 1: +3.5%; fused_qkv runs 81: +5.7% with order 2).
// Everywhere else order 1 measured ahead at every size tried: NeoX (gqa +7%
// at 20 rounds), fp16 (head_dim 64, 3-pass items: +4.4%), head_dim 96 and 192
// (+4.5% and +3.4%).
bool ring_by_rule(const WorkMap &wm) { return wm.u_idx == 1; }
constexpr int kRingSmallCta = 64;         // threads per CTA: ring order 1 on interleaved calls
constexpr int kRingLargeCta = 512;        // threads per CTA: ring order 2 on long calls
constexpr long long kRingLargeCtaRounds = 32;   // rounds of items per warp from which order 2 takes 512

int ring_ahead_by_rule(const Call &c, const WorkMap &wm) {
    const bool light = !c.is_neox && (c.dtype & 0xff) == QKNR_BF16 &&
                       (c.head_dim == 64 || c.head_dim == 128 || c.head_dim == 256);
    if (!light) return 0;
    const long long warps = static_cast<long long>(wm.grid) * (wm.threads / qknr::kWarp);
    return 2 * wm.items >= 13 * warps ? 1 : 0;   // rounds = items / warps >= 6.5
}

// Items are (token, chunk of warp passes); the default is the largest unroll
// class (8 x 16-byte loads in flight per lane, or four passes per ring stage).
// `force` (from qknr_tune's measurements) sets the kernel, the passes per item
// and the prefetch depth; otherwise an explicit qknr_set_tuning value, then a
// work map that qknr_tune chose for this shape, then the fixed rule decide.
int plan_register(DeviceState &st, const Call &c, WorkMap *wm, const TunedMap *force = nullptr) {
    const int d_idx = head_dim_index(c.head_dim);
    const int hpw = heads_per_pass(c.head_dim);
    const int heads = c.n_qo + c.n_kv;
    wm->passes_per_token = (heads + hpw - 1) / hpw;
    TunedMap tm;
    const bool tuned = force ? (tm = *force, true) : tuned_for(st, c, &tm);
    int ppi = force ? force->passes : tune(QKNR_TUNE_PASSES);
    if (ppi <= 0 && tuned) ppi = tm.passes;
    if (ppi <= 0) {
        // a problem too small to give every SM several warps (decode-sized
        // batches) spreads its passes over as many warps as it can
        const long long passes = c.num_tokens * wm->passes_per_token;
        ppi = passes <= 16LL * st.sm_count ? 1 : qknr::kUnrollClass[qknr::kNumUnroll - 1];
    }
    wm->chunks_per_token = (wm->passes_per_token + ppi - 1) / ppi;
    wm->max_passes = (wm->passes_per_token + wm->chunks_per_token - 1) / wm->chunks_per_token;
    wm->u_idx = wm->max_passes <= 2 ? 0 : 1;
    wm->items = c.num_tokens * wm->chunks_per_token;
    const bool auto_threads = threads_index(tune(QKNR_TUNE_THREADS)) < 0;
    int threads = auto_threads ? 256 : tune(QKNR_TUNE_THREADS);
    wm->threads = threads;

    const int dt = (c.dtype & 0xff) == QKNR_FP16 ? 1 : 0;
    const int pos64 = (c.dtype & QKNR_POS_I64) ? 1 : 0;
    const int mode = c.is_neox ? qknr::kNeox : qknr::kInterleaved;
    const int early = (c.dtype & QKNR_INPUTS_READY) ? 1 : 0;
    // rope_dim fixed at compile time where it measured faster (interleaved
    // pairing, 4-pass items, rope_dim = head_dim or head_dim / 2); the table has
    // no such instantiation elsewhere, and then the run-time rope_dim kernel runs
    wm->r_idx = qknr::kRopeRuntime;
    if (mode == qknr::kInterleaved && wm->u_idx == 1)
        wm->r_idx = c.rope_dim == c.head_dim ? qknr::kRopeFull
                    : (2 * c.rope_dim == c.head_dim ? qknr::kRopeHalf : qknr::kRopeRuntime);
    int kind = force ? force->kernel : tune(QKNR_TUNE_KERNEL);
    if (kind == QKNR_KERNEL_AUTO && tuned) kind = tm.kernel;
    if (kind == QKNR_KERNEL_AUTO) kind = ring_by_rule(*wm) ? QKNR_KERNEL_RING : QKNR_KERNEL_REGISTER;
    wm->kind = kind;
    int order = force ? force->ring_order : tune(QKNR_TUNE_RING_ORDER);
    if (order == 0 && tuned) order = tm.ring_order;
    int occ = 0;
    int rc = QKNR_OK;
    if (kind == QKNR_KERNEL_RING) {
        wm->kernel = ring_kernel(dt, early, pos64, d_idx, mode, wm->r_idx);
        if (!wm->kernel && wm->r_idx != qknr::kRopeRuntime) {
            wm->r_idx = qknr::kRopeRuntime;
            wm->kernel = ring_kernel(dt, early, pos64, d_idx, mode, wm->r_idx);
        }
        if (!wm->kernel) return fail(QKNR_ERR_UNSUPPORTED, "no ring kernel for this shape");
        wm->smem = qknr::ring_smem_bytes(threads);
        rc = cached_occupancy(st.ring_occ[early][dt][pos64][d_idx][mode][wm->r_idx][threads_index(threads)],
                              wm->kernel, threads, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(ring)", &occ,
                              wm->smem);
    } else {
        wm->kernel = register_kernel(dt, early, pos64, d_idx, mode, wm->u_idx, wm->r_idx);
        if (!wm->kernel && wm->r_idx != qknr::kRopeRuntime) {
            wm->r_idx = qknr::kRopeRuntime;
            wm->kernel = register_kernel(dt, early, pos64, d_idx, mode, wm->u_idx, wm->r_idx);
        }
        if (!wm->kernel) return fail(QKNR_ERR_UNSUPPORTED, "no kernel for this shape");
        wm->smem = 0;
        rc = resident_ctas(st, dt, pos64, d_idx, mode, wm->u_idx, wm->r_idx, threads, early, wm->kernel, &occ);
    }
    if (rc) return rc;
    const int cap = tune(QKNR_TUNE_CTAS_PER_SM);
    if (cap > 0) occ = std::min(occ, cap);
    wm->ctas_per_sm = occ;
    wm->grid = persistent_grid(wm->items, threads, occ, st.sm_count);
    wm->ring_ahead = kind != QKNR_KERNEL_RING ? 0 : (order == 0 ? ring_ahead_by_rule(c, *wm) : order - 1);
    if (auto_threads && cap <= 0 && kind == QKNR_KERNEL_RING) {
        // The ring kernel's CTA size, at the same 16 resident warps per SM:
        // interleaved calls on issue order 1 measured faster in CTAs of two
        // warps (dit +1.6%, 2304 tokens +2.2%, head_dim 192 +3%; the next
        // launch's CTAs take an SM's slots as soon as two warps of this one
        // are done), calls on order 2 whose warps run at least 32 rounds of
        // items in one CTA per SM (+0.35% to +1%: each SM's warps take
        // consecutive items, a contiguous stretch of q and k per round).
        const long long warps = static_cast<long long>(wm->grid) * (threads / qknr::kWarp);
        int want = threads;
        if (wm->ring_ahead == 0 && !c.is_neox) want = kRingSmallCta;
        if (wm->ring_ahead == 1 && wm->items >= kRingLargeCtaRounds * warps) want = kRingLargeCta;
        if (want != threads) {
            threads = want;
            wm->threads = threads;
            wm->smem = qknr::ring_smem_bytes(threads);
            rc = cached_occupancy(st.ring_occ[early][dt][pos64][d_idx][mode][wm->r_idx][threads_index(threads)],
                                  wm->kernel, threads, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(ring)", &occ,
                                  wm->smem);
            if (rc) return rc;
            wm->ctas_per_sm = occ;
            wm->grid = persistent_grid(wm->items, threads, occ, st.sm_count);
        }
    }
    wm->interleave = tune(QKNR_TUNE_ORDER) == 1 ? 0 : 1;   // interleaved unless asked otherwise
    int pf = force ? force->prefetch : tune(QKNR_TUNE_PREFETCH);
    if (pf == 0 && tuned) pf = tm.prefetch;
    const int auto_pf = kind == QKNR_KERNEL_RING ? kAutoPrefetchRing : kAutoPrefetchItems;
    wm->prefetch_items = pf < 0 ? 0 : (pf > 0 ? pf : auto_pf);
    return QKNR_OK;
}

int plan(DeviceState &st, const Call &c, WorkMap *wm) {
    const int rc = plan_register(st, c, wm);
    if (rc) return rc;
    const int pdl = tune(QKNR_TUNE_PDL);
    wm->pdl = pdl < 0 ? 1 : pdl;
    return QKNR_OK;
}

// One step of the unfused baseline: the register kernel's work map (4 passes
// per item, 256 threads) with the norm-only or rope-only instantiation.
int plan_unfused(DeviceState &st, const Call &c, int op, WorkMap *wm) {
    const int d_idx = head_dim_index(c.head_dim);
    const int hpw = heads_per_pass(c.head_dim);
    wm->kind = QKNR_KERNEL_REGISTER;
    wm->passes_per_token = (c.n_qo + c.n_kv + hpw - 1) / hpw;
    wm->chunks_per_token = (wm->passes_per_token + 3) / 4;
    wm->max_passes = (wm->passes_per_token + wm->chunks_per_token - 1) / wm->chunks_per_token;
    wm->u_idx = 1;
    wm->items = c.num_tokens * wm->chunks_per_token;
    wm->threads = 256;
    const int dt = (c.dtype & 0xff) == QKNR_FP16 ? 1 : 0;
    const int pos64 = (c.dtype & QKNR_POS_I64) ? 1 : 0;
    const int mode = c.is_neox ? qknr::kNeox : qknr::kInterleaved;
    wm->kernel = dt ? qknr::unfused_kernel_fp16(op, pos64, d_idx, mode)
                    : qknr::unfused_kernel_bf16(op, pos64, d_idx, mode);
    if (!wm->kernel) return fail(QKNR_ERR_UNSUPPORTED, "no unfused kernel for this shape");
    int occ = 0;
    const int rc = cached_occupancy(st.unfused_occ[dt][op - 1][pos64][d_idx][mode], wm->kernel, wm->threads,
                                    "cudaOccupancyMaxActiveBlocksPerMultiprocessor(unfused)", &occ);
    if (rc) return rc;
    wm->ctas_per_sm = occ;
    wm->grid = persistent_grid(wm->items, wm->threads, occ, st.sm_count);
    const int pf = tune(QKNR_TUNE_PREFETCH);
    wm->prefetch_items = pf < 0 ? 0 : (pf == 0 ? kAutoPrefetchItems : pf);
    const int pdl = tune(QKNR_TUNE_PDL);
    wm->pdl = pdl < 0 ? 1 : pdl;
    return QKNR_OK;
}

DeviceState *current_state() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (!g_dev[dev].ready.load(std::memory_order_acquire)) return nullptr;
    return &g_dev[dev];
}

// Byte extent of one token row: heads [0, n) with the shared head stride.
long long row_bytes(int n, long long head_stride_b, int head_dim) {
    return static_cast<long long>(n - 1) * head_stride_b + 2LL * head_dim;
}

int validate(const Call &c) {
    const int dtype = c.dtype;
    if ((dtype & ~(0xff | QKNR_POS_I64 | QKNR_INPUTS_READY)) != 0 ||
        ((dtype & 0xff) != QKNR_BF16 && (dtype & 0xff) != QKNR_FP16))
        return fail(QKNR_ERR_INVALID_ARG,
                    "dtype 0x%x is not QKNR_BF16/QKNR_FP16 [| QKNR_POS_I64] [| QKNR_INPUTS_READY]", dtype);
    if (c.num_tokens < 0) return fail(QKNR_ERR_INVALID_ARG, "num_tokens %lld < 0", c.num_tokens);
    if (c.n_qo < 1 || c.n_kv < 1)
        return fail(QKNR_ERR_INVALID_ARG, "head counts n_qo=%d n_kv=%d must be >= 1", c.n_qo, c.n_kv);
    if (static_cast<long long>(c.n_qo) + c.n_kv > kMaxHeads)  // the kernels count a token's heads in an int
        return fail(QKNR_ERR_INVALID_ARG, "n_qo + n_kv = %lld exceeds %d heads per token",
                    static_cast<long long>(c.n_qo) + c.n_kv, kMaxHeads);
    if (!shape_ok(c.head_dim, c.rope_dim, c.is_neox))
        return fail(QKNR_ERR_UNSUPPORTED,
                    "unsupported head_dim=%d rope_dim=%d is_neox=%d (head_dim in {64,80,96,128,192,256}; rope_dim even, "
                    "0 < rope_dim <= head_dim; NeoX needs rope_dim %% 16 == 0 or rope_dim <= 8)",
                    c.head_dim, c.rope_dim, c.is_neox);
    if (!std::isfinite(c.eps) || c.eps < 0.f) return fail(QKNR_ERR_INVALID_ARG, "eps must be a finite value >= 0");
    if (!c.q || !c.k || !c.q_w || !c.k_w || !c.cache || !c.positions)
        return fail(QKNR_ERR_INVALID_ARG, "null pointer argument");
    const long long k_hs = c.k_head_stride < 0 ? c.head_stride : c.k_head_stride;
    if (c.q_stride < 0 || c.k_stride < 0 || c.head_stride < 0) return fail(QKNR_ERR_INVALID_ARG, "negative stride");
    // Every byte offset below (and in the kernels) is a signed 64-bit value.
    // Bound each tensor's extent first, in 128-bit arithmetic, so that none of
    // them can wrap, whatever sizes a caller passes.
    {
        using wide = __int128;
        const wide last = c.num_tokens > 0 ? c.num_tokens - 1 : 0;
        const wide q_ext = last * c.q_stride * 2 + static_cast<wide>(c.n_qo - 1) * c.head_stride * 2 + 2 * c.head_dim;
        const wide k_ext = last * c.k_stride * 2 + static_cast<wide>(c.n_kv - 1) * k_hs * 2 + 2 * c.head_dim;
        const wide limit = kMaxExtentBytes;
        if (q_ext > limit || k_ext > limit || c.q_stride > kMaxExtentBytes || c.k_stride > kMaxExtentBytes ||
            c.head_stride > kMaxExtentBytes || k_hs > kMaxExtentBytes || c.num_tokens > kMaxExtentBytes)
            return fail(QKNR_ERR_INVALID_ARG, "q or k would span more than 2^56 bytes (sizes or strides out of range)");
    }
    if ((c.n_qo > 1 && c.head_stride < c.head_dim) || (c.n_kv > 1 && k_hs < c.head_dim))
        return fail(QKNR_ERR_INVALID_ARG, "head stride %lld < head_dim %d: heads overlap",
                    c.n_qo > 1 && c.head_stride < c.head_dim ? c.head_stride : k_hs, c.head_dim);
    if (!aligned(c.q, 16) || !aligned(c.k, 16) || !aligned(c.q_w, 16) || !aligned(c.k_w, 16))
        return fail(QKNR_ERR_MISALIGNED, "q, k, q_w and k_w must be 16-byte aligned");
    if ((c.q_stride % 8) || (c.k_stride % 8) || (c.head_stride % 8) || (k_hs % 8))
        return fail(QKNR_ERR_MISALIGNED, "q_stride, k_stride and head strides must be multiples of 8 elements");
    if (!aligned(c.cache, 4)) return fail(QKNR_ERR_MISALIGNED, "cos_sin_cache must be 4-byte aligned");
    if (!aligned(c.positions, (dtype & QKNR_POS_I64) ? 8 : 4))
        return fail(QKNR_ERR_MISALIGNED, "positions must be aligned to their element size");

    const long long hs_b = c.head_stride * 2, qs_b = c.q_stride * 2, ks_b = c.k_stride * 2;
    const long long q_row = row_bytes(c.n_qo, hs_b, c.head_dim), k_row = row_bytes(c.n_kv, k_hs * 2, c.head_dim);
    if (c.num_tokens > 1 && (qs_b < q_row || ks_b < k_row))
        return fail(QKNR_ERR_INVALID_ARG, "token stride smaller than one token's heads: rows overlap");
    if (c.num_tokens > 0) {
        // q and k must be disjoint. Either their address ranges do not meet, or
        // they interleave inside rows of one common token stride.
        const uintptr_t qa = reinterpret_cast<uintptr_t>(c.q), ka = reinterpret_cast<uintptr_t>(c.k);
        const uintptr_t q_end = qa + static_cast<uintptr_t>((c.num_tokens - 1) * qs_b + q_row);
        const uintptr_t k_end = ka + static_cast<uintptr_t>((c.num_tokens - 1) * ks_b + k_row);
        const bool apart = q_end <= ka || k_end <= qa;
        if (!apart) {
            bool ok = false;
            if (qs_b == ks_b && qs_b > 0) {
                const long long S = qs_b;
                const long long diff = static_cast<long long>(ka) - static_cast<long long>(qa);
                const long long off = ((diff % S) + S) % S;  // k row start inside a q row period
                ok = off >= q_row && off + k_row <= S;
            }
            if (!ok) return fail(QKNR_ERR_INVALID_ARG, "q and k overlap in memory");
        }
    }
    return QKNR_OK;
}

// QKNR_LOG=1 (environment): one line on stderr per distinct call shape with
// the launch chosen for it.
void log_launch(const WorkMap &wm, const Call &c) {
    static const bool on = [] {
        const char *e = std::getenv("QKNR_LOG");
        return e && *e && std::strcmp(e, "0") != 0;
    }();
    if (!on) return;
    static std::mutex mu;
    static std::set<std::array<long long, 10>> seen;
    const std::array<long long, 10> key = {c.num_tokens, c.n_qo, c.n_kv, c.head_dim, c.rope_dim, c.is_neox,
                                           c.dtype, wm.kind, wm.threads, wm.grid};
    std::lock_guard<std::mutex> lock(mu);
    if (!seen.insert(key).second) return;
    std::fprintf(stderr,
                 "qknr: T=%lld n_qo=%d n_kv=%d head_dim=%d rope_dim=%d %s %s pos%s -> %s kernel, grid %d x %d, "
                 "%d CTAs/SM, %lld items (%d per token), %d passes per token, rope_dim %s, PDL %s\n",
                 c.num_tokens, c.n_qo, c.n_kv, c.head_dim, c.rope_dim, c.is_neox ? "neox" : "interleaved",
                 (c.dtype & 0xff) == QKNR_FP16 ? "fp16" : "bf16", (c.dtype & QKNR_POS_I64) ? "64" : "32",
                 wm.kind == QKNR_KERNEL_RING ? "ring" : "register", wm.grid, wm.threads, wm.ctas_per_sm,
                 wm.items, wm.chunks_per_token, wm.passes_per_token,
                 wm.r_idx == qknr::kRopeRuntime ? "at run time" : "compiled in", wm.pdl ? "on" : "off");
}

int launch(const WorkMap &wm, const Call &c, unsigned long long *status, cudaStream_t stream) {
    log_launch(wm, c);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(wm.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(wm.threads));
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = wm.pdl ? 1 : 0;
    Params prm = {};
    prm.q = static_cast<char *>(c.q);
    prm.k = static_cast<char *>(c.k);
    prm.q_w = static_cast<const uint4 *>(c.q_w);
    prm.k_w = static_cast<const uint4 *>(c.k_w);
    prm.cache = c.cache;
    prm.positions = c.positions;
    prm.status = status;
    prm.q_stride_b = c.q_stride * 2;
    prm.k_stride_b = c.k_stride * 2;
    prm.head_stride_b = c.head_stride * 2;
    prm.num_items = wm.items;
    prm.cache_len = c.cache_len;
    prm.n_qo = c.n_qo;
    prm.n_kv = c.n_kv;
    prm.rope_dim = c.rope_dim;
    prm.chunks_per_token = wm.chunks_per_token;
    prm.passes_per_token = wm.passes_per_token;
    prm.cache_vec = (c.rope_dim % 8 == 0) && aligned(c.cache, 16);
    prm.interleave = wm.interleave;
    prm.prefetch_items = wm.prefetch_items;
    if (wm.chunks_per_token <= qknr::kBoundTable)
        for (int ch = 0; ch <= wm.chunks_per_token; ++ch)
            prm.pass_bound[ch] = static_cast<short>((static_cast<long long>(ch) * wm.passes_per_token) /
                                                    wm.chunks_per_token);
    prm.eps = c.eps;
    prm.inv_d = 1.0f / static_cast<float>(c.head_dim);
    prm.ring_ahead = wm.ring_ahead;
    cfg.dynamicSmemBytes = static_cast<size_t>(wm.smem);
    void *args[] = {&prm};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, wm.kernel, args);
    if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
    return QKNR_OK;
}

// Checked calls: reset the position status, launch, read the status back, report.
int run_checked(DeviceState &st, const WorkMap &wm, const Call &c, cudaStream_t s,
                unsigned long long *host_words) {
    cudaError_t e = cudaMemsetAsync(st.status, 0, sizeof(unsigned long long), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(st.status + 1, 0xff, sizeof(unsigned long long), s);
    if (e != cudaSuccess) return fail_cuda(e, "status reset");
    int rc = launch(wm, c, st.status, s);
    if (rc) return rc;
    e = cudaMemcpyAsync(host_words, st.status, kStatusWords * sizeof(unsigned long long),
                        cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail_cuda(e, "status read-back");
    if (host_words[0]) {
        return fail(QKNR_ERR_POSITION_OOB,
                    "%llu token(s) have positions outside [0, %lld); first bad token index %llu (left untouched)",
                    host_words[0], c.cache_len, host_words[1]);
    }
    return QKNR_OK;
}

int apply_impl(const Call &c, void *stream, bool checked) {
    DeviceState *st = current_state();
    if (!st) return fail(QKNR_ERR_NOT_INITIALIZED, "qknr_init was not called for the current device");
    int rc = validate(c);
    if (rc) return rc;
    if (checked && c.cache_len < 0) return fail(QKNR_ERR_INVALID_ARG, "cache_len %lld < 0", c.cache_len);
    if (c.num_tokens == 0) return QKNR_OK;
    if (checked && c.cache_len == 0)
        return fail(QKNR_ERR_POSITION_OOB, "cache_len is 0: every position is out of range");
    WorkMap wm;
    rc = plan(*st, c, &wm);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!checked) return launch(wm, c, st->status, s);
    std::lock_guard<std::mutex> lock(st->checked_mu);
    return run_checked(*st, wm, c, s, st->status_host);
}

// ---------------------------------------------------------------------------
// Allocation-free checked variant.
//
// Some callers cannot call cudaMalloc at all: code that runs where allocation
// is forbidden or already accounted for (a pre-sized memory pool, an embedded
// runtime that owns every device allocation, a plug-in loaded into a host
// that reserves the allocator for itself). qknr_apply_checked needs a small
// status word, which qknr_init allocates. This variant keeps that word in
// the file-scope array below instead, so it needs neither qknr_init nor any
// allocation. The array is part of the library image: every GPU that loads
// the library holds its 256 bytes until the process exits.
constexpr int kNoAllocStatusWords = 32;  // 256 bytes; one call uses the first kStatusWords
static_assert(kNoAllocStatusWords >= kStatusWords, "static status array too small");
static __device__ __align__(256) unsigned long long g_noalloc_status[kNoAllocStatusWords];

struct NoAllocSlot {
    std::once_flag once;
    int setup_rc = QKNR_OK;
    std::string setup_err;
    DeviceState state;  // status = device address of g_noalloc_status; no host buffer
};
NoAllocSlot g_noalloc[kMaxDevices];

// Once per device, with that device current: resolve the array's device
// address (in host code its name is only a host-side stand-in) and read the
// SM count. Nothing is allocated.
void noalloc_setup(NoAllocSlot &slot, int dev) {
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_status);
    if (e != cudaSuccess) {
        slot.setup_rc = fail_cuda(e, "cudaGetSymbolAddress(static status)");
        slot.setup_err = t_last_error;
        return;
    }
    e = cudaDeviceGetAttribute(&slot.state.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        slot.setup_rc = fail_cuda(e, "cudaDeviceGetAttribute(SM count)");
        slot.setup_err = t_last_error;
        return;
    }
    slot.state.status = static_cast<unsigned long long *>(ptr);
    slot.state.status_host = nullptr;
    slot.state.ready.store(true, std::memory_order_release);
}

int apply_checked_noalloc_impl(const Call &c, void *stream) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(QKNR_ERR_INVALID_ARG, "device %d out of range", dev);
    NoAllocSlot &slot = g_noalloc[dev];
    std::call_once(slot.once, noalloc_setup, std::ref(slot), dev);
    if (slot.setup_rc) return fail(slot.setup_rc, "%s", slot.setup_err.c_str());

    int rc = validate(c);
    if (rc) return rc;
    if (c.cache_len < 0) return fail(QKNR_ERR_INVALID_ARG, "cache_len %lld < 0", c.cache_len);
    if (c.num_tokens == 0) return QKNR_OK;
    if (c.cache_len == 0) return fail(QKNR_ERR_POSITION_OOB, "cache_len is 0: every position is out of range");
    // A call needs kStatusWords words whatever its problem size, so the fixed
    // array always covers it (static_assert above).
    WorkMap wm;
    rc = plan(slot.state, c, &wm);
    if (rc) return rc;
    std::lock_guard<std::mutex> lock(slot.state.checked_mu);
    unsigned long long host_words[kStatusWords] = {0ull, 0ull};
    return run_checked(slot.state, wm, c, static_cast<cudaStream_t>(stream), host_words);
}

// ---------------------------------------------------------------------------
// Host buffers (qknr_apply_host).
//
// q, k and positions start and end in host memory. When the GPU can address
// that memory (mapped pinned or managed memory), one launch works on it in
// place: the loads and stores cross the host link, both directions at once.
// Otherwise the buffers are staged through the caller's device buffers: the
// tokens are cut into
// chunks; chunk i's heads and positions go host -> device on host_in, the
// kernel runs on the caller's stream once they have landed, and the results
// go device -> host on host_out once the kernel is done. The two copy
// directions and the kernels of neighbouring chunks overlap, so a call takes
// about as long as its slower copy direction plus one chunk.
constexpr int kHostMaxChunks = 8;                    // automatic chunking: at most this many chunks
constexpr long long kHostMinChunkBytes = 4LL << 20;  // ... of at least this many head bytes each way

void host_pipe_release(DeviceState &st) {
    if (st.host_in) cudaStreamDestroy(st.host_in);
    if (st.host_out) cudaStreamDestroy(st.host_out);
    for (cudaEvent_t *ev : {&st.ev_start, &st.ev_in, &st.ev_kernel, &st.ev_out}) {
        if (*ev) cudaEventDestroy(*ev);
        *ev = nullptr;
    }
    st.host_in = st.host_out = nullptr;
    st.host_ready = false;
}

// With st.host_mu held and the device current.
int host_pipe_setup(DeviceState &st) {
    if (st.host_ready) return QKNR_OK;
    cudaError_t e = cudaStreamCreateWithFlags(&st.host_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&st.host_out, cudaStreamNonBlocking);
    for (cudaEvent_t *ev : {&st.ev_start, &st.ev_in, &st.ev_kernel, &st.ev_out})
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        host_pipe_release(st);
        return fail_cuda(e, "host pipeline streams and events");
    }
    st.host_ready = true;
    return QKNR_OK;
}

// Copy the heads of n_tok token rows between two buffers of one layout (n
// heads of head_dim elements, head_stride_b apart; rows stride_b apart).
// Only head bytes move: a row's heads form one span when they are adjacent,
// otherwise each head is copied on its own.
cudaError_t copy_heads(char *dst, const char *src, long long n_tok, long long stride_b, int n,
                       long long head_stride_b, int head_dim, cudaMemcpyKind kind, cudaStream_t s) {
    const size_t head_b = 2 * static_cast<size_t>(head_dim);
    const bool span = n == 1 || head_stride_b == static_cast<long long>(head_b);
    const size_t width = span ? n * head_b : head_b;
    const int pieces = span ? 1 : n;
    for (int h = 0; h < pieces; ++h) {
        const size_t off = static_cast<size_t>(h) * static_cast<size_t>(head_stride_b);
        cudaError_t e;
        if (n_tok == 1 || static_cast<size_t>(stride_b) == width)
            e = cudaMemcpyAsync(dst + off, src + off, static_cast<size_t>(n_tok) * width, kind, s);
        else
            e = cudaMemcpy2DAsync(dst + off, static_cast<size_t>(stride_b), src + off, static_cast<size_t>(stride_b),
                                  width, static_cast<size_t>(n_tok), kind, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// The device address of host memory the GPU can reach directly (mapped
// pinned memory or managed memory), checked at both ends of its extent;
// nullptr for anything else (pageable or device memory, or an extent that
// leaves the allocation).
void *device_view(const void *p, long long extent) {
    cudaPointerAttributes a = {};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // a failed query stays the last error otherwise
        return nullptr;
    }
    if ((a.type != cudaMemoryTypeHost && a.type != cudaMemoryTypeManaged) || !a.devicePointer) return nullptr;
    if (extent > 1) {
        cudaPointerAttributes b = {};
        const char *last = static_cast<const char *>(p) + (extent - 1);
        if (cudaPointerGetAttributes(&b, last) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        if (b.type != a.type || !b.devicePointer ||
            static_cast<const char *>(b.devicePointer) - static_cast<const char *>(a.devicePointer) != extent - 1)
            return nullptr;
    }
    return a.devicePointer;
}

int apply_host_impl(const Call &dc, void *h_q, void *h_k, const void *h_pos, long long chunk_tokens, int flags,
                    void *stream) {
    DeviceState *st = current_state();
    if (!st) return fail(QKNR_ERR_NOT_INITIALIZED, "qknr_init was not called for the current device");
    if (!h_q || !h_k || !h_pos) return fail(QKNR_ERR_INVALID_ARG, "null host pointer");
    if (flags != QKNR_HOST_AUTO && flags != QKNR_HOST_STAGED && flags != QKNR_HOST_DIRECT)
        return fail(QKNR_ERR_INVALID_ARG, "flags %d is not QKNR_HOST_AUTO/STAGED/DIRECT", flags);
    if (chunk_tokens < 0) return fail(QKNR_ERR_INVALID_ARG, "chunk_tokens %lld < 0", chunk_tokens);
    Call hc = dc;  // the host buffers: the same layout
    hc.q = h_q;
    hc.k = h_k;
    hc.positions = h_pos;
    int rc = validate(hc);
    if (rc) return rc;
    const long long T = dc.num_tokens;
    const long long hs_b = dc.head_stride * 2, qs_b = dc.q_stride * 2, ks_b = dc.k_stride * 2;
    const long long pos_b = (dc.dtype & QKNR_POS_I64) ? 8 : 4;
    if (T == 0) return QKNR_OK;

    if (flags != QKNR_HOST_STAGED) {
        // direct: the kernel reads and writes the host buffers over the host link
        void *vq = device_view(h_q, (T - 1) * qs_b + row_bytes(dc.n_qo, hs_b, dc.head_dim));
        void *vk = device_view(h_k, (T - 1) * ks_b + row_bytes(dc.n_kv, hs_b, dc.head_dim));
        void *vp = device_view(h_pos, T * pos_b);
        if (vq && vk && vp) {
            Call c = dc;
            c.q = vq;
            c.k = vk;
            c.positions = vp;
            rc = validate(c);
            if (rc) return rc;
            WorkMap wm;
            rc = plan(*st, c, &wm);
            if (rc) return rc;
            return launch(wm, c, st->status, static_cast<cudaStream_t>(stream));
        }
        if (flags == QKNR_HOST_DIRECT)
            return fail(QKNR_ERR_INVALID_ARG,
                        "QKNR_HOST_DIRECT: h_q, h_k and h_positions must be mapped pinned or managed memory");
    }
    if (!dc.q || !dc.k || !dc.positions)
        return fail(QKNR_ERR_INVALID_ARG,
                    "the host buffers are not all device-mapped (pinned or managed memory), so the staged mode "
                    "runs and needs d_q, d_k and d_positions");
    rc = validate(dc);  // staged: the device staging buffers
    if (rc) return rc;
    long long chunk = chunk_tokens;
    if (chunk == 0) {
        const long long tok_b = 2LL * dc.head_dim * (dc.n_qo + dc.n_kv);
        chunk = std::max((T + kHostMaxChunks - 1) / kHostMaxChunks, (kHostMinChunkBytes + tok_b - 1) / tok_b);
    }
    chunk = std::min(chunk, T);

    std::lock_guard<std::mutex> lock(st->host_mu);
    rc = host_pipe_setup(*st);
    if (rc) return rc;
    cudaStream_t user = static_cast<cudaStream_t>(stream);
    // everything before this call on the caller's stream comes first
    cudaError_t e = cudaEventRecord(st->ev_start, user);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st->host_in, st->ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st->host_out, st->ev_start, 0);
    if (e != cudaSuccess) return fail_cuda(e, "host pipeline start");

    const char *what = nullptr;
    for (long long t0 = 0; t0 < T && !rc && e == cudaSuccess; t0 += chunk) {
        const long long n = std::min(chunk, T - t0);
        char *dq = static_cast<char *>(dc.q) + t0 * qs_b, *dk = static_cast<char *>(dc.k) + t0 * ks_b;
        char *hq = static_cast<char *>(h_q) + t0 * qs_b, *hk = static_cast<char *>(h_k) + t0 * ks_b;
        char *dpos = static_cast<char *>(const_cast<void *>(dc.positions)) + t0 * pos_b;
        const char *hpos = static_cast<const char *>(h_pos) + t0 * pos_b;
        what = "host-to-device copy";
        e = copy_heads(dq, hq, n, qs_b, dc.n_qo, hs_b, dc.head_dim, cudaMemcpyHostToDevice, st->host_in);
        if (e == cudaSuccess)
            e = copy_heads(dk, hk, n, ks_b, dc.n_kv, hs_b, dc.head_dim, cudaMemcpyHostToDevice, st->host_in);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dpos, hpos, static_cast<size_t>(n * pos_b), cudaMemcpyHostToDevice, st->host_in);
        if (e == cudaSuccess) e = cudaEventRecord(st->ev_in, st->host_in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(user, st->ev_in, 0);
        if (e != cudaSuccess) break;
        Call cc = dc;
        cc.q = dq;
        cc.k = dk;
        cc.positions = dpos;
        cc.num_tokens = n;
        WorkMap wm;
        rc = plan(*st, cc, &wm);
        if (rc) break;
        wm.pdl = 0;  // each chunk's kernel waits for its copies, not only for the kernel before it
        rc = launch(wm, cc, st->status, user);
        if (rc) break;
        what = "device-to-host copy";
        e = cudaEventRecord(st->ev_kernel, user);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st->host_out, st->ev_kernel, 0);
        if (e == cudaSuccess)
            e = copy_heads(hq, dq, n, qs_b, dc.n_qo, hs_b, dc.head_dim, cudaMemcpyDeviceToHost, st->host_out);
        if (e == cudaSuccess)
            e = copy_heads(hk, dk, n, ks_b, dc.n_kv, hs_b, dc.head_dim, cudaMemcpyDeviceToHost, st->host_out);
    }
    // the caller's stream continues once the last result is on the host (also
    // after an error, so that nothing later on it overtakes what was enqueued)
    cudaError_t e2 = cudaEventRecord(st->ev_out, st->host_out);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(user, st->ev_out, 0);
    if (rc) return rc;
    if (e != cudaSuccess) return fail_cuda(e, what);
    if (e2 != cudaSuccess) return fail_cuda(e2, "host pipeline end");
    return QKNR_OK;
}

// q and k with their own head strides. With one stride (or one head on a
// side, whose stride does not matter) this is qknr_apply's single launch.
// Otherwise the register kernel runs twice on the stream: over the q heads
// alone, then over the k heads alone, each with its own stride; the per-head
// arithmetic is the same, so are the bits.
int apply_strided_impl(const Call &c, void *stream) {
    DeviceState *st = current_state();
    if (!st) return fail(QKNR_ERR_NOT_INITIALIZED, "qknr_init was not called for the current device");
    if (c.k_head_stride < 0) return fail(QKNR_ERR_INVALID_ARG, "negative stride");
    int rc = validate(c);
    if (rc) return rc;
    if (c.num_tokens == 0) return QKNR_OK;
    Call one = c;
    if (c.n_kv == 1 || c.k_head_stride == c.head_stride) {
        one.k_head_stride = -1;
        return apply_impl(one, stream, false);
    }
    if (c.n_qo == 1) {
        one.head_stride = c.k_head_stride;
        one.k_head_stride = -1;
        return apply_impl(one, stream, false);
    }
    Call sides[2] = {c, c};
    sides[0].n_kv = 0;                          // q heads, head_stride apart
    sides[0].k_head_stride = -1;
    sides[1].n_qo = 0;                          // k heads, k_head_stride apart
    sides[1].head_stride = c.k_head_stride;
    sides[1].k_head_stride = -1;
    const int pdl = tune(QKNR_TUNE_PDL);
    for (const Call &side : sides) {
        WorkMap wm;
        rc = plan_register(*st, side, &wm);
        if (rc) return rc;
        wm.pdl = pdl < 0 ? 1 : pdl;
        rc = launch(wm, side, st->status, static_cast<cudaStream_t>(stream));
        if (rc) return rc;
    }
    return QKNR_OK;
}

Call make_call(void *q, void *k, const void *q_w, const void *k_w, const float *cache, long long cache_len,
               const void *positions, long long num_tokens, int n_qo, int n_kv, int head_dim, int rope_dim,
               int is_neox, long long q_stride, long long k_stride, long long head_stride, float eps,
               int dtype) {
    Call c;
    c.q = q;
    c.k = k;
    c.q_w = q_w;
    c.k_w = k_w;
    c.cache = cache;
    c.cache_len = cache_len;
    c.positions = positions;
    c.num_tokens = num_tokens;
    c.n_qo = n_qo;
    c.n_kv = n_kv;
    c.head_dim = head_dim;
    c.rope_dim = rope_dim;
    c.is_neox = is_neox ? 1 : 0;
    c.q_stride = q_stride;
    c.k_stride = k_stride;
    c.head_stride = head_stride;
    c.eps = eps;
    c.dtype = dtype;
    return c;
}

// ---------------------------------------------------------------------------
// Work-map tuning (qknr_tune).
//
// The fixed rule (4-pass items, L2 prefetch of four items) is the best single
// choice over the measured workloads, but the best passes per item and
// prefetch depth differ by shape by up to a few per cent. qknr_tune times the
// candidates on scratch buffers laid out like the caller's call, never on the
// caller's data (the op works in place), and records the fastest for that
// shape; later calls of the same shape and layout use it.
constexpr long long kTuneMaxScratch = 8LL << 30;   // bytes of q and k replicas at most
constexpr int kTuneMaxReplicas = 16;
constexpr int kTuneRounds = 3;
constexpr float kTuneMargin = 0.01f;   // a candidate must beat the rule by this fraction

struct Scratch {
    std::vector<void *> ptrs;
    ~Scratch() {
        for (void *p : ptrs) cudaFree(p);
    }
    cudaError_t alloc(void **out, size_t bytes) {
        cudaError_t e = cudaMalloc(out, bytes);
        if (e == cudaSuccess) ptrs.push_back(*out);
        return e;
    }
};

int tune_impl(const Call &shape, void *stream, TunedMap *best_out, double *best_ms) {
    DeviceState *st = current_state();
    if (!st) return fail(QKNR_ERR_NOT_INITIALIZED, "qknr_init was not called for the current device");
    if (shape.num_tokens < 1) return fail(QKNR_ERR_INVALID_ARG, "num_tokens must be >= 1 to tune");
    // validate the layout on stand-in pointers first: aligned, and far enough
    // apart (each extent is at most 2^56 bytes) that only a bad layout fails
    Call probe = shape;
    probe.q = reinterpret_cast<void *>(uintptr_t(1) << 40);
    probe.k = reinterpret_cast<void *>(uintptr_t(1) << 58);
    probe.q_w = probe.k_w = probe.positions = reinterpret_cast<const void *>(uintptr_t(256));
    probe.cache = reinterpret_cast<const float *>(uintptr_t(256));
    int rc = validate(probe);
    if (rc) return rc;

    const long long T = shape.num_tokens;
    const long long q_bytes = ((T - 1) * shape.q_stride + static_cast<long long>(shape.n_qo - 1) * shape.head_stride +
                               shape.head_dim) * 2;
    const long long k_bytes = ((T - 1) * shape.k_stride + static_cast<long long>(shape.n_kv - 1) * shape.head_stride +
                               shape.head_dim) * 2;
    const long long rep_bytes = q_bytes + k_bytes;
    if (rep_bytes > kTuneMaxScratch)
        return fail(QKNR_ERR_INVALID_ARG, "qknr_tune: q and k span %lld bytes; at most %lld are tuned on scratch",
                    rep_bytes, kTuneMaxScratch);
    int l2 = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute(L2 size)");
    // replicas rotated between launches so that none finds its inputs in L2
    long long n_rep = rep_bytes >= 4LL * l2 ? 1 : (4LL * l2 + rep_bytes - 1) / rep_bytes;
    n_rep = std::min<long long>(std::min<long long>(n_rep, kTuneMaxReplicas), std::max(1LL, kTuneMaxScratch / rep_bytes));

    const long long cache_len = std::min<long long>(T, 65536);
    const bool pos64 = (shape.dtype & QKNR_POS_I64) != 0;
    Scratch mem;
    std::vector<Call> calls(static_cast<size_t>(n_rep), shape);
    void *w = nullptr, *cache = nullptr, *pos = nullptr;
    e = mem.alloc(&w, 2 * 2 * static_cast<size_t>(shape.head_dim));
    if (e == cudaSuccess) e = mem.alloc(&cache, static_cast<size_t>(cache_len) * shape.rope_dim * sizeof(float));
    if (e == cudaSuccess) e = mem.alloc(&pos, static_cast<size_t>(T) * (pos64 ? 8 : 4));
    for (auto &c : calls) {
        if (e == cudaSuccess) e = mem.alloc(&c.q, static_cast<size_t>(q_bytes));
        if (e == cudaSuccess) e = mem.alloc(&c.k, static_cast<size_t>(k_bytes));
    }
    if (e != cudaSuccess) return fail_cuda(e, "qknr_tune: scratch allocation");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // every byte 0x3f: finite, nonzero values in every buffer (bf16 0.746, fp16
    // 1.81, fp32 0.747), so the candidates move and compute what real data
    // does; positions walk the table
    constexpr int kFill = 0x3f;
    e = cudaMemsetAsync(w, kFill, 2 * 2 * static_cast<size_t>(shape.head_dim), s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(cache, kFill, static_cast<size_t>(cache_len) * shape.rope_dim * sizeof(float), s);
    for (auto &c : calls) {
        if (e == cudaSuccess) e = cudaMemsetAsync(c.q, kFill, static_cast<size_t>(q_bytes), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(c.k, kFill, static_cast<size_t>(k_bytes), s);
    }
    if (e == cudaSuccess) {
        std::vector<long long> p64(pos64 ? static_cast<size_t>(T) : 0);
        std::vector<int> p32(pos64 ? 0 : static_cast<size_t>(T));
        for (long long t = 0; t < T; ++t) {
            if (pos64) p64[static_cast<size_t>(t)] = t % cache_len;
            else p32[static_cast<size_t>(t)] = static_cast<int>(t % cache_len);
        }
        e = cudaMemcpy(pos, pos64 ? static_cast<const void *>(p64.data()) : static_cast<const void *>(p32.data()),
                       static_cast<size_t>(T) * (pos64 ? 8 : 4), cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail_cuda(e, "qknr_tune: scratch set-up");
    for (auto &c : calls) {
        c.q_w = c.k_w = w;
        c.cache = static_cast<const float *>(cache);
        c.positions = pos;
        c.cache_len = 0;
    }

    // candidates: the rule's own launch first, then distinct (kernel, passes per
    // item, prefetch depth) triples
    const int hpw = heads_per_pass(shape.head_dim);
    const int ppt = (shape.n_qo + shape.n_kv + hpw - 1) / hpw;
    std::vector<TunedMap> cands(1);
    std::set<int> seen_chunks;
    for (int passes : {4, 3, 2, 1}) {
        const int chunks = (ppt + passes - 1) / passes;
        if (!seen_chunks.insert(chunks).second) continue;
        if (passes < 4 && cands.size() >= 25) break;
        for (int variant : {0, 1, 2})    // register; ring, next after the wait; ring, two ahead
            for (int pf : {4, 2, 1, -1}) {
                TunedMap m;
                m.kernel = variant == 0 ? QKNR_KERNEL_REGISTER : QKNR_KERNEL_RING;
                m.ring_order = variant;
                m.passes = passes;
                m.prefetch = pf;
                cands.push_back(m);
            }
    }
    std::vector<WorkMap> maps(cands.size());
    for (size_t i = 0; i < cands.size(); ++i) {
        rc = plan_register(*st, calls[0], &maps[i], &cands[i]);
        if (rc) return rc;
        const int pdl = tune(QKNR_TUNE_PDL);
        maps[i].pdl = pdl < 0 ? 1 : pdl;
    }
    cudaEvent_t ev[2] = {nullptr, nullptr};
    e = cudaEventCreate(&ev[0]);
    if (e == cudaSuccess) e = cudaEventCreate(&ev[1]);
    if (e != cudaSuccess) {
        for (cudaEvent_t x : ev)
            if (x) cudaEventDestroy(x);
        return fail_cuda(e, "qknr_tune: events");
    }
    size_t next = 0;
    auto run = [&](const WorkMap &m, int n) -> int {
        for (int i = 0; i < n; ++i) {
            const Call &c = calls[next++ % calls.size()];
            const int r = launch(m, c, st->status, s);
            if (r) return r;
        }
        return QKNR_OK;
    };
    // launches per timing: about 2 ms of work, between 5 and 200 launches
    float ms = 0.f;
    rc = run(maps[0], 3);
    if (!rc) e = cudaEventRecord(ev[0], s);
    if (!rc && e == cudaSuccess) rc = run(maps[0], 5);
    if (!rc && e == cudaSuccess) e = cudaEventRecord(ev[1], s);
    if (!rc && e == cudaSuccess) e = cudaEventSynchronize(ev[1]);
    if (!rc && e == cudaSuccess) e = cudaEventElapsedTime(&ms, ev[0], ev[1]);
    int n_iter = 5;
    if (!rc && e == cudaSuccess) n_iter = static_cast<int>(std::min(200.0, std::max(5.0, 2.0 / std::max(1e-4, ms / 5.0))));
    std::vector<std::vector<float>> times(cands.size());
    for (int round = 0; round < kTuneRounds && !rc && e == cudaSuccess; ++round) {
        for (size_t i = 0; i < cands.size() && !rc && e == cudaSuccess; ++i) {
            rc = run(maps[i], 2);                       // settle into this work map
            if (!rc) e = cudaEventRecord(ev[0], s);
            if (!rc && e == cudaSuccess) rc = run(maps[i], n_iter);
            if (!rc && e == cudaSuccess) e = cudaEventRecord(ev[1], s);
            if (!rc && e == cudaSuccess) e = cudaEventSynchronize(ev[1]);
            if (!rc && e == cudaSuccess) e = cudaEventElapsedTime(&ms, ev[0], ev[1]);
            if (!rc && e == cudaSuccess) times[i].push_back(ms / n_iter);
        }
    }
    cudaEventDestroy(ev[0]);
    cudaEventDestroy(ev[1]);
    if (rc) return rc;
    if (e != cudaSuccess) return fail_cuda(e, "qknr_tune: timing");
    // the candidate with the lowest median time per launch; the rule's launch
    // (candidate 0) stays unless another beats it by more than the timing noise
    size_t best = 0;
    float best_t = 0.f, rule_t = 0.f;
    for (size_t i = 0; i < cands.size(); ++i) {
        std::vector<float> v = times[i];
        std::sort(v.begin(), v.end());
        const float med = v[v.size() / 2];
        if (i == 0) rule_t = med;
        if (i == 0 || med < best_t) {
            best = i;
            best_t = med;
        }
    }
    if (best != 0 && best_t > rule_t * (1.0f - kTuneMargin)) {
        best = 0;
        best_t = rule_t;
    }
    {
        std::lock_guard<std::mutex> lock(st->tuned_mu);
        st->tuned[shape_key(shape)] = cands[best];
        st->has_tuned.store(true, std::memory_order_release);
    }
    *best_out = cands[best];
    *best_ms = best_t;
    return QKNR_OK;
}

}  // namespace

extern "C" {

int qknr_version(void) { return kVersion; }

const char *qknr_last_error(void) { return t_last_error.c_str(); }

int qknr_can_use(int head_dim, int rope_dim, int is_neox, int dtype) {
    if ((dtype & ~(0xff | QKNR_POS_I64 | QKNR_INPUTS_READY)) != 0) return 0;
    if ((dtype & 0xff) != QKNR_BF16 && (dtype & 0xff) != QKNR_FP16) return 0;
    return shape_ok(head_dim, rope_dim, is_neox) ? 1 : 0;
}

int qknr_init(int device) {
    int count = 0;
    cudaError_t e = cudaGetDeviceCount(&count);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDeviceCount");
    if (device < 0 || device >= count || device >= kMaxDevices)
        return fail(QKNR_ERR_INVALID_ARG, "device %d does not exist (%d devices)", device, count);
    std::lock_guard<std::mutex> lock(g_init_mu);
    DeviceState &st = g_dev[device];
    if (st.ready.load()) return QKNR_OK;
    int prev = -1;
    e = cudaGetDevice(&prev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (prev != device && (e = cudaSetDevice(device)) != cudaSuccess) return fail_cuda(e, "cudaSetDevice");
    int rc = QKNR_OK;
    const size_t words = kStatusWords * sizeof(unsigned long long);
    e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) rc = fail_cuda(e, "cudaDeviceGetAttribute(SM count)");
    if (!rc && (e = cudaMalloc(&st.status, words)) != cudaSuccess) rc = fail_cuda(e, "cudaMalloc(status)");
    if (!rc && (e = cudaMallocHost(&st.status_host, words)) != cudaSuccess)
        rc = fail_cuda(e, "cudaMallocHost(status)");
    if (!rc && (e = cudaMemset(st.status, 0, words)) != cudaSuccess) rc = fail_cuda(e, "cudaMemset(status)");
    if (!rc) {
        for (auto &e : st.occupancy)
            for (auto &a : e)
                for (auto &b : a)
                    for (auto &c : b)
                        for (auto &d : c)
                            for (auto &u : d)
                                for (auto &r : u)
                                    for (auto &x : r) x.store(0);
        // the ring kernels' cached occupancy goes with the limit on their
        // dynamic shared memory, which a new context no longer has
        std::atomic<int> *ring = &st.ring_occ[0][0][0][0][0][0][0];
        for (size_t i = 0; i < sizeof(st.ring_occ) / sizeof(st.ring_occ[0][0][0][0][0][0][0]); ++i) ring[i].store(0);
        st.ready.store(true, std::memory_order_release);
    } else {
        if (st.status) cudaFree(st.status);
        if (st.status_host) cudaFreeHost(st.status_host);
        st.status = nullptr;
        st.status_host = nullptr;
    }
    if (prev != device && prev >= 0) cudaSetDevice(prev);
    return rc;
}

int qknr_shutdown(void) {
    std::lock_guard<std::mutex> lock(g_init_mu);
    int prev = -1;
    cudaGetDevice(&prev);
    int rc = QKNR_OK;
    for (int d = 0; d < kMaxDevices; ++d) {
        DeviceState &st = g_dev[d];
        if (!st.ready.load()) continue;
        st.ready.store(false);
        cudaSetDevice(d);
        if (st.status && cudaFree(st.status) != cudaSuccess) rc = fail(QKNR_ERR_CUDA, "cudaFree(status) failed");
        if (st.status_host && cudaFreeHost(st.status_host) != cudaSuccess)
            rc = fail(QKNR_ERR_CUDA, "cudaFreeHost(status) failed");
        st.status = nullptr;
        st.status_host = nullptr;
        {
            std::lock_guard<std::mutex> tuned_lock(st.tuned_mu);
            st.tuned.clear();
            st.has_tuned.store(false);
        }
        std::lock_guard<std::mutex> host_lock(st.host_mu);
        host_pipe_release(st);
    }
    if (prev >= 0) cudaSetDevice(prev);
    return rc;
}

int qknr_apply(void *q, void *k, const void *q_w, const void *k_w, const float *cos_sin_cache,
               const void *positions, int64_t num_tokens, int n_qo, int n_kv, int head_dim, int rope_dim,
               int is_neox, int64_t q_stride, int64_t k_stride, int64_t head_stride, float eps, int dtype,
               void *stream) {
    return apply_impl(make_call(q, k, q_w, k_w, cos_sin_cache, 0, positions, num_tokens, n_qo, n_kv, head_dim,
                                rope_dim, is_neox, q_stride, k_stride, head_stride, eps, dtype),
                      stream, false);
}

int qknr_apply_checked(void *q, void *k, const void *q_w, const void *k_w, const float *cos_sin_cache,
                       int64_t cache_len, const void *positions, int64_t num_tokens, int n_qo, int n_kv,
                       int head_dim, int rope_dim, int is_neox, int64_t q_stride, int64_t k_stride,
                       int64_t head_stride, float eps, int dtype, void *stream) {
    return apply_impl(make_call(q, k, q_w, k_w, cos_sin_cache, cache_len, positions, num_tokens, n_qo, n_kv,
                                head_dim, rope_dim, is_neox, q_stride, k_stride, head_stride, eps, dtype),
                      stream, true);
}

int qknr_apply_checked_noalloc(void *q, void *k, const void *q_w, const void *k_w, const float *cos_sin_cache,
                               int64_t cache_len, const void *positions, int64_t num_tokens, int n_qo,
                               int n_kv, int head_dim, int rope_dim, int is_neox, int64_t q_stride,
                               int64_t k_stride, int64_t head_stride, float eps, int dtype, void *stream) {
    return apply_checked_noalloc_impl(make_call(q, k, q_w, k_w, cos_sin_cache, cache_len, positions, num_tokens,
                                                n_qo, n_kv, head_dim, rope_dim, is_neox, q_stride, k_stride,
                                                head_stride, eps, dtype),
                                      stream);
}

int qknr_apply_unfused(void *q, void *k, const void *q_w, const void *k_w, const float *cos_sin_cache,
                       const void *positions, int64_t num_tokens, int n_qo, int n_kv, int head_dim,
                       int rope_dim, int is_neox, int64_t q_stride, int64_t k_stride, int64_t head_stride,
                       float eps, int dtype, void *stream) {
    DeviceState *st = current_state();
    if (!st) return fail(QKNR_ERR_NOT_INITIALIZED, "qknr_init was not called for the current device");
    const Call c = make_call(q, k, q_w, k_w, cos_sin_cache, 0, positions, num_tokens, n_qo, n_kv, head_dim,
                             rope_dim, is_neox, q_stride, k_stride, head_stride, eps, dtype);
    int rc = validate(c);
    if (rc) return rc;
    if (c.num_tokens == 0) return QKNR_OK;
    WorkMap norm, rope;
    rc = plan_unfused(*st, c, qknr::kOpNorm, &norm);
    if (!rc) rc = plan_unfused(*st, c, qknr::kOpRope, &rope);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = launch(norm, c, st->status, s);
    if (!rc) rc = launch(rope, c, st->status, s);
    return rc;
}

int qknr_apply_host(void *h_q, void *h_k, const void *q_w, const void *k_w, const float *cos_sin_cache,
                    const void *h_positions, void *d_q, void *d_k, void *d_positions, int64_t num_tokens,
                    int n_qo, int n_kv, int head_dim, int rope_dim, int is_neox, int64_t q_stride,
                    int64_t k_stride, int64_t head_stride, float eps, int dtype, int64_t chunk_tokens,
                    int flags, void *stream) {
    return apply_host_impl(make_call(d_q, d_k, q_w, k_w, cos_sin_cache, 0, d_positions, num_tokens, n_qo, n_kv,
                                     head_dim, rope_dim, is_neox, q_stride, k_stride, head_stride, eps, dtype),
                           h_q, h_k, h_positions, chunk_tokens, flags, stream);
}

int qknr_apply_strided(void *q, void *k, const void *q_w, const void *k_w, const float *cos_sin_cache,
                       const void *positions, int64_t num_tokens, int n_qo, int n_kv, int head_dim, int rope_dim,
                       int is_neox, int64_t q_stride, int64_t k_stride, int64_t q_head_stride,
                       int64_t k_head_stride, float eps, int dtype, void *stream) {
    Call c = make_call(q, k, q_w, k_w, cos_sin_cache, 0, positions, num_tokens, n_qo, n_kv, head_dim, rope_dim,
                       is_neox, q_stride, k_stride, q_head_stride, eps, dtype);
    c.k_head_stride = k_head_stride;
    return apply_strided_impl(c, stream);
}

int qknr_tune(int64_t num_tokens, int n_qo, int n_kv, int head_dim, int rope_dim, int is_neox, int64_t q_stride,
              int64_t k_stride, int64_t head_stride, int dtype, void *stream, int64_t *out) {
    const Call c = make_call(nullptr, nullptr, nullptr, nullptr, nullptr, 0, nullptr, num_tokens, n_qo, n_kv, head_dim,
                             rope_dim, is_neox, q_stride, k_stride, head_stride, 1e-6f, dtype);
    TunedMap best;
    double ms = 0.0;
    int rc = tune_impl(c, stream, &best, &ms);
    if (rc || !out) return rc;
    DeviceState *st = current_state();
    WorkMap wm;
    Call aligned = c;
    aligned.cache = reinterpret_cast<const float *>(uintptr_t(256));
    rc = plan(*st, aligned, &wm);
    if (rc) return rc;
    out[0] = wm.kind;
    out[1] = wm.grid;
    out[2] = wm.threads;
    out[3] = wm.items;
    out[4] = wm.chunks_per_token;
    out[5] = wm.ctas_per_sm;
    out[6] = wm.pdl;
    out[7] = wm.passes_per_token;
    out[8] = wm.kind == QKNR_KERNEL_RING ? qknr::kRingMaxPasses : qknr::kUnrollClass[wm.u_idx];
    out[9] = wm.interleave ? 2 : 1;
    out[10] = wm.prefetch_items;
    out[11] = wm.r_idx == qknr::kRopeFull ? c.head_dim : (wm.r_idx == qknr::kRopeHalf ? c.head_dim / 2 : 0);
    out[12] = wm.kind == QKNR_KERNEL_RING ? wm.ring_ahead + 1 : 0;
    out[13] = static_cast<int64_t>(ms * 1e6);   // measured nanoseconds per launch
    return QKNR_OK;
}

int qknr_set_tuning(int key, int value) {
    std::call_once(g_env_once, read_env_tuning);
    if (key == QKNR_TUNE_RESET) {
        for (int i = 0; i < kNumTuneKeys; ++i) g_tune[i] = kTuneAuto[i];
        return QKNR_OK;
    }
    int rc = tune_check(key, value);
    if (rc) return rc;
    g_tune[key] = value;
    return QKNR_OK;
}

int qknr_get_tuning(int key, int *value) {
    if (!value) return fail(QKNR_ERR_INVALID_ARG, "value is null");
    if (key != QKNR_TUNE_KERNEL && key != QKNR_TUNE_RING_ORDER && key != QKNR_TUNE_PASSES &&
        key != QKNR_TUNE_THREADS && key != QKNR_TUNE_CTAS_PER_SM &&
        key != QKNR_TUNE_PDL && key != QKNR_TUNE_ORDER && key != QKNR_TUNE_PREFETCH)
        return fail(QKNR_ERR_INVALID_ARG, "unknown tuning key %d", key);
    *value = tune(key);
    return QKNR_OK;
}

int qknr_query_work_map(int64_t num_tokens, int n_qo, int n_kv, int head_dim, int rope_dim, int is_neox,
                        int dtype, int64_t *out) {
    if (!out) return fail(QKNR_ERR_INVALID_ARG, "out is null");
    DeviceState *st = current_state();
    if (!st) return fail(QKNR_ERR_NOT_INITIALIZED, "qknr_init was not called for the current device");
    if (num_tokens < 0 || n_qo < 1 || n_kv < 1 || num_tokens > kMaxExtentBytes ||
        static_cast<long long>(n_qo) + n_kv > kMaxHeads)
        return fail(QKNR_ERR_INVALID_ARG, "bad sizes");
    if (!qknr_can_use(head_dim, rope_dim, is_neox, dtype))
        return fail(QKNR_ERR_UNSUPPORTED, "shape outside the accepted set");
    // the plan depends on the table only through its alignment: use an aligned
    // stand-in; q and k contiguous (the layout a tuned shape is looked up by)
    Call c = make_call(nullptr, nullptr, nullptr, nullptr, reinterpret_cast<const float *>(uintptr_t(256)), 0,
                       nullptr, num_tokens, n_qo, n_kv, head_dim, rope_dim, is_neox,
                       static_cast<long long>(n_qo) * head_dim, static_cast<long long>(n_kv) * head_dim, head_dim,
                       1e-6f, dtype);
    WorkMap wm;
    int rc = plan(*st, c, &wm);
    if (rc) return rc;
    out[0] = wm.kind;
    out[1] = wm.grid;
    out[2] = wm.threads;
    out[3] = wm.items;
    out[4] = wm.chunks_per_token;
    out[5] = wm.ctas_per_sm;
    out[6] = wm.pdl;
    out[7] = wm.passes_per_token;
    out[8] = wm.kind == QKNR_KERNEL_RING ? qknr::kRingMaxPasses : qknr::kUnrollClass[wm.u_idx];
    out[9] = wm.interleave ? 2 : 1;
    out[10] = wm.prefetch_items;
    out[11] = wm.r_idx == qknr::kRopeFull ? head_dim : (wm.r_idx == qknr::kRopeHalf ? head_dim / 2 : 0);
    out[12] = wm.kind == QKNR_KERNEL_RING ? wm.ring_ahead + 1 : 0;
    return QKNR_OK;
}

}  // extern "C"
