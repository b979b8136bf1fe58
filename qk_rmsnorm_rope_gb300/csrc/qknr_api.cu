// qknr_api.cu -- the C ABI (include/qknr.h): validation, work map, launch.
//
// Argument rules follow the tensor contract of the fused_inplace_qknorm_rope
// deep-dive §3 and the host checks of §4.7 (shape/stride/dtype checks before
// launch, int32 or int64 positions, grid sized from occupancy x SM count, the
// CUDA launch error checked), restated for this library's kernels.
#include "../../include/qknr.h"
#include "qknr_dispatch.h"
#include "qknr_kernel.cuh"

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

namespace {

using qknr::Params;

constexpr int kMaxDevices = 64;
constexpr int kVersion = 10000;  // 1.0.0

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

struct DeviceState {
    std::atomic<bool> ready{false};
    int sm_count = 0;
    unsigned long long *status = nullptr;       // device: {bad-token count, first bad token}
    unsigned long long *status_host = nullptr;  // pinned host copy
    std::mutex checked_mu;                      // serialises qknr_apply_checked on this device
    // resident CTAs per SM, by (dtype, pos64, d_idx, mode, u_idx, threads class); 0 = unknown
    std::atomic<int> occupancy[2][2][qknr::kNumHeadDim][2][qknr::kNumUnroll][4];
};

DeviceState g_dev[kMaxDevices];
std::mutex g_init_mu;

// process-wide work-map overrides (0 / -1 = automatic)
std::atomic<int> g_force_ppi{0}, g_force_threads{0}, g_force_ctas_per_sm{0}, g_force_pdl{-1};
std::once_flag g_env_once;

void read_env_overrides() {
    // QKNR_WORK_MAP="passes_per_item,threads_per_cta,ctas_per_sm"
    if (const char *s = std::getenv("QKNR_WORK_MAP")) {
        int a = 0, b = 0, c = 0;
        if (std::sscanf(s, "%d,%d,%d", &a, &b, &c) >= 1) {
            g_force_ppi = std::max(a, 0);
            g_force_threads = std::max(b, 0);
            g_force_ctas_per_sm = std::max(c, 0);
        }
    }
    if (const char *s = std::getenv("QKNR_PDL")) g_force_pdl = std::atoi(s) ? 1 : 0;
}

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

struct WorkMap {
    int grid = 0, threads = 0, chunks_per_token = 0, passes_per_token = 0, max_passes = 0;
    int u_idx = 0, ctas_per_sm = 0, pdl = 1;
    long long items = 0;
    const void *kernel = nullptr;
};

int resident_ctas(DeviceState &st, int dt, int pos64, int d_idx, int mode, int u_idx, int threads,
                  const void *kernel, int *out) {
    std::atomic<int> &slot = st.occupancy[dt][pos64][d_idx][mode][u_idx][threads_index(threads)];
    int v = slot.load(std::memory_order_relaxed);
    if (v == 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kernel, threads, 0);
        if (e != cudaSuccess) return fail_cuda(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        if (v <= 0) return fail(QKNR_ERR_CUDA, "kernel cannot be resident with %d threads", threads);
        slot.store(v, std::memory_order_relaxed);
    }
    *out = v;
    return QKNR_OK;
}

// Choose the launch for one call. Items are (token, chunk of warp passes);
// the default aims at 4 passes per item (8 x 16-byte loads in flight per lane).
int plan(DeviceState &st, long long num_tokens, int n_qo, int n_kv, int head_dim, int is_neox,
         int dtype, WorkMap *wm) {
    std::call_once(g_env_once, read_env_overrides);
    const int d_idx = head_dim_index(head_dim);
    const int lph = head_dim / 16;
    const int hpw = qknr::kWarp / lph;
    const int heads = n_qo + n_kv;
    wm->passes_per_token = (heads + hpw - 1) / hpw;

    int ppi = g_force_ppi.load();
    if (ppi <= 0) ppi = 4;
    ppi = std::min(ppi, qknr::kUnrollClass[qknr::kNumUnroll - 1]);
    wm->chunks_per_token = (wm->passes_per_token + ppi - 1) / ppi;
    wm->max_passes = (wm->passes_per_token + wm->chunks_per_token - 1) / wm->chunks_per_token;
    wm->u_idx = wm->max_passes <= 2 ? 0 : 1;
    wm->items = num_tokens * wm->chunks_per_token;

    int threads = g_force_threads.load();
    if (threads_index(threads) < 0) threads = 256;
    wm->threads = threads;

    const int dt = (dtype & 0xff) == QKNR_FP16 ? 1 : 0;
    const int pos64 = (dtype & QKNR_POS_I64) ? 1 : 0;
    const int mode = is_neox ? qknr::kNeox : qknr::kInterleaved;
    wm->kernel = dt ? qknr::kernel_fp16(pos64, d_idx, mode, wm->u_idx)
                    : qknr::kernel_bf16(pos64, d_idx, mode, wm->u_idx);
    if (!wm->kernel) return fail(QKNR_ERR_UNSUPPORTED, "no kernel for this shape");

    int occ = 0;
    int rc = resident_ctas(st, dt, pos64, d_idx, mode, wm->u_idx, threads, wm->kernel, &occ);
    if (rc) return rc;
    const int force_cps = g_force_ctas_per_sm.load();
    if (force_cps > 0) occ = std::min(occ, force_cps);
    wm->ctas_per_sm = occ;
    const long long warps_per_cta = threads / qknr::kWarp;
    const long long needed = (wm->items + warps_per_cta - 1) / warps_per_cta;
    const long long cap = static_cast<long long>(occ) * st.sm_count;
    wm->grid = static_cast<int>(std::max(1LL, std::min(needed, cap)));
    const int pdl = g_force_pdl.load();
    wm->pdl = pdl < 0 ? 1 : pdl;
    return QKNR_OK;
}

DeviceState *current_state(int *dev_out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (!g_dev[dev].ready.load(std::memory_order_acquire)) return nullptr;
    if (dev_out) *dev_out = dev;
    return &g_dev[dev];
}

// Byte extent of one token row: heads [0, n) with the shared head stride.
long long row_bytes(int n, long long head_stride_b, int head_dim) {
    return static_cast<long long>(n - 1) * head_stride_b + 2LL * head_dim;
}

int validate(void *q, void *k, const void *q_w, const void *k_w, const float *cache,
             const void *positions, long long num_tokens, int n_qo, int n_kv, int head_dim,
             int rope_dim, int is_neox, long long q_stride, long long k_stride,
             long long head_stride, float eps, int dtype) {
    if ((dtype & ~(0xff | QKNR_POS_I64)) != 0 || ((dtype & 0xff) != QKNR_BF16 && (dtype & 0xff) != QKNR_FP16))
        return fail(QKNR_ERR_INVALID_ARG, "dtype 0x%x is not QKNR_BF16/QKNR_FP16 [| QKNR_POS_I64]", dtype);
    if (num_tokens < 0) return fail(QKNR_ERR_INVALID_ARG, "num_tokens %lld < 0", num_tokens);
    if (n_qo < 1 || n_kv < 1) return fail(QKNR_ERR_INVALID_ARG, "head counts n_qo=%d n_kv=%d must be >= 1", n_qo, n_kv);
    if (!shape_ok(head_dim, rope_dim, is_neox))
        return fail(QKNR_ERR_UNSUPPORTED,
                    "unsupported head_dim=%d rope_dim=%d is_neox=%d (head_dim in {64,128,256}; rope_dim even, "
                    "0 < rope_dim <= head_dim; NeoX needs rope_dim %% 16 == 0 or rope_dim <= 8)",
                    head_dim, rope_dim, is_neox);
    if (!std::isfinite(eps) || eps < 0.f) return fail(QKNR_ERR_INVALID_ARG, "eps must be a finite value >= 0");
    if (!q || !k || !q_w || !k_w || !cache || !positions)
        return fail(QKNR_ERR_INVALID_ARG, "null pointer argument");
    if (q_stride < 0 || k_stride < 0 || head_stride < 0)
        return fail(QKNR_ERR_INVALID_ARG, "negative stride");
    if ((n_qo > 1 || n_kv > 1) && head_stride < head_dim)
        return fail(QKNR_ERR_INVALID_ARG, "head_stride %lld < head_dim %d: heads overlap", head_stride, head_dim);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(q_w, 16) || !aligned(k_w, 16))
        return fail(QKNR_ERR_MISALIGNED, "q, k, q_w and k_w must be 16-byte aligned");
    if ((q_stride % 8) || (k_stride % 8) || (head_stride % 8))
        return fail(QKNR_ERR_MISALIGNED, "q_stride, k_stride and head_stride must be multiples of 8 elements");
    if (!aligned(cache, 4)) return fail(QKNR_ERR_MISALIGNED, "cos_sin_cache must be 4-byte aligned");
    if (!aligned(positions, (dtype & QKNR_POS_I64) ? 8 : 4))
        return fail(QKNR_ERR_MISALIGNED, "positions must be aligned to their element size");

    const long long hs_b = head_stride * 2, qs_b = q_stride * 2, ks_b = k_stride * 2;
    const long long q_row = row_bytes(n_qo, hs_b, head_dim), k_row = row_bytes(n_kv, hs_b, head_dim);
    if (num_tokens > 1 && (qs_b < q_row || ks_b < k_row))
        return fail(QKNR_ERR_INVALID_ARG, "token stride smaller than one token's heads: rows overlap");
    if (num_tokens > 0) {
        // q and k must be disjoint. Either their address ranges do not meet, or
        // they interleave inside rows of one common token stride.
        const uintptr_t qa = reinterpret_cast<uintptr_t>(q), ka = reinterpret_cast<uintptr_t>(k);
        const uintptr_t q_end = qa + static_cast<uintptr_t>((num_tokens - 1) * qs_b + q_row);
        const uintptr_t k_end = ka + static_cast<uintptr_t>((num_tokens - 1) * ks_b + k_row);
        const bool apart = q_end <= ka || k_end <= qa;
        if (!apart) {
            bool ok = false;
            if (qs_b == ks_b && qs_b > 0) {
                const long long S = qs_b;
                const long long diff = static_cast<long long>(ka) - static_cast<long long>(qa);
                const long long off = ((diff % S) + S) % S;   // k row start inside a q row period
                ok = off >= q_row && off + k_row <= S;
            }
            if (!ok) return fail(QKNR_ERR_INVALID_ARG, "q and k overlap in memory");
        }
    }
    return QKNR_OK;
}

int launch(DeviceState &st, const WorkMap &wm, const Params &prm, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(wm.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(wm.threads));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = wm.pdl ? 1 : 0;
    void *args[] = {const_cast<Params *>(&prm)};
    cudaError_t e = cudaLaunchKernelExC(&cfg, wm.kernel, args);
    if (e != cudaSuccess) return fail_cuda(e, "kernel launch");
    (void)st;
    return QKNR_OK;
}

int apply_impl(void *q, void *k, const void *q_w, const void *k_w, const float *cache,
               long long cache_len, const void *positions, long long num_tokens, int n_qo,
               int n_kv, int head_dim, int rope_dim, int is_neox, long long q_stride,
               long long k_stride, long long head_stride, float eps, int dtype, void *stream,
               bool checked) {
    int dev = -1;
    DeviceState *st = current_state(&dev);
    if (!st) return fail(QKNR_ERR_NOT_INITIALIZED, "qknr_init was not called for the current device");
    int rc = validate(q, k, q_w, k_w, cache, positions, num_tokens, n_qo, n_kv, head_dim, rope_dim,
                      is_neox, q_stride, k_stride, head_stride, eps, dtype);
    if (rc) return rc;
    if (checked && cache_len < 0) return fail(QKNR_ERR_INVALID_ARG, "cache_len %lld < 0", cache_len);
    if (num_tokens == 0) return QKNR_OK;

    WorkMap wm;
    rc = plan(*st, num_tokens, n_qo, n_kv, head_dim, is_neox, dtype, &wm);
    if (rc) return rc;

    Params prm = {};
    prm.q = static_cast<char *>(q);
    prm.k = static_cast<char *>(k);
    prm.q_w = static_cast<const uint4 *>(q_w);
    prm.k_w = static_cast<const uint4 *>(k_w);
    prm.cache = cache;
    prm.positions = positions;
    prm.status = st->status;
    prm.q_stride_b = q_stride * 2;
    prm.k_stride_b = k_stride * 2;
    prm.head_stride_b = head_stride * 2;
    prm.num_items = wm.items;
    prm.cache_len = 0;
    prm.n_qo = n_qo;
    prm.n_kv = n_kv;
    prm.rope_dim = rope_dim;
    prm.chunks_per_token = wm.chunks_per_token;
    prm.passes_per_token = wm.passes_per_token;
    prm.cache_vec = (rope_dim % 8 == 0) && aligned(cache, 16);
    prm.eps = eps;
    prm.inv_d = 1.0f / static_cast<float>(head_dim);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (!checked) return launch(*st, wm, prm, s);

    if (cache_len == 0) return fail(QKNR_ERR_POSITION_OOB, "cache_len is 0: every position is out of range");
    prm.cache_len = cache_len;
    std::lock_guard<std::mutex> lock(st->checked_mu);
    cudaError_t e = cudaMemsetAsync(st->status, 0, sizeof(unsigned long long), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(st->status + 1, 0xff, sizeof(unsigned long long), s);
    if (e != cudaSuccess) return fail_cuda(e, "status reset");
    rc = launch(*st, wm, prm, s);
    if (rc) return rc;
    e = cudaMemcpyAsync(st->status_host, st->status, 2 * sizeof(unsigned long long),
                        cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail_cuda(e, "status read-back");
    const unsigned long long bad = st->status_host[0], first = st->status_host[1];
    if (bad) {
        return fail(QKNR_ERR_POSITION_OOB,
                    "%llu token(s) have positions outside [0, %lld); first bad token index %llu (left untouched)",
                    bad, cache_len, first);
    }
    return QKNR_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free checked variant.
//
// Some callers cannot call cudaMalloc at all: code that runs where allocation
// is forbidden or already accounted for (a pre-sized memory pool, an embedded
// runtime that owns every device allocation, a plug-in loaded into a host
// that reserves the allocator for itself). qknr_apply_checked needs a 16-byte
// status word, which qknr_init allocates. This variant keeps that word in
// the file-scope array below instead, so it needs neither qknr_init nor any
// allocation. The array is part of the library image: every GPU that loads
// the library holds its 256 bytes until the process exits.
constexpr int kNoAllocStatusWords = 32;  // 256 bytes; one call uses the first 2 words
static __device__ __align__(256) unsigned long long g_noalloc_status[kNoAllocStatusWords];

struct NoAllocSlot {
    std::once_flag once;
    int setup_rc = QKNR_OK;
    std::string setup_err;
    DeviceState state;   // status = device address of g_noalloc_status; no host buffer
    std::mutex call_mu;  // one call at a time per device (the array is shared)
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

int apply_checked_noalloc_impl(void *q, void *k, const void *q_w, const void *k_w,
                               const float *cache, long long cache_len, const void *positions,
                               long long num_tokens, int n_qo, int n_kv, int head_dim,
                               int rope_dim, int is_neox, long long q_stride, long long k_stride,
                               long long head_stride, float eps, int dtype, void *stream) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(QKNR_ERR_INVALID_ARG, "device %d out of range", dev);
    NoAllocSlot &slot = g_noalloc[dev];
    std::call_once(slot.once, noalloc_setup, std::ref(slot), dev);
    if (slot.setup_rc) return fail(slot.setup_rc, "%s", slot.setup_err.c_str());

    int rc = validate(q, k, q_w, k_w, cache, positions, num_tokens, n_qo, n_kv, head_dim, rope_dim,
                      is_neox, q_stride, k_stride, head_stride, eps, dtype);
    if (rc) return rc;
    if (cache_len < 0) return fail(QKNR_ERR_INVALID_ARG, "cache_len %lld < 0", cache_len);
    if (num_tokens == 0) return QKNR_OK;
    if (cache_len == 0) return fail(QKNR_ERR_POSITION_OOB, "cache_len is 0: every position is out of range");
    // The status this call needs is 2 words whatever the problem size, so the
    // fixed array always covers it; guard the invariant all the same.
    static_assert(kNoAllocStatusWords >= 2, "static status array too small");

    WorkMap wm;
    rc = plan(slot.state, num_tokens, n_qo, n_kv, head_dim, is_neox, dtype, &wm);
    if (rc) return rc;

    Params prm = {};
    prm.q = static_cast<char *>(q);
    prm.k = static_cast<char *>(k);
    prm.q_w = static_cast<const uint4 *>(q_w);
    prm.k_w = static_cast<const uint4 *>(k_w);
    prm.cache = cache;
    prm.positions = positions;
    prm.status = slot.state.status;
    prm.q_stride_b = q_stride * 2;
    prm.k_stride_b = k_stride * 2;
    prm.head_stride_b = head_stride * 2;
    prm.num_items = wm.items;
    prm.cache_len = cache_len;
    prm.n_qo = n_qo;
    prm.n_kv = n_kv;
    prm.rope_dim = rope_dim;
    prm.chunks_per_token = wm.chunks_per_token;
    prm.passes_per_token = wm.passes_per_token;
    prm.cache_vec = (rope_dim % 8 == 0) && aligned(cache, 16);
    prm.eps = eps;
    prm.inv_d = 1.0f / static_cast<float>(head_dim);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lock(slot.call_mu);
    // The array keeps the previous call's contents: reset count and first-bad index.
    e = cudaMemsetAsync(slot.state.status, 0, sizeof(unsigned long long), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(slot.state.status + 1, 0xff, sizeof(unsigned long long), s);
    if (e != cudaSuccess) return fail_cuda(e, "static status reset");
    rc = launch(slot.state, wm, prm, s);
    if (rc) return rc;
    unsigned long long host_status[2] = {0ull, 0ull};
    e = cudaMemcpyAsync(host_status, slot.state.status, sizeof host_status, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail_cuda(e, "static status read-back");
    if (host_status[0]) {
        return fail(QKNR_ERR_POSITION_OOB,
                    "%llu token(s) have positions outside [0, %lld); first bad token index %llu (left untouched)",
                    host_status[0], cache_len, host_status[1]);
    }
    return QKNR_OK;
}

}  // namespace

extern "C" {

int qknr_version(void) { return kVersion; }

const char *qknr_last_error(void) { return t_last_error.c_str(); }

int qknr_can_use(int head_dim, int rope_dim, int is_neox, int dtype) {
    if ((dtype & ~(0xff | QKNR_POS_I64)) != 0) return 0;
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
    e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) rc = fail_cuda(e, "cudaDeviceGetAttribute(SM count)");
    if (!rc && (e = cudaMalloc(&st.status, 2 * sizeof(unsigned long long))) != cudaSuccess)
        rc = fail_cuda(e, "cudaMalloc(status)");
    if (!rc && (e = cudaMallocHost(&st.status_host, 2 * sizeof(unsigned long long))) != cudaSuccess)
        rc = fail_cuda(e, "cudaMallocHost(status)");
    if (!rc && (e = cudaMemset(st.status, 0, 2 * sizeof(unsigned long long))) != cudaSuccess)
        rc = fail_cuda(e, "cudaMemset(status)");
    if (!rc) {
        for (auto &a : st.occupancy)
            for (auto &b : a)
                for (auto &c : b)
                    for (auto &d : c)
                        for (auto &u : d)
                            for (auto &x : u) x.store(0);
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
    }
    if (prev >= 0) cudaSetDevice(prev);
    return rc;
}

int qknr_apply(void *q, void *k, const void *q_w, const void *k_w, const float *cos_sin_cache,
               const void *positions, int64_t num_tokens, int n_qo, int n_kv, int head_dim,
               int rope_dim, int is_neox, int64_t q_stride, int64_t k_stride, int64_t head_stride,
               float eps, int dtype, void *stream) {
    return apply_impl(q, k, q_w, k_w, cos_sin_cache, 0, positions, num_tokens, n_qo, n_kv, head_dim,
                      rope_dim, is_neox ? 1 : 0, q_stride, k_stride, head_stride, eps, dtype, stream,
                      false);
}

int qknr_apply_checked(void *q, void *k, const void *q_w, const void *k_w,
                       const float *cos_sin_cache, int64_t cache_len, const void *positions,
                       int64_t num_tokens, int n_qo, int n_kv, int head_dim, int rope_dim,
                       int is_neox, int64_t q_stride, int64_t k_stride, int64_t head_stride,
                       float eps, int dtype, void *stream) {
    return apply_impl(q, k, q_w, k_w, cos_sin_cache, cache_len, positions, num_tokens, n_qo, n_kv,
                      head_dim, rope_dim, is_neox ? 1 : 0, q_stride, k_stride, head_stride, eps,
                      dtype, stream, true);
}

int qknr_set_work_map(int passes_per_item, int threads_per_cta, int ctas_per_sm, int use_pdl) {
    std::call_once(g_env_once, read_env_overrides);
    if (passes_per_item < 0 || passes_per_item > qknr::kUnrollClass[qknr::kNumUnroll - 1])
        return fail(QKNR_ERR_INVALID_ARG, "passes_per_item must be in [0, %d]",
                    qknr::kUnrollClass[qknr::kNumUnroll - 1]);
    if (threads_per_cta != 0 && threads_index(threads_per_cta) < 0)
        return fail(QKNR_ERR_INVALID_ARG, "threads_per_cta must be 0 or one of 64/128/256/512");
    if (ctas_per_sm < 0) return fail(QKNR_ERR_INVALID_ARG, "ctas_per_sm must be >= 0");
    if (use_pdl < -1 || use_pdl > 1) return fail(QKNR_ERR_INVALID_ARG, "use_pdl must be -1, 0 or 1");
    g_force_ppi = passes_per_item;
    g_force_threads = threads_per_cta;
    g_force_ctas_per_sm = ctas_per_sm;
    g_force_pdl = use_pdl;
    return QKNR_OK;
}

int qknr_query_work_map(int64_t num_tokens, int n_qo, int n_kv, int head_dim, int rope_dim,
                        int is_neox, int dtype, int64_t out[8]) {
    if (!out) return fail(QKNR_ERR_INVALID_ARG, "out is null");
    DeviceState *st = current_state(nullptr);
    if (!st) return fail(QKNR_ERR_NOT_INITIALIZED, "qknr_init was not called for the current device");
    if (num_tokens < 0 || n_qo < 1 || n_kv < 1) return fail(QKNR_ERR_INVALID_ARG, "bad sizes");
    if (!qknr_can_use(head_dim, rope_dim, is_neox, dtype))
        return fail(QKNR_ERR_UNSUPPORTED, "shape outside the accepted set");
    WorkMap wm;
    int rc = plan(*st, num_tokens, n_qo, n_kv, head_dim, is_neox, dtype, &wm);
    if (rc) return rc;
    out[0] = wm.grid;
    out[1] = wm.threads;
    out[2] = wm.items;
    out[3] = wm.chunks_per_token;
    out[4] = wm.passes_per_token;
    out[5] = qknr::kUnrollClass[wm.u_idx];
    out[6] = wm.ctas_per_sm;
    out[7] = wm.pdl;
    return QKNR_OK;
}

int qknr_apply_checked_noalloc(void *q, void *k, const void *q_w, const void *k_w,
                               const float *cos_sin_cache, int64_t cache_len, const void *positions,
                               int64_t num_tokens, int n_qo, int n_kv, int head_dim, int rope_dim,
                               int is_neox, int64_t q_stride, int64_t k_stride, int64_t head_stride,
                               float eps, int dtype, void *stream) {
    return apply_checked_noalloc_impl(q, k, q_w, k_w, cos_sin_cache, cache_len, positions, num_tokens,
                                      n_qo, n_kv, head_dim, rope_dim, is_neox ? 1 : 0, q_stride,
                                      k_stride, head_stride, eps, dtype, stream);
}

}  // extern "C"
