// qknr_kernel.cuh -- fused in-place per-head QK RMSNorm + RoPE for sm_103a.
//
// The op (fused_inplace_qknorm_rope deep-dive §2.1-§2.3): per head, sum of
// squares over head_dim in fp32, r = rsqrt(sum/D + eps), n = x*r*w, rotate the
// first rope_dim dims with the token's cos|sin row (interleaved or NeoX
// pairing), round once to the storage dtype and store over the input.
//
// Work map (this library's own design for GB300, not the page's warp-per-head):
//  * A lane owns two 16-byte vectors (8 elements each) of one head, so a head
//    takes D/16 lanes and a warp pass covers 32/(D/16) heads. Loads and stores
//    are 128-bit, streaming (evict-first), and every warp instruction touches
//    whole 32-byte sectors.
//  * The two vectors are chosen so that no pairing needs a lane exchange:
//    interleaved pairs (2j, 2j+1) sit inside one vector; for NeoX with
//    rope_dim % 16 == 0 a lane owns dims [8a, 8a+8) and [8a+R/2, 8a+R/2+8),
//    i.e. both halves of eight rotation pairs; lanes past the rotated span own
//    two tail vectors from the two halves of the tail. The only shuffles are
//    the log2(D/16)-step segmented sum of squares.
//  * A warp item is (token, chunk of up to UMAX passes). By default warp w of
//    W takes items w, w + W, w + 2W, ...: all warps sweep the tensors together,
//    a compact window of memory at any moment. A contiguous range of items per
//    warp is the other order. A warp keeps the current token's cos/sin values
//    in registers and reloads them only when its token changes; positions are
//    read 32 items ahead, so the cos/sin loads never wait for one.
//  * Each item issues all its loads (up to UMAX passes x 2 vectors per lane)
//    before any arithmetic, to keep many bytes in flight per SM.
//  * Grid: persistent, at most one wave of resident CTAs; programmatic
//    dependent launch lets the next kernel in the stream get resident early.
//  * While it waits for the previous grid, each warp prefetches its first
//    items' q/k rows and its first positions into L2 (see the kernel body).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qknr_math.cuh"

namespace qknr {

constexpr int kWarp = 32;
constexpr int kBoundTable = 32;       // items per token up to which pass bounds come from a table

// Kernel parameters, passed by value as a __grid_constant__.
struct Params {
    char *q;                      // head (0,0) of q
    char *k;                      // head (0,0) of k
    const uint4 *q_w;             // [D] weights as 16-byte vectors
    const uint4 *k_w;
    const float *cache;           // [cache_len, R] fp32
    const void *positions;        // [T] int32 / int64
    unsigned long long *status;   // checked variant: {bad-token count, first bad token}
    long long q_stride_b;         // bytes between tokens of q
    long long k_stride_b;
    long long head_stride_b;      // bytes between heads (q and k)
    long long num_items;          // num_tokens * chunks_per_token
    long long cache_len;          // > 0: check positions against it
    int n_qo, n_kv;
    int rope_dim;
    int chunks_per_token;         // items per token
    int passes_per_token;         // ceil((n_qo + n_kv) / heads_per_pass)
    int cache_vec;                // 1: cos/sin rows may be read as float4
    int interleave;               // 1: warp w takes items w, w + W, ... (W warps); 0: a contiguous range
    int prefetch_items;           // items per warp whose q/k rows are prefetched into L2 before the wait
    float eps;
    float inv_d;                  // 1 / head_dim in fp32 (exact for 64, 128 and 256; for 80, 96 and 192
                                  // the rounded reciprocal moves the mean by at most about one ulp)
    short pass_bound[kBoundTable + 1];  // first pass of chunk c, c <= chunks_per_token <= kBoundTable
    int ring_ahead;               // ring kernel's issue order: 0 next item after the wait, 1 two ahead
};

template <class P>
__device__ __forceinline__ long long load_position(const void *positions, long long t) {
    return static_cast<long long>(__ldg(reinterpret_cast<const P *>(positions) + t));
}

// Pull the line holding ptr into L2 (no data comes back to the SM).
__device__ __forceinline__ void prefetch_l2(const void *ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// Before a launch waits for the previous grid in its stream, each warp pulls
// its first p.prefetch_items items' q/k rows and the positions of its first
// 32 items into L2. A prefetch brings nothing back to the SM, and L2 is where
// every store of the previous grid lands, so a line it brings in cannot go
// stale. It uses DRAM time that the previous grid's last warps leave idle, and
// the first loads after the wait hit L2. Not inlined, so that its address
// arithmetic does not take registers from the item loop.
template <class P, int HPW, int UMAX, int OP>
__device__ __noinline__ void prefetch_first_items(const Params &p, long long it_begin, long long it_end,
                                                  long long it_step, int g, int va, int vb, bool active,
                                                  int lane) {
    const int chunks = p.chunks_per_token;
    const int H = p.n_qo + p.n_kv;
    for (int j = 0; j < p.prefetch_items; ++j) {
        const long long itp = it_begin + j * it_step;
        if (itp >= it_end) break;
        const long long tp = itp / chunks;
        const int chp = static_cast<int>(itp - tp * chunks);
        const int pbp = (chp * p.passes_per_token) / chunks;
        const int pep = ((chp + 1) * p.passes_per_token) / chunks;
        const char *q_row = p.q + tp * p.q_stride_b;
        const char *k_row = p.k + tp * p.k_stride_b - static_cast<long long>(p.n_qo) * p.head_stride_b;
        for (int u = 0; u < UMAX; ++u) {
            const int h = (pbp + u) * HPW + g;
            if (pbp + u < pep && h < H && active) {
                const char *base = (h < p.n_qo ? q_row : k_row) + static_cast<long long>(h) * p.head_stride_b;
                prefetch_l2(base + 16 * va);
                prefetch_l2(base + 16 * vb);
            }
        }
    }
    if (OP != kOpNorm) {
        const long long it_j = it_begin + lane * it_step;
        if (it_j < it_end) prefetch_l2(reinterpret_cast<const P *>(p.positions) + it_j / chunks);
    }
}

// Lane geometry of a head: a head's data takes NVH lanes (two 16-byte
// vectors each); its lane group is LPH lanes, NVH rounded up to a power of two
// (head_dim 80, 96 and 192 leave 2 and 4 lanes of the group idle: no loads, no
// stores, zero in the sum); a warp pass covers HPW heads.
template <int D>
struct HeadGeom {
    static constexpr int NVH = D / 16;
    static constexpr int LPH = NVH <= 1 ? 1 : NVH <= 2 ? 2 : NVH <= 4 ? 4 : NVH <= 8 ? 8 : NVH <= 16 ? 16 : 32;
    static constexpr int HPW = kWarp / LPH;
    static_assert(D % 16 == 0 && NVH >= 1 && NVH <= kWarp, "head_dim");
};

// What one lane owns of its head: the two 16-byte vectors (vector v = dims
// [8v, 8v+8)) and their role in the rotation.
struct LaneMap {
    int va, vb;
    bool split;      // NeoX rope_dim % 16 == 0 layout
    bool rot_lane;   // this lane holds rotated dims
    bool active;     // this lane holds data (l < NVH)
};

// Interleaved pairs (2j, 2j+1) sit inside one vector. NeoX with rope_dim % 16
// == 0: a rotating lane owns dims [8a, 8a+8) and [8a+R/2, 8a+R/2+8), both
// halves of eight rotation pairs; lanes past the rotated span own one vector
// from each half of the tail. NeoX with rope_dim <= 8: all of it in vector 0.
template <int D, int MODE>
__device__ __forceinline__ LaneMap lane_map(int l, int R) {
    constexpr int NVH = HeadGeom<D>::NVH;
    LaneMap m;
    m.split = false;
    if (MODE == kNeox && (R & 15) == 0) {
        m.split = true;
        const int rl = R >> 4;          // lanes holding rotation pairs
        if (l < rl) {
            m.va = l;
            m.vb = l + rl;
            m.rot_lane = true;
        } else {
            m.va = (R >> 3) + (l - rl);
            m.vb = m.va + ((D - R) >> 4);
            m.rot_lane = false;
        }
    } else {
        m.va = l;
        m.vb = l + NVH;
        m.rot_lane = (MODE == kNeox) ? (l == 0) : (8 * m.va < R);
    }
    m.active = l < NVH;
    if (!m.active) {
        m.va = 0;
        m.vb = 0;
        m.rot_lane = false;
    }
    return m;
}

// First and end pass of chunk `ch` of a token: from the host's table, or by
// division. An integer division costs about twenty instructions and the
// kernels run their items back to back, so the table is worth 1-2%
// (interleaved); the NeoX instantiations keep the division, which measured
// faster there.
template <int MODE>
__device__ __forceinline__ void item_passes(const Params &p, int chunks, int ch, int &pb, int &pe) {
    if (MODE == kInterleaved && chunks <= kBoundTable) {
        pb = p.pass_bound[ch];
        pe = p.pass_bound[ch + 1];
    } else {
        pb = chunks == 1 ? 0 : (ch * p.passes_per_token) / chunks;
        pe = chunks == 1 ? p.passes_per_token : ((ch + 1) * p.passes_per_token) / chunks;
    }
}

// A new token's position, checked against the cache when the call asks for it
// (cache_len > 0): `ok` becomes false for a position outside the cache, and the
// first chunk's lane 0 counts the bad token once. Otherwise `ok` is left as it is.
__device__ __forceinline__ void check_position(const Params &p, long long pos, long long t, int ch, int lane,
                                               bool &ok) {
    if (p.cache_len > 0) {
        ok = pos >= 0 && pos < p.cache_len;
        if (!ok && ch == 0 && lane == 0) {
            atomicAdd(p.status, 1ull);
            atomicMin(p.status + 1, static_cast<unsigned long long>(t));
        }
    }
}

// The token's cos and (sign-free) sin per owned element. Interleaved:
// c[m]/s[m] serve pair m of vector a (m < 4) and pair m-4 of vector b (m >=
// 4). NeoX split: c[e]/s[e] serve element e of both vectors. NeoX small:
// element e < R/2 of vector 0. Identity (1, 0) wherever nothing rotates.
template <int MODE>
__device__ __forceinline__ void token_cos_sin(const Params &p, long long pos, bool load, int va, int vb, bool split,
                                              int R, int half, float (&c)[8], float (&s)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) { c[e] = 1.f; s[e] = 0.f; }
    if (load) {
        const float *row = p.cache + pos * R;
        if (MODE == kInterleaved) {
            if (p.cache_vec && 8 * va + 8 <= R) {
                const float4 ca = __ldg(reinterpret_cast<const float4 *>(row + 4 * va));
                const float4 sa = __ldg(reinterpret_cast<const float4 *>(row + half + 4 * va));
                c[0] = ca.x; c[1] = ca.y; c[2] = ca.z; c[3] = ca.w;
                s[0] = sa.x; s[1] = sa.y; s[2] = sa.z; s[3] = sa.w;
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j = 4 * va + q;
                    if (2 * j < R) { c[q] = __ldg(row + j); s[q] = __ldg(row + half + j); }
                }
            }
            if (p.cache_vec && 8 * vb + 8 <= R) {
                const float4 cb = __ldg(reinterpret_cast<const float4 *>(row + 4 * vb));
                const float4 sb = __ldg(reinterpret_cast<const float4 *>(row + half + 4 * vb));
                c[4] = cb.x; c[5] = cb.y; c[6] = cb.z; c[7] = cb.w;
                s[4] = sb.x; s[5] = sb.y; s[6] = sb.z; s[7] = sb.w;
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j = 4 * vb + q;
                    if (2 * j < R) { c[4 + q] = __ldg(row + j); s[4 + q] = __ldg(row + half + j); }
                }
            }
        } else if (split) {
            const int j0 = 8 * va;      // dims [j0, j0+8) of the first half
            if (p.cache_vec) {
                const float4 c0 = __ldg(reinterpret_cast<const float4 *>(row + j0));
                const float4 c1 = __ldg(reinterpret_cast<const float4 *>(row + j0 + 4));
                const float4 s0 = __ldg(reinterpret_cast<const float4 *>(row + half + j0));
                const float4 s1 = __ldg(reinterpret_cast<const float4 *>(row + half + j0 + 4));
                c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
                c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
                s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w;
                s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) { c[e] = __ldg(row + j0 + e); s[e] = __ldg(row + half + j0 + e); }
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (e < half) { c[e] = __ldg(row + e); s[e] = __ldg(row + half + e); }
            }
        }
    }
}

// T: storage type (bf16/half); P: position type (int / long long);
// D: head_dim; MODE: pairing; UMAX: max warp passes per item (loads in flight);
// OP: fused (the product) or one step of the unfused baseline;
// EARLY: the caller has promised that the weights and positions were not
// written by the grid this launch depends on (QKNR_INPUTS_READY), so they are
// read before waiting for that grid.
// RC: rope_dim fixed at compile time (0: taken from the parameters at run
// time). Measured worth +0.3-0.8% for interleaved pairing with 4-pass items,
// so the host uses it there for rope_dim = head_dim and head_dim / 2; with NeoX
// pairing it measured slower (the compiler's schedule of the split layout).
template <class T, class P, int D, int MODE, int UMAX, int OP = kOpFused, bool EARLY = false, int RC = 0>
__global__ void __launch_bounds__(512) qknr_fused_kernel(const __grid_constant__ Params p) {
    constexpr int LPH = HeadGeom<D>::LPH;
    constexpr int HPW = HeadGeom<D>::HPW;    // heads per warp pass

    const int lane = threadIdx.x & (kWarp - 1);
    const int g = lane / LPH;           // head slot within the pass
    const int R = RC > 0 ? RC : p.rope_dim;
    const int half = R >> 1;
    const int H = p.n_qo + p.n_kv;
    const LaneMap lm = lane_map<D, MODE>(lane % LPH, R);
    const int va = lm.va, vb = lm.vb;
    const bool split = lm.split, rot_lane = lm.rot_lane, active = lm.active;

    const long long gtid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long warp_id = gtid / kWarp;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) / kWarp;
    // Items of this warp: every nwarps-th item (the default: all warps sweep
    // the tensors together, a compact window of memory at any moment, measured
    // faster on GB300), or a balanced contiguous range.
    const long long it_begin = p.interleave ? warp_id : warp_id * p.num_items / nwarps;
    const long long it_end = p.interleave ? p.num_items : (warp_id + 1) * p.num_items / nwarps;
    const long long it_step = p.interleave ? nwarps : 1;

    // Before waiting for the previous grid: pull this warp's first items' q/k
    // rows and its first positions into L2 (prefetch_first_items).
    if (p.prefetch_items > 0)
        prefetch_first_items<P, HPW, UMAX, OP>(p, it_begin, it_end, it_step, g, va, vb, active, lane);

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 900)
    // Programmatic dependent launch: read nothing before the previous grid in
    // the stream has completed; then let the next grid get resident.
    if (!EARLY) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;");
    }
#endif

    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
    const uint4 wqa = active ? __ldg(p.q_w + va) : zero4, wqb = active ? __ldg(p.q_w + vb) : zero4;
    const uint4 wka = active ? __ldg(p.k_w + va) : zero4, wkb = active ? __ldg(p.k_w + vb) : zero4;

    // the current token's cos and sin per owned element (token_cos_sin)
    float c[8], s[8];
    long long cur_t = -1;
    bool tok_ok = true;
    // Positions read ahead, 32 items at a time: lane j holds the position of
    // the token of the batch's j-th item; jb is the current item's index in
    // the batch.
    long long my_pos = 0;
    int jb = 0;
    if (OP != kOpNorm) {
        const long long it_j = it_begin + lane * it_step;
        if (it_j < it_end) my_pos = load_position<P>(p.positions, it_j / p.chunks_per_token);
    }

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 900)
    // EARLY: the weights and the first positions are in flight; only q, k and
    // the cos|sin rows are read after the previous grid has completed
    if (EARLY) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;");
    }
#endif
    // (token, chunk) of the current item, advanced incrementally: no 64-bit
    // division per item (each one costs dozens of instructions, and a warp
    // runs its items back to back, so every instruction per item shows)
    const int chunks = p.chunks_per_token;
    long long t = it_begin / chunks;
    int ch = static_cast<int>(it_begin - t * chunks);
    const long long step_t = it_step / chunks;
    const int step_c = static_cast<int>(it_step - step_t * chunks);

    for (long long it = it_begin; it < it_end; it += it_step, ++jb) {
        if (OP != kOpNorm && jb == kWarp) {   // next batch of 32 items' positions
            jb = 0;
            const long long it_j = it + lane * it_step;
            my_pos = it_j < it_end ? load_position<P>(p.positions, it_j / chunks) : 0;
        }
        if (it != it_begin) {
            t += step_t;
            ch += step_c;
            if (ch >= chunks) { ch -= chunks; ++t; }
        }
        int pb, pe;                     // the item's passes [pb, pe)
        item_passes<MODE>(p, chunks, ch, pb, pe);

        // this token's rows; k's is shifted back by n_qo heads so that head h
        // (q heads first, then k heads) is row + h * head_stride for both
        char *const q_row = p.q + t * p.q_stride_b;
        char *const k_row = p.k + t * p.k_stride_b - static_cast<long long>(p.n_qo) * p.head_stride_b;
        uint4 xa[UMAX], xb[UMAX];
        char *dst[UMAX];
#pragma unroll
        for (int u = 0; u < UMAX; ++u) {
            const int h = (pb + u) * HPW + g;
            const bool ok = (pb + u < pe) && (h < H) && active;
            char *base = (h < p.n_qo ? q_row : k_row) + static_cast<long long>(h) * p.head_stride_b;
            dst[u] = ok ? base : nullptr;
            if (ok) {
                xa[u] = __ldcs(reinterpret_cast<const uint4 *>(base) + va);
                xb[u] = __ldcs(reinterpret_cast<const uint4 *>(base) + vb);
            } else {
                xa[u] = make_uint4(0u, 0u, 0u, 0u);
                xb[u] = make_uint4(0u, 0u, 0u, 0u);
            }
        }

        // The q/k loads above do not depend on the position; the cos/sin loads
        // below go out while they are in flight (the position itself was
        // read ahead, 32 tokens at a time).
        if (OP != kOpNorm && t != cur_t) {
            cur_t = t;
            const long long pos = __shfl_sync(0xffffffffu, my_pos, jb);
            check_position(p, pos, t, ch, lane, tok_ok);
            token_cos_sin<MODE>(p, pos, tok_ok && rot_lane, va, vb, split, R, half, c, s);
        }
        if (!tok_ok) continue;          // warp-uniform: t is the same for the whole warp

#pragma unroll
        for (int u = 0; u < UMAX; ++u) {
            if (pb + u >= pe) break;    // warp-uniform
            const int h = (pb + u) * HPW + g;
            const bool is_q = h < p.n_qo;
            qknr_head<T, MODE, LPH, OP>(xa[u], xb[u], is_q ? wqa : wka, is_q ? wqb : wkb, c, s, split,
                                        rot_lane, half, p.inv_d, p.eps);
            if (dst[u] != nullptr) {
                __stcs(reinterpret_cast<uint4 *>(dst[u]) + va, xa[u]);
                __stcs(reinterpret_cast<uint4 *>(dst[u]) + vb, xb[u]);
            }
        }
    }
}

}  // namespace qknr
