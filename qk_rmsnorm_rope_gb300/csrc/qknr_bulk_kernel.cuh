// qknr_bulk_kernel.cuh -- the fused op with bulk asynchronous copies (TMA)
// feeding a shared-memory ring, for sm_103a.
//
// Same arithmetic and lane mapping as qknr_fused_kernel (qknr_kernel.cuh);
// only the way bytes reach the SM differs. The register kernel can keep only
// as many loads in flight as its registers hold, and on GB300 that leaves HBM
// idle part of the time. Here one producer warp per CTA streams tiles into an
// S-stage ring with cp.async.bulk, so the bytes in flight per SM are bounded
// by shared memory (up to ~200 KB) instead of registers:
//
//  * tile = (token, chunk of heads). Its smem stage holds the chunk's q heads,
//    then its k heads (D*2 bytes each, densely packed), then the token's fp32
//    cos|sin row (R*4 bytes). With a head stride equal to head_dim the q part
//    and the k part are one bulk copy each; otherwise one copy per head.
//  * the producer warp reads 32 positions at a time (one coalesced load), then
//    for each tile waits for its stage to be free (empty mbarrier), arms the
//    stage's full mbarrier with the byte count and issues the copies. In the
//    checked mode a tile whose position is outside the cache is not copied: it
//    is flagged, counted, and its stage is released at once.
//  * all consumer warps work on every tile, in order: each takes every NC-th
//    warp pass of the tile, two passes at a time with independent dependency
//    chains, computing from shared memory with the register kernel's lane
//    mapping (two 16-byte vectors per lane, no pairing shuffles) and storing
//    128-bit results straight to global memory; the stage is free again once
//    all NC consumers have arrived on its empty mbarrier.
//  * tiles are split across CTAs in balanced contiguous ranges; the grid is
//    persistent (one wave).
//  * every mbarrier wait is bounded by %globaltimer. A wait that runs out sets
//    a watchdog bit in the status word and the warp stops; before the CTA
//    exits, thread 0 waits (bounded again) for every copy it issued.
#pragma once

#include "qknr_kernel.cuh"

namespace qknr {

constexpr unsigned long long kWatchdogNs = 1000000000ull;  // 1 s per wait
constexpr unsigned long long kWatchdogBit = 1ull;          // status[2]: a wait ran out

struct BulkParams {
    char *q;
    char *k;
    const uint4 *q_w;
    const uint4 *k_w;
    const float *cache;
    const void *positions;
    unsigned long long *status;   // [0] bad-token count, [1] first bad token, [2] watchdog bits
    long long q_stride_b;
    long long k_stride_b;
    long long head_stride_b;
    long long num_tiles;          // num_tokens * chunks_per_token
    long long cache_len;          // > 0: check positions against it
    int n_qo, n_kv;
    int rope_dim;
    int chunks_per_token;
    int heads_per_chunk;          // heads in a full chunk (a token's last chunk may hold fewer)
    int stages;                   // ring depth S
    int stage_bytes;              // bytes per stage, a multiple of 128
    int heads_contig;             // head_stride == head_dim: one copy per q / k run
    float eps;
    float inv_d;
};

// Shared-memory layout: S full barriers, S empty barriers, S flags, then the
// stages at a 128-byte boundary.
__host__ __device__ constexpr int bulk_stage_offset(int stages) {
    return ((stages * 20) + 127) / 128 * 128;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity to complete, for at most
// kWatchdogNs. Returns false if the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWatchdogNs) return false;
    }
    return true;
}

// The same wait for a whole warp: every lane polls the barrier (each needs the
// acquire for the data it reads), lane 0's clock decides a time-out for all,
// so the result is warp-uniform.
__device__ __forceinline__ bool mbar_wait_bounded_warp(uint32_t bar, uint32_t parity) {
    bool ok = mbar_try_wait(bar, parity);
    unsigned long long t0 = 0;
    while (!__all_sync(0xffffffffu, ok)) {
        if (!ok) ok = mbar_try_wait(bar, parity);
        const unsigned long long now = global_ns();
        if (t0 == 0) t0 = now;
        const int expired = (now - t0) > kWatchdogNs ? 1 : 0;
        if (__shfl_sync(0xffffffffu, expired, 0)) return false;
    }
    return true;
}

// Global -> shared bulk copy completing on an mbarrier (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint4 lds16(const unsigned char *p) {
    return *reinterpret_cast<const uint4 *>(p);
}

__device__ __forceinline__ float4 lds_f4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}

template <class T, class P, int D, int MODE>
__global__ void __launch_bounds__(544, 1) qknr_bulk_kernel(const __grid_constant__ BulkParams p) {
    constexpr int LPH = D / 16;
    constexpr int HPW = kWarp / LPH;
    static_assert(D % 16 == 0 && LPH >= 1 && LPH <= kWarp && (LPH & (LPH - 1)) == 0, "head_dim");
    extern __shared__ __align__(128) unsigned char smem[];

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 900)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
#endif

    const int S = p.stages;
    unsigned long long *full = reinterpret_cast<unsigned long long *>(smem);
    unsigned long long *empty = full + S;
    int *flags = reinterpret_cast<int *>(empty + S);
    unsigned char *stages = smem + bulk_stage_offset(S);

    const int warp = threadIdx.x / kWarp;
    const int lane = threadIdx.x % kWarp;
    const int n_consumers = static_cast<int>(blockDim.x / kWarp) - 1;
    const long long tb = static_cast<long long>(blockIdx.x) * p.num_tiles / gridDim.x;
    const long long te = static_cast<long long>(blockIdx.x + 1) * p.num_tiles / gridDim.x;
    const int n_local = static_cast<int>(te - tb);
    const int H = p.n_qo + p.n_kv;
    const int R = p.rope_dim;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(full + s), 1);
            mbar_init(smem_u32(empty + s), static_cast<uint32_t>(n_consumers));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    long long issued = 0;  // tiles whose copies thread 0 issued (producer lane 0)

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        bool dead = false;
        for (long long base = tb; base < te && !dead; base += kWarp) {
            long long my_pos = 0;
            const long long my_tile = base + lane;
            if (my_tile < te) my_pos = load_position<P>(p.positions, my_tile / p.chunks_per_token);
            const int nb = static_cast<int>(min(static_cast<long long>(kWarp), te - base));
            for (int j = 0; j < nb; ++j) {
                const long long pos = __shfl_sync(0xffffffffu, my_pos, j);
                if (lane == 0) {
                    const long long i = base + j - tb;
                    const int s = static_cast<int>(i % S);
                    const uint32_t round = static_cast<uint32_t>(i / S);
                    if (!mbar_wait_bounded(smem_u32(empty + s), (round & 1u) ^ 1u)) {
                        atomicOr(p.status + 2, kWatchdogBit);
                        dead = true;
                    } else {
                        const long long tile = base + j;
                        const long long t = tile / p.chunks_per_token;
                        const int c = static_cast<int>(tile - t * p.chunks_per_token);
                        const int h0 = c * p.heads_per_chunk;
                        const int h1 = min(H, h0 + p.heads_per_chunk);
                        const bool bad = p.cache_len > 0 && (pos < 0 || pos >= p.cache_len);
                        flags[s] = bad ? 1 : 0;
                        const uint32_t fb = smem_u32(full + s);
                        if (bad) {
                            if (c == 0) {
                                atomicAdd(p.status, 1ull);
                                atomicMin(p.status + 1, static_cast<unsigned long long>(t));
                            }
                            mbar_arrive(fb);
                        } else {
                            const uint32_t head_b = 2u * D;
                            const uint32_t bytes = static_cast<uint32_t>(h1 - h0) * head_b + 4u * R;
                            mbar_arrive_expect_tx(fb, bytes);
                            const uint32_t dst = smem_u32(stages + static_cast<size_t>(s) * p.stage_bytes);
                            const int qa = h0, qb = min(h1, p.n_qo);
                            if (qb > qa) {
                                const char *src = p.q + t * p.q_stride_b + qa * p.head_stride_b;
                                if (p.heads_contig) {
                                    bulk_g2s(dst, src, static_cast<uint32_t>(qb - qa) * head_b, fb);
                                } else {
                                    for (int h = qa; h < qb; ++h)
                                        bulk_g2s(dst + (h - h0) * head_b,
                                                 p.q + t * p.q_stride_b + h * p.head_stride_b, head_b, fb);
                                }
                            }
                            const int ka = max(h0, p.n_qo), kb = h1;
                            if (kb > ka) {
                                const char *src = p.k + t * p.k_stride_b + (ka - p.n_qo) * p.head_stride_b;
                                if (p.heads_contig) {
                                    bulk_g2s(dst + (ka - h0) * head_b, src,
                                             static_cast<uint32_t>(kb - ka) * head_b, fb);
                                } else {
                                    for (int h = ka; h < kb; ++h)
                                        bulk_g2s(dst + (h - h0) * head_b,
                                                 p.k + t * p.k_stride_b + (h - p.n_qo) * p.head_stride_b,
                                                 head_b, fb);
                                }
                            }
                            bulk_g2s(dst + (h1 - h0) * head_b, p.cache + pos * R, 4u * R, fb);
                        }
                        issued = i + 1;
                    }
                }
                dead = __shfl_sync(0xffffffffu, dead ? 1 : 0, 0) != 0;
                if (dead) break;
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int cw = warp - 1;
        const int g = lane / LPH;
        const int l = lane % LPH;
        const int half = R >> 1;
        int va, vb;
        bool split = false, rot_lane;
        if (MODE == kNeox && (R & 15) == 0) {
            split = true;
            const int rl = R >> 4;
            if (l < rl) {
                va = l;
                vb = l + rl;
                rot_lane = true;
            } else {
                va = (R >> 3) + (l - rl);
                vb = va + ((D - R) >> 4);
                rot_lane = false;
            }
        } else {
            va = l;
            vb = l + LPH;
            rot_lane = (MODE == kNeox) ? (l == 0) : (8 * va < R);
        }
        const uint4 wqa = __ldg(p.q_w + va), wqb = __ldg(p.q_w + vb);
        const uint4 wka = __ldg(p.k_w + va), wkb = __ldg(p.k_w + vb);

        // Every consumer warp takes part in every tile, in tile order: warp cw
        // handles passes cw, cw + NC, ... of the tile, two at a time with
        // independent chains, then arrives on the stage's empty barrier (which
        // counts all NC consumers). A warp waits for tile i only after it has
        // itself seen tile i - S arrive, and tile i + S cannot arrive before
        // this warp released tile i, so the parity it awaits is never stale.
        for (int i = 0; i < n_local; ++i) {
            const int s = i % S;
            const uint32_t round = static_cast<uint32_t>(i / S);
            if (!mbar_wait_bounded_warp(smem_u32(full + s), round & 1u)) {
                if (lane == 0) atomicOr(p.status + 2, kWatchdogBit);
                break;
            }
            if (flags[s] == 0) {
                const long long tile = tb + i;
                const long long t = tile / p.chunks_per_token;
                const int c = static_cast<int>(tile - t * p.chunks_per_token);
                const int h0 = c * p.heads_per_chunk;
                const int h1 = min(H, h0 + p.heads_per_chunk);
                const int npass = (h1 - h0 + HPW - 1) / HPW;
                const unsigned char *st = stages + static_cast<size_t>(s) * p.stage_bytes;
                const float *row = reinterpret_cast<const float *>(st + (h1 - h0) * 2 * D);

                float c8[8], s8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) { c8[e] = 1.f; s8[e] = 0.f; }
                if (rot_lane && cw < npass) {
                    if (MODE == kInterleaved) {
                        // R % 8 == 0 here: a vector rotates entirely or not at all
                        if (8 * va < R) {
                            const float4 ca = lds_f4(row + 4 * va), sa = lds_f4(row + half + 4 * va);
                            c8[0] = ca.x; c8[1] = ca.y; c8[2] = ca.z; c8[3] = ca.w;
                            s8[0] = sa.x; s8[1] = sa.y; s8[2] = sa.z; s8[3] = sa.w;
                        }
                        if (8 * vb < R) {
                            const float4 cb = lds_f4(row + 4 * vb), sb = lds_f4(row + half + 4 * vb);
                            c8[4] = cb.x; c8[5] = cb.y; c8[6] = cb.z; c8[7] = cb.w;
                            s8[4] = sb.x; s8[5] = sb.y; s8[6] = sb.z; s8[7] = sb.w;
                        }
                    } else if (split) {
                        const int j0 = 8 * va;
                        const float4 c0 = lds_f4(row + j0), c1 = lds_f4(row + j0 + 4);
                        const float4 s0 = lds_f4(row + half + j0), s1 = lds_f4(row + half + j0 + 4);
                        c8[0] = c0.x; c8[1] = c0.y; c8[2] = c0.z; c8[3] = c0.w;
                        c8[4] = c1.x; c8[5] = c1.y; c8[6] = c1.z; c8[7] = c1.w;
                        s8[0] = s0.x; s8[1] = s0.y; s8[2] = s0.z; s8[3] = s0.w;
                        s8[4] = s1.x; s8[5] = s1.y; s8[6] = s1.z; s8[7] = s1.w;
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (e < half) { c8[e] = row[e]; s8[e] = row[half + e]; }
                    }
                }

                for (int pp = cw; pp < npass; pp += 2 * n_consumers) {
                    uint4 xa[2], xb[2];
                    int hh[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int h = h0 + (pp + u * n_consumers) * HPW + g;
                        hh[u] = h;
                        xa[u] = make_uint4(0u, 0u, 0u, 0u);
                        xb[u] = xa[u];
                        if (h < h1) {
                            const unsigned char *hp = st + (h - h0) * 2 * D;
                            xa[u] = lds16(hp + 16 * va);
                            xb[u] = lds16(hp + 16 * vb);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const bool is_q = hh[u] < p.n_qo;
                        qknr_head<T, MODE, LPH>(xa[u], xb[u], is_q ? wqa : wka, is_q ? wqb : wkb, c8, s8,
                                                 split, rot_lane, half, p.inv_d, p.eps);
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int h = hh[u];
                        if (h < h1) {
                            char *dstp = h < p.n_qo ? p.q + t * p.q_stride_b + h * p.head_stride_b
                                                    : p.k + t * p.k_stride_b + (h - p.n_qo) * p.head_stride_b;
                            __stcs(reinterpret_cast<uint4 *>(dstp) + va, xa[u]);
                            __stcs(reinterpret_cast<uint4 *>(dstp) + vb, xb[u]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(empty + s));
        }
    }

    // Every thread gets here, also after a wait ran out. Before the CTA exits,
    // make sure no copy issued into this CTA's shared memory is still running.
    __syncthreads();
    if (threadIdx.x == 0 && issued > 0) {
        for (int s = 0; s < S && s < issued; ++s) {
            const long long last = s + static_cast<long long>(S) * ((issued - 1 - s) / S);
            if (!mbar_wait_bounded(smem_u32(full + s), static_cast<uint32_t>(last / S) & 1u))
                atomicOr(p.status + 2, kWatchdogBit);
        }
    }
}

}  // namespace qknr
