// qknr_ring_kernel.cuh -- the fused op with each warp's items double-buffered
// in shared memory by asynchronous copies, for sm_103a.
//
// Same op, items, lane mapping and arithmetic (qknr_head) as the register
// kernel in qknr_kernel.cuh, so both give the same bits; only the way q and k
// reach the lanes differs. The register kernel holds an item's loads in
// registers, so a warp has nothing in flight while it computes. Here each
// warp owns two 4 KB stages of shared memory, and every lane copies its own
// 16-byte vectors of an item into its own slots of a stage with cp.async
// (global -> shared, no registers). A lane later reads back only what it
// copied itself, so completion is the lane's own cp.async group: no mbarrier,
// no spin-wait and no synchronisation between lanes or warps.
//
// Two issue orders (Params::ring_ahead), both measured on GB300:
//  0  the next item is issued right after this item's bytes have landed, so
//     it is in flight while this one is computed; a launch asks for no more
//     at its start than the register kernel does. Best on calls of up to a
//     few hundred MB and on NeoX pairing.
//  1  after the first item, the item two ahead is issued once this item's
//     stores are out, so two items can be in flight. More bytes in flight
//     sustain more bandwidth on large interleaved calls (fused_qkv: 99-99.7%
//     of the measured copy peak); the start is slower.
#pragma once

#include <cstdint>

#include "qknr_kernel.cuh"

namespace qknr {

constexpr int kRingStages = 2;                // per warp
constexpr int kRingStageBytes = 4096;         // up to 4 warp passes of 1 KB
constexpr int kRingMaxPasses = 4;             // warp passes per item

// Dynamic shared memory of a CTA of `threads` threads.
__host__ __device__ constexpr int ring_smem_bytes(int threads) {
    return (threads / kWarp) * kRingStages * kRingStageBytes;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy that bypasses L1 (both addresses 16-byte aligned)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's committed groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// T, P, D, MODE, EARLY, RC as for qknr_fused_kernel; items have at most
// kRingMaxPasses warp passes (the host's work map guarantees it). Needs
// ring_smem_bytes(blockDim.x) bytes of dynamic shared memory, and q, k, their
// strides and the head stride 16-byte aligned (the C ABI's vector rule).
template <class T, class P, int D, int MODE, bool EARLY = false, int RC = 0>
__global__ void __launch_bounds__(512) qknr_ring_kernel(const __grid_constant__ Params p) {
    constexpr int LPH = HeadGeom<D>::LPH;
    constexpr int HPW = HeadGeom<D>::HPW;   // heads per warp pass
    static_assert(2 * kRingMaxPasses * kWarp * 16 <= kRingStageBytes, "an item's slots must fit a stage");

    const int lane = threadIdx.x & (kWarp - 1);
    const int g = lane / LPH;
    const int R = RC > 0 ? RC : p.rope_dim;
    const int half = R >> 1;
    const int H = p.n_qo + p.n_kv;
    const LaneMap lm = lane_map<D, MODE>(lane % LPH, R);
    const int va = lm.va, vb = lm.vb;
    const bool active = lm.active;

    // This lane's slots: vector j of pass u of an item sits at
    // ((2u + j) * 32 + lane) * 16 within the stage, so a warp's 16-byte
    // accesses to one slot row cover 512 consecutive bytes (no bank conflict).
    extern __shared__ __align__(128) unsigned char ring_smem[];
    const uint32_t slots = smem_u32(ring_smem) + (threadIdx.x >> 5) * (kRingStages * kRingStageBytes) + lane * 16;

    const long long gtid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long warp_id = gtid / kWarp;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) / kWarp;
    const long long it_begin = p.interleave ? warp_id : warp_id * p.num_items / nwarps;
    const long long it_end = p.interleave ? p.num_items : (warp_id + 1) * p.num_items / nwarps;
    const long long it_step = p.interleave ? nwarps : 1;

    if (p.prefetch_items > 0)
        prefetch_first_items<P, HPW, kRingMaxPasses, kOpFused>(p, it_begin, it_end, it_step, g, va, vb, active,
                                                               lane);
#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 900)
    if (!EARLY) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;");
    }
#endif
    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
    const uint4 wqa = active ? __ldg(p.q_w + va) : zero4, wqb = active ? __ldg(p.q_w + vb) : zero4;
    const uint4 wka = active ? __ldg(p.k_w + va) : zero4, wkb = active ? __ldg(p.k_w + vb) : zero4;
    float c[8], s[8];
    long long cur_t = -1;
    bool tok_ok = true;
    long long my_pos = 0;   // positions read 32 items ahead, as in the register kernel
    int jb = 0;
    {
        const long long it_j = it_begin + lane * it_step;
        if (it_j < it_end) my_pos = load_position<P>(p.positions, it_j / p.chunks_per_token);
    }
#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 900)
    if (EARLY) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;");
    }
#endif
    const int chunks = p.chunks_per_token;
    long long t = it_begin / chunks;
    int ch = static_cast<int>(it_begin - t * chunks);
    const long long step_t = it_step / chunks;
    const int step_c = static_cast<int>(it_step - step_t * chunks);

    // Issue cursor: the next item to copy in.
    long long ti = t, it_i = it_begin;
    int chi = ch;
    auto issue = [&](int stage_) {
        int b0, b1;
        item_passes<MODE>(p, chunks, chi, b0, b1);
        const uint32_t dst = slots + stage_ * kRingStageBytes;
        const char *q_row = p.q + ti * p.q_stride_b;
        const char *k_row = p.k + ti * p.k_stride_b - static_cast<long long>(p.n_qo) * p.head_stride_b;
#pragma unroll
        for (int u = 0; u < kRingMaxPasses; ++u) {
            const int h = (b0 + u) * HPW + g;
            if (b0 + u < b1 && h < H && active) {
                const char *base = (h < p.n_qo ? q_row : k_row) + static_cast<long long>(h) * p.head_stride_b;
                cp_async16(dst + (2 * u) * (kWarp * 16), base + 16 * va);
                cp_async16(dst + (2 * u + 1) * (kWarp * 16), base + 16 * vb);
            }
        }
        cp_async_commit();
        it_i += it_step;
        ti += step_t;
        chi += step_c;
        if (chi >= chunks) { chi -= chunks; ++ti; }
    };
    if (it_i < it_end) issue(0);

    const bool ahead2 = p.ring_ahead != 0;
    bool next_pending = false;   // the item after this one was already issued (order 1)
    int stage = 0;
    for (long long it = it_begin; it < it_end; it += it_step, ++jb) {
        if (jb == kWarp) {   // next batch of 32 items' positions
            jb = 0;
            const long long it_j = it + lane * it_step;
            my_pos = it_j < it_end ? load_position<P>(p.positions, it_j / chunks) : 0;
        }
        if (it != it_begin) {
            t += step_t;
            ch += step_c;
            if (ch >= chunks) { ch -= chunks; ++t; }
        }
        int pb, pe;
        item_passes<MODE>(p, chunks, ch, pb, pe);
        // the cos|sin loads go out before the wait for the item's q/k bytes
        if (t != cur_t) {
            cur_t = t;
            const long long pos = __shfl_sync(0xffffffffu, my_pos, jb);
            check_position(p, pos, t, ch, lane, tok_ok);
            token_cos_sin<MODE>(p, pos, tok_ok && lm.rot_lane, va, vb, lm.split, R, half, c, s);
        }
        if (next_pending) cp_async_wait<1>();
        else cp_async_wait<0>();
        // order 0: the next item into the other stage (it held the previous
        // item, whose slots this lane has read); order 1 does this once
        if ((!ahead2 || it == it_begin) && it_i < it_end) issue(stage ^ 1);

        if (tok_ok) {
            const uint32_t sbase = slots + stage * kRingStageBytes;
            char *const q_row = p.q + t * p.q_stride_b;
            char *const k_row = p.k + t * p.k_stride_b - static_cast<long long>(p.n_qo) * p.head_stride_b;
#pragma unroll
            for (int u = 0; u < kRingMaxPasses; ++u) {
                if (pb + u >= pe) break;    // warp-uniform
                const int h = (pb + u) * HPW + g;
                const bool ok = (h < H) && active;
                uint4 xa = zero4, xb = zero4;
                if (ok) {
                    xa = lds128(sbase + (2 * u) * (kWarp * 16));
                    xb = lds128(sbase + (2 * u + 1) * (kWarp * 16));
                }
                const bool is_q = h < p.n_qo;
                qknr_head<T, MODE, LPH, kOpFused>(xa, xb, is_q ? wqa : wka, is_q ? wqb : wkb, c, s, lm.split,
                                                  lm.rot_lane, half, p.inv_d, p.eps);
                if (ok) {
                    char *base = (is_q ? q_row : k_row) + static_cast<long long>(h) * p.head_stride_b;
                    __stcs(reinterpret_cast<uint4 *>(base) + va, xa);
                    __stcs(reinterpret_cast<uint4 *>(base) + vb, xb);
                }
            }
        }
        // order 1: the item two ahead into this stage, once its slots are read
        next_pending = false;
        if (ahead2 && it_i < it_end) {
            issue(stage);
            next_pending = true;
        }
        stage ^= 1;
    }
    cp_async_wait<0>();
}

}  // namespace qknr
