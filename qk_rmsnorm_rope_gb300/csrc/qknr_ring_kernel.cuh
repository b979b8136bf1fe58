// qknr_ring_kernel.cuh -- the fused op with each warp's items double-buffered
// in shared memory by bulk asynchronous copies (TMA), for sm_103a.
//
// Same op, lane mapping and arithmetic (qknr_head) as the register kernel in
// qknr_kernel.cuh, so both give the same bits; only the way q and k reach the
// lanes differs. The register kernel holds an item's loads in registers, so a
// warp has nothing in flight while it computes. Here each warp owns two 4 KB
// stages of shared memory and one mbarrier per stage:
//  * one lane issues the item's q/k bytes as one or two cp.async.bulk copies
//    (one per side when the item spans the q/k boundary; one per head when
//    heads are not contiguous) into a stage, with the byte count armed on the
//    stage's mbarrier;
//  * the warp waits for the item's bytes, then at once issues its next item
//    into the other stage, so that item's copy is in flight while this one is
//    computed: per pass each lane reads its two 16-byte vectors from shared
//    memory, runs qknr_head and stores the result straight to global memory;
//  * the first item alone is issued before the loop, so a launch requests no
//    more at its start than the register kernel does.
// There is no synchronisation between warps: stages, barriers and items are
// private to a warp, and items are dealt to warps as in the register kernel.
// Measured on GB300 it is faster than the register kernel on NeoX pairing at
// every size tried and on interleaved calls of up to a few hundred MB; on
// larger interleaved calls the register kernel sustains more bandwidth.
//
// Every mbarrier wait is bounded (kRingWaitNs of %globaltimer). A wait that
// runs out sets the watchdog word of the status block, waits (bounded again)
// for the copy it was waiting on, and the warp returns, leaving its remaining
// items untouched; the host reports it (QKNR_ERR_WATCHDOG) from the checked
// entry points and qknr_sync.
#pragma once

#include <cstdint>

#include "qknr_kernel.cuh"

namespace qknr {

constexpr int kRingStages = 2;                // per warp
constexpr int kRingStageBytes = 4096;         // up to 4 warp passes of at most 1 KB
constexpr int kRingMaxPasses = 4;             // warp passes per item
constexpr int kRingWarpBytes = kRingStages * (kRingStageBytes + 8);  // stages + mbarriers
constexpr unsigned long long kRingWaitNs = 1000000000ull;            // 1 s per wait
constexpr int kStatusWatchdog = 2;            // status word set when a wait ran out

// Dynamic shared memory of a CTA of `threads` threads.
__host__ __device__ constexpr int ring_smem_bytes(int threads) { return (threads / kWarp) * kRingWarpBytes; }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Arrive once on `bar` and add `bytes` to the bytes its phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Global -> shared bulk copy; its bytes complete on `bar`. dst, src and bytes
// are multiples of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// The slow path of mbar_wait: poll until the phase completes or kRingWaitNs
// have passed (false).
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kRingWaitNs) return false;
    }
}

// Wait for the phase of `bar` with parity `parity`; false if it did not
// complete within kRingWaitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity);
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
    constexpr int HB = D * static_cast<int>(sizeof(T));   // bytes of one head
    static_assert(kRingMaxPasses * HPW * HB <= kRingStageBytes, "an item must fit its stage");

    const int lane = threadIdx.x & (kWarp - 1);
    const int g = lane / LPH;
    const int R = RC > 0 ? RC : p.rope_dim;
    const int half = R >> 1;
    const int H = p.n_qo + p.n_kv;
    const LaneMap lm = lane_map<D, MODE>(lane % LPH, R);
    const int va = lm.va, vb = lm.vb;
    const bool active = lm.active;

    // this warp's stages and their mbarriers (one arrival: the issuing lane's)
    extern __shared__ __align__(128) unsigned char ring_smem[];
    const int wib = threadIdx.x >> 5;
    const uint32_t data_s = smem_u32(ring_smem) + wib * (kRingStages * kRingStageBytes);
    const uint32_t bar_s =
        smem_u32(ring_smem) + (blockDim.x >> 5) * (kRingStages * kRingStageBytes) + wib * (kRingStages * 8);
    if (lane == 0) {
#pragma unroll
        for (int s_ = 0; s_ < kRingStages; ++s_) mbar_init(bar_s + 8 * s_, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();

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
    const bool contig = p.head_stride_b == HB;

    // Issue cursor: the next item to copy in, advanced by every lane alike;
    // lane 0 issues the copies.
    long long ti = t, it_i = it_begin;
    int chi = ch;
    auto issue = [&](int stage_) {
        if (lane == 0) {
            int b0, b1;
            item_passes<MODE>(p, chunks, chi, b0, b1);
            const int h0 = b0 * HPW;
            const int h1 = min(b1 * HPW, H);
            const uint32_t dst = data_s + stage_ * kRingStageBytes;
            const uint32_t bar = bar_s + 8 * stage_;
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>((h1 - h0) * HB));
            const char *q_row = p.q + ti * p.q_stride_b;
            const char *k_row = p.k + ti * p.k_stride_b - static_cast<long long>(p.n_qo) * p.head_stride_b;
            if (contig) {
                if (h0 < p.n_qo) {
                    const int he = min(h1, p.n_qo);
                    bulk_load(dst, q_row + static_cast<long long>(h0) * HB, (he - h0) * HB, bar);
                }
                if (h1 > p.n_qo) {
                    const int hk = max(h0, p.n_qo);
                    bulk_load(dst + (hk - h0) * HB, k_row + static_cast<long long>(hk) * HB, (h1 - hk) * HB, bar);
                }
            } else {
                for (int h = h0; h < h1; ++h)
                    bulk_load(dst + (h - h0) * HB, (h < p.n_qo ? q_row : k_row) + h * p.head_stride_b, HB, bar);
            }
        }
        it_i += it_step;
        ti += step_t;
        chi += step_c;
        if (chi >= chunks) { chi -= chunks; ++ti; }
    };
    if (it_i < it_end) issue(0);

    int stage = 0;
    uint32_t parity = 0;
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

        const uint32_t sbase = data_s + stage * kRingStageBytes;
        if (!mbar_wait(bar_s + 8 * stage, parity)) {
            // the only copy this warp has in flight is this item's (the next
            // one is issued after this wait): give it one more bounded wait
            if (lane == 0) atomicOr(p.status + kStatusWatchdog, 1ull);
            mbar_wait(bar_s + 8 * stage, parity);
            return;
        }
        // the other stage held the previous item, whose reads ended at the
        // last __syncwarp: order them before the async proxy writes it again
        if (it_i < it_end) {
            if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(stage ^ 1);
        }
        if (tok_ok) {
            char *const q_row = p.q + t * p.q_stride_b;
            char *const k_row = p.k + t * p.k_stride_b - static_cast<long long>(p.n_qo) * p.head_stride_b;
            const int h0 = pb * HPW;
#pragma unroll
            for (int u = 0; u < kRingMaxPasses; ++u) {
                if (pb + u >= pe) break;    // warp-uniform
                const int h = (pb + u) * HPW + g;
                const bool ok = (h < H) && active;
                uint4 xa = zero4, xb = zero4;
                if (ok) {
                    const uint32_t a = sbase + (h - h0) * HB;
                    xa = lds128(a + 16 * va);
                    xb = lds128(a + 16 * vb);
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
        __syncwarp();
        stage ^= 1;
        parity ^= static_cast<uint32_t>(stage == 0);
    }
}

}  // namespace qknr
