// qknr_async_kernel.cuh -- the fused op with a per-warp cp.async pipeline, for sm_103a.
//
// Same arithmetic and lane mapping as the register kernel (qknr_kernel.cuh):
// a lane owns two 16-byte vectors of one head, a warp pass covers 32/(D/16)
// heads. The register kernel holds its loads in flight in registers, which
// caps the bytes in flight per SM. Here every warp streams its own passes
// into a private S-stage ring in shared memory with cp.async (16-byte
// asynchronous global -> shared copies, completion tracked per thread with
// commit/wait groups), and computes S passes behind the copies, so the bytes
// in flight are bounded by shared memory and registers hold only the pass
// being computed. There is no cross-warp synchronisation and no spin-wait.
//
//  * A warp's work is a balanced contiguous range of (token, pass) units.
//  * Stage = the pass's data (vector a of all 32 lanes, then vector b; 1 KB)
//    + the token's fp32 cos|sin row (R*4 bytes, copied only for a pass that
//    starts a token in the warp's range) + a flag word.
//  * Positions are read 32 tokens at a time (one coalesced load per warp).
//  * In the checked mode a token whose position is outside the cache is not
//    copied and not stored (left untouched), and is counted once.
//  * Needs rope_dim % 8 == 0 and a 16-byte aligned cos|sin table.
#pragma once

#include "qknr_bulk_kernel.cuh"
#include "qknr_kernel.cuh"

namespace qknr {

struct AsyncParams {
    char *q;
    char *k;
    const uint4 *q_w;
    const uint4 *k_w;
    const float *cache;
    const void *positions;
    unsigned long long *status;   // [0] bad-token count, [1] first bad token
    long long q_stride_b;
    long long k_stride_b;
    long long head_stride_b;
    long long num_tokens;
    long long num_passes;         // num_tokens * passes_per_token
    long long cache_len;          // > 0: check positions against it
    int n_qo, n_kv;
    int rope_dim;
    int passes_per_token;
    int stages;                   // S in [2, 8]
    int stage_bytes;              // 1024 + 4 * rope_dim + 16
    float eps;
    float inv_d;
};

constexpr int kAsyncMaxStages = 8;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// wait until at most n of this thread's groups are pending (n is warp-uniform)
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
    switch (n) {
        case 1: cp_async_wait<1>(); break;
        case 2: cp_async_wait<2>(); break;
        case 3: cp_async_wait<3>(); break;
        case 4: cp_async_wait<4>(); break;
        case 5: cp_async_wait<5>(); break;
        case 6: cp_async_wait<6>(); break;
        case 7: cp_async_wait<7>(); break;
        default: cp_async_wait<0>(); break;
    }
}

template <class T, class P, int D, int MODE>
__global__ void __launch_bounds__(256, 3) qknr_async_kernel(const __grid_constant__ AsyncParams p) {
    constexpr int LPH = D / 16;
    constexpr int HPW = kWarp / LPH;
    static_assert(D % 16 == 0 && LPH >= 1 && LPH <= kWarp && (LPH & (LPH - 1)) == 0, "head_dim");
    extern __shared__ __align__(128) unsigned char smem[];

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 900)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
#endif

    const int lane = threadIdx.x % kWarp;
    const int wic = threadIdx.x / kWarp;     // warp in CTA
    const int g = lane / LPH;
    const int l = lane % LPH;
    const int R = p.rope_dim;
    const int half = R >> 1;
    const int H = p.n_qo + p.n_kv;
    const int S = p.stages;
    const int ppt = p.passes_per_token;
    unsigned char *ring = smem + static_cast<size_t>(wic) * S * p.stage_bytes;

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

    const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / kWarp;
    const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) / kWarp;
    const long long u0 = gw * p.num_passes / nw;
    const long long u1 = (gw + 1) * p.num_passes / nw;

    // ---------------------------------------------------------------- issue side
    long long pos_base = -1000000;   // first token of the positions batch held by the lanes
    long long my_pos = 0;            // position of token pos_base + lane
    bool issue_bad = false;          // the token being issued is skipped (checked mode)
    long long issue_u = u0;
    int issue_slot = 0;

    auto issue = [&](long long u, int slot) {
        unsigned char *st = ring + static_cast<size_t>(slot) * p.stage_bytes;
        const long long t = u / ppt;
        const int pl = static_cast<int>(u - t * ppt);
        if (u == u0 || pl == 0) {   // warp-uniform: the pass starts a token
            if (t >= pos_base + kWarp || t < pos_base) {
                pos_base = t;
                my_pos = (t + lane < p.num_tokens) ? load_position<P>(p.positions, t + lane) : 0;
            }
            const long long pos = __shfl_sync(0xffffffffu, my_pos, static_cast<int>(t - pos_base));
            issue_bad = p.cache_len > 0 && (pos < 0 || pos >= p.cache_len);
            if (lane == 0) {
                *reinterpret_cast<int *>(st + 1024 + 4 * R) = issue_bad ? 1 : 0;
                if (issue_bad && pl == 0) {
                    atomicAdd(p.status, 1ull);
                    atomicMin(p.status + 1, static_cast<unsigned long long>(t));
                }
            }
            if (!issue_bad) {
                const float *row = p.cache + pos * R;
                for (int c = lane; c < R / 4; c += kWarp) cp_async16(smem_u32(st + 1024 + 16 * c), row + 4 * c);
            }
        }
        const int h = pl * HPW + g;
        if (!issue_bad && h < H) {
            const char *base = (h < p.n_qo) ? p.q + t * p.q_stride_b + static_cast<long long>(h) * p.head_stride_b
                                            : p.k + t * p.k_stride_b + static_cast<long long>(h - p.n_qo) * p.head_stride_b;
            cp_async16(smem_u32(st + 16 * lane), base + 16 * va);
            cp_async16(smem_u32(st + 512 + 16 * lane), base + 16 * vb);
        }
    };

    // prologue: S passes in flight (a commit group per pass, empty past the range)
    for (int k = 0; k < S; ++k) {
        if (issue_u < u1) issue(issue_u, issue_slot);
        cp_async_commit();
        ++issue_u;
        issue_slot = (issue_slot + 1 == S) ? 0 : issue_slot + 1;
    }

    // ---------------------------------------------------------------- compute side
    float c8[8], s8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) { c8[e] = 1.f; s8[e] = 0.f; }
    bool tok_bad = false;
    int slot = 0;
    for (long long u = u0; u < u1; ++u) {
        cp_async_wait_dyn(S - 1);   // this thread's copies for pass u have landed
        __syncwarp();               // ... and every lane's (the row comes from several lanes)
        const unsigned char *st = ring + static_cast<size_t>(slot) * p.stage_bytes;
        const long long t = u / ppt;
        const int pl = static_cast<int>(u - t * ppt);
        if (u == u0 || pl == 0) {
            tok_bad = *reinterpret_cast<const int *>(st + 1024 + 4 * R) != 0;
            if (!tok_bad && rot_lane) {
                const float *row = reinterpret_cast<const float *>(st + 1024);
                if (MODE == kInterleaved) {
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
        }
        if (!tok_bad) {
            const int h = pl * HPW + g;
            uint4 xa = make_uint4(0u, 0u, 0u, 0u), xb = xa;
            if (h < H) {
                xa = lds16(st + 16 * lane);
                xb = lds16(st + 512 + 16 * lane);
            }
            const bool is_q = h < p.n_qo;
            qknr_head<T, MODE, LPH>(xa, xb, is_q ? wqa : wka, is_q ? wqb : wkb, c8, s8, split, rot_lane,
                                     half, p.inv_d, p.eps);
            if (h < H) {
                char *dst = is_q ? p.q + t * p.q_stride_b + static_cast<long long>(h) * p.head_stride_b
                                 : p.k + t * p.k_stride_b + static_cast<long long>(h - p.n_qo) * p.head_stride_b;
                __stcs(reinterpret_cast<uint4 *>(dst) + va, xa);
                __stcs(reinterpret_cast<uint4 *>(dst) + vb, xb);
            }
        }
        __syncwarp();               // every lane is done reading this stage
        if (issue_u < u1) issue(issue_u, slot);
        cp_async_commit();
        ++issue_u;
        slot = (slot + 1 == S) ? 0 : slot + 1;
    }
    cp_async_wait<0>();
}

}  // namespace qknr
