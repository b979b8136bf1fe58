// qknr_lean_kernel.cuh -- the register kernel with its per-token state in
// shared memory, for sm_103a.
//
// The register kernel's speed on GB300 is set by how many 16-byte loads each
// SM keeps in flight, and that is capped by registers: about 110 registers a
// thread leave room for two 256-thread CTAs per SM. This variant keeps the
// loads in registers exactly as the register kernel does (a warp item = up to
// UMAX passes, all loads issued before any arithmetic) but moves the rest of
// the per-thread state out of registers:
//  * both weight vectors live once per CTA in shared memory;
//  * the current token's fp32 cos|sin row lives in a per-warp shared buffer
//    (copied in when the warp reaches a new token);
//  * every pass re-reads its weight and cos/sin slices with shared loads the
//    compiler may not hoist, and store addresses are recomputed;
// so that three 256-thread CTAs (24 warps) fit an SM. Same lane mapping,
// same arithmetic (qknr_head) and so the same bits as every other kernel.
#pragma once

#include "qknr_kernel.cuh"

namespace qknr {

constexpr int kLeanMaxWarps = 8;     // CTAs of at most 256 threads
constexpr int kLeanMaxRope = 256;    // cos|sin row buffer per warp: 1 KB

__device__ __forceinline__ uint4 lds_volatile_u4(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
    return v;
}

__device__ __forceinline__ float4 lds_volatile_f4(const void *p) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
    return v;
}

__device__ __forceinline__ float lds_volatile_f1(const void *p) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
    return v;
}

// cos/sin for this lane's elements from a cos|sin row in shared memory, in the
// order qknr_head wants them (see qknr_math.cuh); (1, 0) where nothing rotates.
template <int MODE>
__device__ __forceinline__ void lean_cos_sin(const float *row, int R, int half, int va, int vb, bool split,
                                             bool rot_lane, float (&c)[8], float (&s)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) { c[e] = 1.f; s[e] = 0.f; }
    if (!rot_lane) return;
    if (MODE == kInterleaved) {
        // pairs 4va..4va+3 of vector a, 4vb..4vb+3 of vector b; a pair rotates if 2j < R
        if (8 * va + 8 <= R && (R & 7) == 0) {
            const float4 ca = lds_volatile_f4(row + 4 * va), sa = lds_volatile_f4(row + half + 4 * va);
            c[0] = ca.x; c[1] = ca.y; c[2] = ca.z; c[3] = ca.w;
            s[0] = sa.x; s[1] = sa.y; s[2] = sa.z; s[3] = sa.w;
        } else {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int j = 4 * va + m;
                if (2 * j < R) { c[m] = lds_volatile_f1(row + j); s[m] = lds_volatile_f1(row + half + j); }
            }
        }
        if (8 * vb + 8 <= R && (R & 7) == 0) {
            const float4 cb = lds_volatile_f4(row + 4 * vb), sb = lds_volatile_f4(row + half + 4 * vb);
            c[4] = cb.x; c[5] = cb.y; c[6] = cb.z; c[7] = cb.w;
            s[4] = sb.x; s[5] = sb.y; s[6] = sb.z; s[7] = sb.w;
        } else {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int j = 4 * vb + m;
                if (2 * j < R) { c[4 + m] = lds_volatile_f1(row + j); s[4 + m] = lds_volatile_f1(row + half + j); }
            }
        }
    } else if (split) {
        const int j0 = 8 * va;
        const float4 c0 = lds_volatile_f4(row + j0), c1 = lds_volatile_f4(row + j0 + 4);
        const float4 s0 = lds_volatile_f4(row + half + j0), s1 = lds_volatile_f4(row + half + j0 + 4);
        c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
        c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
        s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w;
        s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (e < half) { c[e] = lds_volatile_f1(row + e); s[e] = lds_volatile_f1(row + half + e); }
    }
}

template <class T, class P, int D, int MODE>
__global__ void __launch_bounds__(256, 3) qknr_lean_kernel(const __grid_constant__ Params p) {
    constexpr int LPH = D / 16;
    constexpr int HPW = kWarp / LPH;
    constexpr int UMAX = 4;
    static_assert(D % 16 == 0 && LPH >= 1 && LPH <= kWarp && (LPH & (LPH - 1)) == 0, "head_dim");
    __shared__ __align__(16) uint4 s_w[2][D / 8];                         // q_w, k_w
    __shared__ __align__(16) float s_row[kLeanMaxWarps][kLeanMaxRope];   // cos|sin row per warp

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 900)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
#endif

    for (int i = threadIdx.x; i < 2 * (D / 8); i += blockDim.x)
        s_w[i / (D / 8)][i % (D / 8)] = __ldg((i < D / 8 ? p.q_w : p.k_w) + i % (D / 8));
    __syncthreads();

    const int lane = threadIdx.x & (kWarp - 1);
    const int wic = threadIdx.x / kWarp;
    const int g = lane / LPH;
    const int l = lane % LPH;
    const int R = p.rope_dim;
    const int half = R >> 1;
    const int H = p.n_qo + p.n_kv;
    float *row = s_row[wic];

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

    const long long gtid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long warp_id = gtid / kWarp;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) / kWarp;
    const long long it_begin = warp_id * p.num_items / nwarps;
    const long long it_end = (warp_id + 1) * p.num_items / nwarps;

    long long cur_t = -1;
    bool tok_ok = true;
    long long my_pos = 0;
    int jb = 0;
    if (it_begin + lane < it_end) my_pos = load_position<P>(p.positions, (it_begin + lane) / p.chunks_per_token);

    for (long long it = it_begin; it < it_end; ++it, ++jb) {
        if (jb == kWarp) {
            jb = 0;
            my_pos = it + lane < it_end ? load_position<P>(p.positions, (it + lane) / p.chunks_per_token) : 0;
        }
        const long long t = it / p.chunks_per_token;
        const int ch = static_cast<int>(it - t * p.chunks_per_token);
        const int pb = static_cast<int>(static_cast<long long>(ch) * p.passes_per_token / p.chunks_per_token);
        const int pe = static_cast<int>(static_cast<long long>(ch + 1) * p.passes_per_token / p.chunks_per_token);

        uint4 xa[UMAX], xb[UMAX];
#pragma unroll
        for (int u = 0; u < UMAX; ++u) {
            const int h = (pb + u) * HPW + g;
            xa[u] = make_uint4(0u, 0u, 0u, 0u);
            xb[u] = xa[u];
            if ((pb + u < pe) && (h < H)) {
                const char *base = (h < p.n_qo)
                    ? p.q + t * p.q_stride_b + static_cast<long long>(h) * p.head_stride_b
                    : p.k + t * p.k_stride_b + static_cast<long long>(h - p.n_qo) * p.head_stride_b;
                xa[u] = __ldcs(reinterpret_cast<const uint4 *>(base) + va);
                xb[u] = __ldcs(reinterpret_cast<const uint4 *>(base) + vb);
            }
        }

        if (t != cur_t) {          // warp-uniform: a new token's position and cos|sin row
            cur_t = t;
            const long long pos = __shfl_sync(0xffffffffu, my_pos, jb);
            if (p.cache_len > 0) {
                tok_ok = pos >= 0 && pos < p.cache_len;
                if (!tok_ok && ch == 0 && lane == 0) {
                    atomicAdd(p.status, 1ull);
                    atomicMin(p.status + 1, static_cast<unsigned long long>(t));
                }
            }
            __syncwarp();          // every lane is done with the previous row
            if (tok_ok) {
                const float *grow = p.cache + pos * R;
                if (p.cache_vec) {
                    for (int c = lane; c < R / 4; c += kWarp)
                        reinterpret_cast<float4 *>(row)[c] = __ldg(reinterpret_cast<const float4 *>(grow) + c);
                } else {
                    for (int j = lane; j < R; j += kWarp) row[j] = __ldg(grow + j);
                }
            }
            __syncwarp();
        }
        if (!tok_ok) continue;

#pragma unroll
        for (int u = 0; u < UMAX; ++u) {
            if (pb + u >= pe) break;    // warp-uniform
            const int h = (pb + u) * HPW + g;
            const bool is_q = h < p.n_qo;
            float c8[8], s8[8];
            lean_cos_sin<MODE>(row, R, half, va, vb, split, rot_lane, c8, s8);
            const uint4 wa = lds_volatile_u4(&s_w[is_q ? 0 : 1][va]);
            const uint4 wb = lds_volatile_u4(&s_w[is_q ? 0 : 1][vb]);
            qknr_head<T, MODE, LPH>(xa[u], xb[u], wa, wb, c8, s8, split, rot_lane, half, p.inv_d, p.eps);
            if (h < H) {
                char *dst = is_q ? p.q + t * p.q_stride_b + static_cast<long long>(h) * p.head_stride_b
                                 : p.k + t * p.k_stride_b + static_cast<long long>(h - p.n_qo) * p.head_stride_b;
                __stcs(reinterpret_cast<uint4 *>(dst) + va, xa[u]);
                __stcs(reinterpret_cast<uint4 *>(dst) + vb, xb[u]);
            }
        }
    }
}

}  // namespace qknr
