// qknr_math.cuh -- the per-lane arithmetic of one head, in packed fp32x2.
//
// Every kernel of the library calls qknr_head for the math, so all of them
// produce the same bits. The op per head (fused_inplace_qknorm_rope deep-dive
// §2.1-§2.3): widen to fp32, sum of squares over head_dim, r = rsqrt(sum/D +
// eps), n = x * (w * r), rotate the first rope_dim dims with the token's cos
// and sin, round once to the storage type.
//
// On sm_100+ the FMA pipe executes two fp32 operations per instruction
// (__ffma2_rn / __fmul2_rn, round to nearest like their scalar forms). The op
// is close to instruction-issue bound on GB300 at full HBM bandwidth, so the
// lane's 16 elements are kept as 8 float2 pairs arranged so that every step
// pairs up:
//   interleaved: v[0] = (a0, a2), v[1] = (a1, a3), v[2] = (a4, a6), v[3] = (a5, a7)
//                (a = vector a; v[4..7] the same for vector b). A rotation pair
//                (2j, 2j+1) then sits at the same slot of v[2i] and v[2i+1].
//   NeoX:        v[k] = (a_{2k}, a_{2k+1}), v[4+k] = (b_{2k}, b_{2k+1}). With the
//                split lane layout, element e of vector a and element e of
//                vector b form a rotation pair, i.e. slot-wise v[k] and v[4+k].
// Either way a rotation step is (X, Y) -> (X*C - Y*S, Y*C + X*S) on whole pairs.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace qknr {

enum Mode : int { kInterleaved = 0, kNeox = 1 };

// What a launch computes: the fused op, or one half of the unfused two-kernel
// chain the fused op replaces (RMSNorm alone, then RoPE alone, each in place).
enum Op : int { kOpFused = 0, kOpNorm = 1, kOpRope = 2 };

template <class T>
struct Cvt;

template <>
struct Cvt<__nv_bfloat16> {
    // bf16 -> fp32 is exact: the 16 bits become the high half of a float.
    static __device__ __forceinline__ float lo(uint32_t u) { return __uint_as_float(u << 16); }
    static __device__ __forceinline__ float hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
    static __device__ __forceinline__ uint32_t pack(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // round to nearest even; a -> low half
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

template <>
struct Cvt<__half> {
    static __device__ __forceinline__ float lo(uint32_t u) {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(u & 0xffffu)));
    }
    static __device__ __forceinline__ float hi(uint32_t u) {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(u >> 16)));
    }
    static __device__ __forceinline__ uint32_t pack(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

// 8 storage elements (one 16-byte vector) -> 4 pairs in the mode's arrangement.
template <class T, int MODE>
__device__ __forceinline__ void unpack_pairs(const uint4 &x, float2 *v) {
    if (MODE == kInterleaved) {
        v[0] = make_float2(Cvt<T>::lo(x.x), Cvt<T>::lo(x.y));
        v[1] = make_float2(Cvt<T>::hi(x.x), Cvt<T>::hi(x.y));
        v[2] = make_float2(Cvt<T>::lo(x.z), Cvt<T>::lo(x.w));
        v[3] = make_float2(Cvt<T>::hi(x.z), Cvt<T>::hi(x.w));
    } else {
        v[0] = make_float2(Cvt<T>::lo(x.x), Cvt<T>::hi(x.x));
        v[1] = make_float2(Cvt<T>::lo(x.y), Cvt<T>::hi(x.y));
        v[2] = make_float2(Cvt<T>::lo(x.z), Cvt<T>::hi(x.z));
        v[3] = make_float2(Cvt<T>::lo(x.w), Cvt<T>::hi(x.w));
    }
}

template <class T, int MODE>
__device__ __forceinline__ uint4 pack_pairs(const float2 *v) {
    uint4 x;
    if (MODE == kInterleaved) {
        x.x = Cvt<T>::pack(v[0].x, v[1].x);
        x.y = Cvt<T>::pack(v[0].y, v[1].y);
        x.z = Cvt<T>::pack(v[2].x, v[3].x);
        x.w = Cvt<T>::pack(v[2].y, v[3].y);
    } else {
        x.x = Cvt<T>::pack(v[0].x, v[0].y);
        x.y = Cvt<T>::pack(v[1].x, v[1].y);
        x.z = Cvt<T>::pack(v[2].x, v[2].y);
        x.w = Cvt<T>::pack(v[3].x, v[3].y);
    }
    return x;
}

// element e (0..7) of a 16-byte vector held as pairs, and its inverse
template <int MODE>
__device__ __forceinline__ float &pair_elem(float2 *v, int e) {
    if (MODE == kInterleaved) {
        float2 &p = v[(e >> 2) * 2 + (e & 1)];
        return ((e >> 1) & 1) ? p.y : p.x;
    }
    float2 &p = v[e >> 1];
    return (e & 1) ? p.y : p.x;
}

// (X, Y) -> (X*C - Y*S, Y*C + X*S), slot by slot
__device__ __forceinline__ void rotate_pair(float2 &x, float2 &y, float2 c, float2 s) {
    const float2 x0 = x;
    const float2 ys = __fmul2_rn(y, s);
    const float2 yc = __fmul2_rn(y, c);
    x = __ffma2_rn(x0, c, make_float2(-ys.x, -ys.y));
    y = __ffma2_rn(x0, s, yc);
}

// NeoX with rope_dim <= 8: every rotated dim is in vector a, pairs (e, e+HALF).
template <int HALF>
__device__ __forceinline__ void rotate_small_neox(float2 *va, const float (&c)[8], const float (&s)[8]) {
#pragma unroll
    for (int e = 0; e < HALF; ++e) {
        const float x0 = pair_elem<kNeox>(va, e), x1 = pair_elem<kNeox>(va, e + HALF);
        pair_elem<kNeox>(va, e) = x0 * c[e] - x1 * s[e];
        pair_elem<kNeox>(va, e + HALF) = x1 * c[e] + x0 * s[e];
    }
}

// One head slot of a warp pass for this lane: xa, xb are the lane's two
// 16-byte vectors (storage type) and are replaced by the output. wa, wb are
// the lane's slices of the head's weight vector (storage type). c8, s8: the
// token's cos / sin for the lane's rotated elements in the order the mode's
// pairs need them (interleaved: pair m of vector a at [m], of vector b at
// [4+m]; NeoX split: element e at [e]; NeoX with rope_dim <= 8: element e of
// vector a at [e]); (1, 0) where nothing rotates. Every lane of the warp must
// call it (the sum of squares is reduced across the head's LPH lanes).
template <class T, int MODE, int LPH, int OP = kOpFused>
__device__ __forceinline__ void qknr_head(uint4 &xa, uint4 &xb, const uint4 &wa, const uint4 &wb,
                                          const float (&c8)[8], const float (&s8)[8], bool split,
                                          bool rot_lane, int half, float inv_d, float eps) {
    float2 v[8];
    unpack_pairs<T, MODE>(xa, v);
    unpack_pairs<T, MODE>(xb, v + 4);
    if (OP != kOpRope) {
        float2 acc0 = __fmul2_rn(v[0], v[0]);
        float2 acc1 = __fmul2_rn(v[1], v[1]);
        acc0 = __ffma2_rn(v[2], v[2], acc0);
        acc1 = __ffma2_rn(v[3], v[3], acc1);
        acc0 = __ffma2_rn(v[4], v[4], acc0);
        acc1 = __ffma2_rn(v[5], v[5], acc1);
        acc0 = __ffma2_rn(v[6], v[6], acc0);
        acc1 = __ffma2_rn(v[7], v[7], acc1);
        const float2 acc = __fadd2_rn(acc0, acc1);
        float ss = acc.x + acc.y;
#pragma unroll
        for (int off = LPH / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float r = rsqrtf(fmaf(ss, inv_d, eps));
        const float2 rr = make_float2(r, r);
        float2 w[8];
        unpack_pairs<T, MODE>(wa, w);
        unpack_pairs<T, MODE>(wb, w + 4);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __fmul2_rn(v[k], __fmul2_rn(w[k], rr));
    }
    if (OP != kOpNorm) {
        if (MODE == kInterleaved) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                rotate_pair(v[2 * i], v[2 * i + 1], make_float2(c8[2 * i], c8[2 * i + 1]),
                            make_float2(s8[2 * i], s8[2 * i + 1]));
        } else if (split) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                rotate_pair(v[k], v[4 + k], make_float2(c8[2 * k], c8[2 * k + 1]),
                            make_float2(s8[2 * k], s8[2 * k + 1]));
        } else if (rot_lane) {
            switch (half) {
                case 1: rotate_small_neox<1>(v, c8, s8); break;
                case 2: rotate_small_neox<2>(v, c8, s8); break;
                case 3: rotate_small_neox<3>(v, c8, s8); break;
                default: rotate_small_neox<4>(v, c8, s8); break;
            }
        }
    }
    xa = pack_pairs<T, MODE>(v);
    xb = pack_pairs<T, MODE>(v + 4);
}

}  // namespace qknr
