// qknr_register_table.cuh -- the register kernel's instantiation table for one
// storage type and one choice of EARLY (see qknr_kernel.cuh): the kernel entry
// for (position type, head_dim class, pairing, unroll class, rope_dim class).
#pragma once

#include "qknr_dispatch.h"
#include "qknr_kernel.cuh"

namespace qknr {

template <class T, bool EARLY>
struct RegisterTable {
    template <class P, int D, int MODE, int U, int RC = 0>
    static const void *entry() {
        return reinterpret_cast<const void *>(&qknr_fused_kernel<T, P, D, MODE, U, kOpFused, EARLY, RC>);
    }
    // rope_dim class: kRopeRuntime, or rope_dim fixed at head_dim (kRopeFull) or
    // head_dim / 2 (kRopeHalf); the fixed ones exist for interleaved pairing with
    // 4-pass items and head_dim 64, 128 and 256 only (nullptr elsewhere).
    template <class P, int D, int MODE>
    static const void *by_unroll(int u_idx, int r_idx) {
        if (r_idx != kRopeRuntime) {
            if constexpr (MODE == kInterleaved && (D == 64 || D == 128 || D == 256)) {
                if (u_idx != 1) return nullptr;
                return r_idx == kRopeFull ? entry<P, D, MODE, 4, D>() : entry<P, D, MODE, 4, D / 2>();
            }
            return nullptr;
        }
        switch (u_idx) {
            case 0: return entry<P, D, MODE, 2>();
            case 1: return entry<P, D, MODE, 4>();
            default: return nullptr;
        }
    }
    template <class P, int D>
    static const void *by_mode(int mode, int u_idx, int r_idx) {
        return mode == kNeox ? by_unroll<P, D, kNeox>(u_idx, r_idx) : by_unroll<P, D, kInterleaved>(u_idx, r_idx);
    }
    template <class P>
    static const void *by_head_dim(int d_idx, int mode, int u_idx, int r_idx) {
        switch (d_idx) {   // the order of kHeadDims
            case 0: return by_mode<P, 64>(mode, u_idx, r_idx);
            case 1: return by_mode<P, 96>(mode, u_idx, r_idx);
            case 2: return by_mode<P, 128>(mode, u_idx, r_idx);
            case 3: return by_mode<P, 192>(mode, u_idx, r_idx);
            case 4: return by_mode<P, 256>(mode, u_idx, r_idx);
            case 5: return by_mode<P, 80>(mode, u_idx, r_idx);
            default: return nullptr;
        }
    }
    static const void *get(int pos64, int d_idx, int mode, int u_idx, int r_idx) {
        return pos64 ? by_head_dim<long long>(d_idx, mode, u_idx, r_idx)
                     : by_head_dim<int>(d_idx, mode, u_idx, r_idx);
    }
};

}  // namespace qknr
