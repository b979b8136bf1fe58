// qknr_ring_table.cuh -- the ring kernel's instantiation table for one storage
// type and one choice of EARLY: the kernel entry for (position type, head_dim
// class, pairing, rope_dim class).
#pragma once

#include "qknr_dispatch.h"
#include "qknr_ring_kernel.cuh"

namespace qknr {

template <class T>
struct RingTable {
    template <bool EARLY, class P, int D, int MODE, int RC>
    static const void *entry() {
        return reinterpret_cast<const void *>(&qknr_ring_kernel<T, P, D, MODE, EARLY, RC>);
    }
    // rope_dim fixed at head_dim or head_dim / 2 exists for interleaved pairing
    // and head_dim 64, 128 and 256 only (nullptr elsewhere), as for the
    // register kernel
    template <bool EARLY, class P, int D, int MODE>
    static const void *by_rope(int r_idx) {
        if (r_idx == kRopeRuntime) return entry<EARLY, P, D, MODE, 0>();
        if constexpr (MODE == kInterleaved && (D == 64 || D == 128 || D == 256)) {
            return r_idx == kRopeFull ? entry<EARLY, P, D, MODE, D>() : entry<EARLY, P, D, MODE, D / 2>();
        }
        return nullptr;
    }
    template <bool EARLY, class P, int D>
    static const void *by_mode(int mode, int r_idx) {
        return mode == kNeox ? by_rope<EARLY, P, D, kNeox>(r_idx) : by_rope<EARLY, P, D, kInterleaved>(r_idx);
    }
    template <bool EARLY, class P>
    static const void *by_head_dim(int d_idx, int mode, int r_idx) {
        switch (d_idx) {   // the order of kHeadDims
            case 0: return by_mode<EARLY, P, 64>(mode, r_idx);
            case 1: return by_mode<EARLY, P, 96>(mode, r_idx);
            case 2: return by_mode<EARLY, P, 128>(mode, r_idx);
            case 3: return by_mode<EARLY, P, 192>(mode, r_idx);
            case 4: return by_mode<EARLY, P, 256>(mode, r_idx);
            case 5: return by_mode<EARLY, P, 80>(mode, r_idx);
            default: return nullptr;
        }
    }
    template <bool EARLY>
    static const void *get(int pos64, int d_idx, int mode, int r_idx) {
        return pos64 ? by_head_dim<EARLY, long long>(d_idx, mode, r_idx) : by_head_dim<EARLY, int>(d_idx, mode, r_idx);
    }
};

}  // namespace qknr
