// qknr_inst_fp16.cu -- explicit instantiations of the fused kernel for fp16 storage.
#include "qknr_dispatch.h"
#include "qknr_kernel.cuh"

namespace qknr {
namespace {

template <class P, int D, int MODE, int U>
const void *entry() {
    return reinterpret_cast<const void *>(&qknr_fused_kernel<__half, P, D, MODE, U>);
}

template <class P, int D, int MODE>
const void *by_unroll(int u_idx) {
    switch (u_idx) {
        case 0: return entry<P, D, MODE, 2>();
        case 1: return entry<P, D, MODE, 4>();
        default: return nullptr;
    }
}

template <class P, int D>
const void *by_mode(int mode, int u_idx) {
    return mode == kNeox ? by_unroll<P, D, kNeox>(u_idx) : by_unroll<P, D, kInterleaved>(u_idx);
}

template <class P>
const void *by_head_dim(int d_idx, int mode, int u_idx) {
    switch (d_idx) {
        case 0: return by_mode<P, 64>(mode, u_idx);
        case 1: return by_mode<P, 128>(mode, u_idx);
        case 2: return by_mode<P, 256>(mode, u_idx);
        default: return nullptr;
    }
}

}  // namespace

const void *kernel_fp16(int pos64, int d_idx, int mode, int u_idx) {
    return pos64 ? by_head_dim<long long>(d_idx, mode, u_idx) : by_head_dim<int>(d_idx, mode, u_idx);
}

}  // namespace qknr
