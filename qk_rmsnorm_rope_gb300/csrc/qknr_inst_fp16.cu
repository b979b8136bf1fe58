// qknr_inst_fp16.cu -- explicit instantiations of the fused kernels (register and bulk-copy ring) for fp16 storage.
#include "qknr_dispatch.h"
#include "qknr_async_kernel.cuh"
#include "qknr_bulk_kernel.cuh"
#include "qknr_kernel.cuh"
#include "qknr_lean_kernel.cuh"
#include "qknr_register_table.cuh"

namespace qknr {
namespace {

template <class P, int D>
const void *bulk_by_mode(int mode) {
    return mode == kNeox ? reinterpret_cast<const void *>(&qknr_bulk_kernel<__half, P, D, kNeox>)
                         : reinterpret_cast<const void *>(&qknr_bulk_kernel<__half, P, D, kInterleaved>);
}

template <class P>
const void *bulk_by_head_dim(int d_idx, int mode) {
    switch (d_idx) {   // head_dim 80 / 96 / 192: register kernel only
        case 0: return bulk_by_mode<P, 64>(mode);
        case 2: return bulk_by_mode<P, 128>(mode);
        case 4: return bulk_by_mode<P, 256>(mode);
        default: return nullptr;
    }
}

template <int D>
const void *unfused_by_op(int op, int pos64, int mode) {
    if (op == kOpNorm)
        return reinterpret_cast<const void *>(&qknr_fused_kernel<__half, int, D, kInterleaved, 4, kOpNorm>);
    if (op != kOpRope) return nullptr;
    if (pos64)
        return mode == kNeox
                   ? reinterpret_cast<const void *>(&qknr_fused_kernel<__half, long long, D, kNeox, 4, kOpRope>)
                   : reinterpret_cast<const void *>(&qknr_fused_kernel<__half, long long, D, kInterleaved, 4, kOpRope>);
    return mode == kNeox ? reinterpret_cast<const void *>(&qknr_fused_kernel<__half, int, D, kNeox, 4, kOpRope>)
                         : reinterpret_cast<const void *>(&qknr_fused_kernel<__half, int, D, kInterleaved, 4, kOpRope>);
}

template <class P, int D>
const void *async_by_mode(int mode) {
    return mode == kNeox ? reinterpret_cast<const void *>(&qknr_async_kernel<__half, P, D, kNeox>)
                         : reinterpret_cast<const void *>(&qknr_async_kernel<__half, P, D, kInterleaved>);
}

template <class P>
const void *async_by_head_dim(int d_idx, int mode) {
    switch (d_idx) {   // head_dim 80 / 96 / 192: register kernel only
        case 0: return async_by_mode<P, 64>(mode);
        case 2: return async_by_mode<P, 128>(mode);
        case 4: return async_by_mode<P, 256>(mode);
        default: return nullptr;
    }
}

template <class P, int D>
const void *lean_by_mode(int mode) {
    return mode == kNeox ? reinterpret_cast<const void *>(&qknr_lean_kernel<__half, P, D, kNeox>)
                         : reinterpret_cast<const void *>(&qknr_lean_kernel<__half, P, D, kInterleaved>);
}

template <class P>
const void *lean_by_head_dim(int d_idx, int mode) {
    switch (d_idx) {   // head_dim 80 / 96 / 192: register kernel only
        case 0: return lean_by_mode<P, 64>(mode);
        case 2: return lean_by_mode<P, 128>(mode);
        case 4: return lean_by_mode<P, 256>(mode);
        default: return nullptr;
    }
}

}  // namespace

const void *lean_kernel_fp16(int pos64, int d_idx, int mode) {
    return pos64 ? lean_by_head_dim<long long>(d_idx, mode) : lean_by_head_dim<int>(d_idx, mode);
}

const void *async_kernel_fp16(int pos64, int d_idx, int mode) {
    return pos64 ? async_by_head_dim<long long>(d_idx, mode) : async_by_head_dim<int>(d_idx, mode);
}

const void *unfused_kernel_fp16(int op, int pos64, int d_idx, int mode) {
    switch (d_idx) {
        case 0: return unfused_by_op<64>(op, pos64, mode);
        case 1: return unfused_by_op<96>(op, pos64, mode);
        case 2: return unfused_by_op<128>(op, pos64, mode);
        case 3: return unfused_by_op<192>(op, pos64, mode);
        case 4: return unfused_by_op<256>(op, pos64, mode);
        case 5: return unfused_by_op<80>(op, pos64, mode);
        default: return nullptr;
    }
}

const void *bulk_kernel_fp16(int pos64, int d_idx, int mode) {
    return pos64 ? bulk_by_head_dim<long long>(d_idx, mode) : bulk_by_head_dim<int>(d_idx, mode);
}

const void *kernel_fp16(int pos64, int d_idx, int mode, int u_idx) {
    return RegisterTable<__half, false>::get(pos64, d_idx, mode, u_idx);
}

}  // namespace qknr
