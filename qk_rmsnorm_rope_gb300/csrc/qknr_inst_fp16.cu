// qknr_inst_fp16.cu -- explicit instantiations of the register kernel for fp16 storage: the fused op
// (default reads) and the two steps of the unfused baseline.
#include "qknr_dispatch.h"
#include "qknr_kernel.cuh"
#include "qknr_register_table.cuh"

namespace qknr {
namespace {

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

}  // namespace

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

const void *kernel_fp16(int pos64, int d_idx, int mode, int u_idx, int r_idx) {
    return RegisterTable<__half, false>::get(pos64, d_idx, mode, u_idx, r_idx);
}

}  // namespace qknr
