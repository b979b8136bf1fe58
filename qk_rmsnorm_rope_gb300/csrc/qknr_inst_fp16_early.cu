// qknr_inst_fp16_early.cu -- the register kernel for fp16 storage with EARLY set
// (weights and positions read before waiting for the previous grid; the
// caller's QKNR_INPUTS_READY promise). A translation unit of its own so that
// it compiles in parallel with the others.
#include "qknr_register_table.cuh"

namespace qknr {

const void *kernel_fp16_early(int pos64, int d_idx, int mode, int u_idx, int r_idx) {
    return RegisterTable<__half, true>::get(pos64, d_idx, mode, u_idx, r_idx);
}

}  // namespace qknr
