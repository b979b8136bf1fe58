// qknr_inst_bf16_early.cu -- the register kernel for bf16 storage with EARLY set
// (weights and positions read before waiting for the previous grid; the
// caller's QKNR_INPUTS_READY promise). A translation unit of its own so that
// it compiles in parallel with the others.
#include "qknr_register_table.cuh"

namespace qknr {

const void *kernel_bf16_early(int pos64, int d_idx, int mode, int u_idx, int r_idx) {
    return RegisterTable<__nv_bfloat16, true>::get(pos64, d_idx, mode, u_idx, r_idx);
}

}  // namespace qknr
