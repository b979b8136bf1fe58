// qknr_inst_ring_bf16_early.cu -- the ring kernel for bf16 storage with EARLY set (weights and
// positions read before waiting for the previous grid; the caller's
// QKNR_INPUTS_READY promise). A translation unit of its own so that it
// compiles in parallel with the others.
#include "qknr_dispatch.h"
#include "qknr_ring_table.cuh"

namespace qknr {

const void *ring_kernel_bf16_early(int pos64, int d_idx, int mode, int r_idx) {
    return RingTable<__nv_bfloat16>::get<true>(pos64, d_idx, mode, r_idx);
}

}  // namespace qknr
