// qknr_inst_ring_bf16.cu -- explicit instantiations of the ring kernel for bf16 storage.
// A translation unit of its own so that it compiles in parallel with the others.
#include "qknr_dispatch.h"
#include "qknr_ring_table.cuh"

namespace qknr {

const void *ring_kernel_bf16(int pos64, int d_idx, int mode, int r_idx) {
    return RingTable<__nv_bfloat16>::get<false>(pos64, d_idx, mode, r_idx);
}

}  // namespace qknr
