// qknr_dispatch.h -- kernel table shared by the instantiation units and the C ABI.
#pragma once

namespace qknr {

// Unroll classes: the kernel keeps up to UMAX warp passes of loads in flight.
constexpr int kNumUnroll = 2;
constexpr int kUnrollClass[kNumUnroll] = {2, 4};

// rope_dim classes: taken at run time, or fixed at compile time to head_dim or
// head_dim / 2 (interleaved pairing, 4-pass items, head_dim 64 / 128 / 256)
constexpr int kRopeRuntime = 0, kRopeFull = 1, kRopeHalf = 2;
constexpr int kNumRope = 3;

// head_dim classes (80, 96 and 192 pad their lane groups to a power of two)
constexpr int kNumHeadDim = 6;
constexpr int kHeadDims[kNumHeadDim] = {64, 96, 128, 192, 256, 80};

// Kernel entry for (position type, head_dim class, mode, unroll class, rope_dim
// class), or nullptr. Defined in qknr_inst_bf16.cu / qknr_inst_fp16.cu.
const void *kernel_bf16(int pos64, int d_idx, int mode, int u_idx, int r_idx);
const void *kernel_fp16(int pos64, int d_idx, int mode, int u_idx, int r_idx);
// The same with the weights and positions read before waiting for the previous
// grid (QKNR_INPUTS_READY). Defined in qknr_inst_{bf16,fp16}_early.cu.
const void *kernel_bf16_early(int pos64, int d_idx, int mode, int u_idx, int r_idx);
const void *kernel_fp16_early(int pos64, int d_idx, int mode, int u_idx, int r_idx);

// Ring kernel entry for (position type, head_dim class, mode, rope_dim class),
// or nullptr; items of at most four warp passes. Defined in
// qknr_inst_ring_{bf16,fp16}[_early].cu.
const void *ring_kernel_bf16(int pos64, int d_idx, int mode, int r_idx);
const void *ring_kernel_fp16(int pos64, int d_idx, int mode, int r_idx);
const void *ring_kernel_bf16_early(int pos64, int d_idx, int mode, int r_idx);
const void *ring_kernel_fp16_early(int pos64, int d_idx, int mode, int r_idx);

// One step of the unfused two-kernel baseline (op = kOpNorm or kOpRope), the
// register kernel with 4 passes per item. Norm-only ignores pos64 and mode.
const void *unfused_kernel_bf16(int op, int pos64, int d_idx, int mode);
const void *unfused_kernel_fp16(int op, int pos64, int d_idx, int mode);

}  // namespace qknr
