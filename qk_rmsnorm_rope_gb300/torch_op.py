"""PyTorch custom-op registration of the fused op.

Importing this module registers ``torch.ops.qknr.fused_inplace_qknorm_rope``.
As on the fused_inplace_qknorm_rope deep-dive (§5.3), the op is declared to
mutate q and k and to return nothing, so graph capture (torch.compile,
functionalization) sees the in-place update instead of reusing stale q/k; a
fake implementation lets it trace without running the kernel. The call itself
is the library's C ABI through ``qk_rmsnorm_rope_gb300.apply``.

``can_use_fused_inplace_qknorm_rope`` is the shape gate of §5.2 for this
library's kernels (the library accepts a superset of the page's set); it is
marked as a compile-time constant for torch.compile, as the page does.
"""
from __future__ import annotations

import torch

from . import QKNR_BF16, QKNR_FP16, apply, qknr_can_use

__all__ = ["fused_inplace_qknorm_rope", "can_use_fused_inplace_qknorm_rope"]


@torch.library.custom_op("qknr::fused_inplace_qknorm_rope", mutates_args=("q", "k"))
def fused_inplace_qknorm_rope(q: torch.Tensor, k: torch.Tensor, q_weight: torch.Tensor,
                              k_weight: torch.Tensor, cos_sin_cache: torch.Tensor,
                              positions: torch.Tensor, is_neox: bool, eps: float = 1e-6,
                              head_dim: int = 0, rope_dim: int = 0,
                              inputs_ready: bool = False) -> None:
    apply(q, k, q_weight, k_weight, cos_sin_cache, positions, is_neox=is_neox, eps=eps,
          head_dim=head_dim, rope_dim=rope_dim, inputs_ready=inputs_ready)


@fused_inplace_qknorm_rope.register_fake
def _fused_inplace_qknorm_rope_fake(q, k, q_weight, k_weight, cos_sin_cache, positions,
                                    is_neox, eps=1e-6, head_dim=0, rope_dim=0,
                                    inputs_ready=False) -> None:
    return None


@torch.compiler.assume_constant_result
def can_use_fused_inplace_qknorm_rope(head_dim: int, rope_dim: int, is_neox: bool,
                                      dtype: torch.dtype) -> bool:
    if dtype not in (torch.bfloat16, torch.float16):
        return False
    code = QKNR_BF16 if dtype == torch.bfloat16 else QKNR_FP16
    return bool(qknr_can_use(head_dim, rope_dim, int(is_neox), code))
