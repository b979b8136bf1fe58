"""CPU oracle for the fused per-head QK RMSNorm + RoPE op (double precision).

TEST INFRASTRUCTURE: imported only by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``. The product path never imports it,
and it imports nothing from the product package.

The arithmetic lives in ``qknr_oracle.c`` (plain C, double precision, one head
at a time, straight from the formulas of the fused_inplace_qknorm_rope
deep-dive §2.1-§2.3). This module builds it with gcc, loads it with ctypes and
marshals torch CPU tensors into it. Every function here is pinned by
``tests/test_oracle.py`` against hand-derived values, closed forms, invariants
and an independent complex-exponential evaluation of the rotation.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "qknr_oracle.c")
LIBRARY = os.path.join(_HERE, "libqknr_oracle.so")

# tensor-contract codes (the C ABI's values, restated here on purpose)
BF16, FP16, POS_I64 = 0, 1, 0x100

_lib: Optional[ctypes.CDLL] = None


def build(force: bool = False, source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile the oracle into a shared library (gcc, -O2, no fast-math)."""
    if (not force and os.path.exists(output)
            and os.path.getmtime(output) >= os.path.getmtime(source)):
        return output
    tmp = output + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
                    "-ffp-contract=off", "-o", tmp, source, "-lm"], check=True)
    os.replace(tmp, output)
    return output


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the oracle library (building it first if needed)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(LIBRARY))
    return _lib


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.qknr_oracle_decode.argtypes = [i32, ctypes.c_uint16]
    lib.qknr_oracle_decode.restype = ctypes.c_double
    lib.qknr_oracle_head.argtypes = [vp, vp, vp, vp, i32, i32, i32, ctypes.c_double, i32, vp]
    lib.qknr_oracle_head.restype = i32
    lib.qknr_oracle_apply.argtypes = [vp, vp, vp, vp, vp, i64, vp, i64, i32, i32, i32, i32, i32,
                                      i64, i64, i64, ctypes.c_float, i32, vp, vp]
    lib.qknr_oracle_apply.restype = i32
    return lib


def dtype_code(dt: torch.dtype, pos_dt: torch.dtype = torch.int32) -> int:
    code = {torch.bfloat16: BF16, torch.float16: FP16}[dt]
    if pos_dt == torch.int64:
        code |= POS_I64
    return code


def decode(dtype: int, bits: int, lib: Optional[ctypes.CDLL] = None) -> float:
    return (lib or load()).qknr_oracle_decode(dtype, bits)


def apply(q: torch.Tensor, k: torch.Tensor, q_w: torch.Tensor, k_w: torch.Tensor,
          cos_sin_cache: torch.Tensor, positions: torch.Tensor, *, is_neox: bool,
          eps: float, rope_dim: int = 0, lib: Optional[ctypes.CDLL] = None
          ) -> Tuple[np.ndarray, np.ndarray]:
    """Evaluate the op on CPU tensors; returns unrounded float64 outputs
    q_out [T, n_qo, D] and k_out [T, n_kv, D]. Inputs are not modified."""
    lib = lib or load()
    for t in (q, k, q_w, k_w, cos_sin_cache, positions):
        assert t.device.type == "cpu"
    T, n_qo, D = q.shape
    n_kv = k.shape[1]
    assert k.shape[0] == T and k.shape[2] == D
    assert q.stride(2) == 1 and k.stride(2) == 1
    if n_qo > 1 and n_kv > 1:
        assert q.stride(1) == k.stride(1), "q and k share one head stride"
    head_stride = q.stride(1) if n_qo > 1 else k.stride(1)
    R = rope_dim or cos_sin_cache.shape[-1]
    cache = cos_sin_cache.contiguous()
    assert cache.dtype == torch.float32 and cache.shape[1] == R
    pos = positions.contiguous()
    qw, kw = q_w.contiguous(), k_w.contiguous()
    q_out = np.zeros((T, n_qo, D), dtype=np.float64)
    k_out = np.zeros((T, n_kv, D), dtype=np.float64)
    rc = lib.qknr_oracle_apply(
        q.data_ptr(), k.data_ptr(), qw.data_ptr(), kw.data_ptr(), cache.data_ptr(),
        cache.shape[0], pos.data_ptr(), T, n_qo, n_kv, D, R, int(bool(is_neox)),
        q.stride(0), k.stride(0), head_stride, eps, dtype_code(q.dtype, pos.dtype),
        q_out.ctypes.data, k_out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return q_out, k_out


def head(x: torch.Tensor, w: torch.Tensor, cos_row: torch.Tensor, sin_row: torch.Tensor, *,
         is_neox: bool, eps: float, lib: Optional[ctypes.CDLL] = None) -> np.ndarray:
    """One head x [D] with weight w [D] and half-rows cos/sin [R/2] (fp32)."""
    lib = lib or load()
    x, w = x.contiguous(), w.contiguous()
    c = cos_row.contiguous().to(torch.float32)
    s = sin_row.contiguous().to(torch.float32)
    D, R = x.shape[0], 2 * c.shape[0]
    out = np.zeros(D, dtype=np.float64)
    code = dtype_code(x.dtype)
    # eps is an fp32 argument of the op; widen the fp32 value, as the whole-op entry does
    rc = lib.qknr_oracle_head(x.data_ptr(), w.data_ptr(), c.data_ptr(), s.data_ptr(), D, R,
                              int(bool(is_neox)), float(np.float32(eps)), code, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected the head (code {rc})")
    return out


def tolerance(expected: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Parity bound: 2 ulp-equivalents of the output dtype, relative to the
    oracle value, plus 1e-5 absolute (2^-7 for bf16, 2^-10 for fp16)."""
    rel = 2.0 ** -7 if dtype == torch.bfloat16 else 2.0 ** -10
    return rel * np.abs(expected) + 1e-5


def max_violation(got: np.ndarray, expected: np.ndarray, dtype: torch.dtype) -> float:
    """max(|got - expected| / tol(expected)); <= 1 means within tolerance."""
    err = np.abs(np.asarray(got, dtype=np.float64) - expected)
    return float(np.max(err / tolerance(expected, dtype))) if err.size else 0.0
