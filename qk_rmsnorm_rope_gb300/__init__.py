"""Fused in-place per-head QK RMSNorm + RoPE on GB300 (sm_103a).

Thin Python binding over ``libqknr.so`` (C ABI in ``include/qknr.h``). The
``qknr_*`` functions mirror the C entry points one to one and take raw device
pointers; ``apply`` / ``apply_checked`` marshal torch CUDA tensors into them
the way the fused_inplace_qknorm_rope deep-dive's Python op does (§5.3:
head_dim defaults to q.size(-1), rope_dim to cos_sin_cache.size(-1); the op
returns None and mutates q and k). Every computation runs in the library's
CUDA kernels; there is no other code path. The library is loaded at first
use, and that use raises ImportError when it has not been built (so that the
build step itself can import this package).
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

__all__ = [
    "QKNR_BF16", "QKNR_FP16", "QKNR_POS_I64", "QKNR_INPUTS_READY", "QKNR_HOST_AUTO", "QKNR_HOST_STAGED",
    "QKNR_HOST_DIRECT", "QknrError", "library_path",
    "qknr_init", "qknr_shutdown", "qknr_last_error", "qknr_version", "qknr_can_use",
    "qknr_apply", "qknr_apply_checked", "qknr_apply_checked_noalloc", "qknr_apply_unfused",
    "qknr_apply_host", "qknr_apply_strided", "qknr_tune",
    "qknr_set_tuning", "qknr_get_tuning", "qknr_query_work_map", "TUNE_KEYS",
    "init", "apply", "apply_checked", "apply_unfused", "apply_host", "can_use", "dtype_code",
    "work_map", "set_tuning", "get_tuning", "tune",
]

QKNR_BF16 = 0x000
QKNR_FP16 = 0x001
QKNR_POS_I64 = 0x100
QKNR_INPUTS_READY = 0x200   # caller's promise: weights and positions are not written by the kernel just before

STATUS_NAMES = {
    0: "QKNR_OK", 1: "QKNR_ERR_NOT_INITIALIZED", 2: "QKNR_ERR_INVALID_ARG",
    3: "QKNR_ERR_UNSUPPORTED", 4: "QKNR_ERR_MISALIGNED", 5: "QKNR_ERR_CUDA",
    6: "QKNR_ERR_POSITION_OOB",
}

QKNR_KERNEL_AUTO, QKNR_KERNEL_REGISTER, QKNR_KERNEL_RING = 0, 1, 2
KERNEL_NAMES = {QKNR_KERNEL_REGISTER: "register", QKNR_KERNEL_RING: "ring"}
QKNR_HOST_AUTO, QKNR_HOST_STAGED, QKNR_HOST_DIRECT = 0, 1, 2
HOST_MODES = {"auto": QKNR_HOST_AUTO, "staged": QKNR_HOST_STAGED, "direct": QKNR_HOST_DIRECT}
# QKNR_TUNE_* keys (include/qknr.h)
TUNE_KEYS = {"reset": 0, "kernel": 1, "passes": 2, "threads": 3, "ctas_per_sm": 4, "pdl": 5,
             "ring_order": 6, "order": 9, "prefetch": 10}
WORK_MAP_FIELDS = ["kernel", "grid", "threads", "items", "items_per_token", "ctas_per_sm", "pdl",
                   "passes_per_token", "unroll", "order", "prefetch_items", "rope_dim_compiled",
                   "ring_order"]

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "libqknr.so")


class QknrError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {message}")
        self.code = code
        self.message = message


def _load() -> ctypes.CDLL:
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m qk_rmsnorm_rope_gb300.build` "
            "(nvcc for sm_103a). There is no fallback implementation.")
    lib = ctypes.CDLL(path)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.qknr_init.argtypes = [i32]
    lib.qknr_shutdown.argtypes = []
    lib.qknr_last_error.argtypes = []
    lib.qknr_last_error.restype = ctypes.c_char_p
    lib.qknr_version.argtypes = []
    lib.qknr_can_use.argtypes = [i32, i32, i32, i32]
    lib.qknr_apply.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32,
                               i64, i64, i64, f32, i32, vp]
    lib.qknr_apply_checked.argtypes = [vp, vp, vp, vp, vp, i64, vp, i64, i32, i32, i32, i32, i32,
                                       i64, i64, i64, f32, i32, vp]
    lib.qknr_apply_checked_noalloc.argtypes = lib.qknr_apply_checked.argtypes
    lib.qknr_apply_unfused.argtypes = lib.qknr_apply.argtypes
    lib.qknr_apply_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32,
                                    i64, i64, i64, f32, i32, i64, i32, vp]
    lib.qknr_apply_strided.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32,
                                       i64, i64, i64, i64, f32, i32, vp]
    lib.qknr_tune.argtypes = [i64, i32, i32, i32, i32, i32, i64, i64, i64, i32, vp,
                              ctypes.POINTER(ctypes.c_int64)]
    lib.qknr_set_tuning.argtypes = [i32, i32]
    lib.qknr_get_tuning.argtypes = [i32, ctypes.POINTER(ctypes.c_int)]
    lib.qknr_query_work_map.argtypes = [i64, i32, i32, i32, i32, i32, i32,
                                        ctypes.POINTER(ctypes.c_int64)]
    for name in ("qknr_init", "qknr_shutdown", "qknr_version", "qknr_can_use", "qknr_apply",
                 "qknr_apply_checked", "qknr_apply_checked_noalloc", "qknr_apply_unfused",
                 "qknr_apply_host", "qknr_apply_strided", "qknr_tune", "qknr_set_tuning", "qknr_get_tuning",
                 "qknr_query_work_map"):
        getattr(lib, name).restype = i32
    return lib


_lib: Optional[ctypes.CDLL] = None


def _get_lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def __getattr__(name: str):
    # ``qk_rmsnorm_rope_gb300.lib``: the loaded C library (raw ctypes entry points)
    if name == "lib":
        return _get_lib()
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")


def _check(rc: int) -> None:
    if rc != 0:
        raise QknrError(rc, qknr_last_error())


# --------------------------------------------------------------- raw C entry points
def qknr_init(device: int) -> int:
    return _get_lib().qknr_init(device)


def qknr_shutdown() -> int:
    return _get_lib().qknr_shutdown()


def qknr_last_error() -> str:
    return (_get_lib().qknr_last_error() or b"").decode(errors="replace")


def qknr_version() -> int:
    return _get_lib().qknr_version()


def qknr_can_use(head_dim: int, rope_dim: int, is_neox: int, dtype: int) -> int:
    return _get_lib().qknr_can_use(head_dim, rope_dim, int(is_neox), dtype)


def qknr_apply(q, k, q_w, k_w, cos_sin_cache, positions, num_tokens, n_qo, n_kv, head_dim,
               rope_dim, is_neox, q_stride, k_stride, head_stride, eps, dtype, stream) -> int:
    return _get_lib().qknr_apply(q, k, q_w, k_w, cos_sin_cache, positions, num_tokens, n_qo,
                                 n_kv, head_dim, rope_dim, int(is_neox), q_stride, k_stride,
                                 head_stride, eps, dtype, stream)


def qknr_apply_checked(q, k, q_w, k_w, cos_sin_cache, cache_len, positions, num_tokens, n_qo,
                       n_kv, head_dim, rope_dim, is_neox, q_stride, k_stride, head_stride, eps,
                       dtype, stream) -> int:
    return _get_lib().qknr_apply_checked(q, k, q_w, k_w, cos_sin_cache, cache_len, positions,
                                         num_tokens, n_qo, n_kv, head_dim, rope_dim,
                                         int(is_neox), q_stride, k_stride, head_stride, eps,
                                         dtype, stream)


def qknr_apply_checked_noalloc(q, k, q_w, k_w, cos_sin_cache, cache_len, positions, num_tokens,
                               n_qo, n_kv, head_dim, rope_dim, is_neox, q_stride, k_stride,
                               head_stride, eps, dtype, stream) -> int:
    """The allocation-free checked call (no qknr_init needed); see include/qknr.h."""
    return _get_lib().qknr_apply_checked_noalloc(q, k, q_w, k_w, cos_sin_cache, cache_len,
                                                 positions, num_tokens, n_qo, n_kv, head_dim,
                                                 rope_dim, int(is_neox), q_stride, k_stride,
                                                 head_stride, eps, dtype, stream)


def qknr_apply_unfused(q, k, q_w, k_w, cos_sin_cache, positions, num_tokens, n_qo, n_kv,
                       head_dim, rope_dim, is_neox, q_stride, k_stride, head_stride, eps, dtype,
                       stream) -> int:
    return _get_lib().qknr_apply_unfused(q, k, q_w, k_w, cos_sin_cache, positions, num_tokens,
                                         n_qo, n_kv, head_dim, rope_dim, int(is_neox), q_stride,
                                         k_stride, head_stride, eps, dtype, stream)


def qknr_apply_host(h_q, h_k, q_w, k_w, cos_sin_cache, h_positions, d_q, d_k, d_positions,
                    num_tokens, n_qo, n_kv, head_dim, rope_dim, is_neox, q_stride, k_stride,
                    head_stride, eps, dtype, chunk_tokens, flags, stream) -> int:
    return _get_lib().qknr_apply_host(h_q, h_k, q_w, k_w, cos_sin_cache, h_positions, d_q, d_k,
                                      d_positions, num_tokens, n_qo, n_kv, head_dim, rope_dim,
                                      int(is_neox), q_stride, k_stride, head_stride, eps, dtype,
                                      chunk_tokens, flags, stream)


def qknr_apply_strided(q, k, q_w, k_w, cos_sin_cache, positions, num_tokens, n_qo, n_kv,
                       head_dim, rope_dim, is_neox, q_stride, k_stride, q_head_stride,
                       k_head_stride, eps, dtype, stream) -> int:
    return _get_lib().qknr_apply_strided(q, k, q_w, k_w, cos_sin_cache, positions, num_tokens,
                                         n_qo, n_kv, head_dim, rope_dim, int(is_neox), q_stride,
                                         k_stride, q_head_stride, k_head_stride, eps, dtype, stream)


def qknr_tune(num_tokens, n_qo, n_kv, head_dim, rope_dim, is_neox, q_stride, k_stride, head_stride,
              dtype, stream, out) -> int:
    return _get_lib().qknr_tune(num_tokens, n_qo, n_kv, head_dim, rope_dim, int(is_neox), q_stride,
                                k_stride, head_stride, dtype, stream, out)


def qknr_set_tuning(key: int, value: int) -> int:
    return _get_lib().qknr_set_tuning(key, value)


def qknr_get_tuning(key: int, value) -> int:
    return _get_lib().qknr_get_tuning(key, value)


def qknr_query_work_map(num_tokens, n_qo, n_kv, head_dim, rope_dim, is_neox, dtype, out) -> int:
    return _get_lib().qknr_query_work_map(num_tokens, n_qo, n_kv, head_dim, rope_dim,
                                          int(is_neox), dtype, out)


# --------------------------------------------------------------- torch marshalling
def dtype_code(q_dtype, pos_dtype) -> int:
    import torch
    if q_dtype == torch.bfloat16:
        code = QKNR_BF16
    elif q_dtype == torch.float16:
        code = QKNR_FP16
    else:
        raise QknrError(2, f"q/k dtype {q_dtype} is not bfloat16 or float16")
    if pos_dtype == torch.int64:
        code |= QKNR_POS_I64
    elif pos_dtype != torch.int32:
        raise QknrError(2, f"positions dtype {pos_dtype} is not int32 or int64")
    return code


def init(device: Optional[int] = None) -> None:
    """qknr_init for ``device`` (default: torch's current CUDA device)."""
    import torch
    if device is None:
        device = torch.cuda.current_device()
    _check(qknr_init(int(device)))


def can_use(head_dim: int, rope_dim: int, is_neox: bool, dtype=None) -> bool:
    import torch
    code = dtype_code(dtype or torch.bfloat16, torch.int32)
    return bool(qknr_can_use(head_dim, rope_dim, int(is_neox), code))


def _as_tokens(t, name):
    """A [B, S, H, D] tensor as the [B*S, H, D] view of the same memory (the op
    works in place, so a copy would not do); 3-D tensors as they are."""
    if t.dim() == 4:
        try:
            return t.view(t.shape[0] * t.shape[1], t.shape[2], t.shape[3])
        except RuntimeError:
            raise QknrError(2, f"{name}: a 4-D tensor whose batch and sequence dims do not merge "
                               "into one token dim without a copy") from None
    return t


def _marshal(q, k, q_w, k_w, cos_sin_cache, positions, is_neox, head_dim, rope_dim,
             same_device=True, split_strides=False):
    import torch
    if q.dim() != 3 or k.dim() != 3:
        raise QknrError(2, "q and k must be [num_tokens, heads, head_dim] or [batch, seq, heads, head_dim]")
    T, n_qo, D = q.shape
    if k.shape[0] != T or k.shape[2] != D:
        raise QknrError(2, f"k shape {tuple(k.shape)} does not match q {tuple(q.shape)}")
    n_kv = k.shape[1]
    head_dim = head_dim or D
    rope_dim = rope_dim or cos_sin_cache.size(-1)
    if head_dim != D:
        raise QknrError(2, f"head_dim {head_dim} != q.size(-1) {D}")
    if cos_sin_cache.dim() != 2 or cos_sin_cache.size(-1) != rope_dim:
        raise QknrError(2, "cos_sin_cache must be [cache_len, rope_dim]")
    if cos_sin_cache.dtype != torch.float32 or not cos_sin_cache.is_contiguous():
        raise QknrError(2, "cos_sin_cache must be contiguous float32")
    if positions.dim() != 1 or positions.shape[0] != T or not positions.is_contiguous():
        raise QknrError(2, "positions must be a contiguous [num_tokens] tensor")
    for name, t in (("q", q), ("k", k)):
        if t.stride(2) != 1:
            raise QknrError(4, f"{name} must have unit innermost stride")
    if k.dtype != q.dtype or q_w.dtype != q.dtype or k_w.dtype != q.dtype:
        raise QknrError(2, "q, k, q_w and k_w must share one dtype")
    if q_w.shape != (D,) or k_w.shape != (D,) or not (q_w.is_contiguous() and k_w.is_contiguous()):
        raise QknrError(2, "q_w and k_w must be contiguous [head_dim]")
    devs = {t.device for t in ((q, k, q_w, k_w, cos_sin_cache, positions) if same_device
                               else (q_w, k_w, cos_sin_cache))}
    if len(devs) != 1 or next(iter(devs)).type != "cuda":
        raise QknrError(2, "all tensors must be on one CUDA device")
    if n_qo > 1 and n_kv > 1 and q.stride(1) != k.stride(1) and not split_strides:
        raise QknrError(2, "q and k must share one head stride")
    head_stride = q.stride(1) if n_qo > 1 else (k.stride(1) if n_kv > 1 else D)
    out = (T, n_qo, n_kv, head_dim, rope_dim, q.stride(0), k.stride(0), head_stride,
           dtype_code(q.dtype, positions.dtype))
    if split_strides:
        return out + (k.stride(1) if n_kv > 1 else head_stride,)
    return out


def _prepare(q, positions, stream):
    """The raw stream handle for a call on q's device, and positions as the op
    takes them: int32 or int64, contiguous, on q's device. Positions on another
    device, on the host or of another integer type are converted there first (as
    the page's upstream wrapper does); the call's stream then waits for that copy
    and keeps the converted tensor alive until the kernel has run."""
    import torch
    if q.device.type != "cuda":
        raise QknrError(2, "all tensors must be on one CUDA device (CPU tensors are refused: no CPU path)")
    cur = torch.cuda.current_stream(q.device)
    if stream is None:
        s_obj = cur
    elif isinstance(stream, int):
        s_obj = torch.cuda.ExternalStream(stream, device=q.device)
    else:
        s_obj = stream
    if not (positions.dtype in (torch.int32, torch.int64) and positions.device == q.device
            and positions.is_contiguous()):
        if positions.dtype.is_floating_point or positions.dtype.is_complex or positions.dtype == torch.bool:
            raise QknrError(2, f"positions must be an integer tensor, not {positions.dtype}")
        dt = torch.int32 if positions.dtype == torch.int32 else torch.int64
        with torch.cuda.device(q.device):
            positions = positions.to(device=q.device, dtype=dt).contiguous()
        if s_obj != cur:
            s_obj.wait_stream(cur)
            positions.record_stream(s_obj)
    return positions, s_obj.cuda_stream


def apply(q, k, q_w, k_w, cos_sin_cache, positions, *, is_neox: bool, eps: float = 1e-6,
          head_dim: int = 0, rope_dim: int = 0, stream=None, inputs_ready: bool = False) -> None:
    """In-place fused QK RMSNorm + RoPE on torch CUDA tensors (returns None).

    q [T, n_qo, D] and k [T, n_kv, D] (bf16/fp16, unit innermost stride; or
    [B, S, H, D] when B and S merge into one token dim without a copy) are
    overwritten. Runs on ``stream`` (a torch.cuda.Stream or raw handle),
    default torch's current stream on q's device. q and k may have different
    head strides (qknr_apply_strided); with one shared stride this is
    qknr_apply. Positions may be any integer tensor (see _prepare).
    ``inputs_ready=True`` is the caller's promise that q_w, k_w and positions
    were not written by the kernel enqueued just before on the stream
    (QKNR_INPUTS_READY): the kernel then reads them while that kernel finishes.
    """
    import torch
    q, k = _as_tokens(q, "q"), _as_tokens(k, "k")
    positions, stream = _prepare(q, positions, stream)
    T, n_qo, n_kv, D, R, qs, ks, hs, code, khs = _marshal(
        q, k, q_w, k_w, cos_sin_cache, positions, is_neox, head_dim, rope_dim, split_strides=True)
    if inputs_ready:
        code |= QKNR_INPUTS_READY
    with torch.cuda.device(q.device):
        if khs == hs:
            _check(qknr_apply(q.data_ptr(), k.data_ptr(), q_w.data_ptr(), k_w.data_ptr(),
                              cos_sin_cache.data_ptr(), positions.data_ptr(), T, n_qo, n_kv, D, R,
                              int(bool(is_neox)), qs, ks, hs, float(eps), code, stream))
        else:
            _check(qknr_apply_strided(q.data_ptr(), k.data_ptr(), q_w.data_ptr(), k_w.data_ptr(),
                                      cos_sin_cache.data_ptr(), positions.data_ptr(), T, n_qo,
                                      n_kv, D, R, int(bool(is_neox)), qs, ks, hs, khs,
                                      float(eps), code, stream))


def apply_checked(q, k, q_w, k_w, cos_sin_cache, positions, *, is_neox: bool, eps: float = 1e-6,
                  head_dim: int = 0, rope_dim: int = 0, stream=None) -> None:
    """``apply`` plus a device-side check that every position lies inside the
    cache. Synchronous; raises QknrError (QKNR_ERR_POSITION_OOB) if one does
    not, leaving those tokens untouched."""
    import torch
    q, k = _as_tokens(q, "q"), _as_tokens(k, "k")
    positions, stream = _prepare(q, positions, stream)
    T, n_qo, n_kv, D, R, qs, ks, hs, code = _marshal(q, k, q_w, k_w, cos_sin_cache, positions,
                                                      is_neox, head_dim, rope_dim)
    with torch.cuda.device(q.device):
        _check(qknr_apply_checked(q.data_ptr(), k.data_ptr(), q_w.data_ptr(), k_w.data_ptr(),
                                  cos_sin_cache.data_ptr(), cos_sin_cache.shape[0],
                                  positions.data_ptr(), T, n_qo, n_kv, D, R, int(bool(is_neox)),
                                  qs, ks, hs, float(eps), code, stream))


def apply_unfused(q, k, q_w, k_w, cos_sin_cache, positions, *, is_neox: bool, eps: float = 1e-6,
                  head_dim: int = 0, rope_dim: int = 0, stream=None) -> None:
    """The unfused two-kernel baseline (RMSNorm kernel, then RoPE kernel), in
    place; for measuring what fusion saves. See qknr_apply_unfused."""
    import torch
    q, k = _as_tokens(q, "q"), _as_tokens(k, "k")
    positions, stream = _prepare(q, positions, stream)
    T, n_qo, n_kv, D, R, qs, ks, hs, code = _marshal(q, k, q_w, k_w, cos_sin_cache, positions,
                                                      is_neox, head_dim, rope_dim)
    with torch.cuda.device(q.device):
        _check(qknr_apply_unfused(q.data_ptr(), k.data_ptr(), q_w.data_ptr(), k_w.data_ptr(),
                                  cos_sin_cache.data_ptr(), positions.data_ptr(), T, n_qo, n_kv, D,
                                  R, int(bool(is_neox)), qs, ks, hs, float(eps), code, stream))


def apply_host(h_q, h_k, q_w, k_w, cos_sin_cache, h_positions, d_q=None, d_k=None,
               d_positions=None, *, is_neox: bool, eps: float = 1e-6, head_dim: int = 0,
               rope_dim: int = 0, chunk_tokens: int = 0, mode: str = "auto", stream=None) -> None:
    """The op on host tensors h_q, h_k, h_positions, written back into h_q and
    h_k (see qknr_apply_host). q_w, k_w and cos_sin_cache are device tensors.
    As in ``apply``, q and k may be [B, S, H, D] when B and S merge into one
    token dim without a copy (positions then [B*S]).
    ``mode``: "direct" (the kernel works on pinned, device-mapped host memory
    in place), "staged" (chunked copies through the device tensors d_q, d_k,
    d_positions of the same shapes and strides) or "auto" (direct when
    possible). Asynchronous on ``stream`` (default: torch's current stream on
    q_w's device): synchronise it before reading h_q and h_k."""
    import torch
    if mode not in HOST_MODES:
        raise QknrError(2, f"mode must be one of {sorted(HOST_MODES)}")
    h_q, h_k = _as_tokens(h_q, "h_q"), _as_tokens(h_k, "h_k")
    d_q = _as_tokens(d_q, "d_q") if d_q is not None else None
    d_k = _as_tokens(d_k, "d_k") if d_k is not None else None
    for name, h in (("q", h_q), ("k", h_k), ("positions", h_positions)):
        if h.device.type != "cpu":
            raise QknrError(2, f"h_{name} must be a host (CPU) tensor")
    staged = d_q is not None
    if staged:
        for name, h, d in (("q", h_q, d_q), ("k", h_k, d_k), ("positions", h_positions, d_positions)):
            if d is None or h.shape != d.shape or h.stride() != d.stride() or h.dtype != d.dtype:
                raise QknrError(2, f"d_{name} must match h_{name} in shape, stride and dtype")
        shape_of = (d_q, d_k, d_positions)
    else:
        if mode == "staged":
            raise QknrError(2, "mode 'staged' needs the device tensors d_q, d_k, d_positions")
        # the layout checks of _marshal, on host stand-ins with the same geometry
        shape_of = tuple(torch.empty_strided(h.shape, h.stride(), dtype=h.dtype, device="meta")
                         for h in (h_q, h_k, h_positions))
    T, n_qo, n_kv, D, R, qs, ks, hs, code = _marshal(
        *shape_of[:2], q_w, k_w, cos_sin_cache, shape_of[2], is_neox, head_dim, rope_dim,
        same_device=staged)
    if stream is None:
        stream = torch.cuda.current_stream(q_w.device).cuda_stream
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    ptr = (lambda t: t.data_ptr() if t is not None else 0)
    with torch.cuda.device(q_w.device):
        _check(qknr_apply_host(h_q.data_ptr(), h_k.data_ptr(), q_w.data_ptr(), k_w.data_ptr(),
                               cos_sin_cache.data_ptr(), h_positions.data_ptr(), ptr(d_q), ptr(d_k),
                               ptr(d_positions), T, n_qo, n_kv, D, R, int(bool(is_neox)), qs, ks, hs,
                               float(eps), code, int(chunk_tokens), HOST_MODES[mode], stream))


def set_tuning(**kw) -> None:
    """Set launch tuning keys by name (see TUNE_KEYS); ``reset=True`` first
    returns every key to automatic. ``kernel`` also takes "auto", "register"
    or "ring"."""
    if kw.pop("reset", False):
        _check(qknr_set_tuning(0, 0))
    for name, value in kw.items():
        if name == "kernel" and isinstance(value, str):
            value = {"auto": QKNR_KERNEL_AUTO, "register": QKNR_KERNEL_REGISTER, "ring": QKNR_KERNEL_RING}[value]
        _check(qknr_set_tuning(TUNE_KEYS[name], int(value)))


def get_tuning(name: str) -> int:
    v = ctypes.c_int(0)
    _check(qknr_get_tuning(TUNE_KEYS[name], ctypes.byref(v)))
    return v.value


def tune(q, k, q_w, k_w, cos_sin_cache, positions, *, is_neox: bool, head_dim: int = 0,
         rope_dim: int = 0, stream=None, inputs_ready: bool = False) -> Dict[str, int]:
    """qknr_tune for the call apply() would make with these tensors: only their
    shapes, strides and dtypes are read (the candidates run on scratch
    buffers). Later apply() calls with the same shapes, strides and dtypes use
    the launch it chose. Returns the chosen work map, with ``ns_per_launch``
    measured. A set-up-time call: it allocates scratch and waits for the
    stream."""
    import torch
    q, k = _as_tokens(q, "q"), _as_tokens(k, "k")
    T, n_qo, n_kv, D, R, qs, ks, hs, code = _marshal(
        q, k, q_w, k_w, cos_sin_cache, positions, is_neox, head_dim, rope_dim, same_device=False)
    if q.device.type != "cuda":
        raise QknrError(2, "q must be a CUDA tensor")
    if inputs_ready:
        code |= QKNR_INPUTS_READY
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif not isinstance(stream, int):
        stream = stream.cuda_stream
    out = (ctypes.c_int64 * (len(WORK_MAP_FIELDS) + 1))()
    with torch.cuda.device(q.device):
        _check(qknr_tune(T, n_qo, n_kv, D, R, int(bool(is_neox)), qs, ks, hs, code, stream, out))
    d = dict(zip(WORK_MAP_FIELDS + ["ns_per_launch"], [int(v) for v in out]))
    d["kernel"] = KERNEL_NAMES.get(d["kernel"], d["kernel"])
    d["order"] = {1: "contiguous", 2: "interleaved"}.get(d["order"], d["order"])
    return d


def work_map(num_tokens: int, n_qo: int, n_kv: int, head_dim: int, rope_dim: int,
             is_neox: bool, dtype: int) -> Dict[str, int]:
    """The launch qknr_apply would make (kernel, grid, threads, items, ...)."""
    out = (ctypes.c_int64 * len(WORK_MAP_FIELDS))()
    _check(qknr_query_work_map(num_tokens, n_qo, n_kv, head_dim, rope_dim, int(is_neox), dtype,
                               out))
    d = dict(zip(WORK_MAP_FIELDS, [int(v) for v in out]))
    d["kernel"] = KERNEL_NAMES.get(d["kernel"], d["kernel"])
    d["order"] = {1: "contiguous", 2: "interleaved"}.get(d["order"], d["order"])
    return d
