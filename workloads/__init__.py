"""Seeded synthetic inputs for the fused per-head QK RMSNorm + RoPE op.

This module is shared by the tests, the benchmark and the oracle's checks. It
only *draws* inputs: random Q/K activations, RMSNorm weights, token positions
and the fp32 cos|sin table that the op takes as an input tensor. It holds none
of the op's own arithmetic (no norm, no rotation).

Workloads (sizes and value distributions follow the shapes the
fused_inplace_qknorm_rope deep-dive names for DiT attention pre-processing:
FLUX / Qwen-Image / Z-Image style full rope, LLaMA-style NeoX, GQA with partial
rope, and a fused-QKV buffer viewed as strided q/k):

  tiny       bf16 q,k [16,4,64] ~N(0,1); interleaved R=64; cache [64,64]; pos int32 0..15
  dit        bf16 q,k [4608,24,128] ~2*N(0,1); interleaved R=128; cache [4608,128]; pos int32 arange
  mha_neox   bf16 q,k [8192,24,128] ~N(0,1); NeoX R=128; cache [8192,128]; pos int64 arange
  gqa        fp16 q [16384,32,128], k [16384,8,128] ~N(0,1); NeoX R=64, base 1e6;
             cache [32768,64]; pos int64 uniform in [0,32768)
  fused_qkv  bf16 buffer [65536, 24*256] ~N(0,1); q = heads 0-15, k = heads 16-19
             (token stride 6144 elements); D=256, R=128 interleaved; cache [65536,128];
             pos int32 uniform in [0,65536); eps 1e-5

Weights are 1 + 0.1*N(0,1) drawn in fp32 and rounded to the activation dtype.
Every random tensor has its own stream spawned from one seed (default 0), drawn
in the order q (or the fused buffer), k, q_w, k_w, positions, so a tensor does
not change when another one changes size.

Random values are drawn with numpy's PCG64 generator (platform independent) in
fp32 and rounded to bf16/fp16 with round-to-nearest-even by torch's CPU cast.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np
import torch

__all__ = ["Workload", "WORKLOADS", "get", "make_inputs", "to_device", "build_cos_sin_cache",
           "scaled", "algorithmic_bytes", "algorithmic_read_bytes", "algorithmic_write_bytes",
           "num_heads_total", "describe"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str              # "bf16" | "fp16"
    num_tokens: int
    n_qo: int
    n_kv: int
    head_dim: int
    rope_dim: int
    is_neox: bool
    base: float
    cache_len: int
    pos_dtype: str          # "i32" | "i64"
    pos_kind: str           # "arange" | "uniform"
    eps: float
    x_scale: float = 1.0
    # fused_qkv layout: one buffer [T, total_heads, D]; q = heads [0, n_qo),
    # k = heads [n_qo, n_qo + n_kv). 0 means separate contiguous q and k.
    fused_total_heads: int = 0
    seed: int = 0

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    @property
    def pos_torch_dtype(self) -> torch.dtype:
        return torch.int32 if self.pos_dtype == "i32" else torch.int64


WORKLOADS: Dict[str, Workload] = {
    w.name: w for w in [
        Workload("tiny", "bf16", 16, 4, 4, 64, 64, False, 1e4, 64, "i32", "arange", 1e-6),
        Workload("dit", "bf16", 4608, 24, 24, 128, 128, False, 1e4, 4608, "i32", "arange",
                 1e-6, x_scale=2.0),
        Workload("mha_neox", "bf16", 8192, 24, 24, 128, 128, True, 1e4, 8192, "i64", "arange",
                 1e-6),
        Workload("gqa", "fp16", 16384, 32, 8, 128, 64, True, 1e6, 32768, "i64", "uniform",
                 1e-6),
        Workload("fused_qkv", "bf16", 65536, 16, 4, 256, 128, False, 1e4, 65536, "i32",
                 "uniform", 1e-5, fused_total_heads=24),
    ]
}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def scaled(w: Workload, num_tokens: int, cache_len: Optional[int] = None) -> Workload:
    """The same workload with fewer tokens (and optionally a shorter cache).

    An arange workload keeps positions inside the cache by growing the cache to
    at least ``num_tokens`` rows.
    """
    cl = cache_len if cache_len is not None else w.cache_len
    if w.pos_kind == "arange":
        cl = max(cl, num_tokens, 1)
    return dataclasses.replace(w, num_tokens=num_tokens, cache_len=cl)


def num_heads_total(w: Workload) -> int:
    return (w.n_qo + w.n_kv) * w.num_tokens


def algorithmic_write_bytes(w: Workload) -> int:
    """Bytes the op must write once: every Q/K head."""
    return (w.n_qo + w.n_kv) * w.num_tokens * w.head_dim * 2


def algorithmic_read_bytes(w: Workload) -> int:
    """Bytes the op must read once: every Q/K head, one fp32 cache row and one
    position per token, and both weight vectors."""
    psz = 4 if w.pos_dtype == "i32" else 8
    return (algorithmic_write_bytes(w)
            + w.num_tokens * w.rope_dim * 4
            + w.num_tokens * psz
            + 2 * w.head_dim * 2)


def algorithmic_bytes(w: Workload) -> int:
    """Bytes the op must move once: read + write every Q/K head, one fp32 cache
    row and one position per token, and both weight vectors."""
    return algorithmic_read_bytes(w) + algorithmic_write_bytes(w)


def build_cos_sin_cache(cache_len: int, rope_dim: int, base: float) -> torch.Tensor:
    """The op's fp32 input table: row p = [cos(p*theta_j) for j < R/2 | sin(p*theta_j) for j < R/2]
    with theta_j = base^(-2j/R). Angles and trig in float64, rounded once to fp32."""
    half = rope_dim // 2
    j = np.arange(half, dtype=np.float64)
    theta = np.power(float(base), -2.0 * j / float(rope_dim))
    p = np.arange(cache_len, dtype=np.float64)[:, None]
    ang = p * theta[None, :]
    table = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    return torch.from_numpy(np.ascontiguousarray(table))


def _normal(rng: np.random.Generator, shape, scale: float, dtype: torch.dtype) -> torch.Tensor:
    a = rng.standard_normal(shape, dtype=np.float32)
    if scale != 1.0:
        a *= np.float32(scale)
    return torch.from_numpy(a).to(dtype)


def make_inputs(w: Workload, device: str = "cpu") -> Dict[str, torch.Tensor]:
    """Draw one seeded input set. Returns CPU (or ``device``) tensors:

    q, k          [T, n_qo, D] / [T, n_kv, D] views (strided for fused_qkv)
    buffer        the fused [T, total_heads, D] buffer (fused_qkv only)
    q_w, k_w      [D]
    cos_sin_cache [cache_len, R] fp32
    positions     [T] int32 / int64
    """
    ss = np.random.SeedSequence(w.seed)
    r_x, r_k, r_qw, r_kw, r_pos = [np.random.default_rng(s) for s in ss.spawn(5)]
    T, D, dt = w.num_tokens, w.head_dim, w.torch_dtype
    out: Dict[str, torch.Tensor] = {}
    if w.fused_total_heads:
        buf = _normal(r_x, (T, w.fused_total_heads, D), w.x_scale, dt)
        out["buffer"] = buf
        out["q"] = buf[:, :w.n_qo, :]
        out["k"] = buf[:, w.n_qo:w.n_qo + w.n_kv, :]
    else:
        out["q"] = _normal(r_x, (T, w.n_qo, D), w.x_scale, dt)
        out["k"] = _normal(r_k, (T, w.n_kv, D), w.x_scale, dt)
    out["q_w"] = (1.0 + 0.1 * _normal(r_qw, (D,), 1.0, torch.float32)).to(dt)
    out["k_w"] = (1.0 + 0.1 * _normal(r_kw, (D,), 1.0, torch.float32)).to(dt)
    if w.pos_kind == "arange":
        pos = np.arange(T, dtype=np.int64)
    else:
        pos = r_pos.integers(0, w.cache_len, size=T, dtype=np.int64)
    out["positions"] = torch.from_numpy(pos).to(w.pos_torch_dtype)
    out["cos_sin_cache"] = build_cos_sin_cache(w.cache_len, w.rope_dim, w.base)
    if device != "cpu":
        out = to_device(out, w, device)
    return out


def to_device(inputs: Dict[str, torch.Tensor], w: Workload, device) -> Dict[str, torch.Tensor]:
    """Copy an input set to ``device``, keeping q/k as views of the fused
    buffer for the fused_qkv layout."""
    out: Dict[str, torch.Tensor] = {}
    if w.fused_total_heads:
        buf = inputs["buffer"].to(device)
        out["buffer"] = buf
        out["q"] = buf[:, :w.n_qo, :]
        out["k"] = buf[:, w.n_qo:w.n_qo + w.n_kv, :]
    else:
        out["q"] = inputs["q"].to(device)
        out["k"] = inputs["k"].to(device)
    for key in ("q_w", "k_w", "positions", "cos_sin_cache"):
        out[key] = inputs[key].to(device)
    return out


def describe(w: Workload) -> str:
    lay = (f"fused buffer [{w.num_tokens},{w.fused_total_heads}*{w.head_dim}]"
           if w.fused_total_heads else "contiguous q,k")
    return (f"{w.name}: {w.dtype} T={w.num_tokens} n_qo={w.n_qo} n_kv={w.n_kv} D={w.head_dim} "
            f"R={w.rope_dim} {'neox' if w.is_neox else 'interleaved'} base={w.base:g} "
            f"cache={w.cache_len} pos={w.pos_dtype}/{w.pos_kind} eps={w.eps:g} {lay}")


def _check_tables() -> None:
    # static sanity of the workload table (sizes the op accepts)
    for w in WORKLOADS.values():
        assert w.rope_dim % 2 == 0 and 0 < w.rope_dim <= w.head_dim
        assert not math.isnan(w.eps)


_check_tables()
