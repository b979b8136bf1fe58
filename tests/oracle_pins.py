"""Pins for the CPU oracle: checks against what the method and the mathematics
fix, none of which re-types the oracle's own formulas.

Each ``pin_*`` takes a loaded oracle library (the real one, or a deliberately
broken copy built by ``test_oracle_mutants.py``) and raises AssertionError when
the oracle disagrees. What pins what:

  decode       every bf16 / fp16 bit pattern against torch's and numpy's own casts
  hand cases   tests/golden/hand_cases.json, derived by hand from the formulas of
               the fused_inplace_qknorm_rope deep-dive §2.1-§2.3 (the page prints
               no worked example)
  unit RMS     w = 1, eps = 0: mean(out^2) = 1 for any x and any rope_dim
               (rotations preserve length; the mean runs over head_dim)
  eps          w = 1, identity rotation: mean(out^2) = m / (m + eps), m = mean(x^2)
  scale        eps = 0: out(4x) == out(x) bit for bit
  weights      identity rotation: out(x, w) == w * out(x, 1)
  rotation     out(x, p) equals out(x, 0) turned pair by pair through the angle
               p * base^(-2j/R) as a complex product (a + ib) * e^{i*angle},
               evaluated with Python's cmath, independent of the cos|sin table
  NeoX         NeoX(x, w) = P^-1 Interleaved(P x, P w), P the de-interleave permutation
  layout       strided views == contiguous copies; int32 == int64 positions;
               Q heads use q_w, K heads use k_w; K is read at k's own stride
  relative     <rope(q, p+d), rope(k, p'+d)> == <rope(q, p), rope(k, p')>
  arguments    odd / too large rope_dim and out-of-range positions are rejected
"""
from __future__ import annotations

import cmath
import ctypes
import json
import math
import os

import numpy as np
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_cases.json")


def _rand(shape, seed, dtype=torch.bfloat16, scale=1.0):
    g = np.random.default_rng(seed)
    return torch.from_numpy(g.standard_normal(shape, dtype=np.float32) * np.float32(scale)).to(dtype)


def _weights(D, seed, dtype=torch.bfloat16):
    return (1.0 + 0.1 * _rand((D,), seed, torch.float32)).to(dtype)


def _run(lib, q, k, qw, kw, cache, pos, neox, eps):
    return oracle.apply(q, k, qw, kw, cache, pos, is_neox=neox, eps=eps, lib=lib)


def _identity_row_cache(R, rows=1):
    c = torch.zeros(rows, R, dtype=torch.float32)
    c[:, : R // 2] = 1.0
    return c


# --------------------------------------------------------------------------- decode
def pin_decode_bf16(lib):
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = np.array([lib.qknr_oracle_decode(oracle.BF16, int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_decode_fp16(lib):
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([lib.qknr_oracle_decode(oracle.FP16, int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# --------------------------------------------------------------------------- hand cases
def load_hand_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def pin_hand_cases(lib):
    for case in load_hand_cases():
        dt = torch.bfloat16 if case["dtype"] == "bf16" else torch.float16
        D, R = case["head_dim"], case["rope_dim"]
        x = torch.tensor(case["x"], dtype=torch.float64)
        w = torch.tensor(case["w"], dtype=torch.float64)
        xb, wb = x.to(dt), w.to(dt)
        assert torch.equal(xb.double(), x) and torch.equal(wb.double(), w), case["name"]
        cos = torch.tensor(case["cos"], dtype=torch.float32)
        sin = torch.tensor(case["sin"], dtype=torch.float32)
        exp = np.array(case["expected"], dtype=np.float64)
        # through the single-head entry point
        got = oracle.head(xb, wb, cos, sin, is_neox=case["is_neox"], eps=case["eps"], lib=lib)
        assert np.allclose(got, exp, rtol=1e-14, atol=1e-14), (case["name"], got, exp)
        # through the whole-op entry point: the case as a Q head and as a K head
        cache = torch.cat([cos, sin]).reshape(1, R)
        q = xb.reshape(1, 1, D).clone()
        k = xb.reshape(1, 1, D).clone()
        pos = torch.zeros(1, dtype=torch.int32)
        qo, ko = _run(lib, q, k, wb, wb, cache, pos, case["is_neox"], case["eps"])
        assert np.allclose(qo[0, 0], exp, rtol=1e-14, atol=1e-14), case["name"]
        assert np.allclose(ko[0, 0], exp, rtol=1e-14, atol=1e-14), case["name"]


# --------------------------------------------------------------------------- norm
def pin_unit_rms(lib):
    for D, R, neox in [(64, 64, False), (128, 64, True), (128, 128, True), (256, 128, False),
                       (64, 16, False)]:
        T, H = 5, 3
        q = _rand((T, H, D), 11 + D + R, scale=3.0)
        k = _rand((T, 1, D), 12 + D + R)
        ones = torch.ones(D, dtype=torch.bfloat16)
        cache = workloads.build_cos_sin_cache(64, R, 1e4)
        pos = torch.tensor([0, 1, 7, 33, 63], dtype=torch.int32)
        qo, ko = _run(lib, q, k, ones, ones, cache, pos, neox, 0.0)
        for o in (qo, ko):
            ms = np.mean(o * o, axis=-1)
            # fp32 cos^2 + sin^2 differs from 1 by ~1e-7
            assert np.allclose(ms, 1.0, rtol=0, atol=2e-6), (D, R, neox, ms)


def pin_eps_closed_form(lib):
    D, R, eps = 128, 128, 0.5
    q = _rand((4, 2, D), 21, scale=0.5)
    k = _rand((4, 2, D), 22, scale=2.0)
    ones = torch.ones(D, dtype=torch.bfloat16)
    cache = _identity_row_cache(R)
    pos = torch.zeros(4, dtype=torch.int32)
    qo, ko = _run(lib, q, k, ones, ones, cache, pos, False, eps)
    for x, o in ((q, qo), (k, ko)):
        m = np.mean(x.double().numpy() ** 2, axis=-1)
        assert np.allclose(np.mean(o * o, axis=-1), m / (m + eps), rtol=1e-12, atol=0)


def pin_scale_invariance(lib):
    D, R = 128, 64
    q = _rand((3, 4, D), 31)
    k = _rand((3, 2, D), 32)
    qw, kw = _weights(D, 33), _weights(D, 34)
    cache = workloads.build_cos_sin_cache(16, R, 1e4)
    pos = torch.tensor([3, 0, 9], dtype=torch.int32)
    a = _run(lib, q, k, qw, kw, cache, pos, True, 0.0)
    b = _run(lib, q * 4, k * 4, qw, kw, cache, pos, True, 0.0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def pin_weight_linearity(lib):
    D, R = 64, 64
    q = _rand((3, 2, D), 41)
    k = _rand((3, 3, D), 42)
    qw, kw = _weights(D, 43), _weights(D, 44)
    ones = torch.ones(D, dtype=torch.bfloat16)
    cache = _identity_row_cache(R)
    pos = torch.zeros(3, dtype=torch.int32)
    qo, ko = _run(lib, q, k, qw, kw, cache, pos, False, 1e-6)
    q1, k1 = _run(lib, q, k, ones, ones, cache, pos, False, 1e-6)
    assert np.allclose(qo, q1 * qw.double().numpy(), rtol=1e-15, atol=0)
    assert np.allclose(ko, k1 * kw.double().numpy(), rtol=1e-15, atol=0)


# --------------------------------------------------------------------------- rotation
def _pairs(R, neox):
    half = R // 2
    if neox:
        return [(j, j + half, j) for j in range(half)]
    return [(2 * j, 2 * j + 1, j) for j in range(half)]


def pin_rotation_complex(lib):
    for D, R, neox, base in [(64, 64, False, 1e4), (128, 128, True, 1e4), (128, 64, True, 1e6),
                             (256, 128, False, 1e4), (64, 8, True, 1e4), (64, 4, False, 500.0)]:
        T, cache_len = 6, 4096
        q = _rand((T, 2, D), 51 + D + R)
        k = _rand((T, 1, D), 52 + D + R)
        qw, kw = _weights(D, 53), _weights(D, 54)
        cache = workloads.build_cos_sin_cache(cache_len, R, base)
        pos = torch.tensor([0, 1, 2, 100, 1234, 4095], dtype=torch.int64)
        qo, ko = _run(lib, q, k, qw, kw, cache, pos, neox, 1e-6)
        zero = torch.zeros(T, dtype=torch.int64)
        qn, kn = _run(lib, q, k, qw, kw, cache, zero, neox, 1e-6)   # identity rotation
        for o, n in ((qo, qn), (ko, kn)):
            for t in range(T):
                p = int(pos[t])
                for h in range(o.shape[1]):
                    for ia, ib, j in _pairs(R, neox):
                        angle = p * base ** (-2.0 * j / R)
                        z = complex(n[t, h, ia], n[t, h, ib]) * cmath.exp(1j * angle)
                        got = complex(o[t, h, ia], o[t, h, ib])
                        # the table holds cos/sin rounded to fp32 (rel. error <= 2^-24)
                        assert abs(got - z) <= 2e-7 * abs(z) + 1e-12, (D, R, neox, t, h, j)
                    assert np.array_equal(o[t, h, R:], n[t, h, R:])


def pin_neox_interleaved_permutation(lib):
    for D, R in [(128, 128), (128, 64), (64, 16)]:
        half = R // 2
        perm = list(range(D))      # interleaved position -> NeoX position
        for j in range(half):
            perm[2 * j] = j
            perm[2 * j + 1] = j + half
        perm = torch.tensor(perm)
        q = _rand((4, 3, D), 61 + R)
        k = _rand((4, 2, D), 62 + R)
        qw, kw = _weights(D, 63), _weights(D, 64)
        cache = workloads.build_cos_sin_cache(512, R, 1e4)
        pos = torch.tensor([5, 77, 300, 511], dtype=torch.int32)
        nq, nk = _run(lib, q, k, qw, kw, cache, pos, True, 1e-6)
        iq, ik = _run(lib, q[..., perm].contiguous(), k[..., perm].contiguous(),
                      qw[perm].contiguous(), kw[perm].contiguous(), cache, pos, False, 1e-6)
        inv = torch.argsort(perm).numpy()
        assert np.allclose(iq[..., inv], nq, rtol=1e-13, atol=1e-15)
        assert np.allclose(ik[..., inv], nk, rtol=1e-13, atol=1e-15)


def pin_relative_position(lib):
    D, R = 128, 128
    q = _rand((2, 1, D), 71)
    k = _rand((2, 1, D), 72)
    qw, kw = _weights(D, 73), _weights(D, 74)
    cache = workloads.build_cos_sin_cache(2048, R, 1e4)

    def dot(p, pp):
        pos = torch.tensor([p, pp], dtype=torch.int32)
        qo, ko = _run(lib, q, k, qw, kw, cache, pos, False, 1e-6)
        return float(np.dot(qo[0, 0], ko[1, 0]))
    base = dot(10, 3)
    for d in (1, 17, 500, 1500):
        assert abs(dot(10 + d, 3 + d) - base) <= 1e-5 * max(1.0, abs(base))


# --------------------------------------------------------------------------- layout
def pin_layout(lib):
    w = workloads.scaled(workloads.get("fused_qkv"), 9, cache_len=64)
    inp = workloads.make_inputs(w)
    qv, kv = inp["q"], inp["k"]
    assert not qv.is_contiguous()
    a = _run(lib, qv, kv, inp["q_w"], inp["k_w"], inp["cos_sin_cache"], inp["positions"],
             False, w.eps)
    b = _run(lib, qv.contiguous(), kv.contiguous(), inp["q_w"], inp["k_w"],
             inp["cos_sin_cache"], inp["positions"], False, w.eps)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # int64 positions give the same result as the same values in int32
    c = _run(lib, qv, kv, inp["q_w"], inp["k_w"], inp["cos_sin_cache"],
             inp["positions"].to(torch.int64), False, w.eps)
    assert np.array_equal(a[0], c[0]) and np.array_equal(a[1], c[1])
    # each head kind uses its own weight, token row and stride
    cache, pos = inp["cos_sin_cache"], inp["positions"]
    R = cache.shape[1]
    for t in (0, 4, 8):
        row = cache[int(pos[t])]
        for h in range(qv.shape[1]):
            e = oracle.head(qv[t, h], inp["q_w"], row[: R // 2], row[R // 2:], is_neox=False,
                            eps=w.eps, lib=lib)
            assert np.array_equal(a[0][t, h], e)
        for h in range(kv.shape[1]):
            e = oracle.head(kv[t, h], inp["k_w"], row[: R // 2], row[R // 2:], is_neox=False,
                            eps=w.eps, lib=lib)
            assert np.array_equal(a[1][t, h], e)
    # separate tensors with different token strides
    q = _rand((7, 4, 64), 81)
    kbig = _rand((7, 5, 64), 82)
    k = kbig[:, 1:3, :]
    assert k.stride(0) != q.stride(0)
    cache = workloads.build_cos_sin_cache(16, 64, 1e4)
    pos = torch.arange(7, dtype=torch.int32) * 2
    x = _run(lib, q, k, _weights(64, 83), _weights(64, 84), cache, pos, True, 1e-6)
    y = _run(lib, q, k.contiguous(), _weights(64, 83), _weights(64, 84), cache, pos, True, 1e-6)
    assert np.array_equal(x[1], y[1]) and np.array_equal(x[0], y[0])


def pin_rejects_bad_args(lib):
    D = 8
    x = torch.ones(1, 1, D, dtype=torch.bfloat16)
    wgt = torch.ones(D, dtype=torch.bfloat16)
    out = np.zeros((1, 1, D))
    pos = torch.zeros(1, dtype=torch.int32)
    def call(R, cache_len, p):
        cache = torch.zeros(max(cache_len, 1), max(R, 2), dtype=torch.float32)
        pp = torch.tensor([p], dtype=torch.int32)
        return lib.qknr_oracle_apply(x.data_ptr(), x.data_ptr(), wgt.data_ptr(), wgt.data_ptr(),
                                     cache.data_ptr(), cache_len, pp.data_ptr(), 1, 1, 1, D, R,
                                     0, D, D, D, 1e-6, oracle.BF16, out.ctypes.data,
                                     out.ctypes.data)
    assert call(4, 4, 0) == 0
    assert call(3, 4, 0) != 0          # odd rope_dim
    assert call(10, 4, 0) != 0         # rope_dim > head_dim
    assert call(4, 4, 4) != 0          # position past the cache
    assert call(4, 4, -1) != 0         # negative position
    del pos


ALL_PINS = [pin_decode_bf16, pin_decode_fp16, pin_hand_cases, pin_unit_rms, pin_eps_closed_form,
            pin_scale_invariance, pin_weight_linearity, pin_rotation_complex,
            pin_neox_interleaved_permutation, pin_relative_position, pin_layout,
            pin_rejects_bad_args]
