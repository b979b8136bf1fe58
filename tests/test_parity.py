"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every comparison is element by element on the same seeded inputs, with the
bound max |gpu - oracle| <= 2^-7 |oracle| + 1e-5 (bf16) or 2^-10 |oracle| + 1e-5
(fp16), i.e. two units in the last place of the output dtype at the oracle
value plus 1e-5 absolute; a correctly rounded fp32 evaluation stays inside
half of that.

Sizes: each workload at a reduced token count that spans many warp items and
a ragged tail (whole output compared), and at its full size in the launch
configuration the benchmark times (sampled tokens compared, plus properties
that hold at any size); a grid over head_dim x rope_dim x pairing x position
type x token counts 1/9/129 (the grid the deep-dive's own unit test uses,
"Step4"); GQA head counts; strided and padded layouts; and the edge cases.
"""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import oracle  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qknr():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import qk_rmsnorm_rope_gb300 as q
    torch.cuda.set_device(0)
    q.init(0)
    q.qknr_set_work_map(0, 0, 0, -1)
    yield q
    q.qknr_set_work_map(0, 0, 0, -1)


def _expected(cpu, w):
    return oracle.apply(cpu["q"], cpu["k"], cpu["q_w"], cpu["k_w"], cpu["cos_sin_cache"],
                        cpu["positions"], is_neox=w.is_neox, eps=w.eps)


def _run_gpu(q, dev, w):
    q.apply(dev["q"], dev["k"], dev["q_w"], dev["k_w"], dev["cos_sin_cache"], dev["positions"],
            is_neox=w.is_neox, eps=w.eps)
    torch.cuda.synchronize()


def _assert_close(got, exp, dtype, what):
    v = oracle.max_violation(got, exp, dtype)
    assert v <= 1.0, f"{what}: max error {v:.3f} x tolerance"


def _check_workload(q, w):
    cpu = workloads.make_inputs(w)
    eq, ek = _expected(cpu, w)
    dev = workloads.to_device(cpu, w, "cuda")
    _run_gpu(q, dev, w)
    _assert_close(dev["q"].double().cpu().numpy(), eq, w.torch_dtype, f"{w.name} q")
    _assert_close(dev["k"].double().cpu().numpy(), ek, w.torch_dtype, f"{w.name} k")
    if w.fused_total_heads:
        # heads outside q and k (the V part of the fused buffer) keep every bit
        lo = w.n_qo + w.n_kv
        a = dev["buffer"][:, lo:, :].cpu().view(torch.int16)
        b = cpu["buffer"][:, lo:, :].view(torch.int16)
        assert torch.equal(a, b), "bytes outside q/k changed"
    return cpu, dev


REDUCED = [("tiny", 16), ("dit", 300), ("mha_neox", 257), ("gqa", 513), ("fused_qkv", 129)]


@pytest.mark.parametrize("name,T", REDUCED, ids=[r[0] for r in REDUCED])
def test_workload_reduced(qknr, name, T):
    base = workloads.get(name)
    w = workloads.scaled(base, T, cache_len=min(base.cache_len, 8192))
    _check_workload(qknr, w)


def _sample_tokens(T, n, seed):
    g = np.random.default_rng(seed)
    pick = set(g.choice(T, size=min(n, T), replace=False).tolist())
    pick.update({0, 1, T // 2, T - 2, T - 1})
    return torch.tensor(sorted(t for t in pick if 0 <= t < T), dtype=torch.long)


FULL = ["tiny", "dit", "mha_neox", "gqa", "fused_qkv"]


@pytest.mark.parametrize("name", FULL)
def test_workload_full_size_sampled(qknr, name):
    """Full size, default launch (as the benchmark runs it): sampled tokens
    against the oracle, the rest through properties that hold at any size."""
    w = workloads.get(name)
    cpu = workloads.make_inputs(w)
    dev = workloads.to_device(cpu, w, "cuda")
    _run_gpu(qknr, dev, w)
    idx = _sample_tokens(w.num_tokens, 384, 1)
    sub = {"q": cpu["q"][idx], "k": cpu["k"][idx], "q_w": cpu["q_w"], "k_w": cpu["k_w"],
           "cos_sin_cache": cpu["cos_sin_cache"], "positions": cpu["positions"][idx]}
    eq, ek = _expected(sub, w)
    gq = dev["q"][idx.cuda()].double().cpu().numpy()
    gk = dev["k"][idx.cuda()].double().cpu().numpy()
    _assert_close(gq, eq, w.torch_dtype, f"{name} q (sampled)")
    _assert_close(gk, ek, w.torch_dtype, f"{name} k (sampled)")
    # any size: every output finite, and with these weights (|w| <= ~1.5) every
    # head's RMS is below max|w| (a rotation keeps each pair's length)
    for t, wt in ((dev["q"], cpu["q_w"]), (dev["k"], cpu["k_w"])):
        x = t.float()
        assert torch.isfinite(x).all()
        rms = x.pow(2).mean(-1).sqrt()
        assert float(rms.max()) <= float(wt.float().abs().max()) * 1.01
    if w.fused_total_heads:
        lo = w.n_qo + w.n_kv
        assert torch.equal(dev["buffer"][:, lo:, :].cpu().view(torch.int16),
                           cpu["buffer"][:, lo:, :].view(torch.int16))


def _rope_dims(D, neox):
    if neox:
        return sorted({r for r in (4, 8, 16, 32, 64, D // 2, D) if r <= D})
    return sorted({r for r in (2, 6, 8, 24, 64, D // 2, D - 8, D) if 0 < r <= D})


GRID = [(D, R, neox, pos, T)
        for D in (64, 128, 256)
        for neox in (False, True)
        for R in _rope_dims(D, neox)
        for pos in ("i32", "i64")
        for T in (1, 9, 129)]


def _make(D, R, neox, pos, T, n_qo, n_kv, dtype="bf16", seed=0, cache_len=300, base=1e4,
          pos_kind="uniform", eps=1e-6, x_scale=1.0):
    return workloads.Workload(f"grid_{D}_{R}_{int(neox)}_{pos}_{T}", dtype, T, n_qo, n_kv, D, R,
                              neox, base, cache_len, pos, pos_kind, eps, x_scale=x_scale,
                              seed=seed)


@pytest.mark.parametrize("D,R,neox,pos,T", GRID,
                         ids=[f"D{g[0]}-R{g[1]}-{'neox' if g[2] else 'inter'}-{g[3]}-T{g[4]}"
                              for g in GRID])
def test_shape_grid(qknr, D, R, neox, pos, T):
    w = _make(D, R, neox, pos, T, 4, 2, dtype="bf16" if (D + R + T) % 2 == 0 else "fp16")
    _check_workload(qknr, w)


@pytest.mark.parametrize("n_qo,n_kv", [(1, 1), (8, 1), (32, 8), (5, 3), (1, 7), (64, 64)])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_gqa_head_counts(qknr, n_qo, n_kv, D):
    w = _make(D, D // 2, True, "i64", 33, n_qo, n_kv, dtype="fp16", seed=n_qo * 100 + n_kv)
    _check_workload(qknr, w)


@pytest.mark.parametrize("ppi,threads,ctas", [(1, 64, 1), (2, 128, 0), (3, 256, 2), (4, 512, 0),
                                              (4, 64, 0), (1, 256, 0)])
def test_work_maps_agree_bit_for_bit(qknr, ppi, threads, ctas):
    """Per-head results do not depend on the work map: every forced map gives
    the same bits as the automatic one, and all match the oracle."""
    for name, T in (("mha_neox", 97), ("fused_qkv", 41), ("tiny", 16)):
        base = workloads.get(name)
        w = workloads.scaled(base, T, cache_len=min(base.cache_len, 4096))
        cpu = workloads.make_inputs(w)
        ref = workloads.to_device(cpu, w, "cuda")
        qknr.qknr_set_work_map(0, 0, 0, -1)
        _run_gpu(qknr, ref, w)
        dev = workloads.to_device(cpu, w, "cuda")
        assert qknr.qknr_set_work_map(ppi, threads, ctas, 0) == 0
        try:
            _run_gpu(qknr, dev, w)
        finally:
            qknr.qknr_set_work_map(0, 0, 0, -1)
        assert torch.equal(dev["q"].view(torch.int16), ref["q"].view(torch.int16)), name
        assert torch.equal(dev["k"].view(torch.int16), ref["k"].view(torch.int16)), name
        eq, ek = _expected(cpu, w)
        _assert_close(dev["q"].double().cpu().numpy(), eq, w.torch_dtype, name)
        _assert_close(dev["k"].double().cpu().numpy(), ek, w.torch_dtype, name)


def test_separate_strides_and_padded_heads(qknr):
    """q and k views with different token strides and a head stride > head_dim."""
    T, D, R = 77, 128, 64
    g = np.random.default_rng(5)
    qbuf = torch.from_numpy(g.standard_normal((T, 6, 160), dtype=np.float32)).to(torch.bfloat16)
    kbuf = torch.from_numpy(g.standard_normal((T, 3, 160), dtype=np.float32)).to(torch.bfloat16)
    kbig = torch.from_numpy(g.standard_normal((T, 4, 160), dtype=np.float32)).to(torch.bfloat16)
    kbig[:, :3] = kbuf
    q = qbuf[:, 1:5, :D]
    k = kbig[:, 0:3, :D]
    assert q.stride() == (960, 160, 1) and k.stride() == (640, 160, 1)
    qw = (1 + 0.1 * torch.from_numpy(g.standard_normal(D, dtype=np.float32))).to(torch.bfloat16)
    kw = (1 + 0.1 * torch.from_numpy(g.standard_normal(D, dtype=np.float32))).to(torch.bfloat16)
    cache = workloads.build_cos_sin_cache(128, R, 1e4)
    pos = torch.from_numpy(g.integers(0, 128, T)).to(torch.int32)
    eq, ek = oracle.apply(q, k, qw, kw, cache, pos, is_neox=True, eps=1e-6)
    dq_buf, dk_big = qbuf.cuda(), kbig.cuda()
    dq, dk = dq_buf[:, 1:5, :D], dk_big[:, 0:3, :D]
    qknr.apply(dq, dk, qw.cuda(), kw.cuda(), cache.cuda(), pos.cuda(), is_neox=True, eps=1e-6)
    torch.cuda.synchronize()
    _assert_close(dq.double().cpu().numpy(), eq, torch.bfloat16, "q")
    _assert_close(dk.double().cpu().numpy(), ek, torch.bfloat16, "k")
    # everything outside the two views keeps its bits
    mq = torch.ones(T, 6, 160, dtype=torch.bool)
    mq[:, 1:5, :D] = False
    mk = torch.ones(T, 4, 160, dtype=torch.bool)
    mk[:, 0:3, :D] = False
    assert torch.equal(dq_buf.cpu().view(torch.int16)[mq], qbuf.view(torch.int16)[mq])
    assert torch.equal(dk_big.cpu().view(torch.int16)[mk], kbig.view(torch.int16)[mk])


def test_extreme_values(qknr):
    """Zero heads, tiny and large magnitudes, eps = 0 on non-zero heads."""
    for dtype, scale, eps in (("bf16", 1e-20, 1e-6), ("bf16", 1e15, 1e-6), ("fp16", 3e3, 1e-6),
                              ("fp16", 1e-3, 0.0), ("bf16", 1.0, 0.0)):
        w = _make(128, 128, False, "i32", 50, 3, 2, dtype=dtype, seed=9, x_scale=scale, eps=eps)
        cpu = workloads.make_inputs(w)
        cpu["q"][3].zero_()
        if eps == 0.0:
            cpu["q"][3, :, 0] = 1.0        # keep every head non-zero when eps is 0
        _check_workload_inputs(qknr, w, cpu)


def _check_workload_inputs(q, w, cpu):
    eq, ek = _expected(cpu, w)
    dev = workloads.to_device(cpu, w, "cuda")
    _run_gpu(q, dev, w)
    _assert_close(dev["q"].double().cpu().numpy(), eq, w.torch_dtype, f"{w.name} q")
    _assert_close(dev["k"].double().cpu().numpy(), ek, w.torch_dtype, f"{w.name} k")


def test_position_zero_is_pure_rmsnorm(qknr):
    """Row 0 of the table is cos=1, sin=0: the output is the RMSNorm alone."""
    w = _make(128, 128, True, "i64", 40, 4, 4, seed=3)
    cpu = workloads.make_inputs(w)
    cpu["positions"].zero_()
    _check_workload_inputs(qknr, w, cpu)


def test_empty_and_errors_leave_inputs_untouched(qknr):
    w = _make(128, 64, False, "i32", 16, 2, 2)
    cpu = workloads.make_inputs(w)
    dev = workloads.to_device(cpu, w, "cuda")
    before_q, before_k = dev["q"].clone(), dev["k"].clone()
    s = torch.cuda.current_stream().cuda_stream
    common = (dev["q_w"].data_ptr(), dev["k_w"].data_ptr(), dev["cos_sin_cache"].data_ptr(),
              dev["positions"].data_ptr())
    qp, kp = dev["q"].data_ptr(), dev["k"].data_ptr()
    # num_tokens = 0: OK, nothing launched
    assert qknr.qknr_apply(qp, kp, *common, 0, 2, 2, 128, 64, 0, 256, 256, 128, 1e-6, 0, s) == 0
    # misaligned q
    assert qknr.qknr_apply(qp + 2, kp, *common, 16, 2, 2, 128, 64, 0, 256, 256, 128, 1e-6, 0, s) == 4
    # stride not a multiple of 8 elements
    assert qknr.qknr_apply(qp, kp, *common, 16, 2, 2, 128, 64, 0, 260, 256, 128, 1e-6, 0, s) == 4
    # unsupported shapes
    assert qknr.qknr_apply(qp, kp, *common, 16, 2, 2, 96, 64, 0, 256, 256, 128, 1e-6, 0, s) == 3
    assert qknr.qknr_apply(qp, kp, *common, 16, 2, 2, 128, 24, 1, 256, 256, 128, 1e-6, 0, s) == 3
    # invalid arguments
    assert qknr.qknr_apply(qp, kp, *common, -1, 2, 2, 128, 64, 0, 256, 256, 128, 1e-6, 0, s) == 2
    assert qknr.qknr_apply(qp, kp, *common, 16, 0, 2, 128, 64, 0, 256, 256, 128, 1e-6, 0, s) == 2
    assert qknr.qknr_apply(qp, qp, *common, 16, 2, 2, 128, 64, 0, 256, 256, 128, 1e-6, 0, s) == 2
    assert qknr.qknr_apply(qp, kp, *common, 16, 2, 2, 128, 64, 0, 256, 256, 64, 1e-6, 0, s) == 2
    assert qknr.qknr_apply(0, kp, *common, 16, 2, 2, 128, 64, 0, 256, 256, 128, 1e-6, 0, s) == 2
    assert qknr.qknr_apply(qp, kp, *common, 16, 2, 2, 128, 64, 0, 256, 256, 128, -1.0, 0, s) == 2
    assert qknr.qknr_apply(qp, kp, *common, 16, 2, 2, 128, 64, 0, 256, 256, 128, 1e-6, 7, s) == 2
    torch.cuda.synchronize()
    assert torch.equal(dev["q"], before_q) and torch.equal(dev["k"], before_k)


def test_checked_variant(qknr):
    w = _make(128, 128, False, "i64", 70, 4, 2, cache_len=64, seed=4)
    cpu = workloads.make_inputs(w)
    # all in range: same bits as the unchecked call
    dev_a = workloads.to_device(cpu, w, "cuda")
    dev_b = workloads.to_device(cpu, w, "cuda")
    _run_gpu(qknr, dev_a, w)
    qknr.apply_checked(dev_b["q"], dev_b["k"], dev_b["q_w"], dev_b["k_w"], dev_b["cos_sin_cache"],
                       dev_b["positions"], is_neox=False, eps=w.eps)
    assert torch.equal(dev_a["q"], dev_b["q"]) and torch.equal(dev_a["k"], dev_b["k"])
    # out-of-range tokens are reported and left untouched; the rest are computed
    bad = [5, 17, 69]
    cpu_bad = {k: v.clone() for k, v in cpu.items()}
    cpu_bad["positions"][5] = 64
    cpu_bad["positions"][17] = -3
    cpu_bad["positions"][69] = 10 ** 12
    dev = workloads.to_device(cpu_bad, w, "cuda")
    with pytest.raises(qknr.QknrError) as e:
        qknr.apply_checked(dev["q"], dev["k"], dev["q_w"], dev["k_w"], dev["cos_sin_cache"],
                           dev["positions"], is_neox=False, eps=w.eps)
    assert e.value.code == 6 and "3 token" in e.value.message and "index 5" in e.value.message
    good = torch.tensor([t for t in range(70) if t not in bad])
    badi = torch.tensor(bad)
    assert torch.equal(dev["q"][badi.cuda()].cpu(), cpu["q"][badi])
    assert torch.equal(dev["k"][badi.cuda()].cpu(), cpu["k"][badi])
    sub = {"q": cpu["q"][good], "k": cpu["k"][good], "q_w": cpu["q_w"], "k_w": cpu["k_w"],
           "cos_sin_cache": cpu["cos_sin_cache"], "positions": cpu["positions"][good]}
    eq, ek = _expected(sub, w)
    _assert_close(dev["q"][good.cuda()].double().cpu().numpy(), eq, w.torch_dtype, "q")
    _assert_close(dev["k"][good.cuda()].double().cpu().numpy(), ek, w.torch_dtype, "k")


def test_streams_and_repeat_determinism(qknr):
    """A side stream gives the same bits as the default one; runs repeat exactly."""
    base = workloads.get("gqa")
    w = workloads.scaled(base, 200, cache_len=4096)
    cpu = workloads.make_inputs(w)
    a = workloads.to_device(cpu, w, "cuda")
    b = workloads.to_device(cpu, w, "cuda")
    _run_gpu(qknr, a, w)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        qknr.apply(b["q"], b["k"], b["q_w"], b["k_w"], b["cos_sin_cache"], b["positions"],
                   is_neox=True, eps=w.eps)
    s.synchronize()
    assert torch.equal(a["q"], b["q"]) and torch.equal(a["k"], b["k"])
