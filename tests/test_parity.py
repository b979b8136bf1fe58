"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every comparison is element by element on the same seeded inputs, with the
bound max |gpu - oracle| <= 2^-7 |oracle| + 1e-5 (bf16) or 2^-10 |oracle| + 1e-5
(fp16), i.e. two units in the last place of the output dtype at the oracle
value plus 1e-5 absolute; a correctly rounded fp32 evaluation stays inside
half of that.

Sizes: each workload at a reduced token count that spans many warp items and
a ragged tail, and at its full size in the launch configuration the benchmark
times (every element compared, the oracle running in token chunks over the
host cores); a grid over head_dim x rope_dim x pairing x position
type x token counts 1/9/129 (the grid the deep-dive's own unit test uses,
"Step4"); GQA head counts; strided and padded layouts; and the edge cases.
"""
import dataclasses
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
    q.set_tuning(reset=True)
    yield q
    q.set_tuning(reset=True)


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


def _oracle_violation_chunked(cpu, got_q, got_k, w, chunk_elems=1 << 21):
    """Worst |gpu - oracle| / tolerance over every element of a full-size
    output. The oracle runs on token chunks spread over the host cores (its C
    code runs outside the GIL), so memory stays bounded whatever the size.
    got_q / got_k: the GPU's q and k, copied to the host."""
    import concurrent.futures
    T = w.num_tokens
    per_tok = (w.n_qo + w.n_kv) * w.head_dim
    chunk = max(1, chunk_elems // per_tok)

    def one(t0):
        t1 = min(T, t0 + chunk)
        eq, ek = oracle.apply(cpu["q"][t0:t1], cpu["k"][t0:t1], cpu["q_w"], cpu["k_w"],
                              cpu["cos_sin_cache"], cpu["positions"][t0:t1], is_neox=w.is_neox,
                              eps=w.eps)
        vq = oracle.max_violation(got_q[t0:t1].double().numpy(), eq, w.torch_dtype)
        vk = oracle.max_violation(got_k[t0:t1].double().numpy(), ek, w.torch_dtype)
        return max(vq, vk), t1 - t0

    threads = torch.get_num_threads()
    torch.set_num_threads(1)     # the parallelism is the chunks, not torch's
    try:
        with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
            res = list(ex.map(one, range(0, T, chunk)))
    finally:
        torch.set_num_threads(threads)
    assert sum(n for _, n in res) == T
    return max(v for v, _ in res)


FULL = ["tiny", "dit", "mha_neox", "gqa", "fused_qkv"]


@pytest.mark.parametrize("name", FULL)
def test_workload_full_size_every_element(qknr, name):
    """Full size, in the launch the benchmark times (the default work map):
    every element of q and k against the oracle, and V (fused_qkv) bit for
    bit unchanged."""
    w = workloads.get(name)
    cpu = workloads.make_inputs(w)
    dev = workloads.to_device(cpu, w, "cuda")
    m = qknr.work_map(w.num_tokens, w.n_qo, w.n_kv, w.head_dim, w.rope_dim, w.is_neox,
                      qknr.dtype_code(w.torch_dtype, w.pos_torch_dtype))
    _run_gpu(qknr, dev, w)
    got_q, got_k = dev["q"].cpu(), dev["k"].cpu()
    v = _oracle_violation_chunked(cpu, got_q, got_k, w)
    assert v <= 1.0, f"{name}: max error {v:.3f} x tolerance (work map {m})"
    if w.fused_total_heads:
        lo = w.n_qo + w.n_kv
        assert torch.equal(dev["buffer"][:, lo:, :].cpu().view(torch.int16),
                           cpu["buffer"][:, lo:, :].view(torch.int16))


@pytest.mark.parametrize("name", ["dit", "mha_neox", "gqa", "fused_qkv"])
def test_kernels_agree_at_full_size(qknr, name):
    """Full size: the register kernel and the ring kernel in both issue orders,
    each forced, give the same bits on copies of one input (the default launch
    of each workload is compared with the oracle element by element above, so
    every kernel is pinned to it at the sizes the benchmark runs)."""
    w = workloads.get(name)
    cpu = workloads.make_inputs(w)
    outs = []
    for kernel, ring_order in (("register", 0), ("ring", 1), ("ring", 2)):
        dev = workloads.to_device(cpu, w, "cuda")
        qknr.set_tuning(reset=True, kernel=kernel, ring_order=ring_order)
        try:
            _run_gpu(qknr, dev, w)
        finally:
            qknr.set_tuning(reset=True)
        key = "buffer" if w.fused_total_heads else None
        outs.append([dev[key].view(torch.int16)] if key else [dev["q"].view(torch.int16),
                                                              dev["k"].view(torch.int16)])
        del dev
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            assert torch.equal(a, b), name


def _rope_dims(D, neox):
    if neox:
        return sorted({r for r in (4, 8, 16, 32, 64, D // 2, D) if r <= D and (r % 16 == 0 or r <= 8)})
    return sorted({r for r in (2, 6, 8, 24, 64, D // 2, D - 8, D) if 0 < r <= D})


GRID = [(D, R, neox, pos, T)
        for D in (64, 80, 96, 128, 192, 256)
        for neox in (False, True)
        for R in _rope_dims(D, neox)
        for pos in ("i32", "i64")
        for T in (1, 9, 129)]


def _make(D, R, neox, pos, T, n_qo, n_kv, dtype="bf16", seed=0, cache_len=300, base=1e4,
          pos_kind="uniform", eps=1e-6, x_scale=1.0):
    return workloads.Workload(f"grid_{D}_{R}_{int(neox)}_{pos}_{T}", dtype, T, n_qo, n_kv, D, R,
                              neox, base, cache_len, pos, pos_kind, eps, x_scale=x_scale,
                              seed=seed)


@pytest.mark.parametrize("kernel,order", [("register", "interleaved"), ("register", "contiguous"),
                                          ("ring", "interleaved"), ("ring", "contiguous"),
                                          ("ring2", "interleaved")])
@pytest.mark.parametrize("D,R,neox,pos,T", GRID,
                         ids=[f"D{g[0]}-R{g[1]}-{'neox' if g[2] else 'inter'}-{g[3]}-T{g[4]}"
                              for g in GRID])
def test_shape_grid(qknr, D, R, neox, pos, T, kernel, order):
    """The grid with both kernels forced, in both item orders (interleaved is
    the automatic one), and the ring kernel's second issue order ("ring2")."""
    w = _make(D, R, neox, pos, T, 4, 2, dtype="bf16" if (D + R + T) % 2 == 0 else "fp16")
    qknr.set_tuning(reset=True, kernel=kernel.rstrip("2"), ring_order=2 if kernel == "ring2" else 0,
                    order=2 if order == "interleaved" else 1)
    try:
        _check_workload(qknr, w)
    finally:
        qknr.set_tuning(reset=True)


RING_MULTIPASS = [(D, neox, order) for D in (64, 80, 96, 128, 192, 256) for neox in (False, True)
                  for order in (1, 2)]


@pytest.mark.parametrize("D,neox,order", RING_MULTIPASS,
                         ids=[f"D{c[0]}-{'neox' if c[1] else 'inter'}-order{c[2]}" for c in RING_MULTIPASS])
def test_ring_multi_pass_items(D, neox, order, qknr):
    """The ring kernel on calls large enough for items of three or four warp
    passes (the rule's launch for such calls), at every head_dim, including
    80, 96 and 192 whose lane groups have idle lanes, in both issue orders:
    against the oracle, and bit for bit against the register kernel."""
    R = _neox_half(D) if neox else (D if D % 32 == 0 else D // 2)
    w = _make(D, R, neox, "i64" if neox else "i32", 1200, 24, 8, dtype="fp16" if D % 64 else "bf16",
              seed=D + 7 * order + int(neox), cache_len=2048)
    m = qknr.work_map(w.num_tokens, w.n_qo, w.n_kv, D, R, neox,
                      qknr.dtype_code(w.torch_dtype, w.pos_torch_dtype))
    assert m["unroll"] == 4 and m["kernel"] == "ring", m
    cpu = workloads.make_inputs(w)
    ref = workloads.to_device(cpu, w, "cuda")
    qknr.set_tuning(reset=True, kernel="register")
    try:
        _run_gpu(qknr, ref, w)
        qknr.set_tuning(reset=True, kernel="ring", ring_order=order)
        dev = workloads.to_device(cpu, w, "cuda")
        _run_gpu(qknr, dev, w)
    finally:
        qknr.set_tuning(reset=True)
    assert torch.equal(dev["q"].view(torch.int16), ref["q"].view(torch.int16))
    assert torch.equal(dev["k"].view(torch.int16), ref["k"].view(torch.int16))
    eq, ek = _expected(cpu, w)
    _assert_close(dev["q"].double().cpu().numpy(), eq, w.torch_dtype, "q")
    _assert_close(dev["k"].double().cpu().numpy(), ek, w.torch_dtype, "k")


def _neox_half(D):
    """A NeoX rope_dim near half of head_dim that the op takes (a multiple of 16)."""
    return D // 2 if (D // 2) % 16 == 0 else (D // 2) // 16 * 16


@pytest.mark.parametrize("n_qo,n_kv", [(1, 1), (8, 1), (32, 8), (5, 3), (1, 7), (64, 64)])
@pytest.mark.parametrize("D", [64, 80, 96, 128, 192, 256])
def test_gqa_head_counts(qknr, n_qo, n_kv, D):
    w = _make(D, _neox_half(D), True, "i64", 33, n_qo, n_kv, dtype="fp16", seed=n_qo * 100 + n_kv)
    _check_workload(qknr, w)


TUNINGS = [
    dict(passes=1, threads=64, ctas_per_sm=1),
    dict(passes=2, threads=128),
    dict(passes=3, threads=256, ctas_per_sm=2),
    dict(passes=4, threads=512),
    dict(passes=4, threads=64, pdl=0),
    dict(order=1),
    dict(order=2, passes=1, threads=64, ctas_per_sm=1),
    dict(order=2, passes=3, threads=512),
    dict(ctas_per_sm=1),
    dict(passes=1, pdl=0, order=1),
    dict(prefetch=-1),
    dict(prefetch=1, order=1),
    dict(prefetch=2, passes=1, threads=64),
    dict(prefetch=4, pdl=0),
    dict(kernel=1),
    dict(kernel=2),
    dict(kernel=2, passes=1, threads=64, ctas_per_sm=1),
    dict(kernel=2, passes=2, threads=128),
    dict(kernel=2, passes=3, threads=512),
    dict(kernel=2, order=1, prefetch=-1),
    dict(kernel=2, pdl=0, prefetch=1),
    dict(kernel=2, threads=64, ctas_per_sm=2, prefetch=2),
    dict(kernel=2, ring_order=1, passes=4, threads=512),
    dict(kernel=2, ring_order=2),
    dict(kernel=2, ring_order=2, passes=1, threads=64, ctas_per_sm=1),
    dict(kernel=2, ring_order=2, passes=3, order=1, prefetch=-1),
    dict(kernel=2, ring_order=2, pdl=0, threads=128),
]


@pytest.mark.parametrize("tuning", TUNINGS, ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_tunings_agree_bit_for_bit(qknr, tuning):
    """Per-head results do not depend on the launch tuning: every forced setting
    gives the same bits as the automatic one, and all match the oracle. Covers
    one to four passes per item, several items per token, both item orders,
    one or two CTAs per SM, launches with and without programmatic dependent
    launch, every depth of the L2 prefetch before the wait, and both kernels
    (register and ring) under each kind of setting."""
    for name, T in (("mha_neox", 97), ("fused_qkv", 41), ("tiny", 16), ("gqa", 50)):
        base = workloads.get(name)
        w = workloads.scaled(base, T, cache_len=min(base.cache_len, 4096))
        cpu = workloads.make_inputs(w)
        ref = workloads.to_device(cpu, w, "cuda")
        qknr.set_tuning(reset=True)
        _run_gpu(qknr, ref, w)
        dev = workloads.to_device(cpu, w, "cuda")
        qknr.set_tuning(reset=True, **tuning)
        try:
            _run_gpu(qknr, dev, w)
        finally:
            qknr.set_tuning(reset=True)
        assert torch.equal(dev["q"].view(torch.int16), ref["q"].view(torch.int16)), name
        assert torch.equal(dev["k"].view(torch.int16), ref["k"].view(torch.int16)), name
        eq, ek = _expected(cpu, w)
        _assert_close(dev["q"].double().cpu().numpy(), eq, w.torch_dtype, name)
        _assert_close(dev["k"].double().cpu().numpy(), ek, w.torch_dtype, name)


def test_work_map_choice(qknr):
    """The automatic launch: 4-pass items interleaved over a persistent grid of
    at most one wave of resident CTAs on the ring kernel, which issues each
    item's successor once the item's bytes land (order 1), or, for interleaved
    bf16 calls with head_dim 64/128/256 whose warps run at least 6.5 rounds of
    items, two items ahead (order 2); 1-pass items on the register kernel for a
    call too small to give every SM several warps."""
    bf, fp = qknr.QKNR_BF16, qknr.QKNR_FP16 | qknr.QKNR_POS_I64
    m = qknr.work_map(4608, 24, 24, 128, 128, False, bf)           # DiT: 113 MB of q and k
    assert m["kernel"] == "ring" and m["ring_order"] == 1 and m["order"] == "interleaved"
    assert m["unroll"] == 4 and m["passes_per_token"] == 12 and m["items_per_token"] == 3
    assert m["items"] == 4608 * 3 and m["threads"] == 64 and m["pdl"] == 1     # CTAs of two warps
    assert m["prefetch_items"] == 1 and m["rope_dim_compiled"] == 128
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert m["grid"] <= m["ctas_per_sm"] * sms and m["ctas_per_sm"] == 8
    big = qknr.work_map(65536, 16, 4, 256, 128, False, bf)                      # 1.3 GB
    assert big["kernel"] == "ring" and big["ring_order"] == 2 and big["threads"] == 512   # 81 rounds
    assert big["ctas_per_sm"] == 1 and big["grid"] == sms
    for T in (16384, 65536):                                                   # NeoX: any size
        g = qknr.work_map(T, 32, 8, 128, 64, True, fp)
        assert g["kernel"] == "ring" and g["ring_order"] == 1 and g["threads"] == 256
    warps = m["grid"] * m["threads"] // 32                           # one wave, 3 items per token
    assert warps == 16 * sms
    first = -(-13 * warps // 6)                                      # 3 T / warps >= 6.5
    assert qknr.work_map(first - 1, 24, 24, 128, 128, False, bf)["ring_order"] == 1
    mid = qknr.work_map(first, 24, 24, 128, 128, False, bf)
    assert mid["ring_order"] == 2 and mid["threads"] == 256                       # 6.5 rounds
    long_ = qknr.work_map(-(-32 * warps // 3), 24, 24, 128, 128, False, bf)
    assert long_["ring_order"] == 2 and long_["threads"] == 512
    assert qknr.work_map(4 * first, 24, 24, 128, 128, True, bf)["ring_order"] == 1   # NeoX
    assert qknr.work_map(4 * first, 24, 24, 128, 128, False, qknr.QKNR_FP16)["ring_order"] == 1
    assert qknr.work_map(4 * first, 24, 24, 96, 96, False, bf)["ring_order"] == 1     # idle lanes
    small = qknr.work_map(4, 4, 2, 128, 6, False, bf)
    assert small["kernel"] == "register" and small["items_per_token"] == small["passes_per_token"]
    assert small["ring_order"] == 0 and small["prefetch_items"] == 4
    assert qknr.work_map(4, 4, 2, 128, 64, True, fp)["kernel"] == "register"


KERNELS = {"register": dict(kernel="register"), "ring": dict(kernel="ring", ring_order=1),
           "ring2": dict(kernel="ring", ring_order=2)}


@pytest.mark.parametrize("kernel", list(KERNELS))
def test_separate_strides_and_padded_heads(qknr, kernel):
    """q and k views with different token strides and a head stride > head_dim,
    on each kernel and ring order."""
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
    qknr.set_tuning(reset=True, **KERNELS[kernel])
    try:
        qknr.apply(dq, dk, qw.cuda(), kw.cuda(), cache.cuda(), pos.cuda(), is_neox=True, eps=1e-6)
        torch.cuda.synchronize()
    finally:
        qknr.set_tuning(reset=True)
    _assert_close(dq.double().cpu().numpy(), eq, torch.bfloat16, "q")
    _assert_close(dk.double().cpu().numpy(), ek, torch.bfloat16, "k")
    # everything outside the two views keeps its bits
    mq = torch.ones(T, 6, 160, dtype=torch.bool)
    mq[:, 1:5, :D] = False
    mk = torch.ones(T, 4, 160, dtype=torch.bool)
    mk[:, 0:3, :D] = False
    assert torch.equal(dq_buf.cpu().view(torch.int16)[mq], qbuf.view(torch.int16)[mq])
    assert torch.equal(dk_big.cpu().view(torch.int16)[mk], kbig.view(torch.int16)[mk])


STRIDED = [(6, 2, 0, 32, 128, True), (4, 4, 64, 0, 64, False), (1, 3, 0, 16, 256, False),
           (3, 1, 8, 0, 96, True), (5, 3, 8, 24, 192, False), (24, 24, 0, 128, 128, False)]


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("n_qo,n_kv,q_pad,k_pad,D,neox", STRIDED,
                         ids=[f"q{c[0]}+{c[2]}-k{c[1]}+{c[3]}-D{c[4]}" for c in STRIDED])
def test_independent_head_strides(qknr, n_qo, n_kv, q_pad, k_pad, D, neox, kernel):
    """q and k heads with their own strides (qknr_apply_strided, through the
    raw entry point and through apply()), each kernel and ring order forced:
    the same bits as qknr_apply on contiguous copies, within the oracle's
    tolerance, padding untouched."""
    T, R = 131, D // 2 if neox else D
    g = np.random.default_rng(n_qo * 7 + n_kv + D)
    qbuf = torch.from_numpy(g.standard_normal((T, n_qo, D + q_pad), dtype=np.float32)).to(torch.bfloat16)
    kbuf = torch.from_numpy(g.standard_normal((T, n_kv, D + k_pad), dtype=np.float32)).to(torch.bfloat16)
    qw = (1 + 0.1 * torch.from_numpy(g.standard_normal(D, dtype=np.float32))).to(torch.bfloat16)
    kw = (1 + 0.1 * torch.from_numpy(g.standard_normal(D, dtype=np.float32))).to(torch.bfloat16)
    cache = workloads.build_cos_sin_cache(256, R, 1e4)
    pos = torch.from_numpy(g.integers(0, 256, T)).to(torch.int32)
    qc, kc = qbuf[:, :, :D].contiguous(), kbuf[:, :, :D].contiguous()
    eq, ek = oracle.apply(qc, kc, qw, kw, cache, pos, is_neox=neox, eps=1e-6)
    ref_q, ref_k = qc.cuda(), kc.cuda()
    dw = (qw.cuda(), kw.cuda(), cache.cuda(), pos.cuda())
    qknr.apply(ref_q, ref_k, *dw, is_neox=neox, eps=1e-6)
    for route in ("raw", "apply"):
        dq_buf, dk_buf = qbuf.cuda(), kbuf.cuda()
        dq, dk = dq_buf[:, :, :D], dk_buf[:, :, :D]
        qknr.set_tuning(reset=True, **KERNELS[kernel])
        if route == "raw":
            rc = qknr.qknr_apply_strided(dq.data_ptr(), dk.data_ptr(), dw[0].data_ptr(),
                                         dw[1].data_ptr(), dw[2].data_ptr(), dw[3].data_ptr(), T,
                                         n_qo, n_kv, D, R, int(neox), dq.stride(0), dk.stride(0),
                                         dq.stride(1), dk.stride(1), 1e-6, qknr.QKNR_BF16, None)
            assert rc == 0, qknr.qknr_last_error()
        else:
            qknr.apply(dq, dk, *dw, is_neox=neox, eps=1e-6)
        torch.cuda.synchronize()
        qknr.set_tuning(reset=True)
        assert torch.equal(dq.cpu().view(torch.int16), ref_q.cpu().view(torch.int16)), route
        assert torch.equal(dk.cpu().view(torch.int16), ref_k.cpu().view(torch.int16)), route
        _assert_close(dq.double().cpu().numpy(), eq, torch.bfloat16, "q")
        _assert_close(dk.double().cpu().numpy(), ek, torch.bfloat16, "k")
        assert torch.equal(dq_buf[:, :, D:].cpu(), qbuf[:, :, D:])
        assert torch.equal(dk_buf[:, :, D:].cpu(), kbuf[:, :, D:])


def test_independent_head_strides_errors(qknr):
    T, D = 4, 64
    q = torch.zeros(T, 2, D, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(T, 2, D + 8, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(D, dtype=torch.bfloat16, device="cuda")
    cache = workloads.build_cos_sin_cache(8, D, 1e4).cuda()
    pos = torch.zeros(T, dtype=torch.int32, device="cuda")
    args = (q.data_ptr(), k.data_ptr(), w.data_ptr(), w.data_ptr(), cache.data_ptr(),
            pos.data_ptr(), T, 2, 2, D, D, 0, 2 * D, 2 * (D + 8))
    for q_hs, k_hs, code in ((D, -8, 2), (D, 32, 2), (D, D + 4, 4), (D, D + 8, 0)):
        rc = qknr.qknr_apply_strided(*args, q_hs, k_hs, 1e-6, qknr.QKNR_BF16, None)
        assert rc == code, (q_hs, k_hs, rc, qknr.qknr_last_error())
    torch.cuda.synchronize()


@pytest.mark.parametrize("kernel", ["register", "ring", "ring2"])
@pytest.mark.parametrize("pdl", [-1, 0])
def test_cuda_graph_capture_and_replay(qknr, pdl, kernel):
    """Calls captured into a CUDA graph (two calls on different buffers, with
    programmatic dependent launch on or off, either kernel forced) replay to
    the same bits as eager calls, on new values written into the captured
    buffers."""
    base = workloads.get("gqa")
    ws = [workloads.scaled(base, 70, cache_len=4096), workloads.scaled(workloads.get("dit"), 33)]
    qknr.set_tuning(pdl=pdl, kernel=kernel.rstrip("2"), ring_order=2 if kernel == "ring2" else 0)
    try:
        devs = [workloads.to_device(workloads.make_inputs(w), w, "cuda") for w in ws]
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for w, d in zip(ws, devs):   # warm-up outside capture (plans and occupancy cached)
                qknr.apply(d["q"], d["k"], d["q_w"], d["k_w"], d["cos_sin_cache"], d["positions"],
                           is_neox=w.is_neox, eps=w.eps)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for w, d in zip(ws, devs):
                qknr.apply(d["q"], d["k"], d["q_w"], d["k_w"], d["cos_sin_cache"], d["positions"],
                           is_neox=w.is_neox, eps=w.eps)
        for seed in (11, 12):
            fresh = [workloads.make_inputs(dataclasses.replace(w, seed=seed)) for w in ws]
            refs = []
            for w, d, f in zip(ws, devs, fresh):
                d["q"].copy_(f["q"])
                d["k"].copy_(f["k"])
                r = workloads.to_device(f, w, "cuda")
                qknr.apply(r["q"], r["k"], d["q_w"], d["k_w"], d["cos_sin_cache"], d["positions"],
                           is_neox=w.is_neox, eps=w.eps)
                refs.append(r)
            graph.replay()
            torch.cuda.synchronize()
            for d, r in zip(devs, refs):
                assert torch.equal(d["q"].view(torch.int16), r["q"].view(torch.int16))
                assert torch.equal(d["k"].view(torch.int16), r["k"].view(torch.int16))
    finally:
        qknr.set_tuning(reset=True)


def test_guard_bands_around_q_and_k(qknr):
    """Canary bytes right before q, between q and k and right after k (one
    allocation) keep every bit, for several launch tunings."""
    w = _make(128, 64, True, "i64", 97, 6, 2, dtype="fp16", seed=4)
    cpu = workloads.make_inputs(w)
    eq, ek = _expected(cpu, w)
    nq, nk, pad = cpu["q"].numel(), cpu["k"].numel(), 4096
    for tune in ({}, {"order": 1}, {"passes": 1, "threads": 64}, {"kernel": "ring", "ring_order": 1},
                 {"kernel": "ring", "ring_order": 2, "passes": 3}, {"kernel": "ring", "order": 1, "threads": 64}):
        buf = torch.full((pad + nq + pad + nk + pad,), -31.0, dtype=torch.float16, device="cuda")
        dq = buf[pad:pad + nq].view(cpu["q"].shape)
        dk = buf[2 * pad + nq:2 * pad + nq + nk].view(cpu["k"].shape)
        dq.copy_(cpu["q"])
        dk.copy_(cpu["k"])
        dev = workloads.to_device(cpu, w, "cuda")
        qknr.set_tuning(reset=True, **tune)
        try:
            qknr.apply(dq, dk, dev["q_w"], dev["k_w"], dev["cos_sin_cache"], dev["positions"],
                       is_neox=w.is_neox, eps=w.eps)
            torch.cuda.synchronize()
        finally:
            qknr.set_tuning(reset=True)
        host = buf.cpu()
        for lo, hi in ((0, pad), (pad + nq, 2 * pad + nq), (2 * pad + nq + nk, 3 * pad + nq + nk)):
            assert (host[lo:hi] == -31.0).all(), (tune, lo)
        _assert_close(dq.double().cpu().numpy(), eq, torch.float16, f"q {tune}")
        _assert_close(dk.double().cpu().numpy(), ek, torch.float16, f"k {tune}")


_LOG_SCRIPT = r"""
import sys
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})
import torch, workloads
import qk_rmsnorm_rope_gb300 as q
q.init(0)
w = workloads.scaled(workloads.get("dit"), 40)
d = workloads.to_device(workloads.make_inputs(w), w, "cuda")
for _ in range(3):
    q.apply(d["q"], d["k"], d["q_w"], d["k_w"], d["cos_sin_cache"], d["positions"], is_neox=False)
w2 = workloads.scaled(w, 41)
d2 = workloads.to_device(workloads.make_inputs(w2), w2, "cuda")
q.apply(d2["q"], d2["k"], d2["q_w"], d2["k_w"], d2["cos_sin_cache"], d2["positions"], is_neox=False)
torch.cuda.synchronize()
"""


def test_log_prints_once_per_shape(qknr):
    """QKNR_LOG=1 prints one line per distinct call shape (fresh process)."""
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, QKNR_LOG="1")
    r = subprocess.run([sys.executable, "-c", _LOG_SCRIPT.format(root=root, tests=os.path.dirname(
        os.path.abspath(__file__)))], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("qknr: ")]
    assert len(lines) == 2, r.stderr
    assert "T=40 " in lines[0] and "T=41 " in lines[1] and "register kernel" in lines[0]


def test_pass_bound_table_and_division_agree(qknr):
    """Interleaved items take their passes from a host table when a token has
    at most 32 items, else by division: 160 heads of D=128 give 40 passes per
    token, so one pass per item (decode-sized calls) takes the division and 4
    passes per item take the table. Same bits either way, within tolerance."""
    w = _make(128, 128, False, "i32", 37, 80, 80, dtype="bf16", seed=21)
    cpu = workloads.make_inputs(w)
    eq, ek = _expected(cpu, w)
    outs = []
    for passes in (1, 4):
        qknr.set_tuning(reset=True, passes=passes)
        try:
            m = qknr.work_map(w.num_tokens, w.n_qo, w.n_kv, w.head_dim, w.rope_dim, w.is_neox,
                              qknr.QKNR_BF16)
            assert m["items_per_token"] == (40 if passes == 1 else 10)
            dev = workloads.to_device(cpu, w, "cuda")
            _run_gpu(qknr, dev, w)
        finally:
            qknr.set_tuning(reset=True)
        _assert_close(dev["q"].double().cpu().numpy(), eq, w.torch_dtype, f"q passes={passes}")
        _assert_close(dev["k"].double().cpu().numpy(), ek, w.torch_dtype, f"k passes={passes}")
        outs.append((dev["q"].cpu(), dev["k"].cpu()))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int16), outs[1][1].view(torch.int16))


def _random_case(g):
    D = int(g.choice([64, 80, 96, 128, 192, 256]))
    neox = bool(g.integers(0, 2))
    if neox:
        R = int(g.choice([r for r in (2, 4, 6, 8, 16, 32, 48, 64, 96, 128, 192, 256) if r <= D and
                          (r % 16 == 0 or r <= 8)]))
    else:
        R = int(g.choice([r for r in range(2, D + 1, 2)]))
    return dict(D=D, R=R, neox=neox, T=int(g.integers(1, 70)), n_qo=int(g.integers(1, 20)),
                n_kv=int(g.integers(1, 9)), dtype=str(g.choice(["bf16", "fp16"])),
                pos=str(g.choice(["i32", "i64"])), head_pad=int(g.choice([0, 0, 8, 24])),
                tok_pad=int(g.choice([0, 0, 8, 40])), order=int(g.choice([0, 0, 1, 2, 0])),
                passes=int(g.integers(0, 5)), threads=int(g.choice([0, 64, 128, 256, 512])))


@pytest.mark.parametrize("case", range(40))
def test_random_configurations(qknr, case):
    """Seeded random configurations: head_dim, rope_dim, pairing, dtype,
    position type, GQA head counts, padded head and token strides, launch
    tuning (item order, passes per item, threads) and the early-read flag
    together. Against the oracle, and
    bit for bit against the automatic launch on a contiguous copy."""
    g = np.random.default_rng(1000 + case)
    c = _random_case(g)
    w = _make(c["D"], c["R"], c["neox"], c["pos"], c["T"], c["n_qo"], c["n_kv"], dtype=c["dtype"],
              seed=case, cache_len=97)
    cpu = workloads.make_inputs(w)
    eq, ek = _expected(cpu, w)
    D, hs = c["D"], c["D"] + c["head_pad"]
    dt = w.torch_dtype

    def strided(x, n):
        buf = torch.full((c["T"], n * hs + c["tok_pad"]), -5.0, dtype=dt, device="cuda")
        view = buf[:, :n * hs].view(c["T"], n, hs)[:, :, :D]
        view.copy_(x)
        return buf, view

    qbuf, dq = strided(cpu["q"], c["n_qo"])
    kbuf, dk = strided(cpu["k"], c["n_kv"])
    dev = workloads.to_device(cpu, w, "cuda")
    tune = {"order": c["order"]}
    if c["passes"]:
        tune["passes"] = c["passes"]
    if c["threads"]:
        tune["threads"] = c["threads"]
    # half of the cases take the early-read instantiations (a draw of its own,
    # so that the configurations above stay what they were)
    ready = bool(np.random.default_rng(5000 + case).random() < 0.5)
    c["inputs_ready"] = ready
    qknr.set_tuning(reset=True, **tune)
    try:
        qknr.apply(dq, dk, dev["q_w"], dev["k_w"], dev["cos_sin_cache"], dev["positions"],
                   is_neox=w.is_neox, eps=w.eps, inputs_ready=ready)
        torch.cuda.synchronize()
    finally:
        qknr.set_tuning(reset=True)
    _assert_close(dq.double().cpu().numpy(), eq, dt, f"q {c}")
    _assert_close(dk.double().cpu().numpy(), ek, dt, f"k {c}")
    ref = workloads.to_device(cpu, w, "cuda")
    _run_gpu(qknr, ref, w)
    assert torch.equal(dq.cpu().view(torch.int16), ref["q"].cpu().view(torch.int16)), c
    assert torch.equal(dk.cpu().view(torch.int16), ref["k"].cpu().view(torch.int16)), c
    # bytes outside the heads keep every bit
    for buf, n in ((qbuf, c["n_qo"]), (kbuf, c["n_kv"])):
        host = buf.cpu()
        mask = torch.ones_like(host, dtype=torch.bool)
        mask[:, :n * hs].view(c["T"], n, hs)[:, :, :D] = False
        assert (host[mask] == -5.0).all(), c


def test_positions_are_converted(qknr):
    """apply() takes positions of any integer type, on the host or the device,
    converting them to q's device first (the reference wrapper does the same);
    on a side stream too. Same bits as device int32 positions. Float positions
    are refused."""
    w = _make(128, 64, True, "i32", 61, 8, 2, dtype="bf16", seed=31, cache_len=120)
    cpu = workloads.make_inputs(w)
    ref = workloads.to_device(cpu, w, "cuda")
    _run_gpu(qknr, ref, w)
    p32 = cpu["positions"]
    variants = [p32.to(torch.int64), p32.to(torch.int16), p32.to(torch.uint8), p32,
                p32.cuda().to(torch.int16), p32.to(torch.int64)[::1]]
    side = torch.cuda.Stream()
    for i, pos in enumerate(variants):
        dev = workloads.to_device(cpu, w, "cuda")
        stream = side if i % 2 else None
        qknr.apply(dev["q"], dev["k"], dev["q_w"], dev["k_w"], dev["cos_sin_cache"], pos,
                   is_neox=w.is_neox, eps=w.eps, stream=stream)
        torch.cuda.synchronize()
        assert torch.equal(dev["q"].view(torch.int16), ref["q"].view(torch.int16)), (i, pos.dtype)
        assert torch.equal(dev["k"].view(torch.int16), ref["k"].view(torch.int16)), (i, pos.dtype)
    dev = workloads.to_device(cpu, w, "cuda")
    with pytest.raises(qknr.QknrError):
        qknr.apply(dev["q"], dev["k"], dev["q_w"], dev["k_w"], dev["cos_sin_cache"],
                   p32.float(), is_neox=w.is_neox, eps=w.eps)


def test_four_d_inputs(qknr):
    """[B, S, H, D] q and k whose batch and sequence dims merge without a copy
    run in place (same bits as the 3-D call); ones that do not are refused."""
    w = _make(64, 64, False, "i32", 63, 4, 2, dtype="fp16", seed=41, cache_len=80)
    cpu = workloads.make_inputs(w)
    ref = workloads.to_device(cpu, w, "cuda")
    _run_gpu(qknr, ref, w)
    dev = workloads.to_device(cpu, w, "cuda")
    q4, k4 = dev["q"].view(3, 21, 4, 64), dev["k"].view(3, 21, 2, 64)
    qknr.apply(q4, k4, dev["q_w"], dev["k_w"], dev["cos_sin_cache"], dev["positions"],
               is_neox=False, eps=w.eps)
    torch.cuda.synchronize()
    assert torch.equal(dev["q"].view(torch.int16), ref["q"].view(torch.int16))
    assert torch.equal(dev["k"].view(torch.int16), ref["k"].view(torch.int16))
    qt = dev["q"].view(3, 21, 4, 64).transpose(0, 1)     # [S, B, H, D]: no single token stride
    kt = dev["k"].view(3, 21, 2, 64).transpose(0, 1)
    with pytest.raises(qknr.QknrError, match="merge"):
        qknr.apply(qt, kt, dev["q_w"], dev["k_w"], dev["cos_sin_cache"], dev["positions"],
                   is_neox=False, eps=w.eps)


@pytest.mark.parametrize("order", [2, 1])
def test_offsets_beyond_two_gib(qknr, order):
    """q spans 2.5 GB, so its last tokens sit more than 2^31 bytes from its
    start (64-bit addressing); sampled tokens over the whole range against the
    oracle, in both item orders. Inputs are drawn on the device (seeded),
    samples copied back."""
    T, n_qo, n_kv, D, R, L = 600_000, 16, 4, 128, 128, 4096
    g = torch.Generator(device="cuda").manual_seed(77)
    q = torch.randn(T, n_qo, D, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn(T, n_kv, D, device="cuda", generator=g).to(torch.bfloat16)
    assert (T - 1) * q.stride(0) * 2 > 2 ** 31
    qw = (1 + 0.1 * torch.randn(D, device="cuda", generator=g)).to(torch.bfloat16)
    kw = (1 + 0.1 * torch.randn(D, device="cuda", generator=g)).to(torch.bfloat16)
    cache = workloads.build_cos_sin_cache(L, R, 1e4)
    pos = torch.randint(0, L, (T,), device="cuda", generator=g, dtype=torch.int64)
    idx = _sample_tokens(T, 96, 5)
    idx = torch.cat([idx, torch.arange(T - 8, T)]).unique()
    q0, k0, p0 = q[idx.cuda()].cpu(), k[idx.cuda()].cpu(), pos[idx.cuda()].cpu()
    qknr.set_tuning(reset=True, order=order)
    try:
        qknr.apply(q, k, qw, kw, cache.cuda(), pos, is_neox=False, eps=1e-6)
        torch.cuda.synchronize()
    finally:
        qknr.set_tuning(reset=True)
    eq, ek = oracle.apply(q0, k0, qw.cpu(), kw.cpu(), cache, p0, is_neox=False, eps=1e-6)
    _assert_close(q[idx.cuda()].double().cpu().numpy(), eq, torch.bfloat16, "q beyond 2 GiB")
    _assert_close(k[idx.cuda()].double().cpu().numpy(), ek, torch.bfloat16, "k")
    del q, k


INPUTS_READY_CASES = [("tiny", 16, {}), ("dit", 300, {}), ("mha_neox", 257, {}), ("gqa", 513, {}),
                      ("fused_qkv", 129, {}), ("gqa", 40, {"passes": 1}), ("dit", 77, {"threads": 512}),
                      ("mha_neox", 33, {"passes": 2, "threads": 64})]


@pytest.mark.parametrize("name,T,tune", INPUTS_READY_CASES,
                         ids=[f"{c[0]}-T{c[1]}-{c[2]}" for c in INPUTS_READY_CASES])
def test_inputs_ready_same_bits_and_ordering(qknr, name, T, tune):
    """QKNR_INPUTS_READY only moves the weight and position reads before the
    wait for the previous kernel: the same bits as without it, also when the
    previous kernel wrote q and k (two calls in a row on the same tensors, so
    the second reads what the first wrote), and under graph capture."""
    base = workloads.get(name)
    w = workloads.scaled(base, T, cache_len=min(base.cache_len, 4096))
    cpu = workloads.make_inputs(w)
    qknr.set_tuning(reset=True, **tune)
    try:
        ref = workloads.to_device(cpu, w, "cuda")
        for _ in range(2):
            qknr.apply(ref["q"], ref["k"], ref["q_w"], ref["k_w"], ref["cos_sin_cache"],
                       ref["positions"], is_neox=w.is_neox, eps=w.eps)
        dev = workloads.to_device(cpu, w, "cuda")
        for _ in range(2):
            qknr.apply(dev["q"], dev["k"], dev["q_w"], dev["k_w"], dev["cos_sin_cache"],
                       dev["positions"], is_neox=w.is_neox, eps=w.eps, inputs_ready=True)
        torch.cuda.synchronize()
        assert torch.equal(dev["q"].view(torch.int16), ref["q"].view(torch.int16))
        assert torch.equal(dev["k"].view(torch.int16), ref["k"].view(torch.int16))
        # captured: two calls in one graph, replayed on fresh values
        g_dev = workloads.to_device(cpu, w, "cuda")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            qknr.apply(g_dev["q"], g_dev["k"], g_dev["q_w"], g_dev["k_w"], g_dev["cos_sin_cache"],
                       g_dev["positions"], is_neox=w.is_neox, eps=w.eps, inputs_ready=True)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(2):
                qknr.apply(g_dev["q"], g_dev["k"], g_dev["q_w"], g_dev["k_w"], g_dev["cos_sin_cache"],
                           g_dev["positions"], is_neox=w.is_neox, eps=w.eps, inputs_ready=True)
        g_dev["q"].copy_(cpu["q"].cuda() if not w.fused_total_heads else cpu["q"].to("cuda"))
        g_dev["k"].copy_(cpu["k"].cuda() if not w.fused_total_heads else cpu["k"].to("cuda"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(g_dev["q"].view(torch.int16), ref["q"].view(torch.int16))
        assert torch.equal(g_dev["k"].view(torch.int16), ref["k"].view(torch.int16))
    finally:
        qknr.set_tuning(reset=True)


def test_extreme_values(qknr):
    """Zero heads, tiny and large magnitudes, eps = 0 on non-zero heads, and
    fp16 subnormal inputs (scale 1e-6) that eps = 0 normalises to order one."""
    for dtype, scale, eps in (("bf16", 1e-20, 1e-6), ("bf16", 1e15, 1e-6), ("fp16", 3e3, 1e-6),
                              ("fp16", 1e-3, 0.0), ("bf16", 1.0, 0.0), ("fp16", 1e-6, 0.0)):
        w = _make(128, 128, False, "i32", 50, 3, 2, dtype=dtype, seed=9, x_scale=scale, eps=eps)
        cpu = workloads.make_inputs(w)
        cpu["q"][3].zero_()
        if eps == 0.0:
            cpu["q"][3, :, 0] = 1.0        # keep every head non-zero when eps is 0
        _check_workload_inputs(qknr, w, cpu)


def test_fp16_store_overflow_rounds_to_inf(qknr):
    """Weights of 3e4 on every fourth dim push some outputs past fp16's range.
    Rounding to nearest even sends every value at or beyond 65520 to +-inf, so
    those elements must be infinite with the oracle's sign. Values below 65504
    keep the usual tolerance; the few in between may end as 65504 or inf."""
    w = _make(128, 128, False, "i32", 24, 2, 2, dtype="fp16", seed=11)
    cpu = workloads.make_inputs(w)
    weight = torch.ones(128, dtype=torch.float16)
    weight[::4] = 3.0e4
    cpu["q_w"], cpu["k_w"] = weight.clone(), weight.clone()
    eq, ek = _expected(cpu, w)
    dev = workloads.to_device(cpu, w, "cuda")
    _run_gpu(qknr, dev, w)
    torch.cuda.synchronize()
    for name, got, exp in (("q", dev["q"], eq), ("k", dev["k"], ek)):
        g = got.double().cpu().numpy()
        over = np.abs(exp) > 65520.0 * (1 + 1e-5)
        under = np.abs(exp) < 65504.0
        mid = ~(over | under)
        assert over.sum() > 10 and under.sum() > 1000, (name, over.sum(), under.sum())
        assert np.all(np.isinf(g[over])) and np.all(np.sign(g[over]) == np.sign(exp[over])), name
        _assert_close(g[under], exp[under], w.torch_dtype, f"{name} in range")
        assert np.all((np.abs(g[mid]) == 65504.0) | np.isinf(g[mid])), name


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
    assert qknr.qknr_apply(qp, kp, *common, 16, 2, 2, 72, 64, 0, 256, 256, 128, 1e-6, 0, s) == 3
    assert qknr.qknr_apply(qp, kp, *common, 16, 2, 2, 128, 24, 1, 256, 256, 128, 1e-6, 0, s) == 3
    # invalid arguments
    assert qknr.qknr_apply(qp, kp, *common, -1, 2, 2, 128, 64, 0, 256, 256, 128, 1e-6, 0, s) == 2
    assert qknr.qknr_apply(qp, kp, *common, 16, 0, 2, 128, 64, 0, 256, 256, 128, 1e-6, 0, s) == 2
    assert qknr.qknr_apply(qp, qp, *common, 16, 2, 2, 128, 64, 0, 256, 256, 128, 1e-6, 0, s) == 2
    assert qknr.qknr_apply(qp, kp, *common, 16, 2, 2, 128, 64, 0, 256, 256, 64, 1e-6, 0, s) == 2
    assert qknr.qknr_apply(0, kp, *common, 16, 2, 2, 128, 64, 0, 256, 256, 128, 1e-6, 0, s) == 2
    assert qknr.qknr_apply(qp, kp, *common, 16, 2, 2, 128, 64, 0, 256, 256, 128, -1.0, 0, s) == 2
    assert qknr.qknr_apply(qp, kp, *common, 16, 2, 2, 128, 64, 0, 256, 256, 128, 1e-6, 7, s) == 2
    # sizes whose byte extents would wrap a signed 64-bit offset
    assert qknr.qknr_apply(qp, kp, *common, 2 ** 62, 2, 2, 128, 64, 0, 256, 256, 128, 1e-6, 0, s) == 2
    assert qknr.qknr_apply(qp, kp, *common, 16, 2, 2, 128, 64, 0, 2 ** 62, 256, 128, 1e-6, 0, s) == 2
    assert qknr.qknr_apply(qp, kp, *common, 1, 2, 2, 128, 64, 0, 256, 2 ** 63 - 8, 128, 1e-6, 0, s) == 2
    assert qknr.qknr_apply(qp, kp, *common, 16, 2 ** 20, 2, 128, 64, 0, 256, 256, 2 ** 40, 1e-6, 0, s) == 2
    assert "2^56" in qknr.qknr_last_error()
    assert qknr.qknr_apply(qp, kp, *common, 1, 2 ** 31 - 1, 2 ** 31 - 1, 128, 64, 0, 256, 256, 128, 1e-6, 0,
                           s) == 2
    assert "heads per token" in qknr.qknr_last_error()
    torch.cuda.synchronize()
    assert torch.equal(dev["q"], before_q) and torch.equal(dev["k"], before_k)


@pytest.mark.parametrize("tune", [{}, {"order": 1}, {"passes": 1}], ids=["auto", "contiguous", "one-pass"])
def test_checked_variant(qknr, tune):
    qknr.set_tuning(reset=True, **tune)
    try:
        _checked_variant(qknr)
    finally:
        qknr.set_tuning(reset=True)


def _checked_variant(qknr):
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


def _pair_norms(o, R, neox):
    """Length of the rotation pair each element belongs to (|o| past rope_dim)."""
    pn = np.abs(o).copy()
    half = R // 2
    if neox:
        a, b = o[..., :half], o[..., half:R]
        n = np.sqrt(a * a + b * b)
        pn[..., :half] = n
        pn[..., half:R] = n
    else:
        a, b = o[..., 0:R:2], o[..., 1:R:2]
        n = np.sqrt(a * a + b * b)
        pn[..., 0:R:2] = n
        pn[..., 1:R:2] = n
    return pn


@pytest.mark.parametrize("name,T", REDUCED, ids=[r[0] for r in REDUCED])
def test_unfused_baseline(qknr, name, T):
    """The unfused two-kernel chain (RMSNorm kernel, then RoPE kernel) against
    the oracle. Its stored intermediate adds one rounding before the rotation,
    bounded by u * |(n_a, n_b)| per rotated element (u = 2^-8 bf16, 2^-11
    fp16), so the bound is 2u * pair length + the fused bound."""
    base = workloads.get(name)
    w = workloads.scaled(base, T, cache_len=min(base.cache_len, 8192))
    cpu = workloads.make_inputs(w)
    eq, ek = _expected(cpu, w)
    dev = workloads.to_device(cpu, w, "cuda")
    qknr.apply_unfused(dev["q"], dev["k"], dev["q_w"], dev["k_w"], dev["cos_sin_cache"],
                       dev["positions"], is_neox=w.is_neox, eps=w.eps)
    torch.cuda.synchronize()
    u = 2.0 ** -8 if w.torch_dtype == torch.bfloat16 else 2.0 ** -11
    for got, exp in ((dev["q"], eq), (dev["k"], ek)):
        g = got.double().cpu().numpy()
        tol = 2 * u * _pair_norms(exp, w.rope_dim, w.is_neox) + oracle.tolerance(exp, w.torch_dtype)
        assert np.all(np.abs(g - exp) <= tol), float(np.max(np.abs(g - exp) / tol))
    if w.fused_total_heads:
        lo = w.n_qo + w.n_kv
        assert torch.equal(dev["buffer"][:, lo:, :].cpu().view(torch.int16),
                           cpu["buffer"][:, lo:, :].view(torch.int16))


def test_unfused_norm_step_is_the_fused_op_at_position_zero(qknr):
    """With every position 0 the RoPE step is the identity, so the unfused
    chain must give exactly the fused op's bits."""
    w = _make(128, 64, True, "i32", 77, 6, 2, seed=12)
    cpu = workloads.make_inputs(w)
    cpu["positions"].zero_()
    a = workloads.to_device(cpu, w, "cuda")
    b = workloads.to_device(cpu, w, "cuda")
    _run_gpu(qknr, a, w)
    qknr.apply_unfused(b["q"], b["k"], b["q_w"], b["k_w"], b["cos_sin_cache"], b["positions"],
                       is_neox=True, eps=w.eps)
    torch.cuda.synchronize()
    assert torch.equal(a["q"], b["q"]) and torch.equal(a["k"], b["k"])


def test_planned_passes_cover_every_head(qknr):
    """The host's passes per token must match the kernels' lane groups: a head
    takes head_dim/16 lanes rounded up to a power of two, so a pass covers
    32 / that many heads (head_dim 80, 96 and 192 pad their groups)."""
    for D in (64, 80, 96, 128, 192, 256):
        group = 1
        while group < D // 16:
            group *= 2
        per_pass = 32 // group
        for n_qo, n_kv in ((1, 1), (8, 1), (4, 2), (1, 7), (24, 24), (32, 8), (13, 5)):
            H = n_qo + n_kv
            m = qknr.work_map(33, n_qo, n_kv, D, _neox_half(D), True, qknr.QKNR_FP16)
            passes = m["passes_per_token"]
            assert (passes - 1) * per_pass < H <= passes * per_pass, (D, n_qo, n_kv, passes)


def test_split_rope_pair_mapping(qknr):
    """A QK-norm + split-RoPE call in the style the KDA overview lists for
    LTX2 (one call over q and k, each a contiguous [B, S, H*D] bf16 tensor,
    per-head norm, rotate-half pairing of dims i and i + D/2, one cos|sin pair
    of D/2 values per token) maps onto this op as: the [B*S, H, D] view,
    is_neox=True, rope_dim = head_dim, a table whose row s holds sequence
    position s's cos then sin, and positions t mod S. The per-token angles
    here are arbitrary (not base^(-2j/R)), as a video model's 3-D positions
    give. Against the oracle, element by element."""
    B, S, H, D = 2, 45, 6, 128
    g = np.random.default_rng(808)
    q3 = torch.from_numpy(g.standard_normal((B, S, H * D), dtype=np.float32)).to(torch.bfloat16)
    k3 = torch.from_numpy(g.standard_normal((B, S, H * D), dtype=np.float32)).to(torch.bfloat16)
    qw = (1 + 0.1 * torch.from_numpy(g.standard_normal(D, dtype=np.float32))).to(torch.bfloat16)
    kw = (1 + 0.1 * torch.from_numpy(g.standard_normal(D, dtype=np.float32))).to(torch.bfloat16)
    ang = g.uniform(-np.pi, np.pi, size=(S, D // 2))
    table = torch.from_numpy(np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32))
    pos = torch.arange(B * S, dtype=torch.int32) % S
    qv, kv = q3.view(B * S, H, D), k3.view(B * S, H, D)
    eq, ek = oracle.apply(qv, kv, qw, kw, table, pos, is_neox=True, eps=1e-6)
    dq, dk = q3.cuda(), k3.cuda()
    qknr.apply(dq.view(B * S, H, D), dk.view(B * S, H, D), qw.cuda(), kw.cuda(), table.cuda(),
               pos.cuda(), is_neox=True, eps=1e-6)
    torch.cuda.synchronize()
    _assert_close(dq.view(B * S, H, D).double().cpu().numpy(), eq, torch.bfloat16, "q")
    _assert_close(dk.view(B * S, H, D).double().cpu().numpy(), ek, torch.bfloat16, "k")


COMPILED_R = [(D, R, dt, pos) for D in (64, 128, 256) for R in (D, D // 2)
              for dt, pos in (("bf16", "i32"), ("fp16", "i64"))]


@pytest.mark.parametrize("D,R,dtype,pos", COMPILED_R, ids=[f"D{c[0]}-R{c[1]}-{c[2]}-{c[3]}" for c in COMPILED_R])
def test_compiled_rope_dim_kernels(qknr, D, R, dtype, pos):
    """Interleaved pairing with 4-pass items runs an instantiation with
    rope_dim compiled in when rope_dim is head_dim or head_dim / 2; 2-pass
    items run the one that reads rope_dim at run time. Same bits, and the
    oracle's bound; other rope_dims keep the run-time kernel."""
    # 32 heads: at least 4 warp passes per token for every head_dim here, so
    # that 4-pass items take the 4-pass class
    w = _make(D, R, False, pos, 131, 20, 12, dtype=dtype, seed=D + R)
    code = qknr.dtype_code(w.torch_dtype, w.pos_torch_dtype)
    cpu = workloads.make_inputs(w)
    eq, ek = _expected(cpu, w)
    outs = {}
    for passes in (4, 2):
        qknr.set_tuning(reset=True, passes=passes)
        try:
            m = qknr.work_map(w.num_tokens, w.n_qo, w.n_kv, D, R, False, code)
            assert m["rope_dim_compiled"] == (R if passes == 4 else 0), m
            dev = workloads.to_device(cpu, w, "cuda")
            _run_gpu(qknr, dev, w)
        finally:
            qknr.set_tuning(reset=True)
        _assert_close(dev["q"].double().cpu().numpy(), eq, w.torch_dtype, f"q passes={passes}")
        _assert_close(dev["k"].double().cpu().numpy(), ek, w.torch_dtype, f"k passes={passes}")
        outs[passes] = dev
    assert torch.equal(outs[4]["q"].view(torch.int16), outs[2]["q"].view(torch.int16))
    assert torch.equal(outs[4]["k"].view(torch.int16), outs[2]["k"].view(torch.int16))
    qknr.set_tuning(reset=True, passes=4)
    try:
        other = qknr.work_map(w.num_tokens, w.n_qo, w.n_kv, D, R - 2, False, code)
        neox = qknr.work_map(w.num_tokens, w.n_qo, w.n_kv, D, D, True, code)
    finally:
        qknr.set_tuning(reset=True)
    assert other["rope_dim_compiled"] == 0 and neox["rope_dim_compiled"] == 0
