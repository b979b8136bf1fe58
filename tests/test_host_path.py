"""GPU tests of qknr_apply_host: q, k and positions in host memory.

Two modes. Direct: the buffers are pinned and mapped into the device's
address space, and the kernel reads and writes them in place. Staged: they
are copied to caller-owned device buffers in chunks, transformed there and
copied back, with copies and kernels overlapping.

The results must be the same bits as qknr_apply on the same inputs (the same
kernel runs on each chunk, and every token is independent of the others), and
within the oracle's tolerance. Layouts: contiguous q/k, the strided fused QKV
buffer (whose V heads must come back untouched), and heads with padding
between them (the padding must come back untouched too). Chunkings: automatic,
one token, a ragged 7 tokens, everything in one chunk. Pageable memory: the
automatic mode stages it, the direct mode refuses it before any launch.
"""
import os
import sys

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
    torch.cuda.synchronize()


def _host_inputs(cpu, w, pad):
    """Pinned host q, k (views of the buffers returned alongside them) and positions."""
    if w.fused_total_heads:
        buf = cpu["buffer"].clone().pin_memory()
        return buf[:, :w.n_qo, :], buf[:, w.n_qo:w.n_qo + w.n_kv, :], [buf]
    bufs, views = [], []
    for key, n in (("q", w.n_qo), ("k", w.n_kv)):
        b = torch.full((w.num_tokens, n, w.head_dim + pad), -7.0, dtype=w.torch_dtype).pin_memory()
        b[:, :, :w.head_dim] = cpu[key]
        bufs.append(b)
        views.append(b[:, :, :w.head_dim])
    return views[0], views[1], bufs


def _staging(h):
    """A device tensor with h's shape and strides, filled with NaN (so that a
    copy that does not happen shows)."""
    size = max(1, sum((s - 1) * st for s, st in zip(h.shape, h.stride())) + 1) if h.numel() else 1
    base = torch.full((size,), float("nan"), dtype=h.dtype, device="cuda")
    return base.as_strided(h.shape, h.stride())


CASES = [("dit", 300, 0, 0, "staged"), ("dit", 300, 0, 1, "staged"), ("mha_neox", 257, 0, 7, "staged"),
         ("gqa", 513, 0, 0, "staged"), ("fused_qkv", 129, 0, 0, "staged"),
         ("fused_qkv", 129, 0, 129, "staged"), ("tiny", 16, 0, 3, "staged"),
         ("mha_neox", 33, 16, 5, "staged"), ("dit", 1, 8, 0, "staged"),
         ("dit", 300, 0, 0, "direct"), ("mha_neox", 257, 0, 0, "direct"), ("gqa", 513, 0, 0, "direct"),
         ("fused_qkv", 129, 0, 0, "direct"), ("tiny", 16, 0, 0, "direct"),
         ("mha_neox", 33, 16, 0, "direct"), ("dit", 1, 8, 0, "direct"), ("gqa", 77, 0, 0, "auto")]


@pytest.mark.parametrize("name,T,pad,chunk,mode", CASES,
                         ids=[f"{c[0]}-T{c[1]}-pad{c[2]}-chunk{c[3]}-{c[4]}" for c in CASES])
def test_host_path_matches_device_call(qknr, name, T, pad, chunk, mode):
    base = workloads.get(name)
    w = workloads.scaled(base, T, cache_len=min(base.cache_len, 8192))
    cpu = workloads.make_inputs(w)
    # reference: the device entry point on the same values
    ref = workloads.to_device(cpu, w, "cuda")
    qknr.apply(ref["q"], ref["k"], ref["q_w"], ref["k_w"], ref["cos_sin_cache"], ref["positions"],
               is_neox=w.is_neox, eps=w.eps)
    h_q, h_k, bufs = _host_inputs(cpu, w, pad)
    before = [b.clone() for b in bufs]
    h_pos = cpu["positions"].clone().pin_memory()
    d_q, d_k = _staging(h_q), _staging(h_k)
    d_pos = torch.empty_like(h_pos, device="cuda")
    dev = workloads.to_device(cpu, w, "cuda")
    qknr.apply_host(h_q, h_k, dev["q_w"], dev["k_w"], dev["cos_sin_cache"], h_pos, d_q, d_k, d_pos,
                    is_neox=w.is_neox, eps=w.eps, chunk_tokens=chunk, mode=mode)
    torch.cuda.synchronize()
    for got, exp in ((h_q, ref["q"]), (h_k, ref["k"])):
        assert torch.equal(got.cpu().view(torch.int16), exp.cpu().view(torch.int16))
    if mode == "staged":        # the staging buffers hold the results too
        for got, exp in ((d_q, ref["q"]), (d_k, ref["k"])):
            assert torch.equal(got.cpu().view(torch.int16), exp.cpu().view(torch.int16))
    elif mode == "direct":      # ... and are not used at all
        assert torch.isnan(d_q.float()).all() and torch.isnan(d_k.float()).all()
    eq, ek = oracle.apply(cpu["q"], cpu["k"], cpu["q_w"], cpu["k_w"], cpu["cos_sin_cache"],
                          cpu["positions"], is_neox=w.is_neox, eps=w.eps)
    assert oracle.max_violation(h_q.double().numpy(), eq, w.torch_dtype) <= 1.0
    assert oracle.max_violation(h_k.double().numpy(), ek, w.torch_dtype) <= 1.0
    # host bytes outside the heads keep every bit: V of the fused buffer, padding
    for b, b0 in zip(bufs, before):
        mask = torch.ones(b.shape, dtype=torch.bool)
        if w.fused_total_heads:
            mask[:, :w.n_qo + w.n_kv, :] = False
        else:
            mask[:, :, :w.head_dim] = False
        assert torch.equal(b.view(torch.int16)[mask], b0.view(torch.int16)[mask])


def test_host_path_two_calls_and_stream_order(qknr):
    """Two calls in a row on one stream: the second transforms the first's
    results (stream order holds across calls), as two device calls would."""
    base = workloads.get("gqa")
    w = workloads.scaled(base, 200, cache_len=min(base.cache_len, 8192))
    cpu = workloads.make_inputs(w)
    ref = workloads.to_device(cpu, w, "cuda")
    for _ in range(2):
        qknr.apply(ref["q"], ref["k"], ref["q_w"], ref["k_w"], ref["cos_sin_cache"],
                   ref["positions"], is_neox=w.is_neox, eps=w.eps)
    h_q, h_k = cpu["q"].clone().pin_memory(), cpu["k"].clone().pin_memory()
    h_pos = cpu["positions"].clone().pin_memory()
    d_q, d_k, d_pos = _staging(h_q), _staging(h_k), torch.empty_like(h_pos, device="cuda")
    dev = workloads.to_device(cpu, w, "cuda")
    s = torch.cuda.Stream()
    for mode in ("staged", "direct"):
        hq, hk = h_q.clone().pin_memory(), h_k.clone().pin_memory()
        for _ in range(2):
            qknr.apply_host(hq, hk, dev["q_w"], dev["k_w"], dev["cos_sin_cache"], h_pos, d_q, d_k,
                            d_pos, is_neox=w.is_neox, eps=w.eps, chunk_tokens=64, mode=mode,
                            stream=s)
        s.synchronize()
        assert torch.equal(hq.view(torch.int16), ref["q"].cpu().view(torch.int16)), mode
        assert torch.equal(hk.view(torch.int16), ref["k"].cpu().view(torch.int16)), mode


def test_host_path_four_d_inputs(qknr):
    """[B, S, H, D] host (and staging) tensors: the same bits as the device call
    on the [B*S, H, D] layout, in both modes; a 4-D view whose batch and
    sequence dims do not merge without a copy is refused before any work."""
    base = workloads.get("gqa")
    w = workloads.scaled(base, 96, cache_len=min(base.cache_len, 8192))
    cpu = workloads.make_inputs(w)
    ref = workloads.to_device(cpu, w, "cuda")
    qknr.apply(ref["q"], ref["k"], ref["q_w"], ref["k_w"], ref["cos_sin_cache"], ref["positions"],
               is_neox=w.is_neox, eps=w.eps)
    torch.cuda.synchronize()
    dev = workloads.to_device(cpu, w, "cuda")
    four_d = (lambda t: t.view(4, 24, t.shape[1], t.shape[2]))
    for mode in ("staged", "direct"):
        hq = four_d(cpu["q"].clone().pin_memory())
        hk = four_d(cpu["k"].clone().pin_memory())
        h_pos = cpu["positions"].clone().pin_memory()
        staging = ((four_d(torch.empty_like(cpu["q"], device="cuda")),
                    four_d(torch.empty_like(cpu["k"], device="cuda")),
                    torch.empty_like(h_pos, device="cuda")) if mode == "staged" else (None, None, None))
        qknr.apply_host(hq, hk, dev["q_w"], dev["k_w"], dev["cos_sin_cache"], h_pos, *staging,
                        is_neox=w.is_neox, eps=w.eps, mode=mode)
        torch.cuda.synchronize()
        assert torch.equal(hq.reshape(ref["q"].shape).view(torch.int16), ref["q"].cpu().view(torch.int16)), mode
        assert torch.equal(hk.reshape(ref["k"].shape).view(torch.int16), ref["k"].cpu().view(torch.int16)), mode
    # [S, B, ...] storage seen as [B, S, ...]: no single token stride, so refused
    hq = cpu["q"].clone().pin_memory().view(24, 4, w.n_qo, w.head_dim).transpose(0, 1)
    hk = cpu["k"].clone().pin_memory().view(24, 4, w.n_kv, w.head_dim).transpose(0, 1)
    before = hq.clone()
    with pytest.raises(qknr.QknrError):
        qknr.apply_host(hq, hk, dev["q_w"], dev["k_w"], dev["cos_sin_cache"],
                        cpu["positions"].clone().pin_memory(), is_neox=w.is_neox, eps=w.eps)
    assert torch.equal(hq, before)


def test_host_path_pageable_memory(qknr):
    """Pageable host memory is not mapped: the automatic mode stages it (and
    gets the same bits), the direct mode refuses it before any launch."""
    w = workloads.scaled(workloads.get("dit"), 100)
    cpu = workloads.make_inputs(w)
    ref = workloads.to_device(cpu, w, "cuda")
    qknr.apply(ref["q"], ref["k"], ref["q_w"], ref["k_w"], ref["cos_sin_cache"], ref["positions"],
               is_neox=w.is_neox, eps=w.eps)
    h_q, h_k, h_pos = cpu["q"].clone(), cpu["k"].clone(), cpu["positions"].clone()
    assert not h_q.is_pinned()
    dev = workloads.to_device(cpu, w, "cuda")
    d_q, d_k, d_pos = _staging(h_q), _staging(h_k), torch.empty_like(h_pos, device="cuda")
    with pytest.raises(qknr.QknrError, match="mapped pinned"):
        qknr.apply_host(h_q, h_k, dev["q_w"], dev["k_w"], dev["cos_sin_cache"], h_pos, d_q, d_k,
                        d_pos, is_neox=w.is_neox, eps=w.eps, mode="direct")
    assert torch.equal(h_q, cpu["q"])       # refused: nothing ran
    qknr.apply_host(h_q, h_k, dev["q_w"], dev["k_w"], dev["cos_sin_cache"], h_pos, d_q, d_k, d_pos,
                    is_neox=w.is_neox, eps=w.eps, mode="auto")
    torch.cuda.synchronize()
    assert torch.equal(h_q.view(torch.int16), ref["q"].cpu().view(torch.int16))
    assert torch.equal(h_k.view(torch.int16), ref["k"].cpu().view(torch.int16))


def test_host_path_registered_memory(qknr):
    """Pageable buffers registered with cudaHostRegister (mapped) run in the
    direct mode: the staging buffers stay untouched and the bits match."""
    w = workloads.scaled(workloads.get("mha_neox"), 90, cache_len=4096)
    cpu = workloads.make_inputs(w)
    ref = workloads.to_device(cpu, w, "cuda")
    qknr.apply(ref["q"], ref["k"], ref["q_w"], ref["k_w"], ref["cos_sin_cache"], ref["positions"],
               is_neox=w.is_neox, eps=w.eps)
    h_q, h_k, h_pos = cpu["q"].clone(), cpu["k"].clone(), cpu["positions"].clone()
    cudart = torch.cuda.cudart()
    regs = []
    try:
        for t in (h_q, h_k, h_pos):
            rc = cudart.cudaHostRegister(t.data_ptr(), t.numel() * t.element_size(), 2)  # mapped
            assert int(rc) == 0, rc
            regs.append(t)
        d_q, d_k = _staging(h_q), _staging(h_k)
        d_pos = torch.empty_like(h_pos, device="cuda")
        dev = workloads.to_device(cpu, w, "cuda")
        qknr.apply_host(h_q, h_k, dev["q_w"], dev["k_w"], dev["cos_sin_cache"], h_pos, d_q, d_k,
                        d_pos, is_neox=w.is_neox, eps=w.eps, mode="auto")
        torch.cuda.synchronize()
        assert torch.equal(h_q.view(torch.int16), ref["q"].cpu().view(torch.int16))
        assert torch.equal(h_k.view(torch.int16), ref["k"].cpu().view(torch.int16))
        assert torch.isnan(d_q.float()).all()      # direct: staging untouched
    finally:
        for t in regs:
            cudart.cudaHostUnregister(t.data_ptr())


def test_host_path_errors(qknr):
    w = workloads.scaled(workloads.get("tiny"), 8)
    cpu = workloads.make_inputs(w)
    dev = workloads.to_device(cpu, w, "cuda")
    h_q, h_k = cpu["q"].clone().pin_memory(), cpu["k"].clone().pin_memory()
    h_pos = cpu["positions"].clone().pin_memory()
    args = (dev["q_w"], dev["k_w"], dev["cos_sin_cache"])
    with pytest.raises(qknr.QknrError):     # negative chunk size
        qknr.apply_host(h_q, h_k, *args, h_pos, dev["q"], dev["k"], dev["positions"],
                        is_neox=False, chunk_tokens=-1)
    with pytest.raises(qknr.QknrError):     # staged without staging buffers
        qknr.apply_host(h_q, h_k, *args, h_pos, is_neox=False, mode="staged")
    # pageable host memory in the automatic mode without staging buffers: a clear refusal
    with pytest.raises(qknr.QknrError, match="staged mode"):
        qknr.apply_host(cpu["q"].clone(), cpu["k"].clone(), *args, cpu["positions"].clone(),
                        is_neox=False, mode="auto")
    with pytest.raises(qknr.QknrError):     # host tensor on the device
        qknr.apply_host(dev["q"], h_k, *args, h_pos, dev["q"], dev["k"], dev["positions"],
                        is_neox=False)
    rc = qknr.qknr_apply_host(None, h_k.data_ptr(), dev["q_w"].data_ptr(), dev["k_w"].data_ptr(),
                              dev["cos_sin_cache"].data_ptr(), h_pos.data_ptr(),
                              dev["q"].data_ptr(), dev["k"].data_ptr(), dev["positions"].data_ptr(),
                              8, 4, 4, 64, 64, 0, 256, 256, 64, 1e-6, 0, 0, 0, None)
    assert rc == 2 and "null host pointer" in qknr.qknr_last_error()
    rc = qknr.qknr_apply_host(h_q.data_ptr(), h_k.data_ptr(), dev["q_w"].data_ptr(),
                              dev["k_w"].data_ptr(), dev["cos_sin_cache"].data_ptr(),
                              h_pos.data_ptr(), 0, 0, 0, 8, 4, 4, 64, 64, 0, 256, 256, 64, 1e-6, 0, 0,
                              3, None)
    assert rc == 2 and "flags" in qknr.qknr_last_error()
    # zero tokens: nothing to do, OK
    assert qknr.qknr_apply_host(h_q.data_ptr(), h_k.data_ptr(), dev["q_w"].data_ptr(),
                                dev["k_w"].data_ptr(), dev["cos_sin_cache"].data_ptr(),
                                h_pos.data_ptr(), dev["q"].data_ptr(), dev["k"].data_ptr(),
                                dev["positions"].data_ptr(), 0, 4, 4, 64, 64, 0, 256, 256, 64,
                                1e-6, 0, 0, 0, None) == 0


def test_concurrent_calls_from_threads(qknr):
    """Four host threads, each on its own stream and buffers, call apply,
    apply_checked and apply_host (staged and direct) at the same time; every
    result equals the same call made alone."""
    import threading
    cases = [("gqa", 97), ("dit", 60), ("fused_qkv", 33), ("mha_neox", 41)]
    ws = [workloads.scaled(workloads.get(n), T, cache_len=min(workloads.get(n).cache_len, 4096))
          for n, T in cases]
    cpus = [workloads.make_inputs(w) for w in ws]
    refs = []
    for w, cpu in zip(ws, cpus):
        r = workloads.to_device(cpu, w, "cuda")
        qknr.apply(r["q"], r["k"], r["q_w"], r["k_w"], r["cos_sin_cache"], r["positions"],
                   is_neox=w.is_neox, eps=w.eps)
        refs.append((r["q"].cpu(), r["k"].cpu()))
    torch.cuda.synchronize()
    errors = []

    def worker(i):
        try:
            w, cpu = ws[i], cpus[i]
            s = torch.cuda.Stream()
            for it in range(12):
                kind = (i + it) % 4
                dev = workloads.to_device(cpu, w, "cuda")
                torch.cuda.synchronize()
                if kind == 0:
                    qknr.apply(dev["q"], dev["k"], dev["q_w"], dev["k_w"], dev["cos_sin_cache"],
                               dev["positions"], is_neox=w.is_neox, eps=w.eps, stream=s)
                    s.synchronize()
                    got = (dev["q"].cpu(), dev["k"].cpu())
                elif kind == 1:
                    qknr.apply_checked(dev["q"], dev["k"], dev["q_w"], dev["k_w"],
                                       dev["cos_sin_cache"], dev["positions"], is_neox=w.is_neox,
                                       eps=w.eps, stream=s)
                    got = (dev["q"].cpu(), dev["k"].cpu())
                else:
                    h_q, h_k, _ = _host_inputs(cpu, w, 0)
                    h_pos = cpu["positions"].clone().pin_memory()
                    d_q, d_k = _staging(h_q), _staging(h_k)
                    d_pos = torch.empty_like(h_pos, device="cuda")
                    qknr.apply_host(h_q, h_k, dev["q_w"], dev["k_w"], dev["cos_sin_cache"], h_pos,
                                    d_q, d_k, d_pos, is_neox=w.is_neox, eps=w.eps, chunk_tokens=16,
                                    mode="staged" if kind == 2 else "direct", stream=s)
                    s.synchronize()
                    got = (h_q.clone(), h_k.clone())
                for a, b in zip(got, refs[i]):
                    if not torch.equal(a.contiguous().view(torch.int16), b.view(torch.int16)):
                        errors.append((i, it, kind))
        except Exception as e:   # noqa: BLE001 - reported below
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(ws))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=600)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors[:5]
