"""The allocation-free checked entry point, qknr_apply_checked_noalloc.

It serves callers that cannot call cudaMalloc (a runtime that owns every
device allocation, a pre-sized pool, a plug-in whose host keeps the allocator
to itself): it keeps its status word in a static device array of the library
instead of memory from qknr_init. This test calls it through the C ABI twice
in a row, first on inputs with out-of-range positions and then on valid ones
(so the second call only passes if the first call's status was cleared), and
checks each output against qknr_apply_checked's on the same inputs, within the
parity tolerance the other tests use. The no-alloc calls come before any
qknr_init in this module, so a fresh process also shows that they need none;
a second test makes the same two calls in a child process that never calls
qknr_init at all, whatever ran before it in this one. Collected last on
purpose: it needs nothing from the other tests and, run after them, shares the
process with everything they did.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import oracle  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


def _args(q, dev, w, stream):
    T, n_qo, D = dev["q"].shape
    hs = dev["q"].stride(1)
    return (dev["q"].data_ptr(), dev["k"].data_ptr(), dev["q_w"].data_ptr(), dev["k_w"].data_ptr(),
            dev["cos_sin_cache"].data_ptr(), dev["cos_sin_cache"].shape[0],
            dev["positions"].data_ptr(), T, n_qo, dev["k"].shape[1], D, w.rope_dim,
            int(w.is_neox), dev["q"].stride(0), dev["k"].stride(0), hs, w.eps,
            q.dtype_code(dev["q"].dtype, dev["positions"].dtype), stream)


def _close(got, ref, dtype):
    g = got.double().cpu().numpy()
    r = ref.double().cpu().numpy()
    assert oracle.max_violation(g, r, dtype) <= 1.0


def _inputs():
    w = workloads.scaled(workloads.get("gqa"), 301, cache_len=2048)
    good = workloads.make_inputs(w)
    bad = {k: v.clone() for k, v in good.items()}
    bad["positions"][[7, 150, 300]] = torch.tensor([2048, -1, 10 ** 9], dtype=torch.int64)
    return w, good, bad


def test_noalloc_matches_checked_twice_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import qk_rmsnorm_rope_gb300 as q
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream().cuda_stream
    w, good, bad = _inputs()

    # no-alloc calls first (no qknr_init yet in a fresh process)
    na_bad = workloads.to_device(bad, w, "cuda")
    rc1 = q.qknr_apply_checked_noalloc(*_args(q, na_bad, w, stream))
    msg1 = q.qknr_last_error()
    na_good = workloads.to_device(good, w, "cuda")
    rc2 = q.qknr_apply_checked_noalloc(*_args(q, na_good, w, stream))
    torch.cuda.synchronize()
    assert rc1 == 6 and "3 token(s)" in msg1 and "index 7" in msg1, msg1
    assert rc2 == 0, q.qknr_last_error()

    # the existing checked entry point on the same inputs
    q.init(0)
    ref_bad = workloads.to_device(bad, w, "cuda")
    assert q.qknr_apply_checked(*_args(q, ref_bad, w, stream)) == 6
    ref_good = workloads.to_device(good, w, "cuda")
    assert q.qknr_apply_checked(*_args(q, ref_good, w, stream)) == 0
    torch.cuda.synchronize()

    for got, ref in ((na_bad, ref_bad), (na_good, ref_good)):
        _close(got["q"], ref["q"], w.torch_dtype)
        _close(got["k"], ref["k"], w.torch_dtype)
    # tokens with bad positions were left untouched by both
    idx = torch.tensor([7, 150, 300], device="cuda")
    assert torch.equal(na_bad["q"][idx].cpu(), bad["q"][idx.cpu()])
    # and the valid call matches the oracle too
    eq, ek = oracle.apply(good["q"], good["k"], good["q_w"], good["k_w"], good["cos_sin_cache"],
                          good["positions"], is_neox=w.is_neox, eps=w.eps)
    assert oracle.max_violation(na_good["q"].double().cpu().numpy(), eq, w.torch_dtype) <= 1.0
    assert oracle.max_violation(na_good["k"].double().cpu().numpy(), ek, w.torch_dtype) <= 1.0
    assert np.isfinite(na_good["q"].float().cpu().numpy()).all()


_CHILD = r"""
import sys
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})
import torch
import qk_rmsnorm_rope_gb300 as q
import test_zz_no_alloc as t
torch.cuda.set_device(0)
stream = torch.cuda.current_stream().cuda_stream
w, good, bad = t._inputs()
na_bad = t.workloads.to_device(bad, w, "cuda")
rc1 = q.qknr_apply_checked_noalloc(*t._args(q, na_bad, w, stream))
msg1 = q.qknr_last_error()
na_good = t.workloads.to_device(good, w, "cuda")
rc2 = q.qknr_apply_checked_noalloc(*t._args(q, na_good, w, stream))
torch.cuda.synchronize()
# this process never called qknr_init: the entry points that need it refuse
rc_init = q.qknr_apply_checked(*t._args(q, t.workloads.to_device(good, w, "cuda"), w, stream))
torch.save({{"rc1": rc1, "msg1": msg1, "rc2": rc2, "rc_init": rc_init,
            "bad_q": na_bad["q"].cpu(), "bad_k": na_bad["k"].cpu(),
            "good_q": na_good["q"].cpu(), "good_k": na_good["k"].cpu()}}, {out!r})
"""


def test_noalloc_in_a_process_without_init(tmp_path):
    """The two calls in a child process that never calls qknr_init; their
    outputs against qknr_apply_checked's in this process."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import qk_rmsnorm_rope_gb300 as q
    here = os.path.dirname(os.path.abspath(__file__))
    out = str(tmp_path / "child.pt")
    r = subprocess.run([sys.executable, "-c", _CHILD.format(root=os.path.dirname(here), tests=here,
                                                            out=out)],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    got = torch.load(out)
    assert got["rc_init"] == 1                       # QKNR_ERR_NOT_INITIALIZED: no qknr_init there
    assert got["rc1"] == 6 and "3 token(s)" in got["msg1"], got["msg1"]
    assert got["rc2"] == 0
    torch.cuda.set_device(0)
    q.init(0)
    stream = torch.cuda.current_stream().cuda_stream
    w, good, bad = _inputs()
    ref_bad = workloads.to_device(bad, w, "cuda")
    assert q.qknr_apply_checked(*_args(q, ref_bad, w, stream)) == 6
    ref_good = workloads.to_device(good, w, "cuda")
    assert q.qknr_apply_checked(*_args(q, ref_good, w, stream)) == 0
    torch.cuda.synchronize()
    for key, ref in (("bad_q", ref_bad["q"]), ("bad_k", ref_bad["k"]), ("good_q", ref_good["q"]),
                     ("good_k", ref_good["k"])):
        _close(got[key], ref, w.torch_dtype)
