"""Work-map tuning (qknr_tune): candidates timed on scratch buffers, the
fastest kept per call shape and used by later calls of that shape.

GPU: the choice is one of the candidates and the work map of the shape
reports it; later calls give the same bits as untuned ones and match the
oracle; explicit qknr_set_tuning values still win; a bad layout is refused
before anything is allocated; qknr_shutdown forgets the choices. The caller's
tensors are never touched by tuning."""
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
    q.set_tuning(reset=True)


def _apply(q, d, w):
    q.apply(d["q"], d["k"], d["q_w"], d["k_w"], d["cos_sin_cache"], d["positions"],
            is_neox=w.is_neox, eps=w.eps)
    torch.cuda.synchronize()


CASES = [("dit", 4608), ("gqa", 3000), ("fused_qkv", 5000), ("mha_neox", 700)]


@pytest.mark.parametrize("name,T", CASES, ids=[f"{c[0]}-T{c[1]}" for c in CASES])
def test_tune_records_a_candidate_and_later_calls_use_it(qknr, name, T):
    base = workloads.get(name)
    w = workloads.scaled(base, T, cache_len=min(base.cache_len, 8192))
    cpu = workloads.make_inputs(w)
    untuned = workloads.to_device(cpu, w, "cuda")
    _apply(qknr, untuned, w)
    dev = workloads.to_device(cpu, w, "cuda")
    before_q = dev["q"].clone()
    m = qknr.tune(dev["q"], dev["k"], dev["q_w"], dev["k_w"], dev["cos_sin_cache"], dev["positions"],
                  is_neox=w.is_neox)
    torch.cuda.synchronize()
    assert torch.equal(dev["q"], before_q)                      # tuning ran on scratch only
    passes_item = -(-m["passes_per_token"] // m["items_per_token"])
    assert passes_item in (1, 2, 3, 4) and m["prefetch_items"] in (0, 1, 2, 4), m
    assert m["kernel"] in ("register", "ring") and m["ns_per_launch"] > 0
    if not w.fused_total_heads:
        # the work map of the (contiguous) shape reports the tuned choice
        wm = qknr.work_map(w.num_tokens, w.n_qo, w.n_kv, w.head_dim, w.rope_dim, w.is_neox,
                           qknr.dtype_code(w.torch_dtype, w.pos_torch_dtype))
        assert (wm["kernel"], wm["items_per_token"], wm["prefetch_items"]) == (
            m["kernel"], m["items_per_token"], m["prefetch_items"])
    _apply(qknr, dev, w)
    assert torch.equal(dev["q"].view(torch.int16), untuned["q"].view(torch.int16))
    assert torch.equal(dev["k"].view(torch.int16), untuned["k"].view(torch.int16))
    eq, ek = oracle.apply(cpu["q"], cpu["k"], cpu["q_w"], cpu["k_w"], cpu["cos_sin_cache"],
                          cpu["positions"], is_neox=w.is_neox, eps=w.eps)
    assert oracle.max_violation(dev["q"].double().cpu().numpy(), eq, w.torch_dtype) <= 1.0
    assert oracle.max_violation(dev["k"].double().cpu().numpy(), ek, w.torch_dtype) <= 1.0


def test_explicit_tuning_wins_and_shutdown_forgets(qknr):
    w = workloads.scaled(workloads.get("dit"), 2000)
    dev = workloads.make_inputs(w, device="cuda")
    code = qknr.dtype_code(w.torch_dtype, w.pos_torch_dtype)
    rule = qknr.work_map(w.num_tokens, w.n_qo, w.n_kv, w.head_dim, w.rope_dim, False, code)
    m = qknr.tune(dev["q"], dev["k"], dev["q_w"], dev["k_w"], dev["cos_sin_cache"], dev["positions"],
                  is_neox=False)
    qknr.set_tuning(passes=1, prefetch=-1)
    try:
        forced = qknr.work_map(w.num_tokens, w.n_qo, w.n_kv, w.head_dim, w.rope_dim, False, code)
    finally:
        qknr.set_tuning(reset=True)
    assert forced["items_per_token"] == forced["passes_per_token"] and forced["prefetch_items"] == 0
    tuned = qknr.work_map(w.num_tokens, w.n_qo, w.n_kv, w.head_dim, w.rope_dim, False, code)
    assert (tuned["kernel"], tuned["items_per_token"], tuned["prefetch_items"]) == (
        m["kernel"], m["items_per_token"], m["prefetch_items"])
    # another token count is another shape: the fixed rule
    other = qknr.work_map(w.num_tokens + 1, w.n_qo, w.n_kv, w.head_dim, w.rope_dim, False, code)
    assert other["prefetch_items"] == rule["prefetch_items"]
    assert qknr.qknr_shutdown() == 0
    qknr.init(0)
    again = qknr.work_map(w.num_tokens, w.n_qo, w.n_kv, w.head_dim, w.rope_dim, False, code)
    assert (again["kernel"], again["items_per_token"], again["prefetch_items"]) == (
        rule["kernel"], rule["items_per_token"], rule["prefetch_items"])


def test_tune_refuses_bad_layouts(qknr):
    out = None
    # heads overlap (head stride < head_dim), stride not a multiple of 8, unsupported head_dim, no tokens
    assert qknr.qknr_tune(64, 4, 4, 128, 128, 0, 512, 512, 64, 0, None, out) == 2
    assert qknr.qknr_tune(64, 4, 4, 128, 128, 0, 516, 512, 128, 0, None, out) == 4
    assert qknr.qknr_tune(64, 4, 4, 72, 64, 0, 288, 288, 72, 0, None, out) == 3
    assert qknr.qknr_tune(0, 4, 4, 128, 128, 0, 512, 512, 128, 0, None, out) == 2
    # more scratch than the limit
    assert qknr.qknr_tune(1 << 26, 32, 32, 256, 256, 0, 64 * 256, 64 * 256, 256, 0, None, out) == 2
    assert "scratch" in qknr.qknr_last_error()
