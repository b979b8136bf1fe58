"""The PyTorch custom-op registration (torch.ops.qknr.fused_inplace_qknorm_rope).

CPU: the schema declares q and k as mutated and the op returns nothing; the
shape gate agrees with the C ABI's. GPU: the op matches the CPU oracle element
by element and gives the same bits as the direct call, eagerly and under
torch.compile (aot_eager backend, one graph), where the mutation must be
visible to the code after the op."""
import os
import sys

import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import oracle  # noqa: E402
import workloads  # noqa: E402
from qk_rmsnorm_rope_gb300 import torch_op  # noqa: E402


def _assert_oracle(got_q, got_k, cpu, w):
    eq, ek = oracle.apply(cpu["q"], cpu["k"], cpu["q_w"], cpu["k_w"], cpu["cos_sin_cache"],
                          cpu["positions"], is_neox=w.is_neox, eps=w.eps)
    for got, exp, what in ((got_q, eq, "q"), (got_k, ek, "k")):
        v = oracle.max_violation(got.reshape(exp.shape).double().cpu().numpy(), exp, w.torch_dtype)
        assert v <= 1.0, f"{what}: max error {v:.3f} x tolerance"


def test_schema_declares_mutation():
    schema = str(torch.ops.qknr.fused_inplace_qknorm_rope.default._schema)
    assert "Tensor(a0!) q" in schema and "Tensor(a1!) k" in schema
    assert schema.endswith("-> ()")


def test_can_use_gate():
    assert torch_op.can_use_fused_inplace_qknorm_rope(128, 64, True, torch.float16)
    assert torch_op.can_use_fused_inplace_qknorm_rope(256, 128, False, torch.bfloat16)
    assert torch_op.can_use_fused_inplace_qknorm_rope(96, 64, False, torch.bfloat16)
    assert not torch_op.can_use_fused_inplace_qknorm_rope(72, 64, False, torch.bfloat16)
    assert not torch_op.can_use_fused_inplace_qknorm_rope(128, 64, False, torch.float32)


@pytest.mark.gpu
def test_op_matches_direct_call_eager_and_compiled():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import qk_rmsnorm_rope_gb300 as q
    torch.cuda.set_device(0)
    q.init(0)
    w = workloads.scaled(workloads.get("gqa"), 64, cache_len=1024)
    cpu = workloads.make_inputs(w)
    ref = workloads.to_device(cpu, w, "cuda")
    q.apply(ref["q"], ref["k"], ref["q_w"], ref["k_w"], ref["cos_sin_cache"], ref["positions"],
            is_neox=w.is_neox, eps=w.eps)
    eager = workloads.to_device(cpu, w, "cuda")
    torch.ops.qknr.fused_inplace_qknorm_rope(eager["q"], eager["k"], eager["q_w"], eager["k_w"],
                                             eager["cos_sin_cache"], eager["positions"],
                                             w.is_neox, w.eps)

    def step(qq, kk, qw, kw, cache, pos):
        qq = qq * 1.0          # a fresh tensor that the op then mutates inside the graph
        kk = kk * 1.0
        torch.ops.qknr.fused_inplace_qknorm_rope(qq, kk, qw, kw, cache, pos, True, w.eps)
        return qq + 0.0, kk + 0.0

    compiled = torch.compile(step, backend="aot_eager", fullgraph=True)
    src = workloads.to_device(cpu, w, "cuda")
    cq, ck = compiled(src["q"], src["k"], src["q_w"], src["k_w"], src["cos_sin_cache"],
                      src["positions"])
    torch.cuda.synchronize()
    _assert_oracle(eager["q"], eager["k"], cpu, w)
    _assert_oracle(cq, ck, cpu, w)
    for d in (eager,):
        assert torch.equal(d["q"], ref["q"]) and torch.equal(d["k"], ref["k"])
    assert torch.equal(cq, ref["q"]) and torch.equal(ck, ref["k"])
    # the compiled function worked on copies: its inputs keep their values
    assert torch.equal(src["q"].cpu(), cpu["q"])


@pytest.mark.gpu
def test_op_takes_model_layout_and_host_positions():
    """The registered op on [B, S, H, D] q/k and positions given on the host
    (converted like the reference wrapper does): within the oracle's bound,
    and the bits of the 3-D call."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import qk_rmsnorm_rope_gb300 as q
    q.init(0)
    w = workloads.scaled(workloads.get("dit"), 48)
    cpu = workloads.make_inputs(w)
    ref = workloads.to_device(cpu, w, "cuda")
    q.apply(ref["q"], ref["k"], ref["q_w"], ref["k_w"], ref["cos_sin_cache"], ref["positions"],
            is_neox=False, eps=w.eps)
    dev = workloads.to_device(cpu, w, "cuda")
    q4 = dev["q"].view(4, 12, w.n_qo, w.head_dim)
    k4 = dev["k"].view(4, 12, w.n_kv, w.head_dim)
    torch.ops.qknr.fused_inplace_qknorm_rope(q4, k4, dev["q_w"], dev["k_w"], dev["cos_sin_cache"],
                                             cpu["positions"].to(torch.int64), False, w.eps)
    torch.cuda.synchronize()
    _assert_oracle(q4, k4, cpu, w)
    assert torch.equal(dev["q"].view(torch.int16), ref["q"].view(torch.int16))
    assert torch.equal(dev["k"].view(torch.int16), ref["k"].view(torch.int16))
