"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point ``include/qknr.h`` declares, agrees with the header's
constants, applies its shape gate, validates arguments, and refuses to run
without a device instead of falling back to anything else."""
import ctypes
import os
import re
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qknr.h")

import qk_rmsnorm_rope_gb300 as qknr  # noqa: E402


def _header_text():
    with open(HEADER) as f:
        return re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)


def declared_functions():
    return sorted(set(re.findall(r"\b(qknr_\w+)\s*\(", _header_text())))


def declared_constants():
    return {m.group(1): int(m.group(2), 0)
            for m in re.finditer(r"#define\s+(QKNR_\w+)\s+(0x[0-9a-fA-F]+|\d+)", _header_text())}


def test_header_declares_the_abi():
    names = declared_functions()
    for must in ("qknr_init", "qknr_apply", "qknr_shutdown", "qknr_last_error"):
        assert must in names


def test_library_exports_every_declared_function():
    lib = ctypes.CDLL(qknr.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_mirrors_every_declared_function():
    for n in declared_functions():
        assert callable(getattr(qknr, n)), n


def test_constants_match_header():
    c = declared_constants()
    assert c["QKNR_BF16"] == qknr.QKNR_BF16
    assert c["QKNR_FP16"] == qknr.QKNR_FP16
    assert c["QKNR_POS_I64"] == qknr.QKNR_POS_I64
    assert c["QKNR_INPUTS_READY"] == qknr.QKNR_INPUTS_READY
    for name in ("QKNR_HOST_AUTO", "QKNR_HOST_STAGED", "QKNR_HOST_DIRECT"):
        assert c[name] == getattr(qknr, name)
    for code, name in qknr.STATUS_NAMES.items():
        assert c[name] == code


def test_version():
    assert qknr.qknr_version() >= 10000


def _page_accepts(D, R, neox):
    """The shape set of the fused_inplace_qknorm_rope deep-dive §5.2 (can_use):
    head_dim in {64,128,256}; 0 < R <= D; R % (D/32) == 0; for NeoX the rotary
    lanes R/(D/32) are a power of two and at least 2."""
    if D not in (64, 128, 256) or not (0 < R <= D) or R % (D // 32):
        return False
    if neox:
        lanes = R // (D // 32)
        return lanes >= 2 and (lanes & (lanes - 1)) == 0
    return True


def test_can_use_contains_the_pages_set():
    for D in (64, 128, 256):
        for R in range(1, D + 1):
            for neox in (0, 1):
                if _page_accepts(D, R, neox):
                    for dt in (qknr.QKNR_BF16, qknr.QKNR_FP16,
                               qknr.QKNR_BF16 | qknr.QKNR_POS_I64):
                        assert qknr.qknr_can_use(D, R, neox, dt) == 1, (D, R, neox, dt)


def test_can_use_rejects():
    assert qknr.qknr_can_use(72, 64, 0, 0) == 0          # head_dim outside {64,80,96,128,192,256}
    assert qknr.qknr_can_use(80, 32, 1, 0) == 1          # Phi-2-like: head_dim 80, NeoX rotary 32
    assert qknr.qknr_can_use(96, 64, 1, 0) == 1          # head_dim 96
    assert qknr.qknr_can_use(192, 96, 1, 0) == 1
    assert qknr.qknr_can_use(128, 0, 0, 0) == 0          # rope_dim 0
    assert qknr.qknr_can_use(128, 130, 0, 0) == 0        # rope_dim > head_dim
    assert qknr.qknr_can_use(128, 63, 0, 0) == 0         # odd rope_dim
    assert qknr.qknr_can_use(128, 24, 1, 0) == 0         # NeoX half crosses 16-byte vectors
    assert qknr.qknr_can_use(128, 64, 0, 2) == 0         # unknown element type
    assert qknr.qknr_can_use(128, 64, 0, 0x400) == 0     # unknown flag
    assert qknr.qknr_can_use(128, 64, 0, qknr.QKNR_INPUTS_READY) == 1
    assert qknr.qknr_can_use(128, 8, 1, 0) == 1
    assert qknr.qknr_can_use(64, 2, 0, 0) == 1


def test_set_tuning_validation():
    K = qknr.TUNE_KEYS
    bad = [(K["passes"], 5), (K["threads"], 96), (K["ctas_per_sm"], -1), (K["ctas_per_sm"], 33),
           (K["pdl"], 2), (K["order"], 3), (K["prefetch"], -2), (K["prefetch"], 5), (K["kernel"], 3),
           (K["kernel"], -1), (K["ring_order"], 3), (K["ring_order"], -1), (7, 8), (8, 4096), (99, 0)]
    for key, value in bad:
        assert qknr.qknr_set_tuning(key, value) == 2, (key, value)
    assert "tuning key" in qknr.qknr_last_error()
    v = ctypes.c_int(0)
    assert qknr.qknr_get_tuning(7, ctypes.byref(v)) == 2      # keys of retired kernels are unknown
    qknr.set_tuning(passes=2, threads=128, ctas_per_sm=3, pdl=0, order=1, prefetch=-1, kernel="ring",
                    ring_order=2)
    assert qknr.get_tuning("ring_order") == 2
    assert qknr.get_tuning("passes") == 2 and qknr.get_tuning("threads") == 128
    assert qknr.get_tuning("pdl") == 0 and qknr.get_tuning("order") == 1
    assert qknr.get_tuning("prefetch") == -1 and qknr.get_tuning("kernel") == qknr.QKNR_KERNEL_RING
    qknr.set_tuning(kernel="register")
    assert qknr.get_tuning("kernel") == qknr.QKNR_KERNEL_REGISTER
    qknr.set_tuning(reset=True)
    assert qknr.get_tuning("passes") == 0 and qknr.get_tuning("pdl") == -1
    assert qknr.get_tuning("order") == 0 and qknr.get_tuning("prefetch") == 0
    assert qknr.get_tuning("kernel") == qknr.QKNR_KERNEL_AUTO and qknr.get_tuning("ring_order") == 0


def test_apply_rejects_cpu_tensors():
    """No CPU fallback: CPU tensors are refused before any launch."""
    q = torch.zeros(2, 2, 64, dtype=torch.bfloat16)
    k = torch.zeros(2, 2, 64, dtype=torch.bfloat16)
    w = torch.ones(64, dtype=torch.bfloat16)
    cache = torch.zeros(4, 64)
    pos = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(qknr.QknrError) as e:
        qknr.apply(q, k, w, w, cache, pos, is_neox=False)
    assert e.value.code == 2


def test_marshalling_rejects_bad_tensors():
    q = torch.zeros(2, 2, 64, dtype=torch.float32)
    k = torch.zeros(2, 2, 64, dtype=torch.float32)
    w = torch.ones(64, dtype=torch.float32)
    with pytest.raises(qknr.QknrError):
        qknr.apply(q, k, w, w, torch.zeros(4, 64), torch.zeros(2, dtype=torch.int32),
                   is_neox=False)
    with pytest.raises(qknr.QknrError):
        qknr.dtype_code(torch.bfloat16, torch.int16)


_UNINIT_SCRIPT = r"""
import sys
sys.path.insert(0, {root!r})
import ctypes
import qk_rmsnorm_rope_gb300 as q
rc = q.qknr_apply(16, 16, 16, 16, 16, 16, 1, 1, 1, 128, 128, 0, 128, 128, 128, 1e-6, 0, None)
print(rc, q.qknr_last_error())
rc2 = q.qknr_apply_checked(16, 16, 16, 16, 16, 4, 16, 1, 1, 1, 128, 128, 0, 128, 128, 128, 1e-6, 0, None)
out = (ctypes.c_int64 * 12)()
rc3 = q.qknr_query_work_map(8, 1, 1, 128, 128, 0, 0, out)
rc4 = q.qknr_apply_unfused(16, 16, 16, 16, 16, 16, 1, 1, 1, 128, 128, 0, 128, 128, 128, 1e-6, 0, None)
rc5 = q.qknr_apply_host(16, 16, 16, 16, 16, 16, 16, 16, 16, 1, 1, 1, 128, 128, 0, 128, 128, 128, 1e-6, 0,
                        0, 0, None)
rc6 = q.qknr_apply_strided(16, 16, 16, 16, 16, 16, 1, 1, 1, 128, 128, 0, 128, 128, 128, 128, 1e-6, 0, None)
rc7 = q.qknr_tune(64, 4, 4, 128, 128, 0, 512, 512, 128, 0, None, None)
print(rc2, rc3, rc4, rc5, rc6, rc7)
"""


def test_calls_before_init_are_refused():
    """Without qknr_init every compute entry point returns
    QKNR_ERR_NOT_INITIALIZED (checked in a fresh process)."""
    r = subprocess.run([sys.executable, "-c", _UNINIT_SCRIPT.format(root=ROOT)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    first, second = r.stdout.strip().splitlines()[-2:]
    assert first.startswith("1 ") and "qknr_init" in first
    assert second.split() == ["1", "1", "1", "1", "1", "1"]


def test_four_d_inputs_view_or_refuse():
    """[B, S, H, D] tensors become the [B*S, H, D] view of the same memory when
    B and S merge; otherwise they are refused (a copy would not be in place)."""
    x = torch.zeros(3, 5, 4, 64, dtype=torch.bfloat16)
    v = qknr._as_tokens(x, "q")
    assert v.shape == (15, 4, 64) and v.data_ptr() == x.data_ptr()
    assert qknr._as_tokens(v, "q") is v                      # 3-D: as it is
    with pytest.raises(qknr.QknrError, match="merge"):
        qknr._as_tokens(x.transpose(0, 1), "q")
    # the host-buffer entry point takes the same path, before any device work
    w_ = torch.ones(64, dtype=torch.bfloat16)
    cache = torch.zeros(8, 64)
    with pytest.raises(qknr.QknrError, match="merge"):
        qknr.apply_host(x.transpose(0, 1), x.transpose(0, 1), w_, w_, cache,
                        torch.zeros(15, dtype=torch.int32), is_neox=False)


def test_float_positions_refused_before_any_device_work():
    q = torch.zeros(2, 2, 64, dtype=torch.bfloat16)
    w = torch.ones(64, dtype=torch.bfloat16)
    with pytest.raises(qknr.QknrError):
        qknr.apply(q, q, w, w, torch.zeros(4, 64), torch.zeros(2), is_neox=False)
