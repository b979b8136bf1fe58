"""Host logic of bench.py on the CPU: the multi-rank timing reduction (gloo,
world size 2), rank-0-only output, the reference arm's JSON line, and the
roofline-traffic lookup that must ignore summaries taken on other sources."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_path):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    dist = bench.init_dist(w, "gloo")
    try:
        bench.barrier(dist)
        mx = bench.max_over_ranks(dist, 10.0 + rank, torch.device("cpu"))
        with open(f"{out_path}.{rank}", "w") as f:
            f.write(repr(mx))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2(tmp_path):
    port = _free_port()
    out = str(tmp_path / "mx")
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        with open(f"{out}.{r}") as f:
            assert float(f.read()) == 11.0


def _run_bench(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)


def test_reference_arm_line():
    r = _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "5", "--warmup", "3"])
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["config"]["workload"] == "tiny"


def test_reference_arm_other_ranks_are_silent():
    r = _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "5", "--warmup", "3",
                    "--gpus", "2"], {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_warmup_floor():
    r = _run_bench(["--impl", "reference", "--steps", "5", "--warmup", "2"])
    assert r.returncode != 0 and "warmup" in r.stderr


def test_profiled_traffic_requires_matching_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "qk_rmsnorm_rope_gb300").symlink_to(os.path.join(ROOT, "qk_rmsnorm_rope_gb300"))
    f = prof / "qknr_fused_kernel_dit.txt"
    f.write_text(f"source_sha256: {bench.kernel_source_hash('qknr_fused_kernel')}\n"
                 "dram_read_bytes_per_launch: 100\ndram_write_bytes_per_launch: 23\n")
    assert bench.profiled_traffic("qknr_fused_kernel", "dit") == {"read": 100.0, "write": 23.0,
                                                                  "total": 123.0}
    # a summary without the read/write split is not used
    f.write_text(f"source_sha256: {bench.kernel_source_hash('qknr_fused_kernel')}\n"
                 "traffic_bytes_per_launch: 123\n")
    assert bench.profiled_traffic("qknr_fused_kernel", "dit") is None
    f.write_text("source_sha256: 00\ndram_read_bytes_per_launch: 100\ndram_write_bytes_per_launch: 23\n")
    assert bench.profiled_traffic("qknr_fused_kernel", "dit") is None
    assert bench.profiled_traffic("qknr_fused_kernel", "gqa") is None
    assert bench.profiled_traffic("qknr_other_kernel", "dit") is None


def test_reference_arm_config_matches_ours():
    """Both arms name the workload with the same dict (the reference arm's
    token sample per step is reported beside it, not inside it)."""
    r = _run_bench(["--impl", "reference", "--workload", "dit", "--steps", "3", "--warmup", "3"])
    assert r.returncode == 0, r.stderr
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][0])
    w = bench.workloads.get("dit")
    assert d["config"] == bench.config_of(w)
    assert set(d["config"]) == {"workload", "shape", "storage_dtype", "bytes_per_step", "heads_per_step"}
    assert d["config"]["bytes_per_step"] == bench.workloads.algorithmic_bytes(w)
    assert d["sample_tokens_per_step"] >= 1


def test_default_workload_is_every_config_with_the_largest_as_headline():
    assert bench.CONFIGS == ["tiny", "dit", "mha_neox", "gqa", "fused_qkv"]
    sizes = {n: bench.workloads.algorithmic_bytes(bench.workloads.get(n)) for n in bench.CONFIGS}
    assert bench.HEADLINE == max(sizes, key=sizes.get)


def test_algorithmic_read_write_split():
    for n in bench.CONFIGS:
        w = bench.workloads.get(n)
        rd, wr = bench.workloads.algorithmic_read_bytes(w), bench.workloads.algorithmic_write_bytes(w)
        assert rd + wr == bench.workloads.algorithmic_bytes(w)
        assert wr == 2 * (w.n_qo + w.n_kv) * w.num_tokens * w.head_dim


def test_source_hash_ignores_comments_only():
    """The profile hash follows the code: comments and layout do not change it,
    a code change does."""
    src = "int f(int x) {\n  return x + 1;  // one\n}\n/* block\n comment */\n"
    same = "int f(int x) { return x + 1; }\n// another comment\n"
    other = "int f(int x) { return x + 2; }\n"
    assert bench.code_tokens(src) == bench.code_tokens(same)
    assert bench.code_tokens(src) != bench.code_tokens(other)
    h = bench.kernel_source_hash("qknr_fused_kernel")
    assert h == bench.kernel_source_hash("qknr_fused_kernel", read=lambda n: open(
        os.path.join(ROOT, "qk_rmsnorm_rope_gb300", "csrc", n)).read() + "\n// trailing note\n")
