"""The bench's JSON line.  The reference arm times the oracle on CPU (no GPU
needed) and prints the contract's line on rank 0 only; the GPU arm's line
carries the roofline, per-kernel, end-to-end, clock and CPU-baseline records."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMALL = ["--impl", "reference", "--workload", "qwen_t512", "--T", "16", "--E", "8",
         "--steps", "2", "--warmup", "1"]


def _run(extra_env=None):
    env = dict(os.environ)
    env.update(extra_env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *SMALL], cwd=ROOT,
                          env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_the_contract_line():
    r = _run({"CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench
    assert d["metric"] == bench.METRIC
    assert d["impl"] == "reference"
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 2, 1)
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["config"]["T"] == 16 and d["config"]["E"] == 8
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["unit"] == "tokens/s" and "of the workload's 16 tokens" in cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == "tokens/s"
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_prints_nothing_on_other_ranks():
    r = _run({"CUDA_VISIBLE_DEVICES": "", "RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


# ---------------------------------------------------------------- on a GPU
@pytest.mark.gpu
def test_gpu_arm_prints_the_contract_line():
    args = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "qwen_t512", "--T",
            "64", "--E", "16", "--steps", "5", "--warmup", "3", "--cpu-budget", "1"]
    r = subprocess.run(args, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    d = json.loads(lines[-1])
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["n_gpus"] == 1
    assert d["steps"] == 5 and d["warmup"] >= 3 and d["dtype"] == "bf16"
    rf = d["roofline"]
    assert rf["bound"] in ("hbm", "tensor") and rf["peak"] > 0
    assert rf["achieved"] > 0 and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert d["gpu_launches"] > 0
    assert d["kernels"] and all(v["launches"] > 0 for v in d["kernels"].values())
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] == 64 * 4096 * 2
    assert e2e["d2h_bytes_per_step"] == 64 * 4096 * 4
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1


@pytest.mark.gpu
def test_gpu_arm_runs_every_workload_in_one_line():
    """The default run: every workload, bf16 and Q8_0 experts, one after another
    in one process (small shapes here), the headline being the Qwen-layout one."""
    args = [sys.executable, os.path.join(ROOT, "bench.py"), "--T", "64", "--E", "16", "--steps",
            "4", "--warmup", "3", "--no-cpu-baseline"]
    r = subprocess.run(args, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([l for l in r.stdout.splitlines() if l.strip()][-1])
    sys.path.insert(0, ROOT)
    import bench
    w = d["workloads"]
    assert set(w) == set(bench.SUITE) | {n + "+q8_0" for n in bench.SUITE}
    assert d["value"] == w[bench.HEADLINE]["tokens_per_s"]
    for name, rec in w.items():
        assert rec["tokens_per_s"] > 0 and rec["ms_per_step"] > 0, name
        assert rec["expert_weights"] == ("q8_0" if name.endswith("+q8_0") else "dense")
        assert rec["roofline"]["frac"] > 0 and rec["layer_roofline"]["t_star_ms"] > 0
        assert rec["e2e"]["value"] > 0 and rec["gpu_launches"] > 0
        assert "sm_mhz" in rec["clocks"]


# ---------------------------------------------------------------- roofline logic (CPU)
def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_roofline_bound_follows_the_kernels_bytes_and_flops():
    bench = _bench()
    pk = {"hbm_gbs": 6790.7, "bf16_tflops": 1939.5, "bf16_tflops_sustained": 1708.6}
    # default workload: 6.49 GB against 0.1 TFLOP of gate/up -> bound by HBM
    cfg = bench.workload("qwen_t512", None, None)
    r = bench.kernel_roofline(cfg, "ffn_gateup_tc", cfg.E, 0.95, pk, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == pk["hbm_gbs"]
    assert abs(r["achieved"] - r["algorithmic_bytes_per_launch"] / 0.95e-3 / 1e9) < 1e-6
    # skewed prefill: 3.3 TFLOP against 7.9 GB -> bound by the (sustained) tensor peak
    cfg = bench.workload("skewed_zipf", None, None)
    r = bench.kernel_roofline(cfg, "ffn_gateup_tc", cfg.E, 2.26, pk, "measured")
    P = cfg.T * (cfg.k + cfg.S)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["peak"] == pk["bf16_tflops_sustained"]
    assert r["algorithmic_flops_per_launch"] == 4.0 * cfg.d * cfg.I * P
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12
    # the down GEMM does half the flops of gate/up per row
    assert bench.kernel_flops(cfg, "ffn_down_tc") * 2 == bench.kernel_flops(cfg, "ffn_gateup_tc")


def test_source_hash_ignores_comments_only():
    bench = _bench()
    a = "int f(int x) {  // doubles\n  return 2 * x; /* result */ }\n"
    b = "int f(int x) {\n  /* a longer\n     note */ return 2 * x;   }"
    c = "int f(int x) { return 3 * x; }"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_tier_record_host_memory_queries():
    # the tier record's placement fields: the sampled pages' NUMA nodes (shares
    # summing to one) and the nodes of the CPUs this process may run on
    import torch

    bench = _bench()
    ts = [torch.ones(1 << 20, dtype=torch.uint8), torch.ones(1 << 18, dtype=torch.bfloat16)]
    numa = bench.host_pages_numa(ts, samples=16)
    nodes = bench.cpu_numa_nodes()
    if not sys.platform.startswith("linux") or numa is None or nodes is None:
        pytest.skip("no NUMA query here")
    assert abs(sum(numa.values()) - 1.0) < 1e-9
    assert "error" not in numa
    assert nodes and all(isinstance(n, int) and n >= 0 for n in nodes)
