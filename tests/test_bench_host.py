"""Host-side logic of bench.py: algorithmic work per unit and the multi-rank
reduction (world size 2 over gloo on the CPU)."""
import json
import os
import socket

import pytest
import torch.multiprocessing as tmp

import bench


def test_work_per_unit():
    c = dict(H=2048, E=256, I=512, top_k=8)
    # 8 routed + 1 shared expert at 1,769,472 B each, W_r, g, x, out
    assert bench.expert_bytes(2048, 512) == 1769472
    assert bench.decode_bytes(c) == 18038784
    # 2 * 3 * H * I * (k + 1) FLOP per token = 56.6 MFLOP
    per_tok = (bench.gemm_flops(c, 4096, "gate_up") + bench.gemm_flops(c, 4096, "down")) / 4096
    assert per_tok == 2 * 3 * 2048 * 512 * 9
    # one-byte codes: 3 * H * I code bytes plus the same scales and biases per expert
    assert bench.expert_bytes(2048, 512, bits=8) == 3 * 2048 * 512 + 4 * 3 * 2048 * 512 // 64 == 3342336
    assert bench.decode_bytes(c, 1, bits=8) == 9 * 3342336 + 2048 * 256 * 4 + 2048 * 4 + 2 * 2048 * 2 == 32194560
    # T rows reading each of `distinct` selected experts once, plus the shared one
    assert bench.decode_bytes_rows(c, 4, 25) == 26 * 1769472 + 2048 * 256 * 4 + 2048 * 4 + 2 * 4 * 2048 * 2


def test_variant_summary_fractions():
    """The format-variant summary divides the algorithmic work by the measured
    times and the peaks it is given."""
    c = dict(H=2048, E=256, I=512, top_k=8)
    pk = dict(hbm_gbs=6000.0, bf16_tflops=1800.0, bf16_tflops_sustained=1500.0)
    w = dict(t_pre=0.5e-3, t_dec=16e-6, bits=8, k_pre={"gemm_gate_up": 250e-6, "gemm_down": 150e-6})
    v = bench.variant_summary(c, w, 4096, 1, pk)
    flops = bench.gemm_flops(c, 4096, "gate_up") + bench.gemm_flops(c, 4096, "down")
    assert abs(v["prefill"]["tensor_tflops"] - flops / 0.5e-3 / 1e12) < 1e-9
    assert abs(v["prefill"]["frac_of_burst_peak"] - flops / 0.5e-3 / 1e12 / 1800.0) < 1e-12
    assert abs(v["prefill"]["frac_of_sustained_peak"] - flops / 0.5e-3 / 1e12 / 1500.0) < 1e-12
    assert abs(v["prefill"]["gemm_frac_of_burst_peak"]["down"]
               - bench.gemm_flops(c, 4096, "down") / 150e-6 / 1e12 / 1800.0) < 1e-12
    assert v["decode_T1"]["bytes_per_call"] == 32194560
    assert abs(v["decode_T1"]["frac_of_hbm"] - 32194560 / 16e-6 / 1e9 / 6000.0) < 1e-12


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist = bench.init_dist(world, "gloo")
    t = bench.reduce_max(1.0 + rank, dist, "cpu")
    v = bench.job_value(100, world, t)
    q.put((rank, t, v))
    dist.destroy_process_group()


def test_reduce_max_two_ranks():
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
    assert [r[1] for r in res] == [2.0, 2.0]           # every rank sees the slowest rank's time
    assert [r[2] for r in res] == [100.0, 100.0]       # 2 ranks x 100 units / 2 s


def test_measured_traffic_follows_the_sources(tmp_path, monkeypatch):
    """A captured DRAM figure is reported only while the kernel's sources are unchanged."""
    import hashlib
    src = tmp_path / "bit_quantized_sparse_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k.cu").write_text("kernel v1\n")
    (tmp_path / "profiles").mkdir()
    digest = hashlib.sha256(b"kernel v1\n").hexdigest()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"kernels": [
        {"kernel": "my_kernel", "sources": ["csrc/k.cu"], "sha256": digest, "dram_bytes_per_launch": 12345,
         "capture": "a capture"}]}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("my_kernel") == 12345
    assert bench.measured_traffic("other_kernel") is None
    (src / "k.cu").write_text("kernel v2\n")          # the kernel changed after the capture
    assert bench.measured_traffic("my_kernel") is None


def test_spread_percentiles():
    """Per-replay spread: median and the 10th / 90th percentiles, scaled."""
    sp = bench.spread([3.0, 1.0, 2.0, 4.0, 5.0], 1e3)
    assert sp["median"] == 3000.0 and sp["replays"] == 5
    assert abs(sp["p10"] - 1400.0) < 1e-9 and abs(sp["p90"] - 4600.0) < 1e-9
    assert bench.spread([]) is None


def test_spread_bootstrap_interval():
    """The median's bootstrap interval holds the median, lies inside the sample's
    range, is reproducible (seeded) and narrows as the replays grow."""
    import numpy as np
    rng = np.random.default_rng(5)
    small = list(rng.normal(1.0, 0.1, 20))
    big = list(rng.normal(1.0, 0.1, 2000))
    a, b = bench.spread(small), bench.spread(small)
    assert a["median_ci95"] == b["median_ci95"]
    lo, hi = a["median_ci95"]
    assert min(small) <= lo <= a["median"] <= hi <= max(small)
    lo2, hi2 = bench.spread(big)["median_ci95"]
    assert hi2 - lo2 < hi - lo


def test_paired_ratio():
    """Paired rounds: an alternative that always takes twice as long gives a ratio
    of exactly 2 with a degenerate interval; with noise the interval holds the
    median ratio, is reproducible, and the per-arm medians are in ms."""
    import numpy as np
    p = bench.paired_ratio([1e-3, 2e-3, 3e-3], [2e-3, 4e-3, 6e-3])
    assert p["ratio_median"] == 2.0 and p["ratio_ci95"] == [2.0, 2.0] and p["rounds"] == 3
    assert p["a_ms"] == 2.0 and p["b_ms"] == 4.0
    rng = np.random.default_rng(3)
    a = rng.normal(1.0, 0.05, 40)
    b = a * 1.3 + rng.normal(0.0, 0.02, 40)
    q, q2 = bench.paired_ratio(a, b), bench.paired_ratio(a, b)
    assert q["ratio_ci95"] == q2["ratio_ci95"]
    lo, hi = q["ratio_ci95"]
    assert lo <= q["ratio_median"] <= hi and 1.2 < lo and hi < 1.4
