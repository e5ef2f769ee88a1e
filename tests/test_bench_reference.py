"""bench.py --impl reference: the oracle timed as the reference arm (CPU only)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "single_head_n256_d64",
                          "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOPS"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["higher_is_better"] is True
    assert "full runs of the workload" in line["cpu_baseline"]["sample"]   # small enough to run in full


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "single_head_n256_d64",
                          "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=120,
                         env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_paged_cache_layout_reproduces_the_keys():
    """bench --path paged scatters K/V into pages; reading them back through
    the block table must give the contiguous tensors (CPU, no kernel)."""
    torch = __import__("pytest").importorskip("torch")
    sys.path.insert(0, ROOT)
    import bench
    B, H, Nk, d, bs = 3, 2, 150, 8, 16
    g = torch.Generator().manual_seed(5)
    k = torch.randn(B, H, Nk, d, generator=g)
    v = torch.randn(B, H, Nk, d, generator=g)
    kc, vc, table = bench.paged_cache(k, v, bs, seed=11)
    nb = -(-Nk // bs)
    assert kc.shape == (B * nb, H, bs, d) and table.shape == (B, nb) and table.dtype == torch.int32
    assert sorted(table.flatten().tolist()) == list(range(B * nb))   # a permutation of the pages
    for b in range(B):
        for pos in range(Nk):
            phy = int(table[b, pos // bs])
            assert torch.equal(kc[phy, :, pos % bs], k[b, :, pos])
            assert torch.equal(vc[phy, :, pos % bs], v[b, :, pos])
    tail = Nk % bs
    assert torch.count_nonzero(kc[int(table[0, nb - 1]), :, tail:]) == 0


def test_clock_summary_reads_reason_bits():
    """The clock record of the timed region: median SM clock and the names of
    the clock-event reason bits seen (NVML's bit values), CPU only."""
    sys.path.insert(0, ROOT)
    import bench
    sampler = bench.ClockSampler.__new__(bench.ClockSampler)
    sampler.source, sampler.period, sampler.proc = "nvml", 2.5e-4, None
    sampler.samples = [(10.0 + i * 1e-3, 2070.0 - (i % 3), 2070.0, 0x4 if i == 5 else 0) for i in range(20)]
    out = sampler.summary(10.0, 10.0195)
    assert out["samples"] == 20 and out["window"] == "timed region"
    assert out["sm_mhz"] == 2069.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    sampler.samples.append((10.01, 1400.0, 2070.0, 0x8 | 0x40))
    assert set(sampler.summary(10.0, 10.0195)["reasons"]) == {"sw_power_cap", "hw_slowdown", "hw_thermal_slowdown"}
