"""Host-side logic of bench.py (CPU only): the roofline object of the bench
line and the clock record taken during the timed region."""

import json
import os

import pytest

import attn_inputs
import bench


def _traffic(tmp_path, kernels, source_hash="abc"):
    os.makedirs(tmp_path / "profiles", exist_ok=True)
    rec = {"workload": "w", "command": "c", "source_hash": source_hash, "kernels": kernels}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))


def test_roofline_takes_the_dominant_kernel_and_scales_traffic_by_heads(tmp_path, monkeypatch):
    w = attn_inputs.WORKLOADS["wide_head_b2h16_n16384_d128"]
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    _traffic(tmp_path, {"bob_pass2": {"bytes_per_launch": 344e6, "heads": 8, "N": w.N, "d": w.d, "duration_ms": 4.4}})
    kernels = {"bob_pass2": (10, 175.0, 0, 0), "attn_fwd": (10, 31.0, 0, 0)}
    r = bench.roofline(w, kernels, 1700.0)
    assert r["kernel"] == "bob_pass2" and r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    flops = 8 * 2.0 * w.N * w.N * w.d * w.B * w.H          # pass 2 owns 8 counted GEMMs
    assert r["counted_flops_per_launch"] == pytest.approx(flops)
    assert r["achieved"] == pytest.approx(flops / 17.5e-3 / 1e12, rel=1e-4)
    assert r["frac"] == pytest.approx(r["achieved"] / 1700.0, rel=1e-3)
    assert r["traffic"] == pytest.approx(344e6 * (w.B * w.H) / 8)
    # pass 2 re-reads Q, UQ, dO (bf16) and L, D, alpha, E (fp32) once per key block of 128
    N, d, h = w.N, w.d, w.B * w.H
    assert r["ledger_bytes"] == pytest.approx(h * (16 * N * d + (6 * d + 16) * N * N / 128))
    assert r["compulsory_bytes"] == pytest.approx(h * (22 * N * d + 16 * N))
    assert r["traffic_over_ledger"] == pytest.approx(r["traffic"] / r["ledger_bytes"], abs=1e-4)
    assert r["traffic_over_compulsory"] == pytest.approx(r["traffic"] / r["compulsory_bytes"], abs=1e-4)


@pytest.mark.parametrize("why", ["stale_hash", "causal", "other_d", "other_kernel"])
def test_roofline_traffic_is_null_unless_it_matches(tmp_path, monkeypatch, why):
    w = attn_inputs.WORKLOADS["wide_head_b2h16_n16384_d128"]
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    rec = {"bytes_per_launch": 1e8, "heads": 8, "N": w.N, "d": w.d if why != "other_d" else 64, "duration_ms": 1.0}
    name = "bob_pass2" if why != "other_kernel" else "attn_fwd"
    _traffic(tmp_path, {name: rec}, source_hash="old" if why == "stale_hash" else "abc")
    pairs = bench.causal_fraction(w.N) if why == "causal" else 1.0
    r = bench.roofline(w, {"bob_pass2": (10, 175.0, 0, 0)}, 1700.0, pairs)
    assert r["traffic"] is None


def test_roofline_without_records_is_null_and_causal_counts_unmasked_pairs():
    w = attn_inputs.WORKLOADS["wide_head_b2h16_n16384_d128"]
    assert bench.roofline(w, {}, 1700.0) is None
    assert bench.causal_fraction(1) == 1.0
    assert bench.causal_fraction(4) == pytest.approx(10 / 16)     # 4 + 3 + 2 + 1 of 16 pairs


class _FakeNvml:
    def __init__(self, samples):
        self.samples = list(samples)

    def sample(self):
        return self.samples.pop(0) if len(self.samples) > 1 else self.samples[0]

    def max_sm(self):
        return 2070.0


def test_clocks_nvml_record_is_median_and_union_of_reasons(tmp_path, monkeypatch):
    monkeypatch.setenv("FBOB_CLOCK_DIR", str(tmp_path / "logs"))
    seq = [(2070.0, []), (1980.0, ["sw_power_cap"]), (2070.0, []), (2055.0, ["sw_power_cap"])]
    monkeypatch.setattr(bench, "_Nvml", lambda index: _FakeNvml(seq))
    c = bench.Clocks(0)
    c.start()
    c.begin()
    import time
    time.sleep(0.05)
    rec = c.stop()
    assert rec["source"] == "nvml" and rec["sm_max_mhz"] == 2070.0
    assert rec["samples"] >= len(seq)
    assert rec["reasons"] == ["sw_power_cap"]
    assert 1980.0 <= rec["sm_mhz"] <= 2070.0
    assert (tmp_path / "logs" / "clocks_rank0.csv").read_text().startswith("sm_mhz,sm_max_mhz,reasons")


def test_clocks_nvml_records_nothing_before_the_timed_region(tmp_path, monkeypatch):
    monkeypatch.setenv("FBOB_CLOCK_DIR", str(tmp_path))
    monkeypatch.setattr(bench, "_Nvml", lambda index: _FakeNvml([(1000.0, ["hw_slowdown"])]))
    c = bench.Clocks(0)
    c.start()
    import time
    time.sleep(0.02)
    assert c.stop() is None          # begin() never called: no sample is taken


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def test_clocks_nvidia_smi_fallback_parses_reasons(tmp_path, monkeypatch):
    monkeypatch.setenv("FBOB_CLOCK_DIR", str(tmp_path))
    c = bench.Clocks(0)
    os.makedirs(os.path.dirname(c.path), exist_ok=True)
    rows = ["0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1995, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2070, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage line"]
    with open(c.path, "w") as f:
        f.write("\n".join(rows) + "\n")
    c.nvml, c.proc, c.f = None, _FakeProc(), open(os.devnull, "w")
    rec = c.stop()
    assert rec == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3,
                   "source": "nvidia-smi"}


def test_bob_ledger_is_the_pages_formula_in_bytes_and_the_kernels_add_the_z_sweep(tmp_path, monkeypatch):
    """Theorem 4.3's ledger (evolve.pub review, Strengths "Theory honestly
    scoped"): 12Nd + 4N + 4dN^2/B_r + (3d+4)N^2/B_c words per head; here in
    bytes with bf16 inputs (Q, K, V, dO, UQ, UK, UV) and fp32 O, vectors and
    outputs.  The kernels as built add the Z sweep: K, V streamed once more
    per row block, Q, dO, L, D, (alpha, E) read again and U1 round-tripped."""
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))   # no committed counters
    for d in (64, 128):
        w = attn_inputs.small(1, 1, 1024, d, "bf16")
        N = w.N
        led = bench.bob_ledger(w)
        words = {"Q dO UQ K V UK UV (bf16)": 7 * N * d * 2, "O (fp32)": N * d * 4, "outputs (fp32)": 4 * N * d * 4,
                 "L D in, alpha E out": 4 * N * 4, "pass 1 streams": 4 * d * N * N / 128 * 2,
                 "pass 2 streams": (3 * d * 2 + 4 * 4) * N * N / 128}
        assert led["pages_ledger_bytes"] == pytest.approx(sum(words.values()))
        # d = 64: pass 1 is one sweep, exactly the pages' schedule; d = 128: plus the Z sweep
        z_sweep = 2 * d * N * N / 128 * 2 + (2 * N * d * 2 + 4 * N * 4) + 2 * N * d * 4 if d > 64 else 0
        assert led["kernels_ledger_bytes"] == pytest.approx(led["pages_ledger_bytes"] + z_sweep)
        assert led["measured_dram_bytes"] is None and "measured_over_ledger" not in led
        assert led["compulsory_bytes"] < led["kernels_ledger_bytes"]


def test_gpus_must_match_the_launched_ranks():
    bench.check_gpus(1, 1)
    bench.check_gpus(4, 4)
    with pytest.raises(SystemExit):
        bench.check_gpus(8, 1)
