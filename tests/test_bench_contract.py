"""bench.py's JSON contract, roofline units and measurement hygiene, on the CPU.

- The algorithmic work per launch, which every roofline fraction divides by, is
  checked against counts taken from the tensor shapes of the workload.
- Stored ncu DRAM traffic is reported only while the kernel's source is the one
  it was captured from.
- The clock summary flags throttle reasons from nvidia-smi's CSV.
- The reference arm (the oracle timed on host cores) prints one line with the
  contract's keys.

No GPU is used. The oracle's timing sample is replaced by fixed timings, so no
oracle arithmetic runs here.
"""
import hashlib
import json

import pytest

import bench


def test_decode_bytes_count():
    # One decode launch of the mix: 32 sequences x 32 v-heads (16 k-heads), d = 128.
    n, hv, hk, d = 32, 32, 16, 128
    state = n * hv * d * d * 4 * 2          # S float32, read and written once
    inputs = n * (2 * hk * d + hv * d) * 2  # q, k (per k-head) and v, BF16
    gates = n * hv * 4 * 2                  # a and b, float32
    out = n * hv * d * 2                    # o, BF16
    assert bench.decode_delta_bytes(n) == state + inputs + gates + out == 135_012_352


def test_conv_bytes_count():
    C = 8192
    # 2048-token step of 2 sequences: x in, y out (BF16), taps [C, 4], state [2, C, 3] in + out.
    assert bench.conv_prefill_bytes(2048, 2) == 2048 * C * 2 * 2 + C * 4 * 2 + 2 * C * 3 * 2 * 2
    # 32-sequence decode step: x in, y out, state in + out, taps.
    assert bench.conv_update_bytes(32) == 32 * C * 2 * 2 + 32 * C * 3 * 2 * 2 + C * 4 * 2
    assert bench.conv_update_bytes(32) == 4_259_840


def test_prefill_flops_per_chunk_head():
    # A full 64-token chunk of one head at d = 128 is about 11.6 MFLOP; the
    # count is additive over chunks and heads, and a partial chunk costs less.
    one = bench.prefill_flops([64], d=128, hv=1)
    assert 11.6e6 < one < 11.7e6
    assert bench.prefill_flops([64] * 32, d=128, hv=32) == pytest.approx(32 * 32 * one)
    assert bench.prefill_flops([13], d=128, hv=1) < one
    # Chunks of one token: 5 d + 3 d^2 + 1/6 MACs, twice for flops.
    assert bench.prefill_flops([1], d=128, hv=1) == pytest.approx(2 * (5 * 128 + 3 * 128 * 128 + 1 / 6))


def test_stored_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("__global__ void k() {}\n")
    (tmp_path / "profiles").mkdir()
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(
        {"delta_decode": {"source": "kernel.cu", "source_sha256_16": digest,
                          "dram_bytes_per_launch": 123.0}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.stored_traffic("delta_decode") == 123.0
    assert bench.stored_traffic("conv_prefill") is None
    src.write_text("__global__ void k() { /* changed */ }\n")
    assert bench.stored_traffic("delta_decode") is None


def test_clock_summary_flags_throttle_reasons():
    s = bench.ClockSampler(0)
    s.lines = [
        "2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "2055, 2070, 1390.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "1980, 2070, 1399.0, 0x0000000000000020, Not Active, Active, Not Active, Active",
    ]
    out = s.summary()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2055.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert bench.ClockSampler(0).summary()["samples"] == 0


def test_reference_arm_prints_one_contract_line(monkeypatch, capsys):
    calls = []

    def fake_sample(seconds):
        calls.append(seconds)
        return 2e-3, 5e-4, 0.0            # oracle seconds per decode / prefill token-layer

    def fake_all_cores(seconds, pre, dec):
        calls.append(seconds)
        # four workers, each at the one-thread rate
        return 4 * bench.mix_tokens_per_s(2e-3, 5e-4, pre, dec), 4, 0.0

    monkeypatch.setattr(bench, "cpu_oracle_sample", fake_sample)
    monkeypatch.setattr(bench, "cpu_oracle_all_cores", fake_all_cores)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    assert bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1"]) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in rec, key
    assert rec["impl"] == "reference" and rec["steps"] == 2 and rec["warmup"] == 1
    assert len(calls) == 3                # one warm-up sample, then one all-cores run per step
    from gated_deltanet_linear_build_gb300 import synth
    pre = int(sum(int(x) for x in synth.serving_mix_lengths(bench.rank_lengths_seed(0))))
    dec = bench.DECODE_STEPS * bench.N_SEQS
    # the line's numbers carry six significant digits
    assert rec["value"] == pytest.approx(4 * bench.mix_tokens_per_s(2e-3, 5e-4, pre, dec),
                                         rel=1e-5)
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["value"] == rec["value"]
    assert rec["cpu_baseline"]["cores"] == 4
    assert rec["e2e"] == {"value": rec["value"], "unit": rec["unit"], "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}


def test_cpu_baseline_runs_on_every_core():
    """The all-cores oracle leg spawns one worker per host core (no CUDA context
    is inherited) and sums their rates; zero seconds means one sample each."""
    import os
    value, cores, wall = bench.cpu_oracle_all_cores(0.0, 100, 10)
    assert cores == (os.cpu_count() or 1)
    assert value > 0 and wall > 0


def test_packed_layer_inputs_tile_the_buffer_without_overlap():
    # The end-to-end leg copies each layer's x | z_a | z_b as one buffer: the
    # three views must cover it exactly, in order, aligned for the kernels'
    # 16-byte row loads, at a prefill layer's size and at a decode layer's
    # offset inside a step buffer.
    import torch
    per_tok = bench.E2E_BYTES_PER_TOKEN
    assert per_tok == bench.C * 2 + 2 * bench.HV * 4
    for n, base, layers in ((2048, 0, 1), (1810, 0, 1), (bench.N_SEQS, 0, 3)):
        buf = torch.zeros(layers * n * per_tok, dtype=torch.uint8)
        spans = []
        for l in range(layers):
            x, za, zb = bench.packed_layer_inputs(buf, n, base + l * n * per_tok)
            assert x.shape == (n, bench.C) and x.dtype == torch.bfloat16
            assert za.shape == zb.shape == (n, bench.HV) and za.dtype == torch.float32
            for t in (x, za, zb):
                assert t.is_contiguous()
                off = t.data_ptr() - buf.data_ptr()
                assert off % 16 == 0
                spans.append((off, off + t.numel() * t.element_size()))
        assert spans[0][0] == 0 and spans[-1][1] == buf.numel()
        assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
        # writes through the views land in disjoint bytes
        for l in range(layers):
            x, za, zb = bench.packed_layer_inputs(buf, n, base + l * n * per_tok)
            x.fill_(1.0)
            za.fill_(2.0)
            zb.fill_(3.0)
        for l in range(layers):
            x, za, zb = bench.packed_layer_inputs(buf, n, base + l * n * per_tok)
            assert bool((x == 1.0).all()) and bool((za == 2.0).all()) and bool((zb == 3.0).all())


def test_compact_keeps_six_significant_digits():
    out = bench.compact({"a": 276078.08729208616, "b": [0.9070752634563363, 3],
                         "c": {"d": 1e-7 / 3, "e": "text", "f": None, "g": True}})
    assert out == {"a": 276078.0, "b": [0.907075, 3],
                   "c": {"d": 3.33333e-08, "e": "text", "f": None, "g": True}}
