"""Host logic of the measurement, on CPU.

The bandwidth figures the bench reports are algorithmic bytes divided by
measured time, so the byte counts are checked here against the per-layer
figures worked out by hand from each workload's shape: predictor weights
(W1 is h x d, W2 is f x h, plus one fp32 bias per neuron where the workload
places activity with b2), plus every FFN row of each active neuron (up, gate
for the gated activations, and the transposed down row), plus x and y. The
DRAM-traffic figure is a stored ncu capture scaled by the active rows; the
bench reports none once the kernel's sources no longer match the capture.
The clock summary is read from nvidia-smi samples; a fake sample file stands
in for them here.
"""

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from activation_sparse_ffn_gb300 import workload as W  # noqa: E402


@pytest.mark.parametrize("name,count,pred_bytes,row_bytes,with_b2", [
    # d 512, f 2048, h 64, fp32, ReLU, ~205 active: W1 64*512*4 + W2 2048*64*4 + b2 2048*4; 205 x 2 rows of 2 KB
    ("relu_d512_f2048_fp32", 205, 131072 + 524288 + 8192, 205 * 2 * 2048, True),
    # d 4096, f 16384, h 1024, fp16, ReLU, ~1311 active: 8.4 MB + 33.6 MB; 1311 x 2 rows of 8 KB
    ("opt6.7b_relu_d4096_f16384_fp16", 1311, 8388608 + 33554432, 1311 * 2 * 8192, False),
    # d 8192, f 28672, h 1024, bf16, ReGLU, ~2867 active: 16.8 MB + 58.7 MB; 2867 x 3 rows of 16 KB
    ("llama2_70b_reglu_d8192_f28672_bf16_8l", 2867, 16777216 + 58720256, 2867 * 3 * 16384, False),
    # d 4096, f 11008, h 512, bf16, SwiGLU, ~5504 active: 4.2 MB + 11.3 MB; 5504 x 3 rows of 8 KB
    ("swiglu7b_d4096_f11008_bf16_32l", 5504, 4194304 + 11272192, 5504 * 3 * 8192, False),
])
def test_layer_bytes_match_the_shapes(name, count, pred_bytes, row_bytes, with_b2):
    spec = W.WORKLOADS[name]
    b = bench.layer_bytes(spec, count, with_b2)
    assert b["metric"] == pred_bytes + row_bytes + 2 * spec.d * 4
    k = b["kernels"]
    # the FFN kernel's share: the rows plus x and the mask words
    assert k["ffn"] == row_bytes + spec.d * 4 + spec.f // 8
    assert k["pred_hidden"] + k["pred_scores"] >= pred_bytes


def test_zero_skip_counts_only_the_down_rows_read():
    spec = W.WORKLOADS["llama2_70b_reglu_d8192_f28672_bf16_8l"]
    full = bench.layer_bytes(spec, 1000, False)
    half = bench.layer_bytes(spec, 1000, False, kept=500)
    row = spec.d * spec.wbytes
    assert full["metric"] - half["metric"] == 500 * row
    assert bench.layer_bytes(spec, 1000, False, kept=1000)["metric"] == full["metric"]


def test_quantized_rows_count_codes_and_scales():
    q8 = W.WORKLOADS["llama2_70b_reglu_d8192_f28672_q8_8l"]
    q4 = W.WORKLOADS["llama2_70b_reglu_d8192_f28672_q4_8l"]
    bf = W.WORKLOADS["llama2_70b_reglu_d8192_f28672_bf16_8l"]
    n = 100
    pred = bench.layer_bytes(bf, 0, False)["metric"]
    assert bench.layer_bytes(q8, n, False)["metric"] - pred == n * 3 * (8192 + 4)
    assert bench.layer_bytes(q4, n, False)["metric"] - pred == n * 3 * (4096 + 4)


def test_batch_cost_at_one_token_equals_the_single_token_metric():
    spec = W.WORKLOADS["falcon40b_relu_d8192_f32768_fp16_batch"]
    for u in (0, 1, 2294, 13107):
        assert bench.batch_layer_cost(spec, u, 1, False)["metric"] == bench.layer_bytes(spec, u, False)["metric"]
    # every extra token adds only its x and y
    assert (bench.batch_layer_cost(spec, 500, 32, False)["metric"]
            - bench.batch_layer_cost(spec, 500, 1, False)["metric"]) == 31 * 2 * spec.d * 4


def _write_capture(tmp_path):
    src = tmp_path / "k.cu"
    src.write_text("kernel source v1\n")
    d = {
        "launches": [{"active_neurons": 1000, "dram_read": 48_000_000 + 16_000_000, "dram_write": 1_000_000}],
        "l2_prefetch_bytes_per_launch": 16_000_000,
        "bench_workload": "some_layer",
        "sources": [str(src)],
    }
    d["sources_sha256"] = bench.sources_sha256(d["sources"])      # absolute paths join to themselves
    cap = tmp_path / "cap_some_layer.json"
    cap.write_text(json.dumps(d))
    return src, cap


def test_traffic_scales_by_active_rows_only_for_its_workload_and_sources(tmp_path, monkeypatch):
    src, cap = _write_capture(tmp_path)
    monkeypatch.setitem(bench.TRAFFIC_FILES, "ffn", str(tmp_path / "cap_{workload}.json"))
    # 49 KB per neuron once the 16 MB prefetch is taken out; the prefetch is added back when on
    assert bench.measured_traffic("ffn", 2000, False, "some_layer") == pytest.approx(2000 * 49_000)
    assert bench.measured_traffic("ffn", 2000, True, "some_layer") == pytest.approx(2000 * 49_000 + 16_000_000)
    # bytes per neuron of one layer shape say nothing about another (no capture of it)
    assert bench.measured_traffic("ffn", 2000, True, "another_layer") is None
    cap.rename(tmp_path / "cap_another_layer.json")      # a capture filed under the wrong workload
    assert bench.measured_traffic("ffn", 2000, True, "another_layer") is None
    cap = (tmp_path / "cap_another_layer.json").rename(tmp_path / "cap_some_layer.json")
    src.write_text("kernel source v2\n")
    assert bench.measured_traffic("ffn", 2000, True, "some_layer") is None
    assert bench.measured_traffic("no_such_kernel", 2000, True, "some_layer") is None



class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler_with(tmp_path, rows):
    path = tmp_path / "clocks.csv"
    path.write_text("".join(", ".join(r) + "\n" for r in rows))
    s = bench.ClockSampler(0)
    s.proc, s.path, s.fh = _DoneProc(), str(path), open(path, "a")
    return s


def _row(sm, util, hw="Not Active", sw_power="Not Active"):
    # timestamp, index, clocks.sm, clocks.max.sm, power.draw, utilization.gpu, active mask,
    # hw_slowdown, hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    return ["2026/01/01 00:00:00.000", "0", str(sm), "2070", "650.5", str(util), "0x0", hw,
            "Not Active", "Not Active", sw_power]


def test_clock_summary_uses_busy_samples_and_names_throttle_reasons(tmp_path):
    rows = [_row(1980, 0), _row(2070, 97), _row(2055, 99), _row(2040, 98, sw_power="Active"), _row(900, 5)]
    out = _sampler_with(tmp_path, rows).stop()
    assert out["sm_mhz"] == 2055 and out["sm_max_mhz"] == 2070 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]
    # a slowdown during the timed region is reported by name
    out = _sampler_with(tmp_path, [_row(1500, 99, hw="Active"), _row(1490, 99)]).stop()
    assert out["reasons"] == ["hw_slowdown"] and out["sm_mhz"] == 1495


def test_clock_summary_without_nvidia_smi():
    out = bench.ClockSampler(0).stop()
    assert out["samples"] == 0 and out["sm_mhz"] is None and out["reasons"] == ["nvidia-smi unavailable"]


def test_normalize_stand_in_is_x_over_rms():
    """The --normalize harness op divides by the root mean square with no
    epsilon and no learned scale (reading R24), whatever routine computes it."""
    import torch
    g = torch.Generator().manual_seed(3)
    x = torch.randn(3, 4096, generator=g, dtype=torch.float64) * torch.tensor([[1e-3], [1.0], [1e3]], dtype=torch.float64)
    rms = torch.sqrt((x * x).mean(dim=-1, keepdim=True))
    assert torch.allclose(bench.rms_normalize(x), x / rms, rtol=1e-12, atol=0)


def test_profile_steps_must_be_positive(monkeypatch):
    """The roofline line comes from the traced pass, so zero traced steps is refused up front."""
    monkeypatch.setattr(sys, "argv", ["bench.py", "--profile-steps", "0"])
    with pytest.raises(SystemExit):
        bench.parse_args()
    monkeypatch.setattr(sys, "argv", ["bench.py", "--profile-steps", "1"])
    assert bench.parse_args().profile_steps == 1
