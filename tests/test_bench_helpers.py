"""Host-side arithmetic of bench.py (no GPU): the algorithmic bytes behind every GB/s figure of the bench
line, the whole-job throughput and the aggregation of a traced pass into per-kernel medians."""
import importlib.util
import os

import pytest

import ssd_inputs as si

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(_ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)

CFG = si.CONFIGS["llama3_8b"]
LM_HEAD = 2 * 128256 * 4096  # bf16 vocabulary x d_model


def test_layer_bytes_is_the_four_projections_in_16_bits():
    # QKV: (32 query + 2 x 8 KV heads) x 128 rows of 4096; O: 4096 x 4096; gate/up: 2 x 14336 x 4096; down: 4096 x 14336
    assert bench.layer_bytes(CFG) == 2 * (6144 * 4096 + 4096 * 4096 + 2 * 14336 * 4096 + 4096 * 14336) == 436_207_616


def test_pass_bytes_of_the_traffic_capture_forward():
    # the draft forward whose DRAM traffic ncu measured: 2 kept layers, the lm_head, and the fp32 K and V
    # (8 KV heads x 128 x 4 bytes x 2 per layer and token) of 512 visible keys plus the new row
    kv = 2 * 8 * 128 * 4 * 513
    assert bench.pass_bytes(CFG, 2, 512, 1) == 2 * 436_207_616 + LM_HEAD + 2 * kv == 1_931_493_376


def test_pass_bytes_of_the_verify_pass():
    # 32 layers, the lm_head, 7 rows at the generation's mean context of 640 keys (the bench line's figure)
    assert bench.pass_bytes(CFG, 32, 640, 7) == 15_178_924_032


def test_job_throughput_counts_every_rank_over_the_slowest_time():
    assert bench.job_throughput(255, 1, 3264.0) == pytest.approx(78.125, rel=1e-9)
    assert bench.job_throughput(255, 4, 3264.0) == pytest.approx(4 * 78.125, rel=1e-9)


def test_kernel_timeline_medians_and_rates():
    trace, t = [], 1000

    def launch(kind, us):
        nonlocal t
        trace.append((kind, t - 500, t, t + int(us * 1000)))  # (kind, resident, running, end) in ns
        t += int(us * 1000) + 2000

    for scale in (1.0, 1.1, 0.9):  # three layers: the medians are the scale-1.0 layer's times
        launch(10, 12 * scale)  # QKV
        launch(2, 7 * scale)  # attention
        launch(11, 8 * scale)  # residual projection after attention: O
        launch(12, 40 * scale)  # gate/up
        launch(11, 20 * scale)  # residual projection after gate/up: down
    launch(13, 150)  # lm_head
    trace.append((10, 0, 0, 0))  # a slot no CTA wrote is skipped
    out = bench.kernel_timeline(CFG, trace)
    for name, us in (("qkv", 12), ("attention", 7), ("o", 8), ("gate_up", 40), ("down", 20), ("lm_head", 150)):
        assert out[name]["median_us"] == pytest.approx(us), name
    assert out["qkv"]["launches"] == 3 and out["o"]["launches"] == 3 and out["lm_head"]["launches"] == 1
    assert "gbs" not in out["attention"]
    assert out["gate_up"]["gbs"] == pytest.approx(4 * 14336 * 4096 / 40 / 1e3, rel=1e-3)
    assert out["lm_head"]["gbs"] == pytest.approx(LM_HEAD / 150 / 1e3, rel=1e-3)
