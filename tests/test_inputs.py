"""Pins of the seeded input generator (shared by the oracle and the GPU path)."""
import math
import os

import numpy as np
import pytest

import ssd_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_ints(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [int(l) for l in f if l.strip() and not l.startswith("#")]


def test_splitmix64_reference_vector():
    gamma = 0x9E3779B97F4A7C15
    want = _golden_ints("splitmix64.txt")
    got = [si.mix(1234567 + k * gamma) for k in range(len(want))]
    assert got == want


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_normal_moments_and_shape(dtype):
    cfg = si.CONFIGS["tiny"].replace(dtype=dtype)
    spec = si.TensorSpec("t", 12345, (200000,), 0.0, 0.02)
    x = si.widen(si.host_values(spec, cfg), dtype)
    n = x.size
    assert abs(x.mean()) < 5 * 0.02 / math.sqrt(n)
    assert abs(x.std() / 0.02 - 1.0) < 0.01
    # symmetric tails: fraction beyond 2 sigma ~ 4.55 %
    frac = np.mean(np.abs(x) > 0.04)
    assert abs(frac - 0.0455) < 0.003


def test_normal_ks():
    scipy_stats = pytest.importorskip("scipy.stats")
    cfg = si.CONFIGS["tiny"]
    spec = si.TensorSpec("t", 777, (20000,), 0.0, 1.0)
    x = si.widen(si.host_values(spec, cfg), "bf16")
    assert scipy_stats.kstest(x, "norm").pvalue > 1e-3


def test_offset_slices_agree():
    cfg = si.CONFIGS["tiny"]
    spec = si.TensorSpec("t", 99, (1000,), 0.0, 0.02)
    full = si.host_values(spec, cfg)
    part = si.host_values(spec, cfg, offset=123, count=400)
    assert np.array_equal(full[123:523], part)


def test_streams_differ_by_tensor_and_seed():
    cfg = si.CONFIGS["tiny"]
    a = si.host_values(si.TensorSpec("a", 1, (64,), 0.0, 0.02), cfg)
    b = si.host_values(si.TensorSpec("b", 2, (64,), 0.0, 0.02), cfg)
    c = si.host_values(si.TensorSpec("a", 1, (64,), 0.0, 0.02), cfg.replace(seed=1))
    assert not np.array_equal(a, b) and not np.array_equal(a, c)


def test_bf16_rounding_is_round_half_even():
    torch = pytest.importorskip("torch")
    vals = [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 0.1, -0.02, 3.0e-5, 1.0 + 2.0 ** -9]
    for v in vals:
        want = torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
        assert si.const_bits(v, "bf16") == want, v


def test_fp16_rounding_matches_ieee():
    vals = [1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 0.1, -0.02, 3.0e-5, 6.0e-8, 65504.0]
    for v in vals:
        want = int(np.array([np.float32(v)]).astype(np.float16).view(np.uint16)[0])
        assert si.const_bits(v, "fp16") == want, v


def test_prompt_tokens_uniform():
    cfg = si.CONFIGS["tiny"]
    p = si.prompt(cfg, 50000)
    assert p.min() >= 0 and p.max() < cfg.vocab
    counts = np.bincount(p, minlength=cfg.vocab)
    exp = p.size / cfg.vocab
    chi2 = np.sum((counts - exp) ** 2 / exp)
    assert chi2 < cfg.vocab + 6 * math.sqrt(2 * cfg.vocab)


def test_workload_skip_sets():
    c8 = si.CONFIGS["llama3_8b"]
    assert c8.skip == tuple(range(1, 32, 2))
    c13 = si.CONFIGS["llama2_13b_cascade"]
    (l1, i1), (l2, i2), (l3, i3) = c13.levels
    assert l2 == (1, 5, 8, 11, 15, 18, 21, 25, 28, 31, 35, 38) and i2
    assert len(l1) == 28 and set(l2) <= set(l1) and not i1
    assert tuple(i for i in range(40) if i not in l1) == (2, 4, 7, 12, 14, 17, 22, 24, 27, 32, 34, 37)
    assert l3 == () and i3
    assert si.CONFIGS["tiny"].skip == (1, 2)


def test_output_projection_scale():
    cfg = si.CONFIGS["llama3_8b"]
    specs = {s.name: s for s in si.layer_specs(cfg, 3)}
    assert specs["wo"].sigma == pytest.approx(0.02 / 8.0)
    assert specs["wd"].sigma == pytest.approx(0.02 / 8.0)
    assert specs["wq"].sigma == 0.02 and specs["g_attn"].sigma == 0.0 and specs["g_attn"].mean == 1.0
