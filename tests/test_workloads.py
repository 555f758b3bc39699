"""Host-side checks of the seeded input recipes (no GPU, no method arithmetic)."""

import numpy as np
import torch

from workloads import (IGNORE_INDEX, WORKLOADS, bf16_bits_from_f32, bf16_bits_to_f32, generate,
                       workload)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 37.0,
                        np.array([1.0 + 2**-8, 1.0 + 3 * 2**-8, -1.0 - 2**-8, 0.0, -0.0], np.float32)])
    ours = bf16_bits_from_f32(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_five_workloads_listed():
    assert len(WORKLOADS) == 5
    assert workload("lmhead").T == 65536 and workload("lmhead").V == 124160
    assert workload("long").Hd == 4096 and workload("long").reduction == "sum"
    assert workload("rlpg").n_seq == 8 and workload("rlpg").reduction == "none"
    assert workload("lmhead").flops == 8 * 65536 * 2048 * 124160


def test_generation_is_deterministic_and_shaped():
    a = generate("tiny")
    b = generate("tiny")
    assert np.array_equal(a.H_bits, b.H_bits) and np.array_equal(a.W_bits, b.W_bits)
    assert np.array_equal(a.targets, b.targets)
    assert a.H_bits.shape == (256, 256) and a.W_bits.shape == (4096, 256)
    assert a.targets.dtype == np.int64 and a.H_bits.dtype == np.uint16
    assert a.targets.min() >= 0 and a.targets.max() < 4096
    c = generate("tiny", seed=1)
    assert not np.array_equal(a.H_bits, c.H_bits)
    w = bf16_bits_to_f32(a.W_bits)
    assert abs(float(w.std()) - 0.02) < 0.001


def test_ignore_and_zipf_recipe():
    inp = generate("medium", T=4000, Hd=64, V=5000)
    assert int((inp.targets == IGNORE_INDEX).sum()) == 200
    valid = inp.targets[inp.targets != IGNORE_INDEX]
    assert valid.min() >= 0 and valid.max() < 5000
    # bounded Zipf(1.1): rank 1 carries p1 = 1 / H_{5000,1.1} of the mass
    p1 = 1.0 / np.sum(np.arange(1, 5001, dtype=np.float64) ** -1.1)
    assert abs(np.mean(valid == 0) - p1) < 0.03


def test_outlier_recipe():
    inp = generate("lmhead", T=512, Hd=256, V=300)
    h = np.abs(bf16_bits_to_f32(inp.H_bits))
    frac_big = np.mean(h > 8.0)
    assert 0.0004 < frac_big < 0.002


def test_policy_gradient_recipe():
    inp = generate("rlpg", T=8 * 100, Hd=64, V=1000)
    L = 100
    for s in range(8):
        seg = inp.targets[s * L:(s + 1) * L]
        assert np.all(seg[:30] == IGNORE_INDEX) and np.all(seg[30:] >= 0)
        d = inp.dloss[s * L:(s + 1) * L]
        assert np.all(d == d[0])
    assert inp.dloss.shape == (800,) and inp.reduction == "none"
