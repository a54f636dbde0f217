"""The seeded input generators (shared by tests, oracle and benchmark)."""
import numpy as np
import torch

import synth


def test_splitmix64_published_outputs():
    # First outputs of SplitMix64 seeded with 0 (reference implementation by Vigna).
    z = synth.splitmix64(0, 4)
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                   0x06C45D188009454F, 0xF88BB8A8724C81EC]
    assert int(synth.splitmix64(0, 2, start=2)[0]) == 0x06C45D188009454F


def test_uniform_and_normal_moments():
    u = synth.uniform01(123, 1 << 20)
    assert u.min() > 0 and u.max() < 1 and abs(u.mean() - 0.5) < 2e-3
    n = synth.normal(5, 1 << 20)
    assert abs(n.mean()) < 5e-3 and abs(n.std() - 1) < 5e-3


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(100000) * np.exp2(rng.integers(-20, 20, 100000))).astype(np.float32)
    ours = synth.f32_to_bf16_bits(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(synth.bf16_bits_to_f32(ours), torch.from_numpy(v).to(torch.bfloat16).float().numpy())


def test_activation_outlier_channels():
    x = synth.activations(64, 4096, seed=0, label="t")
    xf = synth.bf16_bits_to_f32(x)
    col_amax = np.abs(xf).max(axis=0)
    cols = synth.pick(0, "t/outlier-channels/4096", 4096, 4)
    assert cols.size == 4
    assert np.all(col_amax[cols] > 20) and np.median(col_amax) < 5


def test_weights_outlier_rows_and_sigma():
    w = synth.weights(512, 256, seed=1, label="t", sigma=0.015, outlier_rows=8)
    wf = synth.bf16_bits_to_f32(w).astype(np.float64)
    rows = synth.pick(1, "t/outlier-rows/512", 512, 8)
    normal_rows = np.setdiff1d(np.arange(512), rows)
    assert abs(wf[normal_rows].std() - 0.015) < 1e-3
    assert abs(wf[rows].std() - 0.3) < 0.03


def test_router_top2():
    tok, off = synth.route_top2(4096, 8, seed=0)
    assert off[0] == 0 and off[-1] == 8192 and np.all(np.diff(off) >= 0)
    counts = np.diff(off)
    assert counts.min() > 800 and counts.max() < 1250 and len(set(counts.tolist())) > 1
    # each token appears exactly twice, with two distinct experts
    expert_of_row = np.repeat(np.arange(8), counts)
    pairs = {}
    for t, e in zip(tok, expert_of_row):
        pairs.setdefault(int(t), []).append(int(e))
    assert len(pairs) == 4096 and all(len(v) == 2 and v[0] != v[1] for v in pairs.values())
    # stable: rows of one expert keep token order
    for e in range(8):
        seg = tok[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)


def test_deterministic():
    a = synth.activations(3, 256, seed=9)
    b = synth.activations(3, 256, seed=9)
    c = synth.activations(3, 256, seed=10)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
