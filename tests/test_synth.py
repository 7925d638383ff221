"""The seeded input generators: shapes, distributions, bf16 rounding (no GPU)."""
import numpy as np
import torch

import synth


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 3
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0]       # ties to even
    bits = synth.round_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)
    back = synth.bf16_bits_to_f32(bits)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_tiny_workload():
    inp = synth.make_inputs("tiny")
    assert inp.X.shape == (6, 64) and inp.W.shape == (16, 64) and inp.X_bits is None
    assert inp.targets.min() >= 0 and inp.targets.max() < 16
    again = synth.make_inputs("tiny")
    assert np.array_equal(inp.X, again.X) and np.array_equal(inp.targets, again.targets)


def test_zipf_and_ignore():
    wl = synth.WORKLOADS["v152k"]
    inp = synth.make_inputs(synth.Workload("z", 4000, 16, 1000, 8, "bf16", 0.02, "zipf",
                                           ignore_frac=0.1, seed=3))
    y = inp.targets
    assert (y == synth.IGNORE_INDEX).sum() == 400
    v = y[y >= 0]
    assert v.max() < 1000
    # Zipf(1.1): id 0 most frequent, frequencies fall with the id
    c = np.bincount(v, minlength=1000)
    assert c[0] > c[1] > c[10] and c[0] > 10 * c[100]
    assert wl.ignore_frac == 0.1


def test_page_t4_setup_shape():
    z, y = synth.page_t4_simulation()
    assert z.shape == (6, 16) and y.shape == (6,) and y.min() >= 0 and y.max() < 16
