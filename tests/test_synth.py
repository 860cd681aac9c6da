"""The seeded input generators: bf16 rounding, determinism and workload shapes."""
import numpy as np
import torch

import synth


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    f = (rng.standard_normal(100_000) * np.exp2(rng.uniform(-30, 30, 100_000))).astype(np.float32)
    f[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]       # ties to even both ways
    ours = synth.bf16_bits_from_f32(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = synth.f32_from_bf16_bits(ours)
    assert np.array_equal(back, torch.from_numpy(ours.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_generators_are_seeded_and_shaped():
    a1, b1, c1 = synth.tiny_end_to_end(seed=1)
    a2, b2, c2 = synth.tiny_end_to_end(seed=1)
    assert a1.shape == (256, 512) and b1.shape == (512, 256) and len(c1) == 4
    assert np.array_equal(a1, a2) and np.array_equal(b1, b2) and np.array_equal(c1, c2)
    x, cols = synth.activation(2, 64, 7168)
    assert x.shape == (64, 7168) and len(cols) == 72
    xf = synth.f32_from_bf16_bits(x)
    assert np.abs(xf[:, cols]).mean() > 50 * np.abs(np.delete(xf, cols, axis=1)).mean()


def test_moe_routing_is_zipf_and_padded():
    counts, offsets = synth.moe_routing(5)
    assert counts.sum() == 16384 * 8
    assert counts[0] == counts.max() and counts[0] > 30000
    pad = np.diff(offsets)
    assert np.all(pad % 128 == 0) and np.all(pad >= counts) and np.all(pad - counts < 128)
    assert offsets[0] == 0 and offsets.dtype == np.int32
