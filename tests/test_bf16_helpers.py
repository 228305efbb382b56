"""The test-side bf16 helpers (used to compare the workspace's bf16 operand rows bit for bit)
against torch's own fp32 -> bf16 conversion, which rounds to nearest, ties to even."""
import numpy as np
import torch

from gpu_helpers import bf16_rn_bits, bf16_to_f32, decode_dpre, split_planes


def test_round_to_nearest_even_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 1, 10000), rng.normal(0, 1e-30, 1000),
                        rng.normal(0, 1e30, 1000), [0.0, -0.0, 1.0, 1.00390625, 1.01171875]])
    x = x.astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16_rn_bits(x), want)
    assert np.array_equal(bf16_to_f32(want), torch.from_numpy(want.view(np.int16)).view(
        torch.bfloat16).float().numpy())


def test_two_term_split_carries_sixteen_bits():
    rng = np.random.default_rng(1)
    d = rng.normal(0, 1, (3, 2, 4, 5)).astype(np.float32)
    raw = split_planes(d, mp=24)
    assert raw.shape == (3, 2, 2, 24) and not raw[..., 20:].any()
    back = decode_dpre(raw.view(np.int16), 5, 0)
    assert np.max(np.abs(back - d) / np.abs(d)) <= 2.0 ** -16
    one = decode_dpre(raw.view(np.int16), 5, 1)
    assert 2.0 ** -12 < np.max(np.abs(one - d) / np.abs(d)) <= 2.0 ** -8
