"""Input generator checks (CPU): determinism, slicing, distribution, the
derived overlap parameter of the M = 10 recipe."""
import json
import os

import numpy as np
import torch

from moe_decode_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_slices_equal_full_tensor():
    full = synth.all_expert_weights(synth.TINY, 0)
    for e in (0, 7, 15):
        part = synth.expert_weights(synth.TINY, 0, e)
        for a, b in zip(full, part):
            assert torch.equal(a[e], b)


def test_deterministic_and_distinct_streams():
    a = synth.normal_f32(5, synth.T_W1, 100, 1000, 1.0)
    b = synth.normal_f32(5, synth.T_W1, 100, 1000, 1.0)
    c = synth.normal_f32(5, synth.T_W3, 100, 1000, 1.0)
    d = synth.normal_f32(6, synth.T_W1, 100, 1000, 1.0)
    assert torch.equal(a, b)
    assert not torch.equal(a, c) and not torch.equal(a, d)


def test_moments():
    v = synth.normal_f32(1000, synth.T_W2, 0, 1 << 20, 0.02).double()
    assert abs(v.mean().item()) < 1e-4
    assert abs(v.std().item() - 0.02) < 2e-4
    kurt = (((v - v.mean()) / v.std()) ** 4).mean().item()
    assert abs(kurt - 2.7) < 0.02  # Irwin-Hall n = 4


def test_overlap_rho_matches_derivation_record():
    rec = json.load(open(os.path.join(GOLDEN, "overlap_rho.json")))
    assert rec["rho"] == synth.RHO_OVERLAP_M10
    assert abs(rec["mean_consecutive_overlap"] - 4.0) <= 0.25


def test_overlap_recipe_is_linear_mix():
    x = synth.x_overlap(synth.LING, 3, 10).float()
    assert x.shape == (10, 2560)
    # tokens share a component: pairwise correlation close to rho
    c = np.corrcoef(x.numpy())
    off = c[~np.eye(10, dtype=bool)]
    assert abs(off.mean() - synth.RHO_OVERLAP_M10) < 0.05


def test_fp8_input_quantiser_matches_the_oracle_definition():
    """The generator's FP8 encoding of synthetic weights (torch float8
    conversion) gives the oracle quantiser's codes and scales bit for bit,
    including an all-zero block and values at the top of the range."""
    import oracle
    oracle.build()
    w = synth.normal_bf16(71, 1, 0, 6 * 384, 0.02).view(6, 384).clone()
    w[2, :128] = 0
    w[4, 5] = 3.0
    c, s = synth.fp8_quantize(w)
    co, so = oracle.fp8_quantize(synth.to_u16(w), 128)
    assert np.array_equal(c.numpy(), co)
    assert np.array_equal(s.numpy().view(np.uint32), so.view(np.uint32))
