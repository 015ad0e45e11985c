"""Pins for the fp32 emulation of the tiled online softmax with the conditional rescale.

The pages claim the conditional rescale changes nothing in the result (the final O / l
division is the one exact correction).  The emulation, run with tau = 0 (rescale
whenever the maximum grows) and tau = 8, must agree with the fp64 oracle to fp32
rounding, and tau = 8 must skip rescales on the outlier workload.
"""
import numpy as np
import pytest

import oracle
from oracle.tiled import tiled_attn
from attn_inputs import make_inputs


@pytest.mark.parametrize("recipe", ["normal", "outliers"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tau", [0.0, 8.0])
def test_tiled_matches_oracle(recipe, causal, tau):
    B, Hq, Hkv, N, d = 1, 2, 1, 320, 64     # 3 key tiles, the last one ragged
    x = make_inputs(71, B, Hq, Hkv, N, d, recipe=recipe)
    scale = 1 / 8
    heads = [(0, 0), (0, 1)]
    O, L, st = tiled_attn(x["q"], x["k"], x["v"], causal, scale, tau, heads)
    Or, Lr = oracle.attn_fwd(x["q"], x["k"], x["v"], causal, scale, heads=heads)
    # fp32 arithmetic on |O| <= max|V|: a few ulp of accumulated rounding per key tile.
    np.testing.assert_allclose(O, Or, rtol=0, atol=2e-5)
    np.testing.assert_allclose(L, Lr, rtol=0, atol=2e-5 * max(1.0, np.abs(Lr).max()))


def test_threshold_skips_rescales():
    x = make_inputs(72, 1, 1, 1, 1024, 64, recipe="outliers")
    heads = [(0, 0)]
    _, _, st0 = tiled_attn(x["q"], x["k"], x["v"], True, 1 / 8, 0.0, heads)
    _, _, st8 = tiled_attn(x["q"], x["k"], x["v"], True, 1 / 8, 8.0, heads)
    assert st0["rescales"] == st0["max_grew"] > 0
    assert st8["rescales"] < st0["rescales"]
    assert st8["inits"] == st0["inits"] == 1024
