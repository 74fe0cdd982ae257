"""The comparison rules of tests/parity.py themselves (no GPU).

The forward output y = (x * rstd) * gain has no cancellation, so it is held
to the specification's rule as written: one ulp everywhere and 99.9% of all
elements bit-identical.  These tests check that the helper enforces exactly
that (a two-ulp element fails even where the cancellation floor would have
let it pass), that the relaxed rule stays confined to outputs marked as
cancelling, and that fp32 arithmetic in the kernels' order -- emulated
here in numpy float32 -- meets the strict rule at the 4096-wide bf16
workload's distribution.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import rms_norm as orm
from oracle import rounding

import parity as P


def _bf16_next_up(v: np.ndarray, k: int = 1) -> np.ndarray:
    """The bf16 value k steps above v (v bf16, positive)."""
    bits = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
    return (bits + k).view(torch.bfloat16).to(torch.float64).numpy()


def test_strict_rule_rejects_two_ulps_the_floor_would_accept():
    ref = np.full((4, 256), 1.0)
    ref[0, 0] = 1e-6                       # tiny element, far below the row rms
    ref = rounding.round_to(ref, "bf16")
    got = ref.copy()
    got[0, 0] = _bf16_next_up(ref[:1, :1], 2)[0, 0]
    # relaxed: within 1e-5 of the row rms, so it passes
    P.check_rows(got, ref, "bf16", None, "dx", cancels=True)
    with pytest.raises(AssertionError, match="out of tolerance"):
        P.check_rows(got, ref, "bf16", None, "y")


def test_strict_rate_counts_every_element():
    ref = rounding.round_to(np.linspace(0.5, 1.5, 4000).reshape(2, 2000), "bf16")
    got = ref.copy()
    # five one-ulp differences in 4000 elements: 99.875% identical
    for j in range(5):
        got[0, 17 * j] = _bf16_next_up(ref[:1, 17 * j:17 * j + 1])[0, 0]
    with pytest.raises(AssertionError, match="bit-identical"):
        P.check_rows(got, ref, "bf16", None, "y")
    got[0, 68] = ref[0, 68]               # four left: exactly the 0.1% allowed
    stats = P.check_rows(got, ref, "bf16", None, "y")
    assert stats["counted"] == 4000 and stats["max_ulp"] == 1


def test_terms_only_with_cancellation():
    ref = np.ones((1, 8))
    with pytest.raises(AssertionError, match="terms only apply"):
        P.check_rows(ref, ref, "f32", None, "y", terms=ref)


def test_fp32_strict_relative_to_the_element():
    ref = np.array([[1.0, 1e-3, 0.0]])
    got = ref * (1 + 2e-5)
    with pytest.raises(AssertionError):
        P.check_rows(got, ref, "f32", None, "y")
    P.check_rows(ref * (1 + 5e-6), ref, "f32", None, "y")


@pytest.mark.parametrize("cast_mode", [orm.ROUND_ONCE, orm.ROUND_TWICE])
def test_fp32_kernel_order_meets_the_strict_rule(cast_mode):
    """rstd from an fp32 sum, x_hat = x * rstd and the gain product in fp32,
    one rounding to bf16 (two for round twice): within one ulp of the
    oracle everywhere, and well over 99.9% identical."""
    w = W.LLAMA_BF16_4096x4096.with_(rows=64, cast_mode=cast_mode)
    inp = W.make_inputs(w)
    x32 = inp["x"].float().numpy()
    g32 = inp["gamma"].float().numpy()
    ss = np.sum(x32.astype(np.float32) ** 2, axis=1, dtype=np.float32)
    rs = (1.0 / np.sqrt(ss / np.float32(w.hidden) + np.float32(w.eps))).astype(np.float32)
    xh = (x32 * rs[:, None]).astype(np.float32)
    if cast_mode == orm.ROUND_TWICE:
        xh = torch.from_numpy(xh).to(torch.bfloat16).float().numpy()
    y32 = (xh * g32[None, :]).astype(np.float32)
    got = torch.from_numpy(y32).to(torch.bfloat16).double().numpy()
    xd, gd = W.as_float64(inp["x"]), W.as_float64(inp["gamma"])
    ref, _ = orm.forward(xd, gd, w.eps, 0, "bf16", cast_mode)
    alt = None
    if cast_mode == orm.ROUND_TWICE:
        x_hat = xd * orm.rstd_exact(xd, w.eps)[:, None]
        mask, lo, hi = P.round_twice_alternatives(x_hat, gd[None, :], "bf16")
        alt = [(mask, lo), (mask, hi)]
    stats = P.check_rows(got, ref, "bf16", alt, "y")
    assert stats["bit_identical"] > 0.9995
