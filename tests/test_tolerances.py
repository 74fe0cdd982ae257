"""The parity tolerances against what fp32 arithmetic in the kernels' order
can reach (no GPU).

The kernels sum a row in fp32 as per-thread partial sums over at most a few
hundred elements, combined by a fixed tree (warp butterfly, then the
CTA's warps, then cluster ranks).  Emulated here in numpy float32 against
the float64 oracle, that order keeps rstd within the 1e-6 relative
tolerance at the widest rows (65536), while a plain sequential fp32 sum of
the same squares drifts further -- the tolerance separates the two.  The
dW tolerance (1e-3 relative) is checked the same way for the fixed-order
column sum over per-CTA partials at the largest row count.
"""
import numpy as np

from oracle import rms_norm as orm


def tree_sum_f32(v: np.ndarray, threads: int) -> np.ndarray:
    """Row sums of v [rows, n] in float32: thread t adds elements t,
    t + threads, ... in order, then the thread sums are added pairwise
    (a butterfly over a power-of-two count)."""
    rows, n = v.shape
    per = -(-n // threads)
    pad = np.zeros((rows, per * threads), np.float32)
    pad[:, :n] = v
    acc = np.zeros((rows, threads), np.float32)
    for k in range(per):
        acc = (acc + pad[:, k * threads:(k + 1) * threads]).astype(np.float32)
    while acc.shape[1] > 1:
        half = acc.shape[1] // 2
        acc = (acc[:, :half] + acc[:, half:]).astype(np.float32)
    return acc[:, 0]


def sequential_sum_f32(v: np.ndarray) -> np.ndarray:
    return np.cumsum(v, axis=1, dtype=np.float32)[:, -1]


def rstd_f32(ss: np.ndarray, n: int, eps: float) -> np.ndarray:
    ms = (ss / np.float32(n)).astype(np.float32)
    return (np.float32(1) / np.sqrt(ms + np.float32(eps))).astype(np.float32)


def test_tree_order_meets_the_rstd_tolerance_at_the_widest_rows():
    rng = np.random.default_rng(7)
    n, eps = 65536, 1e-5
    for scale, shift in ((1.0, 0.0), (8.0, 0.0), (1.0, 3.0), (64.0, 10.0)):
        x = (rng.standard_normal((8, n)) * scale + shift).astype(np.float32)
        exact = orm.rstd_exact(x.astype(np.float64), eps)
        sq = (x * x).astype(np.float32)
        tree = rstd_f32(tree_sum_f32(sq, 1024), n, eps)
        seq = rstd_f32(sequential_sum_f32(sq), n, eps)
        err_tree = np.max(np.abs(tree / exact - 1.0))
        err_seq = np.max(np.abs(seq / exact - 1.0))
        assert err_tree <= 1e-6, (scale, shift, err_tree)
        # the tolerance rejects the sequential order (about 2e-6 to 7e-6 here)
        assert err_seq > 1e-6, (scale, shift, err_seq)


def test_column_sum_order_meets_the_dw_tolerance_at_the_largest_batch():
    """dW over 16384 rows: 152 CTAs each add ~108 rows' dy * x_hat in order,
    then the 152 partial rows are added in a fixed order, all in fp32."""
    rng = np.random.default_rng(11)
    rows, n, ctas = 16384, 256, 152
    prod = (rng.standard_normal((rows, n)) * rng.standard_normal((rows, n))).astype(np.float32)
    exact = prod.astype(np.float64).sum(axis=0)
    bounds = [c * rows // ctas for c in range(ctas + 1)]
    parts = np.stack([np.cumsum(prod[bounds[c]:bounds[c + 1]], axis=0,
                                dtype=np.float32)[-1] for c in range(ctas)])
    got = np.cumsum(parts, axis=0, dtype=np.float32)[-1].astype(np.float64)
    floor = np.sqrt(np.mean(exact ** 2))
    rel = np.abs(got - exact) / np.maximum(np.abs(exact), floor)
    assert np.max(rel) <= 1e-3
    # the bound is loose for this order: the error sits far below it
    assert np.max(rel) < 1e-4
