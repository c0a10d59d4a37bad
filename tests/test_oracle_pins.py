"""Pins for the fp64 CPU oracle: each check ties it to something other than
itself (the pages' worked examples, closed forms, exact rational arithmetic,
an independent library routine, or invariants of the definition), chosen so
that a dropped term, a wrong sign, a wrong index, a swapped gamma/beta, an
N-1 divisor or a missing eps fails at least one of them. CPU only."""
import itertools
import math
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


# ---------------------------------------------------------------- worked examples

def test_series_true_variance(golden):
    """'第 7 章 LayerNorm 与 RMSNorm' §7.3: mean 1000.0055, var 8.25e-6."""
    g = golden("series_1000.txt")
    x = np.array(g["values"], np.float64)
    mean, var = oracle.row_moments(x)
    assert abs(mean - g["mean"][0]) <= 1e-9
    assert abs(var - g["var"][0]) <= 1e-15


def test_series_fp32_inputs_exact(golden):
    """The same series rounded to fp32 first: the oracle's fp32-input path
    equals the exact rational moments of those fp32 values."""
    xs = np.array(golden("series_1000.txt")["values"], np.float32)
    fr = [Fraction(float(v)) for v in xs]
    mu = sum(fr) / len(fr)
    var = sum((v - mu) ** 2 for v in fr) / len(fr)
    m, v = oracle.row_moments(xs)
    assert abs(m - float(mu)) <= 1e-12
    assert abs(v - float(var)) <= 1e-12 * float(var)
    # the fp32 rounding of the inputs moves the variance off 8.25e-6
    assert abs(float(var) - 8.248128e-6) < 1e-12


def _naive_f32_var(values):
    """E[x^2] - E[x]^2 with every operation rounded to fp32 (the formula the
    pages forbid); used only as a negative control."""
    s = np.float32(0)
    q = np.float32(0)
    for v in values:
        s = np.float32(s + v)
        q = np.float32(q + np.float32(v * v))
    n = np.float32(len(values))
    m = np.float32(s / n)
    return float(np.float32(np.float32(q / n) - np.float32(m * m)))


def test_series_naive_fp32_negative_control(golden):
    """The naive fp32 formula gives only 0 or 0.25 on the series (§7.3), far
    outside any tolerance the parity tests use, while the oracle is exact."""
    g = golden("series_1000.txt")
    xs = [np.float32(v) for v in g["values"]]
    rng = random.Random(0)
    seen = set()
    for _ in range(500):
        rng.shuffle(xs)
        seen.add(_naive_f32_var(xs))
    assert seen <= set(g["naive_f32_outcomes"])
    _, var = oracle.row_moments(np.array(xs, np.float32))
    for bad in seen:
        assert abs(bad - var) > 0.5 * var


def test_mask_example(golden):
    """'T3 讲解' §②, trap 1: N=5 gives var 1.2; the unmasked padded sum 10.8."""
    g = golden("mask_n5.txt")
    x = np.array(g["values"], np.float64)
    mean, var = oracle.row_moments(x)
    assert mean == g["mean"][0]
    assert abs(var - g["var"][0]) <= 1e-15
    # negative control: the padding bug the page describes
    pad = np.zeros(int(g["block_n"][0]))
    pad[: x.size] = x
    unmasked = float(np.sum((pad - pad.sum() / x.size) ** 2) / x.size)
    assert abs(unmasked - g["unmasked_var"][0]) <= 1e-12
    assert abs(unmasked - var) > 1.0


# ---------------------------------------------------------------- Welford / Chan

def _two_pass(vals):
    mu = sum(vals) / len(vals)
    return mu, sum((v - mu) ** 2 for v in vals) / len(vals)


def _trees(items):
    """Every binary merge tree over `items` in the given leaf order."""
    if len(items) == 1:
        yield items[0]
        return
    for k in range(1, len(items)):
        for left in _trees(items[:k]):
            for right in _trees(items[k:]):
                yield (left, right)


def _eval_tree(t):
    if isinstance(t, tuple):
        return oracle.chan_combine(_eval_tree(t[0]), _eval_tree(t[1]))
    return oracle.welford_update(oracle.Welford(0.0, 0.0, 0.0), t)


def test_welford_update_matches_two_pass():
    rng = np.random.default_rng(1)
    for N in range(1, 9):
        for _ in range(20):
            x = rng.normal(rng.uniform(-50, 50), rng.uniform(0.01, 5), N)
            s = oracle.Welford(0.0, 0.0, 0.0)
            for v in x:
                s = oracle.welford_update(s, v)
            mu, var = oracle.row_moments(x)
            assert s.n == N
            assert abs(s.mean - mu) <= 1e-12 * max(1.0, abs(mu))
            assert abs(s.m2 / N - var) <= 1e-12 * max(var, 1e-300) + 1e-13


def test_chan_combine_every_merge_order():
    """Every permutation of the leaves and every tree shape reach the
    two-pass result (the merge is a monoid, '第 7 章' §7.4.1)."""
    rng = np.random.default_rng(2)
    for N in range(1, 6):
        x = list(rng.normal(10.0, 2.0, N))
        mu, var = oracle.row_moments(np.array(x))
        for perm in itertools.permutations(x):
            for t in _trees(list(perm)):
                s = _eval_tree(t)
                assert s.n == N
                assert abs(s.mean - mu) <= 1e-12 * abs(mu)
                assert abs(s.m2 / N - var) <= 1e-11 * var


def test_chan_combine_empty_is_identity():
    a = oracle.Welford(3.0, 1.5, 2.0)
    e = oracle.Welford(0.0, 0.0, 0.0)
    for r in (oracle.chan_combine(a, e), oracle.chan_combine(e, a)):
        assert (r.n, r.mean, r.m2) == (3.0, 1.5, 2.0)
    r = oracle.chan_combine(e, e)
    assert (r.n, r.mean, r.m2) == (0.0, 0.0, 0.0)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("eps", [1e-5, 1e-6])
@pytest.mark.parametrize("N", [1, 7, 4096])
def test_constant_rows(eps, N):
    """var = 0 exactly, rstd = eps^-1/2, LayerNorm y = beta exactly."""
    rng = np.random.default_rng(N)
    for c in (0.0, 1.0, -3.25, 812.5):
        x = np.full((2, N), c, np.float32)
        gamma = rng.uniform(0.5, 1.5, N).astype(np.float32)
        beta = rng.uniform(-0.1, 0.1, N).astype(np.float32)
        e = oracle.eps_as_f32(eps)
        y, mean, rstd = oracle.ln_fwd(x, gamma, beta, e)
        assert np.all(mean == c)
        assert np.all(rstd == 1.0 / math.sqrt(e))
        assert np.array_equal(y, np.broadcast_to(beta.astype(np.float64), y.shape))
        yr, rr = oracle.rms_fwd(x, gamma, e)
        assert np.allclose(rr, 1.0 / math.sqrt(c * c + e), rtol=1e-15)


def test_textbook_cases():
    # [0, 2]: mean 1, var 1; with gamma=1, beta=0, eps=0 the output is [-1, 1]
    x = np.array([[0.0, 2.0]])
    one, zero = np.ones(2), np.zeros(2)
    y, mean, rstd = oracle.ln_fwd(x, one, zero, 0.0)
    assert mean[0] == 1.0 and rstd[0] == 1.0 and list(y[0]) == [-1.0, 1.0]
    # RMS of a row of +-a is 1/sqrt(a^2 + eps) whatever the signs
    a, eps = 3.0, 1e-6
    x = np.array([[a, -a, -a, a, a]])
    w = np.array([1.0, 2.0, 0.5, 1.0, -1.0])
    y, rstd = oracle.rms_fwd(x, w, eps)
    r = 1.0 / math.sqrt(a * a + eps)
    assert abs(rstd[0] - r) <= 1e-16
    assert np.allclose(y[0], x[0] * r * w, rtol=1e-15, atol=0)


@pytest.mark.parametrize("N", [2, 3, 10, 257, 1000])
def test_arithmetic_progression_closed_form(N):
    """x_i = a + b*i: mean = a + b(N-1)/2, var = b^2 (N^2-1)/12."""
    a, b = 3.0, 0.5
    x = a + b * np.arange(N, dtype=np.float64)
    mean, var = oracle.row_moments(x)
    assert abs(mean - (a + b * (N - 1) / 2)) <= 1e-13 * abs(mean)
    assert abs(var - b * b * (N * N - 1) / 12) <= 1e-13 * var


def test_exact_rational_tiny_rows():
    """Brute force: moments of random fp32 rows in exact rational arithmetic."""
    rng = np.random.default_rng(3)
    for N in range(1, 13):
        for _ in range(10):
            x = rng.normal(rng.uniform(-1000, 1000), rng.uniform(1e-3, 10), N).astype(np.float32)
            fr = [Fraction(float(v)) for v in x]
            mu = sum(fr) / N
            var = sum((v - mu) ** 2 for v in fr) / N
            m, v = oracle.row_moments(x)
            assert abs(m - float(mu)) <= 1e-15 * abs(float(mu)) + 1e-300
            assert abs(v - float(var)) <= 1e-9 * float(var) + 1e-18


# ---------------------------------------------------------------- library routine

@pytest.mark.parametrize("N", [1, 5, 33, 1000, 4099])
def test_ln_matches_torch_fp64(N):
    """Independent library routine: torch's CPU LayerNorm in fp64 returns the
    same y, mean and rstd (its mean/rstd via native_layer_norm)."""
    g = torch.Generator().manual_seed(N)
    x = torch.randn(6, N, generator=g, dtype=torch.float64) * 4 + 7
    gamma = torch.rand(N, generator=g, dtype=torch.float64) + 0.5
    beta = torch.rand(N, generator=g, dtype=torch.float64) - 0.5
    eps = 1e-5
    y_t, mean_t, rstd_t = torch.native_layer_norm(x, [N], gamma, beta, eps)
    y, mean, rstd = oracle.ln_fwd(x.numpy(), gamma.numpy(), beta.numpy(), eps)
    assert np.allclose(y, y_t.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(mean, mean_t.numpy().ravel(), rtol=1e-13, atol=1e-13)
    assert np.allclose(rstd, rstd_t.numpy().ravel(), rtol=1e-12, atol=0)


@pytest.mark.parametrize("N", [1, 5, 64, 4099])
def test_rms_matches_torch_fp64(N):
    if not hasattr(torch.nn.functional, "rms_norm"):
        pytest.skip("torch without F.rms_norm")
    g = torch.Generator().manual_seed(100 + N)
    x = torch.rand(6, N, generator=g, dtype=torch.float64) * 2 - 1
    w = torch.rand(N, generator=g, dtype=torch.float64)
    eps = 1e-6
    y_t = torch.nn.functional.rms_norm(x, [N], w, eps)
    y, rstd = oracle.rms_fwd(x.numpy(), w.numpy(), eps)
    assert np.allclose(y, y_t.numpy(), rtol=1e-12, atol=1e-13)
    ms = (x * x).mean(dim=1)
    assert np.allclose(rstd, (1.0 / torch.sqrt(ms + eps)).numpy(), rtol=1e-13)


# ---------------------------------------------------------------- invariants

def test_ln_invariants_and_affine_roles():
    """gamma scales and beta shifts (not the other way round); with gamma=1,
    beta=0 each row has mean 0 and mean square var/(var+eps)."""
    rng = np.random.default_rng(4)
    M, N, eps = 5, 300, 1e-5
    x = rng.normal(2.0, 0.01, (M, N))
    one, zero = np.ones(N), np.zeros(N)
    xhat, mean, rstd = oracle.ln_fwd(x, one, zero, eps)
    var = 1.0 / rstd ** 2 - eps
    assert np.allclose(xhat.mean(axis=1), 0.0, atol=1e-12)
    assert np.allclose((xhat ** 2).mean(axis=1), var / (var + eps), rtol=1e-12)
    gamma = rng.uniform(0.5, 1.5, N)
    beta = rng.uniform(-0.1, 0.1, N)
    y, _, _ = oracle.ln_fwd(x, gamma, beta, eps)
    assert np.allclose(y, xhat * gamma + beta, rtol=1e-13, atol=1e-14)
    # shifting the row leaves the normalised output unchanged
    y2, mean2, rstd2 = oracle.ln_fwd(x + 1000.0, gamma, beta, eps)
    assert np.allclose(mean2, mean + 1000.0, rtol=1e-15)
    assert np.allclose(y2, y, atol=1e-8)


def test_rms_invariants():
    """w=1: mean of y^2 is ms/(ms+eps); scaling x by k>0 and eps by k^2
    leaves y unchanged; no mean is subtracted."""
    rng = np.random.default_rng(5)
    M, N, eps = 4, 513, 1e-6
    x = rng.uniform(-1, 1, (M, N)) + 5.0
    y, rstd = oracle.rms_fwd(x, np.ones(N), eps)
    ms = (x ** 2).mean(axis=1)
    assert np.allclose((y ** 2).mean(axis=1), ms / (ms + eps), rtol=1e-12)
    assert np.all(y > 0)  # a positive row stays positive: nothing was subtracted
    y2, _ = oracle.rms_fwd(x * 8.0, np.ones(N), eps * 64.0)
    assert np.allclose(y2, y, rtol=1e-13)


def test_dtypes_widen_exactly():
    vals = np.array([[1.0, 2.0, -0.5, 3.75]], np.float32)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)  # exact in bf16
    g = np.array([1.5, 0.5, 1.0, 2.0], np.float32)
    b = np.array([0.25, -0.125, 0.0, 1.0], np.float32)
    gb = (g.view(np.uint32) >> 16).astype(np.uint16)
    bb = (b.view(np.uint32) >> 16).astype(np.uint16)
    r32 = oracle.ln_fwd(vals, g, b, 1e-5)
    r16 = oracle.ln_fwd(bits, gb, bb, 1e-5)
    r64 = oracle.ln_fwd(vals.astype(np.float64), g.astype(np.float64), b.astype(np.float64), 1e-5)
    for a, c, d in zip(r32, r16, r64):
        assert np.array_equal(a, c) and np.array_equal(a, d)


# ---------------------------------------------------------------- rounding

def _bf16_to_f64(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def test_round_bf16_ties_and_specials():
    cases = [
        (1.0, 0x3F80),
        (1.0 + 2.0 ** -8, 0x3F80),                 # tie -> even (down)
        (1.0 + 3 * 2.0 ** -8, 0x3F82),             # tie -> even (up)
        (-(1.0 + 2.0 ** -8), 0xBF80),
        (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),    # just above the tie
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (2.0 ** -133, 0x0001),                     # smallest bf16 subnormal
        (2.0 ** -134, 0x0000),                     # half of it: tie -> even (zero)
        (3 * 2.0 ** -134, 0x0002),
        (float("inf"), 0x7F80),
        (-float("inf"), 0xFF80),
        (3.3961e38, 0x7F7F),                       # below the overflow midpoint
        ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),    # the midpoint: tie -> even = inf
        (3.3963e38, 0x7F80),                       # past the midpoint
        (3.3895313892515355e38, 0x7F7F),           # largest finite bf16
    ]
    got = oracle.round_bf16(np.array([v for v, _ in cases]))
    assert [int(v) for v in got] == [b for _, b in cases]
    assert int(oracle.round_bf16(np.array([float("nan")]))[0]) & 0x7FC0 == 0x7FC0


def test_round_bf16_matches_torch_on_fp32_values():
    """Library routine: torch's fp32->bf16 conversion is round-to-nearest-even."""
    rng = np.random.default_rng(6)
    bits = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f) & (np.abs(f) < 3.38e38)]
    t = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    o = oracle.round_bf16(f.astype(np.float64))
    assert np.array_equal(o, t)


def test_round_bf16_nearest_on_doubles():
    """Doubles with more bits than fp32: the result is the nearest bf16 (ties
    to an even last bit), checked against both neighbours."""
    rng = np.random.default_rng(7)
    v = rng.normal(0, 1, 50000) * np.exp2(rng.integers(-30, 30, 50000))
    r = _bf16_to_f64(oracle.round_bf16(v))
    # ulp of the binade of |v|
    ulp = np.exp2(np.floor(np.log2(np.abs(v))) - 7)
    assert np.all(np.abs(v - r) <= ulp / 2)
    tie = np.abs(v - r) == ulp / 2
    assert np.all((oracle.round_bf16(v[tie]) & 1) == 0)


def test_round_f32_matches_numpy():
    rng = np.random.default_rng(8)
    v = rng.normal(0, 1, 100000) * np.exp2(rng.integers(-60, 60, 100000))
    assert np.array_equal(oracle.round_f32(v), v.astype(np.float32))


# ---------------------------------------------------------------- residual add

def test_add_round_matches_torch():
    """Library routine: torch adds fp32 tensors with one IEEE rounding and
    bf16 tensors in fp32 then rounds to bf16 (which equals one rounding of
    the exact sum, fp32 having more than 2*8+2 bits)."""
    g = torch.Generator().manual_seed(11)
    x = torch.randn(4096, generator=g) * torch.exp2(torch.randint(-20, 20, (4096,), generator=g).float())
    r = torch.randn(4096, generator=g) * torch.exp2(torch.randint(-20, 20, (4096,), generator=g).float())
    h = oracle.add_round(x.numpy(), r.numpy())
    assert np.array_equal(h, (x + r).numpy())
    xb, rb = x.to(torch.bfloat16), r.to(torch.bfloat16)
    hb = oracle.add_round(xb.view(torch.int16).numpy().view(np.uint16), rb.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(hb, (xb + rb).view(torch.int16).numpy().view(np.uint16))


def test_add_round_exact_cases():
    one = np.array([1.0], np.float32)
    assert oracle.add_round(one, np.array([2.0 ** -24], np.float32))[0] == 1.0          # tie to even
    assert oracle.add_round(one, np.array([3 * 2.0 ** -24], np.float32))[0] == np.float32(1 + 2.0 ** -22)
    b = lambda v: (np.array([v], np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert int(oracle.add_round(b(1.0), b(2.0 ** -8))[0]) == 0x3F80                       # tie to even (down)
    assert int(oracle.add_round(b(1.0 + 2.0 ** -7), b(2.0 ** -8))[0]) == 0x3F82           # tie to even (up)


def test_fused_add_is_norm_of_the_sum():
    rng = np.random.default_rng(12)
    x = rng.normal(0, 1, (3, 257)).astype(np.float32)
    r = rng.normal(5, 2, (3, 257)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, 257).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, 257).astype(np.float32)
    h, y, mean, rstd = oracle.ln_fwd_add(x, r, g, b, 1e-5)
    assert np.array_equal(h, x + r)
    y2, mean2, rstd2 = oracle.ln_fwd(x + r, g, b, 1e-5)
    assert np.array_equal(y, y2) and np.array_equal(mean, mean2) and np.array_equal(rstd, rstd2)
    h, y, rstd = oracle.rms_fwd_add(x, r, g, 1e-6)
    assert np.array_equal(y, oracle.rms_fwd(x + r, g, 1e-6)[0])


# ---------------------------------------------------------------- backward

def _loss_ln(x, g, b, dy, eps):
    """L = sum dy * y with y the (pinned) forward oracle: its gradient is
    what the backward oracle must return."""
    return float((oracle.ln_fwd(x, g, b, eps)[0] * dy).sum())


def _loss_rms(x, w, dy, eps):
    return float((oracle.rms_fwd(x, w, eps)[0] * dy).sum())


def _fd(f, a, h):
    """Central differences of f with respect to every entry of `a`."""
    out = np.empty(a.shape)
    for idx in np.ndindex(a.shape):
        ap, am = a.copy(), a.copy()
        ap[idx] += h
        am[idx] -= h
        out[idx] = (f(ap) - f(am)) / (2 * h)
    return out


@pytest.mark.parametrize("M,N,eps", [(1, 1, 1e-5), (2, 2, 1e-5), (3, 5, 1e-5), (2, 8, 0.3), (4, 17, 1e-5)])
def test_ln_bwd_is_the_gradient_of_the_forward(M, N, eps):
    """'第 7 章' §7.7 formulas against finite differences of the forward
    definition (step 1e-5: truncation ~1e-10, rounding ~1e-11)."""
    rng = np.random.default_rng(M * 100 + N)
    x = rng.normal(1.0, 2.0, (M, N))
    g = rng.uniform(0.5, 1.5, N)
    b = rng.uniform(-0.5, 0.5, N)
    dy = rng.normal(0, 1, (M, N))
    dx, dg, db = oracle.ln_bwd(dy, x, g, eps)
    h = 1e-5
    assert np.allclose(dx, _fd(lambda a: _loss_ln(a, g, b, dy, eps), x, h), rtol=1e-6, atol=1e-7)
    assert np.allclose(dg, _fd(lambda a: _loss_ln(x, a, b, dy, eps), g, h), rtol=1e-6, atol=1e-7)
    assert np.allclose(db, _fd(lambda a: _loss_ln(x, g, a, dy, eps), b, h), rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("M,N,eps", [(1, 1, 1e-6), (2, 3, 1e-6), (3, 8, 0.5), (4, 19, 1e-6)])
def test_rms_bwd_is_the_gradient_of_the_forward(M, N, eps):
    rng = np.random.default_rng(M * 10 + N)
    x = rng.normal(0.5, 1.5, (M, N))
    w = rng.uniform(0.2, 1.2, N)
    dy = rng.normal(0, 1, (M, N))
    dx, dw = oracle.rms_bwd(dy, x, w, eps)
    h = 1e-5
    assert np.allclose(dx, _fd(lambda a: _loss_rms(a, w, dy, eps), x, h), rtol=1e-6, atol=1e-7)
    assert np.allclose(dw, _fd(lambda a: _loss_rms(x, a, dy, eps), w, h), rtol=1e-6, atol=1e-7)


def test_gamma_outside_the_bracket_is_caught():
    """§7.7 warns that gamma multiplies dy inside the bracket; the formula
    with gamma pulled out (the common mistake) fails the finite-difference
    check that the oracle passes: a negative control of that pin."""
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, (2, 9))
    g = rng.uniform(0.2, 2.0, 9)
    b = np.zeros(9)
    dy = rng.normal(0, 1, (2, 9))
    fd = _fd(lambda a: _loss_ln(a, g, b, dy, 1e-5), x, 1e-5)
    mu = x.mean(1, keepdims=True)
    rs = 1 / np.sqrt(((x - mu) ** 2).mean(1, keepdims=True) + 1e-5)
    xh = (x - mu) * rs
    wrong = rs * g * (dy - dy.mean(1, keepdims=True) - xh * (dy * xh).mean(1, keepdims=True))
    assert np.abs(wrong - fd).max() > 1e-2
    assert np.allclose(oracle.ln_bwd(dy, x, g, 1e-5)[0], fd, rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_ln_bwd_matches_torch_autograd(dtype):
    """Library routine: torch's fp64 layer_norm backward (autograd)."""
    rng = np.random.default_rng(21)
    M, N = 7, 333
    x = rng.normal(3, 2, (M, N)).astype(dtype)
    g = rng.uniform(0.5, 1.5, N).astype(dtype)
    b = rng.uniform(-0.1, 0.1, N).astype(dtype)
    dy = rng.normal(0, 1, (M, N)).astype(dtype)
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    gt = torch.tensor(g, dtype=torch.float64, requires_grad=True)
    bt = torch.tensor(b, dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.layer_norm(xt, (N,), gt, bt, 1e-5)
    y.backward(torch.tensor(dy, dtype=torch.float64))
    dx, dg, db = oracle.ln_bwd(dy, x, g, 1e-5)
    assert np.allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(dg, gt.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(db, bt.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_rms_bwd_matches_torch_autograd():
    rng = np.random.default_rng(22)
    M, N = 6, 250
    x = rng.normal(0, 1, (M, N))
    w = rng.uniform(0, 1, N)
    dy = rng.normal(0, 1, (M, N))
    xt = torch.tensor(x, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    ms = (xt * xt).mean(-1, keepdim=True)
    y = xt * torch.rsqrt(ms + 1e-6) * wt   # written out: RMSNorm by its definition, differentiated by autograd
    y.backward(torch.tensor(dy))
    dx, dw = oracle.rms_bwd(dy, x, w, 1e-6)
    assert np.allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(dw, wt.grad.numpy(), rtol=1e-10, atol=1e-12)
    if hasattr(torch.nn.functional, "rms_norm"):
        xt.grad = None
        wt.grad = None
        torch.nn.functional.rms_norm(xt, (N,), wt, 1e-6).backward(torch.tensor(dy))
        assert np.allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
        assert np.allclose(dw, wt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_bwd_invariants():
    """LayerNorm: sum_i dx_i = 0 for any dy and gamma (xhat sums to zero),
    and with eps = 0 also sum_i dx_i xhat_i = 0 (y does not change when x is
    scaled about its mean). RMSNorm with eps = 0: sum_i dx_i x_i = 0 (y does
    not change when x is scaled)."""
    rng = np.random.default_rng(23)
    M, N = 5, 1000
    x = rng.normal(2, 3, (M, N))
    g = rng.uniform(0.5, 1.5, N)
    dy = rng.normal(0, 1, (M, N))
    dx, _, _ = oracle.ln_bwd(dy, x, g, 1e-5)
    scale = np.abs(dx).sum(1)
    assert np.all(np.abs(dx.sum(1)) <= 1e-13 * scale)
    dx0, _, _ = oracle.ln_bwd(dy, x, g, 0.0)
    xh = (x - x.mean(1, keepdims=True)) / x.std(1, keepdims=True)
    assert np.all(np.abs((dx0 * xh).sum(1)) <= 1e-12 * np.abs(dx0 * xh).sum(1))
    dxr, _ = oracle.rms_bwd(dy, x, g, 0.0)
    assert np.all(np.abs((dxr * x).sum(1)) <= 1e-12 * np.abs(dxr * x).sum(1))


def test_bwd_special_cases():
    """Constant dy with gamma = 1: g is constant, so dx = 0; dbeta_i = M c;
    dgamma_i = c * sum_n xhat_ni. dy = 0: every gradient is zero."""
    rng = np.random.default_rng(24)
    M, N, c = 4, 64, 0.75
    x = rng.normal(0, 1, (M, N))
    dy = np.full((M, N), c)
    dx, dg, db = oracle.ln_bwd(dy, x, np.ones(N), 1e-5)
    assert np.abs(dx).max() <= 1e-13
    assert np.allclose(db, M * c, rtol=0, atol=1e-13)
    mu = x.mean(1, keepdims=True)
    xh = (x - mu) / np.sqrt(((x - mu) ** 2).mean(1, keepdims=True) + 1e-5)
    assert np.allclose(dg, c * xh.sum(0), rtol=1e-12, atol=1e-13)
    z = np.zeros((M, N))
    for v in oracle.ln_bwd(z, x, rng.uniform(0, 1, N), 1e-5) + oracle.rms_bwd(z, x, rng.uniform(0, 1, N), 1e-6):
        assert not v.any()


def test_bwd_bf16_inputs_widen_exactly():
    """bf16 inputs give the gradient of their exact fp32 values."""
    rng = np.random.default_rng(25)
    x = rng.normal(0, 1, (3, 40)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, 40).astype(np.float32)
    dy = rng.normal(0, 1, (3, 40)).astype(np.float32)
    bf = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)
    back = lambda u: (u.astype(np.uint32) << 16).view(np.float32)
    for got, want in zip(oracle.ln_bwd(bf(dy), bf(x), bf(g), 1e-5),
                         oracle.ln_bwd(back(bf(dy)), back(bf(x)), back(bf(g)), 1e-5)):
        assert np.array_equal(got, want)
    for got, want in zip(oracle.rms_bwd(bf(dy), bf(x), bf(g), 1e-6),
                         oracle.rms_bwd(back(bf(dy)), back(bf(x)), back(bf(g)), 1e-6)):
        assert np.array_equal(got, want)


# ---------------------------------------------------------------- fp16

def test_f16_widening_matches_numpy():
    """fp16 patterns (every 7th of the 65536) widen to numpy's value (an
    independent decoder), NaNs to NaN."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    h = bits.view(np.float16)
    got = np.array([oracle.row_moments(h[i:i + 1])[0] for i in range(0, 65536, 7)])
    want = h[::7].astype(np.float64)
    both_nan = np.isnan(got) & np.isnan(want)
    assert np.array_equal(got[~both_nan], want[~both_nan])


def test_round_f16_matches_numpy():
    """Library routine: numpy's float64 -> float16 conversion rounds to
    nearest even; over random magnitudes spanning subnormals to overflow,
    ties, and every fp16 value and midpoint."""
    rng = np.random.default_rng(16)
    v = rng.normal(0, 1, 200000) * np.exp2(rng.integers(-30, 18, 200000))
    allh = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    fin = allh[np.isfinite(allh)].astype(np.float64)
    fin = np.unique(fin)
    mids = (fin[:-1] + fin[1:]) / 2           # exact ties (fp64 holds them)
    for arr in (v, fin, mids, np.array([65504.0, 65519.99, 65520.0, 1e9, -65520.0, 2.0 ** -25, 2.0 ** -26,
                                        3 * 2.0 ** -26, 0.0, -0.0])):
        got = oracle.round_f16(arr)
        with np.errstate(over="ignore"):
            want = arr.astype(np.float16)
        assert np.array_equal(got.view(np.uint16), want.view(np.uint16))


def test_f16_oracle_paths_equal_widened_inputs():
    """fp16 inputs give exactly the results of their widened values."""
    rng = np.random.default_rng(17)
    x = rng.normal(3, 2, (4, 300)).astype(np.float16)
    r = rng.normal(0, 1, (4, 300)).astype(np.float16)
    g = rng.uniform(0.5, 1.5, 300).astype(np.float16)
    b = rng.uniform(-0.1, 0.1, 300).astype(np.float16)
    w = lambda a: a.astype(np.float64)
    for got, want in zip(oracle.ln_fwd(x, g, b, 1e-5), oracle.ln_fwd(w(x), w(g), w(b), 1e-5)):
        assert np.array_equal(got, want)
    for got, want in zip(oracle.ln_bwd(r, x, g, 1e-5), oracle.ln_bwd(w(r), w(x), w(g), 1e-5)):
        assert np.array_equal(got, want)
    h = oracle.add_round(x, r)
    assert h.dtype == np.float16 and np.array_equal(h, (x.astype(np.float32) + r.astype(np.float32)).astype(np.float16))


# ---------------------------------------------------------------- FP8 (E4M3) output

def _torch_e4m3(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch():
    """All 256 codes decode to torch's float8_e4m3fn values (an independent
    library routine), NaN codes to NaN."""
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_values(codes)
    theirs = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    nan = np.isnan(theirs)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2
    assert np.array_equal(ours[~nan], theirs[~nan])
    assert oracle.e4m3_values(np.array([0x7E]))[0] == 448.0 and oracle.e4m3_values(np.array([1]))[0] == 2.0 ** -9


def test_e4m3_rounding_matches_torch_in_range():
    """Nearest-even rounding against torch's cast, on random values below
    the saturation point, every code value, and every midpoint (ties)."""
    rng = np.random.default_rng(8)
    v = rng.normal(0, 1, 100000) * np.exp2(rng.integers(-12, 9, 100000))
    v = v[np.abs(v) < 448]
    vals = np.unique(oracle.e4m3_values(np.arange(256, dtype=np.uint8)))
    vals = vals[np.isfinite(vals)]
    mids = (vals[:-1] + vals[1:]) / 2
    for arr in (v, vals, mids, -mids, np.array([447.0, 447.99, 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -11])):
        arr = arr.astype(np.float32).astype(np.float64)   # torch casts from fp32: give both the same value
        assert np.array_equal(oracle.quant_e4m3(arr, 1.0), _torch_e4m3(arr)), arr[:4]


def test_e4m3_saturates_and_scales():
    """Magnitudes from 448 up give +-448 (0x7E / 0xFE): the saturating form
    the GEMM input takes; NaN stays NaN; the scale divides."""
    big = np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e30, np.inf, -448.5, -np.inf])
    q = oracle.quant_e4m3(big, 1.0)
    assert q.tolist() == [0x7E] * 7 + [0xFE, 0xFE]
    assert oracle.quant_e4m3(np.array([np.nan]), 1.0)[0] == 0x7F
    y = np.array([1.0, -3.0, 0.5])
    assert np.array_equal(oracle.quant_e4m3(y, 0.25), oracle.quant_e4m3(y * 4, 1.0))
    assert oracle.e4m3_values(oracle.quant_e4m3(np.array([2.0]), 1 / 64.0))[0] == 128.0
