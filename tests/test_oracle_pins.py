"""Pins for the CPU oracle, against things other than the oracle itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a transposed operand, g broadcast along the wrong axis, a double
rounding) fails at least one of them:

* exact rational arithmetic (fractions.Fraction) on tiny random inputs, for
  the dense definition AND for the factored three-term identity;
* closed forms: B = 0 / A = 0 / s = 0, W = 0, rank one, orthonormal A with W
  orthogonal to its row space, W = -sBA (clamp and eps branch);
* small-integer inputs, where every float64 step is exact;
* hand-worked fixtures under tests/golden/ with their citations;
* an independent bf16 rounding implementation (bit arithmetic on float32)
  and torch's float32 -> bf16 cast, on float32-representable values.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from synthetic import configs, gen

RNG = np.random.default_rng(1234)


# ------------------------------------------------------------ helpers
def _exact_dense_sq(W, A, B, s):
    """sum_k (W_jk + s * sum_l B_jl A_lk)^2 in exact rationals, per row."""
    d_out, d_in = W.shape
    r = A.shape[0]
    s = Fraction(s)
    out = []
    for j in range(d_out):
        acc = Fraction(0)
        for k in range(d_in):
            v = Fraction(W[j, k]) + s * sum(Fraction(B[j, l]) * Fraction(A[l, k]) for l in range(r))
            acc += v * v
        out.append(acc)
    return out


def _exact_factored_sq(W, A, B, s):
    """||W_j||^2 + 2s rowsum(B o U)_j + s^2 rowsum((BG) o B)_j, exact rationals."""
    d_out, d_in = W.shape
    r = A.shape[0]
    s = Fraction(s)
    Wf = [[Fraction(x) for x in row] for row in W]
    Af = [[Fraction(x) for x in row] for row in A]
    Bf = [[Fraction(x) for x in row] for row in B]
    G = [[sum(Af[a][k] * Af[b][k] for k in range(d_in)) for b in range(r)] for a in range(r)]
    out = []
    for j in range(d_out):
        base = sum(x * x for x in Wf[j])
        U = [sum(Wf[j][k] * Af[l][k] for k in range(d_in)) for l in range(r)]
        cross = sum(Bf[j][l] * U[l] for l in range(r))
        ba = sum(Bf[j][a] * G[a][b] * Bf[j][b] for a in range(r) for b in range(r))
        out.append(base + 2 * s * cross + s * s * ba)
    return out


def _read_golden(path):
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line or "=" not in line:
                continue
            k, v = (t.strip() for t in line.split("=", 1))
            rows = [[float(x) for x in part.split()] for part in v.split(";")]
            vals[k] = np.array(rows) if len(rows) > 1 else np.array(rows[0])
    return vals


# ------------------------------------------------------------ norm: exact arithmetic
@pytest.mark.parametrize("shape", [(5, 7, 3), (4, 9, 1), (6, 5, 4), (3, 24, 2)])
def test_dense_norm_matches_exact_rationals(shape):
    d_out, d_in, r = shape
    W = RNG.standard_normal((d_out, d_in))
    A = RNG.standard_normal((r, d_in))
    B = RNG.standard_normal((d_out, r))
    s = 1.75
    exact = _exact_dense_sq(W, A, B, s)
    got = oracle.row_norm(W, A, B, s)
    for j in range(d_out):
        want = math.sqrt(float(exact[j]))
        assert abs(got[j] - want) <= 4e-15 * want, (j, got[j], want)


@pytest.mark.parametrize("shape", [(5, 7, 3), (4, 6, 2)])
def test_factored_identity_exact(shape):
    """The three-term decomposition the GPU path relies on equals the dense
    definition exactly (English summary, "Factored Norm"); and the oracle,
    which uses only the dense form, agrees with both."""
    d_out, d_in, r = shape
    W = RNG.standard_normal((d_out, d_in))
    A = RNG.standard_normal((r, d_in))
    B = RNG.standard_normal((d_out, r))
    s = -0.625
    dense = _exact_dense_sq(W, A, B, s)
    fact = _exact_factored_sq(W, A, B, s)
    assert dense == fact
    got = oracle.row_norm(W, A, B, s)
    np.testing.assert_allclose(got ** 2, [float(x) for x in fact], rtol=1e-14)


def test_small_integer_inputs_are_exact():
    d_out, d_in, r = 6, 10, 3
    W = RNG.integers(-3, 4, (d_out, d_in)).astype(np.float64)
    A = RNG.integers(-3, 4, (r, d_in)).astype(np.float64)
    B = RNG.integers(-3, 4, (d_out, r)).astype(np.float64)
    exact = _exact_dense_sq(W, A, B, 2)
    got = oracle.row_norm(W, A, B, 2.0)
    for j in range(d_out):
        assert exact[j].denominator == 1
        assert got[j] == math.sqrt(int(exact[j]))


# ------------------------------------------------------------ norm: closed forms
@pytest.mark.parametrize("zero", ["B", "A", "s"])
def test_no_adapter_gives_plain_row_norm(zero):
    d_out, d_in, r = 7, 33, 5
    W = RNG.standard_normal((d_out, d_in))
    A = RNG.standard_normal((r, d_in)) * (zero != "A")
    B = RNG.standard_normal((d_out, r)) * (zero != "B")
    s = 0.0 if zero == "s" else 1.5
    got = oracle.row_norm(W, A, B, s)
    for j in range(d_out):
        want = math.sqrt(math.fsum(x * x for x in W[j]))
        assert abs(got[j] - want) <= 2e-16 * want * 4


def test_zero_base_weight_gives_gram_form():
    d_out, d_in, r = 5, 11, 3
    W = np.zeros((d_out, d_in))
    A = RNG.standard_normal((r, d_in))
    B = RNG.standard_normal((d_out, r))
    s = -1.25
    Af = [[Fraction(x) for x in row] for row in A]
    G = [[sum(Af[a][k] * Af[b][k] for k in range(d_in)) for b in range(r)] for a in range(r)]
    got = oracle.row_norm(W, A, B, s)
    for j in range(d_out):
        bgb = sum(Fraction(B[j, a]) * G[a][b] * Fraction(B[j, b]) for a in range(r) for b in range(r))
        want = abs(s) * math.sqrt(float(bgb))
        assert abs(got[j] - want) <= 4e-15 * want


def test_rank_one_closed_form():
    d_out, d_in = 6, 40
    W = RNG.standard_normal((d_out, d_in))
    a = RNG.standard_normal(d_in)
    b = RNG.standard_normal(d_out)
    s = 0.8
    got = oracle.row_norm(W, a[None, :], b[:, None], s)
    aa = math.fsum(x * x for x in a)
    for j in range(d_out):
        ww = math.fsum(x * x for x in W[j])
        wa = math.fsum(x * y for x, y in zip(W[j], a))
        want = math.sqrt(ww + 2 * s * b[j] * wa + s * s * b[j] ** 2 * aa)
        assert abs(got[j] - want) <= 1e-14 * want


def test_orthonormal_adapter_orthogonal_weight():
    d_out, d_in, r = 8, 30, 4
    Q, _ = np.linalg.qr(RNG.standard_normal((d_in, r)))
    A = Q.T                                          # orthonormal rows: A A^T = I
    W = RNG.standard_normal((d_out, d_in))
    W = W - (W @ A.T) @ A                            # rows orthogonal to rowspace(A)
    B = RNG.standard_normal((d_out, r))
    s = 1.3
    got = oracle.row_norm(W, A, B, s)
    want = np.sqrt(np.array([math.fsum(x * x for x in W[j]) for j in range(d_out)])
                   + s * s * np.array([math.fsum(x * x for x in B[j]) for j in range(d_out)]))
    np.testing.assert_allclose(got, want, rtol=1e-13)


def test_cancelling_adapter_hits_clamp_and_eps():
    """W = -s B A exactly: every row norm is 0, so g = m / eps
    (Chinese write-up section 1.2.2: clamp at 0 under the root, eps before the divide)."""
    d_out, d_in, r = 4, 9, 2
    A = RNG.integers(-3, 4, (r, d_in)).astype(np.float64)
    B = RNG.integers(-3, 4, (d_out, r)).astype(np.float64)
    s = 2.0
    W = -s * (B @ A)
    wn = oracle.row_norm(W, A, B, s)
    assert np.all(wn == 0.0)
    m = np.array([1.0, 2.0, -3.0, 0.5])
    g = oracle.magnitude_scale(m, wn, 1e-6)
    np.testing.assert_array_equal(g, m / 1e-6)


def test_magnitude_scale_uses_eps_only_below_it():
    wn = np.array([0.0, 1e-7, 1e-6, 2.0])
    m = np.array([1.0, 1.0, 1.0, 3.0])
    g = oracle.magnitude_scale(m, wn, 1e-6)
    np.testing.assert_array_equal(g, [1e6, 1e6, 1e6, 1.5])


def test_golden_tiny_norm(golden_dir):
    gd = _read_golden(os.path.join(golden_dir, "tiny_norm_example.txt"))
    W, A, B = gd["norm.W"], gd["norm.A"][None, :], gd["norm.B"].reshape(-1, 1)
    wn = oracle.row_norm(W, A, B, float(gd["norm.s"][0]))
    # every intermediate is a small integer, so the root is of the exact square
    np.testing.assert_array_equal(wn, np.sqrt(gd["norm.wnorm_sq"]))
    g = oracle.magnitude_scale(gd["norm.m"], wn, float(gd["norm.eps"][0]))
    np.testing.assert_allclose(g, gd["norm.m"] / np.sqrt(gd["norm.wnorm_sq"]), rtol=1e-15)


def test_norm_and_scale_decodes_bf16_rows_independently():
    """Rows are independent: evaluating a subset of rows gives the same values
    as the full evaluation (the sampled checks at large sizes rely on this)."""
    cfg = configs.get(0)
    full = gen.norm_inputs(cfg)
    wn, g = oracle.norm_and_scale(full["W"], full["A"], full["B"], full["m"], cfg.s, cfg.eps, cfg.dtype)
    rows = [0, 5, 63, 17]
    sub = gen.norm_inputs(cfg, rows=rows)
    wn2, g2 = oracle.norm_and_scale(sub["W"], sub["A"], sub["B"], sub["m"], cfg.s, cfg.eps, cfg.dtype)
    np.testing.assert_array_equal(wn2, wn[rows])
    np.testing.assert_array_equal(g2, g[rows])


def test_dora_init_puts_g_near_one():
    """At DoRA's initialisation (B = 0, m = ||W||_row) g is 1 up to the
    magnitude jitter: with m drawn as ||W||_row (1 + N(0, 0.0015)), g has mean
    1 and spread 0.0015 (the concentration the Chinese write-up reports in
    section 2.1.1)."""
    cfg = configs.get(2)
    x = gen.norm_inputs(cfg, rows=range(0, 8192, 8))
    Bz = np.zeros_like(x["B"])
    _, g = oracle.norm_and_scale(x["W"], x["A"], Bz, x["m"], cfg.s, cfg.eps, cfg.dtype)
    assert abs(np.mean(g) - 1.0) < 3e-4
    assert 0.0012 < np.std(g) < 0.0018


# ------------------------------------------------------------ compose
def test_golden_tiny_compose(golden_dir):
    gd = _read_golden(os.path.join(golden_dir, "tiny_norm_example.txt"))
    out = oracle.compose(gd["compose.base"], gd["compose.lora"], gd["compose.g"],
                         float(gd["compose.s"][0]))
    np.testing.assert_array_equal(out, gd["compose.out"])


def _compose_case(dtype, T=16, d=24):
    base = RNG.standard_normal((T, d)).astype(np.float32)
    lora = (0.05 * RNG.standard_normal((T, d))).astype(np.float32)
    if dtype == oracle.BF16:
        base_s, lora_s = gen.f32_to_bf16_bits(base), gen.f32_to_bf16_bits(lora)
    else:
        base_s, lora_s = base, lora
    return base_s, lora_s


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.F32])
def test_compose_special_cases(dtype):
    base_s, lora_s = _compose_case(dtype)
    base, lora = oracle.decode(base_s, dtype), oracle.decode(lora_s, dtype)
    d = base.shape[1]
    s = 2.0
    # g = 1: out = s * lora exactly (s a power of two)
    out = oracle.compose_stored(base_s, lora_s, np.ones(d, np.float32), s, dtype)
    np.testing.assert_array_equal(out, oracle.round_to(s * lora, dtype))
    # g = 0: out = -base exactly
    out = oracle.compose_stored(base_s, lora_s, np.zeros(d, np.float32), s, dtype)
    np.testing.assert_array_equal(oracle.decode(out, dtype), -base)
    # base = 0: out = round(g * s * lora)
    g = (1 + 0.01 * RNG.standard_normal(d)).astype(np.float32)
    zero = np.zeros_like(base_s)
    out = oracle.compose_stored(zero, lora_s, g, s, dtype)
    np.testing.assert_array_equal(out, oracle.round_to(g.astype(np.float64)[None, :] * (s * lora), dtype))
    # s = 0: out = round((g - 1) * base)
    out = oracle.compose_stored(base_s, lora_s, g, 0.0, dtype)
    np.testing.assert_array_equal(out, oracle.round_to((g.astype(np.float64)[None, :] - 1) * base, dtype))


def test_compose_broadcasts_g_per_output_feature():
    base = np.arange(12, dtype=np.float64).reshape(3, 4)
    lora = np.zeros((3, 4))
    g = np.array([1.0, 2.0, 3.0, 4.0])
    out = oracle.compose(base, lora, g, 1.0)
    np.testing.assert_array_equal(out, base * (g - 1)[None, :])


def test_naive_form_is_worse_near_one():
    """The stable form evaluated in float32 has a smaller peak error than the
    naive g*(s*lora+base)-base on the g ~ N(1, 0.0015) distribution (Chinese
    write-up section 2.1.1)."""
    T, d = 256, 512
    base = RNG.standard_normal((T, d)).astype(np.float32)
    lora = (0.05 * RNG.standard_normal((T, d))).astype(np.float32)
    g = (1 + 0.0015 * RNG.standard_normal(d)).astype(np.float32)
    s = 1.0
    ref = oracle.compose(base, lora, g, s)
    naive = oracle.naive_compose_f32(base, lora, g, s).astype(np.float64)
    g32 = g[None, :]
    stable32 = ((g32 - np.float32(1)) * base + g32 * (np.float32(s) * lora)).astype(np.float64)
    err_naive = np.max(np.abs(naive - ref))
    err_stable = np.max(np.abs(stable32 - ref))
    assert err_stable < err_naive / 2


def _read_naive_golden(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "naive_compose_f32.txt")) as f:
        for ln in f:
            if not ln.strip() or ln.startswith("#"):
                continue
            p = ln.split()
            rows.append((float.fromhex(p[0]), float.fromhex(p[1]), float.fromhex(p[2]),
                         float.fromhex(p[3]), int(p[4], 16)))
    return rows


def _naive_pins_hold(naive, golden_dir):
    """Every pin of the naive comparator, for the function `naive`:

    * the hand-worked binary32 rows of tests/golden/naive_compose_f32.txt, bit
      for bit (cancellation near g = 1, a rounding tie, the sign of the final
      subtraction, the scale s);
    * small dyadic inputs where every binary32 step of g*(s*lora+base)-base is
      exact, so the result must equal the float64 compose of the oracle bit
      for bit, on a [T x d] block with T != d (g per output feature)."""
    for base, lora, g, s, bits in _read_naive_golden(golden_dir):
        got = naive(np.array([[base]], np.float32), np.array([[lora]], np.float32),
                    np.array([g], np.float32), s)
        if np.asarray(got, np.float32).reshape(()).view(np.uint32) != bits:
            return False
    rng = np.random.default_rng(77)
    T, d = 24, 40
    base = rng.integers(-8, 9, (T, d)).astype(np.float32)
    lora = rng.integers(-8, 9, (T, d)).astype(np.float32)
    g = rng.choice([0.0, 0.5, 1.0, 1.5, 2.0, 3.0], d).astype(np.float32)
    for s in (0.5, 1.0, 2.0):
        want = oracle.compose(base, lora, g, s)        # exact: every value is a small dyadic
        got = np.asarray(naive(base, lora, g, s))
        if got.shape != want.shape or got.dtype != np.float32:
            return False
        if not np.array_equal(got.astype(np.float64), want):
            return False
    return True


def test_naive_comparator_pinned(golden_dir):
    """The naive comparator (Chinese write-up section 2.1.1) against hand-worked
    binary32 results and against exact small-dyadic cases."""
    assert _naive_pins_hold(oracle.naive_compose_f32, golden_dir)


def test_naive_pins_catch_planted_mistakes(golden_dir):
    """Mistakes planted in copies of the naive comparator (on the CPU) fail the
    pins: the final subtraction flipped, s dropped, g broadcast over tokens
    instead of features, the stable form in its place, float64 intermediates."""
    f32 = np.float32

    def plus_base(b, l, g, s):
        return f32(g)[None, :] * (f32(s) * l + b) + b

    def no_scale(b, l, g, s):
        return g.astype(f32)[None, :] * (l.astype(f32) + b) - b

    def by_token(b, l, g, s):
        gg = np.resize(g.astype(f32), b.shape[0])[:, None]
        return gg * (f32(s) * l + b) - b

    def stable_form(b, l, g, s):
        g = g.astype(f32)[None, :]
        return (g - f32(1)) * b + g * (f32(s) * l)

    def in_float64(b, l, g, s):
        return oracle.compose(b, l, g, s).astype(f32)

    for mutant in (plus_base, no_scale, by_token, stable_form, in_float64):
        assert not _naive_pins_hold(mutant, golden_dir), mutant.__name__


# ------------------------------------------------------------ rounding
def test_bf16_rounding_golden(golden_dir):
    with open(os.path.join(golden_dir, "bf16_rne.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    vals = np.array([float(r[0]) for r in rows])
    want = np.array([int(r[1], 16) for r in rows], dtype=np.uint16)
    np.testing.assert_array_equal(oracle.round_to_bf16_bits(vals), want)


def test_bf16_rounding_matches_independent_casts_on_f32_inputs():
    import torch
    x = np.concatenate([
        RNG.standard_normal(20000).astype(np.float32),
        (RNG.standard_normal(2000) * 1e-38).astype(np.float32),   # subnormal bf16 range
        (RNG.standard_normal(2000) * 1e30).astype(np.float32),
    ])
    ours = oracle.round_to_bf16_bits(x.astype(np.float64))
    bits = gen.f32_to_bf16_bits(x)
    np.testing.assert_array_equal(ours, bits)
    t = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, t)


def test_decode_is_exact():
    bits = np.array([0x3F80, 0x3F81, 0xC000, 0x0001, 0x7F7F], dtype=np.uint16)
    np.testing.assert_array_equal(
        oracle.decode(bits, oracle.BF16),
        [1.0, 1.0078125, -2.0, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127])


# ------------------------------------------------------------ memory figures
def test_memory_figures_from_the_pages(golden_dir):
    with open(os.path.join(golden_dir, "memory_figures.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    MB = float(1 << 20)
    for row in rows:
        kind = row[0]
        if kind == "dense_ba_mb":
            d_out, d_in, r, want = int(row[1]), int(row[2]), int(row[3]), float(row[4])
            assert oracle.dense_ba_bytes(d_out, d_in, 4) / MB == pytest.approx(want, abs=0.05)
        elif kind == "factored_mb":
            d_out, d_in, r, want = int(row[1]), int(row[2]), int(row[3]), float(row[4])
            assert oracle.factored_intermediate_bytes(d_out, r, 4) / MB == pytest.approx(want, abs=0.05)
        elif kind == "ratio":
            d_out, d_in, r, want = int(row[1]), int(row[2]), int(row[3]), float(row[4])
            ratio = oracle.dense_ba_bytes(d_out, d_in, 4) / oracle.factored_intermediate_bytes(d_out, r, 4)
            assert ratio == pytest.approx(want, abs=0.05)
        elif kind == "gram_mb":
            r, want = int(row[1]), float(row[2])
            assert oracle.factored_intermediate_bytes(0, r, 4) / MB == pytest.approx(want, abs=0.05)
        elif kind == "gram_max_mb":
            r, want = int(row[1]), float(row[2])
            assert oracle.factored_intermediate_bytes(0, r, 4) / MB <= want


# ------------------------------------------------------------ d_in-sharded norm
def _exact_partials(W, A, B):
    """base, cross, G by their definitions, in exact rationals."""
    d_out, d_in = W.shape
    r = A.shape[0]
    base = [sum(Fraction(W[j, k]) ** 2 for k in range(d_in)) for j in range(d_out)]
    cross = [sum(Fraction(B[j, l]) * sum(Fraction(W[j, k]) * Fraction(A[l, k]) for k in range(d_in))
                 for l in range(r)) for j in range(d_out)]
    G = [[sum(Fraction(A[a, k]) * Fraction(A[b, k]) for k in range(d_in)) for b in range(r)]
         for a in range(r)]
    return base, cross, G


@pytest.mark.parametrize("cuts", [(), (5,), (0, 3), (2, 2, 7), (1, 4, 9)])
def test_partials_are_the_definitions_and_add_up_exactly(cuts):
    """Small integers: every float64 step is exact, so the shares of each
    column slice equal the rational definitions, the shares of the slices
    (empty ones included) add up to the whole module's, and the identity of
    section 1.2.1 applied to the summed shares gives exactly the dense norm."""
    rng = np.random.default_rng(len(cuts) + 17)
    d_out, d_in, r, s = 5, 10, 3, 2.0
    W = rng.integers(-3, 4, (d_out, d_in)).astype(np.float64)
    A = rng.integers(-3, 4, (r, d_in)).astype(np.float64)
    B = rng.integers(-3, 4, (d_out, r)).astype(np.float64)
    bounds = [0, *cuts, d_in]
    tot_b = np.zeros(d_out)
    tot_c = np.zeros(d_out)
    tot_g = np.zeros((r, r))
    for k0, k1 in zip(bounds[:-1], bounds[1:]):
        b, c, g = oracle.norm_partials(W[:, k0:k1], A[:, k0:k1], B)
        eb, ec, eg = _exact_partials(W[:, k0:k1], A[:, k0:k1], B)
        assert [Fraction(x) for x in b] == eb
        assert [Fraction(x) for x in c] == ec
        assert [[Fraction(x) for x in row] for row in g] == eg
        tot_b += b
        tot_c += c
        tot_g += g
    whole = oracle.norm_partials(W, A, B)
    np.testing.assert_array_equal(tot_b, whole[0])
    np.testing.assert_array_equal(tot_c, whole[1])
    np.testing.assert_array_equal(tot_g, whole[2])
    wn = oracle.norm_from_partials(tot_b, tot_c, tot_g, B, s)
    exact_sq = _exact_dense_sq(W, A, B, s)
    np.testing.assert_array_equal(wn, np.sqrt(np.array([float(x) for x in exact_sq])))


def test_partials_norm_matches_dense_on_random_slices():
    """Real-valued inputs split into four slices of unequal width: the norm from
    the summed shares equals the dense definition to float64 rounding."""
    rng = np.random.default_rng(5)
    d_out, d_in, r, s = 40, 300, 12, -0.75
    W = 0.02 * rng.standard_normal((d_out, d_in))
    A = rng.standard_normal((r, d_in)) / np.sqrt(d_in)
    B = 0.01 * rng.standard_normal((d_out, r))
    parts = [oracle.norm_partials(W[:, a:b], A[:, a:b], B)
             for a, b in ((0, 64), (64, 64), (64, 200), (200, 300))]
    base = sum(p[0] for p in parts)
    cross = sum(p[1] for p in parts)
    G = sum(p[2] for p in parts)
    wn = oracle.norm_from_partials(base, cross, G, B, s)
    ref = oracle.row_norm(W, A, B, s)
    assert np.max(np.abs(wn - ref) / ref) < 1e-13


def test_partials_pins_catch_planted_mistakes():
    """Mistakes planted in copies of norm_from_partials (on the CPU) break the
    exact identity: 2s dropped to s, s^2 to s, the clamp removed on a
    cancelling row."""
    W = np.array([[2.0, -1.0, 0.0], [1.0, 1.0, 1.0]])
    A = np.array([[1.0, 0.0, 1.0]])
    B = np.array([[1.0], [-1.0]])
    s = 2.0
    base, cross, G = oracle.norm_partials(W, A, B)
    exact = np.sqrt(np.array([float(x) for x in _exact_dense_sq(W, A, B, s)]))
    np.testing.assert_array_equal(oracle.norm_from_partials(base, cross, G, B, s), exact)
    ba = np.sum((B @ G) * B, axis=1)
    for wrong in (base + s * cross + s * s * ba, base + 2 * s * cross + s * ba,
                  base + 2 * s * cross):
        assert not np.array_equal(np.sqrt(np.maximum(wrong, 0)), exact)
    # a row with W = -s B A cancels to exactly zero; without the clamp a
    # negative rounding residue would give NaN, with it the norm is 0
    Wc = -s * (B @ A)
    bc, cc, gc = oracle.norm_partials(Wc, A, B)
    assert np.all(oracle.norm_from_partials(bc, cc, gc, B, s) == 0.0)
