"""Pins for the FP64 oracle that do not rely on the oracle itself.

* exact rational arithmetic on tiny shapes (brute force);
* probe rows: a row of x holding one power-of-two entry reproduces a scaled
  weight column exactly (muse_bf16_proj guide, ch. 1, §1.5);
* closed forms: one-hot rows, zero rows, negation and linearity;
* the unpooler slice rule (guide ch. 1, §1.1 table);
* the correctness contract itself, with planted mistakes.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import oracle
from gemv_projection_layers_gb300 import workloads as wl

U = 2.0 ** -53


def _bf16_fraction(b):
    return Fraction(float(wl.bf16_bits_to_f32(np.array([b], np.uint16))[0]))


def _rand_bf16(rng, shape, scale=1.0):
    return wl.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(scale))


@pytest.mark.parametrize("m,N,K", [(1, 5, 7), (3, 7, 13), (9, 32, 64), (4, 3, 1)])
def test_bf16_matches_exact_rational(m, N, K):
    rng = np.random.default_rng(1000 + m * 31 + N * 7 + K)
    x = _rand_bf16(rng, (m, K))
    W = _rand_bf16(rng, (N, K), 0.3)
    # Mix in some extreme magnitudes (tiny, huge, subnormal) so a dropped or
    # misdecoded bit pattern cannot hide.
    W.ravel()[::5] = wl.f32_to_bf16_bits(np.array([3.0e-39, -1.0e30, 7.5e-41, 2.0 ** -20, -65504.0],
                                                  np.float32))[np.arange(W.size)[::5] % 5]
    ref = oracle.reference("pooler", x, W)
    for i in range(m):
        for n in range(N):
            terms = [_bf16_fraction(x[i, k]) * _bf16_fraction(W[n, k]) for k in range(K)]
            exact = sum(terms, Fraction(0))
            bound = K * U * float(sum(abs(t) for t in terms))
            assert abs(Fraction(ref[i, n]) - exact) <= Fraction(bound) + Fraction(0), (i, n)


@pytest.mark.parametrize("m,N,K", [(2, 6, 11), (5, 4, 33)])
def test_router_form_matches_exact_rational(m, N, K):
    rng = np.random.default_rng(7 + m + N + K)
    x = _rand_bf16(rng, (m, K))
    W = (rng.standard_normal((N, K)) / 3.0).astype(np.float32)   # full 24-bit mantissas
    ref = oracle.reference("router", x, W)
    for i in range(m):
        for n in range(N):
            terms = [_bf16_fraction(x[i, k]) * Fraction(float(W[n, k])) for k in range(K)]
            exact = sum(terms, Fraction(0))
            bound = K * U * float(sum(abs(t) for t in terms))
            assert abs(Fraction(ref[i, n]) - exact) <= Fraction(bound), (i, n)


def test_operand_orientation_is_x_times_W_transpose():
    # out[i, n] uses row n of W, not column n: a transposed operand fails here.
    x = wl.f32_to_bf16_bits(np.array([[1, 2, 3]], np.float32))
    W = wl.f32_to_bf16_bits(np.array([[1, 0, 0], [0, 0, 1]], np.float32))
    ref = oracle.reference("o", x, W)
    assert ref.tolist() == [[1.0, 3.0]]


@pytest.mark.parametrize("layer", ["qkv_gate", "router"])
def test_probe_rows_reproduce_scaled_weight_column(layer):
    spec = wl.LAYER_BY_NAME[layer]
    rng = np.random.default_rng(5)
    K, N = spec.K, 64
    if spec.weight_dtype == "fp32":
        W = (rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32)
        wcol = lambda k: W[:, k].astype(np.float64)
    else:
        W = _rand_bf16(rng, (N, K), 1 / np.sqrt(K))
        wcol = lambda k: oracle.bf16_bits_to_f64(W[:, k])
    act = wl.make_activations(layer, 16, seed=1, outliers=True)
    ref = oracle.reference(layer, act.x_bits, W)
    assert len(act.probe_rows) == 2
    for r, c, e, s in zip(act.probe_rows, act.probe_cols, act.probe_exp, act.probe_sign):
        expect = float(s) * 2.0 ** int(e) * wcol(int(c))
        assert np.array_equal(ref[r], expect)


def test_closed_forms_onehot_zero_negation_linearity():
    rng = np.random.default_rng(11)
    K, N = 96, 40
    W = _rand_bf16(rng, (N, K), 0.1)
    one = wl.f32_to_bf16_bits(np.eye(K, dtype=np.float32)[[3, 50, 95]])
    ref = oracle.reference("pooler", one, W)
    for row, k in enumerate([3, 50, 95]):
        assert np.array_equal(ref[row], oracle.bf16_bits_to_f64(W[:, k]))
    zero = np.zeros((2, K), np.uint16)
    assert not oracle.reference("pooler", zero, W).any()
    x = _rand_bf16(rng, (3, K))
    neg = x ^ np.uint16(0x8000)
    assert np.array_equal(oracle.reference("pooler", neg, W), -oracle.reference("pooler", x, W))
    # Linearity within the FP64 bound: x1 + x2 formed exactly (x2 = x1).
    two = wl.f32_to_bf16_bits(2.0 * wl.bf16_bits_to_f32(x))
    r1 = oracle.reference("pooler", x, W)
    assert np.array_equal(oracle.reference("pooler", two, W), 2.0 * r1)


def test_unpooler_slice_rule():
    assert oracle.out_rows("unpooler", 8192, 8) == 1024
    assert oracle.out_rows("unpooler", 8192, 9) == 8192
    assert oracle.out_rows("pooler", 4096, 1) == 4096
    W = wl.make_weights("unpooler", 0)
    x8 = wl.make_activations("unpooler", 8, 0).x_bits
    r8 = oracle.reference("unpooler", x8, W)
    assert r8.shape == (8, 1024)
    # The slice is the first 1024 rows of the full product.
    idx_n = np.array([0, 1, 511, 1023])
    idx_i = np.array([0, 3, 7, 5])
    full = oracle.reference_entries(x8, W, idx_i, idx_n)
    assert np.array_equal(full, r8[idx_i, idx_n])


def test_entries_agree_with_full_reference_and_numpy():
    rng = np.random.default_rng(3)
    x = _rand_bf16(rng, (7, 200))
    W = _rand_bf16(rng, (50, 200), 0.07)
    ref = oracle.reference("qkv_gate", x, W)
    ii = rng.integers(0, 7, 30)
    nn = rng.integers(0, 50, 30)
    assert np.array_equal(oracle.reference_entries(x, W, ii, nn), ref[ii, nn])
    # A library routine computes the same definition (different summation
    # order): agreement within the FP64 bound.
    xd = oracle.bf16_bits_to_f64(x)
    Wd = oracle.bf16_bits_to_f64(W)
    lib = xd @ Wd.T
    bound = 200 * U * (np.abs(xd) @ np.abs(Wd).T)
    assert np.all(np.abs(lib - ref) <= 2 * bound)


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(9)
    x = _rand_bf16(rng, (3, 1024))
    W = _rand_bf16(rng, (300, 1024), 0.03)
    n0 = oracle.threads()
    try:
        oracle.set_threads(1)
        a = oracle.reference("o", x, W)
        oracle.set_threads(max(2, n0))
        b = oracle.reference("o", x, W)
    finally:
        oracle.set_threads(n0)
    assert np.array_equal(a, b)


# --- the contract (guide ch. 1, §1.5), with planted mistakes ----------------

def _ref_and_probe():
    rng = np.random.default_rng(21)
    ref = rng.standard_normal((16, 300))
    return ref, [2, 9]


def test_check_accepts_small_error_and_rejects_planted_mistakes():
    ref, probes = _ref_and_probe()
    rng = np.random.default_rng(22)
    noise = rng.standard_normal(ref.shape)
    ok = ref + 0.004 * np.abs(ref).mean() * noise
    ok[probes] = ref[probes]
    assert oracle.check("pooler", ok, ref, probes)["ok"]
    # global 2 % error
    bad = ref + 0.02 * np.abs(ref).mean() * noise * 1.3
    assert not oracle.check("pooler", bad, ref, probes)["ok"]
    # one row off by 6 % (global ratio still under 1 %)
    row = ok.copy()
    row[5] = ref[5] * 1.06
    r = oracle.check("pooler", row, ref, probes)
    assert r["rel_l2"] < 0.02 and not r["ok"]
    # a probe row off by 0.2 %
    pr = ok.copy()
    pr[9] = ref[9] * 1.002
    assert not oracle.check("pooler", pr, ref, probes)["ok"]
    # NaN
    nan = ok.copy()
    nan[0, 0] = np.nan
    assert not oracle.check("pooler", nan, ref, probes)["ok"]
    # router bound is 100x tighter
    rr = ref + 2e-4 * ref
    assert oracle.check("pooler", rr, ref, [])["ok"]
    assert not oracle.check("router", rr, ref, [])["ok"]
    # transposed / wrong shape
    assert not oracle.check("pooler", ref.T, ref, [])["ok"]
