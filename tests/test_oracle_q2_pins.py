"""Pins of the oracle's Q2_0 (ternary) row product against things other than itself.

The pages name Q2_0 as the ternary sibling format and the next GPU kernel
(bankML "docs/modules/gpu.md", "Advantages and efficiency" and "Limitations")
without giving its layout or its arithmetic; the oracle's readings OPEN-10
(34-byte block: fp16 scale + 2-bit codes 0/1/2 = -1/0/+1) and OPEN-11 (the
Q1_0 chain over ternary lane sums) are the contract.  Pins:
  - codes in {0, 2} only (no zero weight): identical bits to the Q1_0 oracle,
    which has its own pins, on the same signs and scales;
  - all scales 1.0: the exact integer dot product with the i8 wrap;
  - all codes 1 (every weight 0): +0 for every row;
  - swapping codes 0 and 2 (negating every weight) with no -128 quant:
    the negated output, bit for bit;
  - format: the weight of every element equals the numpy-decoded code times
    the numpy-decoded scale;
  - general scales: within the f32 chain's error bound of the exact rational
    value.
"""
from fractions import Fraction

import numpy as np
import pytest

from decode_q1_gemv_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def unpack_codes(tblocks):
    """uint8 codes [rows, n] decoded with numpy (element j: byte j//4, bits 2*(j%4))."""
    rows, nb, _ = tblocks.shape
    b = tblocks[:, :, 2:].astype(np.uint8)
    c = np.stack([(b >> (2 * i)) & 3 for i in range(4)], axis=-1)   # [rows, nb, 32, 4]
    return c.reshape(rows, nb * 128)


def ternary_contrib(codes, q):
    """Per-element contribution: +q for code 2, wrapped -q for code 0, 0 for code 1."""
    q = q.astype(np.int64)
    neg = -q
    neg[neg == 128] = -128
    return np.where(codes == 2, q, np.where(codes == 0, neg, 0))


def scales_f64(tblocks):
    s = tblocks[:, :, 0].astype(np.uint16) | (tblocks[:, :, 1].astype(np.uint16) << 8)
    return s.view(np.float16).astype(np.float64)


def test_format_brute_force(oracle_mod):
    rng = synth.rng_for(301)
    tb = synth.ternary_blocks(rng, 3, 256)
    codes = unpack_codes(tb)
    sc = scales_f64(tb)
    for r in range(3):
        for j in range(0, 256, 7):
            want = float(np.float32((int(codes[r, j]) - 1) * sc[r, j // 128]))
            assert oracle_mod.q2_weight(tb, r, j) == want
    bad = tb.copy()
    bad[0, 0, 2] |= 3  # element 0 gets code 3
    assert np.isnan(oracle_mod.q2_weight(bad, 0, 0))


def test_lane_sums_brute_force(oracle_mod):
    rng = synth.rng_for(302)
    tb = synth.ternary_blocks(rng, 3, 512)
    q, _ = synth.raw_quants(rng, 1, 512, m128_frac=0.1)
    want = ternary_contrib(unpack_codes(tb), q.reshape(1, -1)).reshape(3, 4, 4, 8, 4).sum(axis=-1)
    for r in range(3):
        assert np.array_equal(oracle_mod.q2_lane_sums(tb[r], q[0]), want[r])


@pytest.mark.parametrize("regime", ["halfnormal", "lognormal"])
def test_no_zero_weights_equals_q1_0(oracle_mod, regime):
    """Codes 0/2 only: the same signs as a Q1_0 block (code 2 = bit 1), so the
    two oracles must agree bit for bit."""
    rng = synth.rng_for(303, len(regime))
    rows, n = 40, 1024
    nb = n // 128
    bits = rng.integers(0, 2, size=(rows, nb, 128)).astype(np.uint8)
    scales = synth.block_scales(rng, (rows, nb), regime)
    tb = synth.assemble_ternary_blocks(scales, 2 * bits)
    b1 = synth.assemble_blocks(scales, synth.sign_bytes_from_bits(bits))
    q, d = synth.raw_quants(rng, 1, n, scale=regime, m128_frac=0.03)
    got = oracle_mod.q2_gemv(tb, q[0], d[0])
    want = oracle_mod.gemv(b1, q[0], d[0])
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("m128", [0.0, 0.05])
def test_unit_scales_equal_integer_dot(oracle_mod, m128):
    rng = synth.rng_for(304, int(m128 * 100))
    rows, n = 48, 4096
    tb = synth.ternary_blocks(rng, rows, n, "ones")
    q, d = synth.raw_quants(rng, 1, n, scale="ones", m128_frac=m128)
    if m128 == 0.0:
        q[q == -128] = -127
    got = oracle_mod.q2_gemv(tb, q[0], d[0])
    want = ternary_contrib(unpack_codes(tb), q.reshape(1, -1)).sum(axis=1)
    assert np.array_equal(got.astype(np.float64), want.astype(np.float64))


def test_all_zero_weights_give_plus_zero(oracle_mod):
    rng = synth.rng_for(305)
    rows, n = 8, 512
    scales = synth.block_scales(rng, (rows, n // 128), "lognormal")
    tb = synth.assemble_ternary_blocks(scales, np.ones((rows, n // 128, 128), dtype=np.uint8))
    q, d = synth.raw_quants(rng, 1, n, m128_frac=0.05)
    got = oracle_mod.q2_gemv(tb, q[0], d[0])
    assert np.array_equal(got.view(np.uint32), np.zeros(rows, dtype=np.uint32))


def test_negating_weights_negates_bitwise(oracle_mod):
    rng = synth.rng_for(306)
    rows, n = 24, 1024
    tb = synth.ternary_blocks(rng, rows, n, "lognormal")
    q, d = synth.raw_quants(rng, 1, n, scale="lognormal", m128_frac=0.0)
    q[q == -128] = -127
    codes = unpack_codes(tb).reshape(rows, n // 128, 128)
    neg = synth.assemble_ternary_blocks(tb[:, :, 0].astype(np.uint16) | (tb[:, :, 1].astype(np.uint16) << 8),
                                        2 - codes)
    a = oracle_mod.q2_gemv(tb, q[0], d[0])
    b = oracle_mod.q2_gemv(neg, q[0], d[0])
    nz = a != 0
    assert np.array_equal((-a[nz]).view(np.uint32), b[nz].view(np.uint32))


def test_error_bound_against_exact(oracle_mod):
    rng = synth.rng_for(307)
    rows, n = 10, 1024
    nb = n // 128
    tb = synth.ternary_blocks(rng, rows, n, "lognormal")
    q, d = synth.raw_quants(rng, 1, n, scale="lognormal", m128_frac=0.02)
    got = oracle_mod.q2_gemv(tb, q[0], d[0])
    s = ternary_contrib(unpack_codes(tb), q.reshape(1, -1)).reshape(rows, nb, 4, 8, 4).sum(axis=-1)
    d0 = scales_f64(tb)
    d1 = d[0].view(np.float16).astype(np.float64)
    u = Fraction(1, 2 ** 24)
    for r in range(rows):
        total, absum = Fraction(0), Fraction(0)
        for b in range(nb):
            for k in range(4):
                f = Fraction(float(d0[r, b])) * Fraction(float(d1[4 * b + k]))
                for ll in range(8):
                    t = f * int(s[r, b, k, ll])
                    total += t
                    absum += abs(t)
        assert abs(Fraction(float(got[r])) - total) <= (nb + 8) * u * absum, r


def test_rows_sampled_matches_gemv(oracle_mod):
    rng = synth.rng_for(308)
    tb = synth.ternary_blocks(rng, 50, 640)
    q, d = synth.raw_quants(rng, 1, 640, m128_frac=0.02)
    full = oracle_mod.q2_gemv(tb, q[0], d[0])
    idx = np.array([0, 7, 49, 13, 13])
    assert np.array_equal(oracle_mod.q2_rows_sampled(tb, idx, q[0], d[0]).view(np.uint32),
                          full[idx].view(np.uint32))


@pytest.mark.parametrize("threads", [1, 2, 3, 5])
def test_q2_threaded_thread_count_invariance(oracle_mod, threads):
    """The threaded Q2_0 product equals the single-thread one at 1, 2, 3 and 5
    threads (par.md, "How it is verified")."""
    rng = synth.rng_for(61)
    tb = synth.ternary_blocks(rng, 181, 256, p_zero=1 / 3, scale="lognormal")
    q, d = synth.raw_quants(rng, 1, 256, m128_frac=0.02)
    for rows in (1, 16, 17, 181):
        got = oracle_mod.q2_gemv_threaded(tb[:rows], q[0], d[0], threads)
        want = oracle_mod.q2_gemv(tb[:rows], q[0], d[0])
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
