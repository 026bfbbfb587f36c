"""Pins of the oracle's MXFP4 quantizer against what the MXAttention pages fix.

* E2M1 grid and thresholds: "MXAttention" Eq. (9), (20), (67)-(68) -> tests/golden/e2m1_grid.txt
* round-to-nearest with saturation at +-6: Eq. (10); ties to even: reading R1
* UOS exponent e = ceil(log2(M/7.25)): Eq. (13), (19), Algorithm 1
* worked example M = 14.5 -> e = 1, scale 2 (explainer page), and
  e(1) = -2, Q*(1) = 1 (Appendix J) -> tests/golden/uos_worked_example.txt
* normalised maximum in (3.625, 7.25]: text after Algorithm 1
* OCP floor rule maps maxima into [4, 8) (Eq. 11, 97); TFS into (3, 6] (Eq. 14)
* all-zero block -> sigma = 1, codes 0: section 2, last paragraph
* V blocks of 32 consecutive tokens; Q/K blocks of 32 channels: MatX note
"""
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.split() for l in f if l.strip() and not l.startswith("#")]


def test_e2m1_grid_values(orc):
    g = dict((l[0], [float(x) for x in l[1:]]) for l in _golden_lines("e2m1_grid.txt"))
    mags = [orc.e2m1_value(c) for c in range(8)]
    assert mags == g["grid"]
    assert [orc.e2m1_value(c | 8) for c in range(8)] == [-m for m in g["grid"]]


def test_e2m1_thresholds_and_ties(orc):
    g = dict((l[0], [float(x) for x in l[1:]]) for l in _golden_lines("e2m1_grid.txt"))
    grid, th = g["grid"], g["thresholds"]
    for k, t in enumerate(th):
        below, above = np.nextafter(t, -np.inf), np.nextafter(t, np.inf)
        assert orc.e2m1_value(int(orc.e2m1_code(below))) == grid[k]
        assert orc.e2m1_value(int(orc.e2m1_code(above))) == grid[k + 1]
        # exact tie: the neighbour whose code has mantissa bit 0 (even code)
        tie = grid[k] if k % 2 == 0 else grid[k + 1]
        assert orc.e2m1_value(int(orc.e2m1_code(t))) == tie, t


def test_e2m1_brute_force_nearest(orc):
    """Dense sweep of [-8, 8]: the code's value is a nearest signed grid point;
    beyond +-6 it saturates."""
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6.0])
    signed = np.unique(np.concatenate([-grid, grid]))
    v = np.concatenate([np.linspace(-8, 8, 4001), np.linspace(-0.3, 0.3, 601)])
    codes = orc.e2m1_code(v)
    vals = np.array([orc.e2m1_value(int(c)) for c in codes])
    dist = np.abs(v[:, None] - signed[None, :]).min(axis=1)
    inside = np.abs(v) <= 6
    assert np.all(np.abs(vals - v)[inside] == dist[inside])
    assert np.all(vals[~inside] == np.sign(v[~inside]) * 6)


def test_e2m1_saturation_and_sign(orc):
    for v in [6.0, 6.5, 7.0, 7.25, 8.0, 100.0, 1e30]:
        assert int(orc.e2m1_code(v)) == 7
        assert int(orc.e2m1_code(-v)) == 15
    assert int(orc.e2m1_code(0.0)) == 0
    assert int(orc.e2m1_code(-0.0)) == 8
    assert int(orc.e2m1_code(-0.1)) == 8      # negative value rounding to zero keeps its sign
    assert int(orc.e2m1_code(0.1)) == 0


def test_uos_worked_examples(orc):
    rows = _golden_lines("uos_worked_example.txt")
    for M, e, s in rows:
        M, e, s = float(M), int(e), float(s)
        assert orc.scale_exponent(M, orc.UOS) == e
        assert 2.0 ** e == s
    # Appendix J: Q*(1) = 1 exactly
    codes, scales = orc.rotate_quantize_qk(_bf16_bits(np.array([[1.0] + [0.0] * 127])), rotate=False)
    assert scales[0, 0] == 127 - 2 and orc.e2m1_value(int(codes[0, 0])) * 2.0 ** -2 == 1.0


def test_uos_boundaries_and_ceil(orc):
    for k in range(-40, 41):
        M = 7.25 * 2.0 ** k
        assert orc.scale_exponent(M, orc.UOS) == k                       # normalized max exactly 7.25
        assert orc.scale_exponent(np.nextafter(M, np.inf), orc.UOS) == k + 1
    rng = np.random.default_rng(0)
    for M in np.exp2(rng.uniform(-60, 60, 20000)):
        z = math.log2(M / 7.25)
        if abs(z - round(z)) < 1e-9:
            continue
        assert orc.scale_exponent(M, orc.UOS) == math.ceil(z)


def test_normalized_max_ranges(orc):
    rng = np.random.default_rng(1)
    M = np.exp2(rng.uniform(-100, 100, 50000))
    for rule, lo, hi, lo_open, hi_open in [(orc.UOS, 3.625, 7.25, True, False),
                                           (orc.OCP, 4.0, 8.0, False, True),
                                           (orc.TFS, 3.0, 6.0, True, False)]:
        x = np.array([m / 2.0 ** orc.scale_exponent(m, rule) for m in M])
        assert np.all(x > lo) if lo_open else np.all(x >= lo)
        assert np.all(x < hi) if hi_open else np.all(x <= hi)


def test_ocp_overflow_probability_log_uniform(orc):
    """Eq. (15)/(85): under a log-uniform phase, Pr(OCP-normalised max >= 7) = log2(8/7)."""
    p_ref = float([l for l in _golden_lines("uos_closed_forms.txt") if l[0] == "p_overflow"][0][1])
    assert abs(p_ref - math.log2(8 / 7)) < 1e-15
    rng = np.random.default_rng(2)
    M = np.exp2(rng.uniform(0, 1, 40000) + rng.integers(-30, 30, 40000))
    x = np.array([m / 2.0 ** orc.scale_exponent(m, orc.OCP) for m in M])
    p = np.mean(x >= 7.0)
    assert abs(p - p_ref) < 4 * math.sqrt(p_ref * (1 - p_ref) / M.size)


def _bf16_bits(x):
    import torch

    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_qk_block_quantization_without_rotation(orc):
    """Algorithm 1 per 32-channel block, checked block by block."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 128)) * np.exp2(rng.integers(-8, 8, (64, 1)))
    x[5, 32:64] = 0.0  # an all-zero block
    bits = _bf16_bits(x)
    xb = bits.astype(np.uint32) << 16
    xf = xb.view(np.float32).astype(np.float64)
    codes, scales = orc.rotate_quantize_qk(bits, rotate=False)
    for r in range(64):
        for b in range(4):
            blk = xf[r, 32 * b: 32 * b + 32]
            M = np.abs(blk).max()
            if M == 0:
                assert scales[r, b] == 127 and np.all(codes[r, 32 * b: 32 * b + 32] == 0)
                continue
            e = int(scales[r, b]) - 127
            assert e == math.ceil(math.log2(M / 7.25)) or abs(math.log2(M / 7.25) - round(math.log2(M / 7.25))) < 1e-12
            deq = np.array([orc.e2m1_value(int(c)) for c in codes[r, 32 * b: 32 * b + 32]]) * 2.0 ** e
            # each element is a nearest grid point of blk / 2^e (saturated)
            grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6.0])
            signed = np.concatenate([-grid, grid])
            y = blk / 2.0 ** e
            best = np.abs(y[:, None] - signed[None, :]).min(axis=1)
            assert np.all(np.abs(deq / 2.0 ** e - y) <= best + 1e-12)


def test_v_token_blocks_and_short_tail(orc):
    """V is blocked along tokens (32 consecutive tokens per channel); the last block is short."""
    rng = np.random.default_rng(4)
    N = 100
    v = rng.standard_normal((2, N, 128))
    v[1, 96:, 7] = 1e-3 * np.array([1, -2, 3, -4])  # tail block of channel 7, head 1
    v[0, 40, 9] = 50.0                               # a spike in block 1 of channel 9
    bits = _bf16_bits(v)
    codes, scales = orc.quantize_v(bits)
    assert codes.shape == (2, N, 128) and scales.shape == (2, 128, 4)
    vf = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    tail = vf[1, 96:, 7]
    assert int(scales[1, 7, 3]) - 127 == orc.scale_exponent(np.abs(tail).max())
    assert int(scales[0, 9, 1]) - 127 == orc.scale_exponent(np.abs(vf[0, 32:64, 9]).max())
    assert int(scales[0, 9, 0]) - 127 == orc.scale_exponent(np.abs(vf[0, 0:32, 9]).max())
    # dequantized spike is within one grid step
    deq = orc.dequant_v(codes, scales)
    assert abs(deq[0, 40, 9] - vf[0, 40, 9]) <= 0.5 * 2.0 ** (int(scales[0, 9, 1]) - 127) * 2 + 1e-12


def test_ceil_q_rule_defines_the_qmax_sweep(orc):
    """Section 5.5.1 sweeps Q_max over [6.00, 8.00] in steps of 0.05: e = ceil(log2(M / q))
    is the smallest exponent that brings the block maximum to at most q, so the
    normalized maximum lies in (q/2, q]; exact boundaries M = q * 2^k give e = k and one
    ulp above gives k + 1. q = 7.25 is UOS and q = 6 is TFS."""
    rng = np.random.default_rng(11)
    M = np.exp2(rng.uniform(-40, 40, 100000))
    for q in np.round(np.arange(6.0, 8.0001, 0.05), 2):
        e = np.array([orc.scale_exponent(m, orc.CEIL_Q, q) for m in M[:4000]])
        x = M[:4000] / np.exp2(e)
        assert np.all(x <= q) and np.all(x > q / 2), q
        for k in (-20, -3, 0, 5, 30):
            b = q * 2.0 ** k
            assert orc.scale_exponent(b, orc.CEIL_Q, q) == k
            assert orc.scale_exponent(np.nextafter(b, np.inf), orc.CEIL_Q, q) == k + 1
    for m in M[:20000:7]:
        assert orc.scale_exponent(m, orc.CEIL_Q, 7.25) == orc.scale_exponent(m, orc.UOS)
        assert orc.scale_exponent(m, orc.CEIL_Q, 6.0) == orc.scale_exponent(m, orc.TFS)


def test_rotate_then_quantize_composition(orc):
    """Algorithm 2's Q/K steps in order: rotate each token with R_H (the pinned
    binary32 butterfly, orc.hadamard_fp32), then Algorithm 1 on each 32-channel
    block of the rotated row. orc.rotate_quantize_qk(rotate=True) must equal that
    composition code for code and scale for scale, assembled here from the
    separately pinned pieces (scale exponent, E2M1 code)."""
    rng = np.random.default_rng(21)
    x = rng.standard_normal((24, 128)) * np.exp2(rng.integers(-6, 6, (24, 1)))
    x[3] = 0.0                                  # all-zero row: every block sigma = 1
    x[4, :] = 0.0; x[4, 17] = 5.0               # one-hot rows rotate to +-5/sqrt(128)
    bits = _bf16_bits(x)
    codes, scales = orc.rotate_quantize_qk(bits, rotate=True)
    y = orc.hadamard_fp32(bits).astype(np.float64)
    for r in range(x.shape[0]):
        for b in range(4):
            blk = y[r, 32 * b: 32 * b + 32]
            M = np.abs(blk).max()
            if M == 0:
                assert scales[r, b] == 127 and np.all(codes[r, 32 * b: 32 * b + 32] == 0)
                continue
            e = orc.scale_exponent(M, orc.UOS)
            assert scales[r, b] == e + 127
            ref = orc.e2m1_code(blk / 2.0 ** e)
            assert np.array_equal(codes[r, 32 * b: 32 * b + 32], ref)
    # without the rotation the same rows give different codes (the branch is live)
    c0, _ = orc.rotate_quantize_qk(bits, rotate=False)
    assert not np.array_equal(c0, codes)


def test_rotated_basis_vectors_exact(orc):
    """Integer inputs whose rotation is exact: x = e_j rotates to the j-th row of
    H_128 times fl32(2^-3.5), entries +-0.0883883..., so every block maximum is
    that value, e = ceil(log2(0.08839 / 7.25)) = -6 (scale byte 121), and every
    element is +-5.657 in scale units, saturating to code 7 (6.0) with the sign
    of (-1)^popcount(i & j) (the Sylvester entry, section 4.3 rotation)."""
    for j in (0, 1, 5, 64, 127):
        x = np.zeros((1, 128)); x[0, j] = 1.0
        codes, scales = orc.rotate_quantize_qk(_bf16_bits(x), rotate=True)
        assert np.all(scales == 121)
        signs = np.array([bin(i & j).count("1") & 1 for i in range(128)])
        assert np.array_equal(codes[0], (7 | (signs << 3)).astype(np.uint8))
