"""Pins of the oracle's fixed Hadamard rotation ("MXAttention" section 4.3,
Algorithm 2 (section 4.3), rotation step; explainer page step 1 and glossary).

* the rotation matrix recovered from the oracle is +-2^-3.5 times a Sylvester
  Hadamard matrix: H H^T = 128 I exactly (integer check), H[i][j] = (-1)^popcount(i&j)
* on small-integer inputs the binary32 butterfly equals the exact product H x
* R_H is orthogonal, so the rotated full-precision Q K^T equals Q K^T
"""
import numpy as np
import torch


def _bf16_bits(x):
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _bits_to_f64(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _recover_matrix(orc):
    eye = _bf16_bits(np.eye(128))
    cols = orc.hadamard_fp32(eye)  # row j = R_H^T e_j ... i.e. e_j R_H
    return cols.astype(np.float64)


def test_hadamard_is_sylvester_and_orthogonal(orc):
    R = _recover_matrix(orc)
    c = np.float32(2.0 ** -3.5)
    assert np.all(np.abs(R) == np.float64(c))
    H = np.sign(R).astype(np.int64)
    assert np.array_equal(H @ H.T, 128 * np.eye(128, dtype=np.int64))
    i = np.arange(128)
    syl = np.array([[(-1) ** bin(a & b).count("1") for b in i] for a in i])
    assert np.array_equal(H, syl)


def test_butterfly_exact_on_integers(orc):
    rng = np.random.default_rng(5)
    x = rng.integers(-64, 65, size=(200, 128))
    y = orc.hadamard_fp32(_bf16_bits(x))
    i = np.arange(128)
    H = np.array([[(-1) ** bin(a & b).count("1") for b in i] for a in i], dtype=np.int64)
    z = x @ H  # exact
    expect = (z.astype(np.float32) * np.float32(2.0 ** -3.5)).astype(np.float32)
    assert np.array_equal(y, expect)


def test_rotation_preserves_dot_products(orc):
    rng = np.random.default_rng(6)
    q = _bf16_bits(rng.standard_normal((64, 128)) * 3)
    k = _bf16_bits(rng.standard_normal((64, 128)) * 3)
    R = _recover_matrix(orc)
    H = np.sign(R)
    Rexact = H / np.sqrt(128.0)
    qf, kf = _bits_to_f64(q), _bits_to_f64(k)
    # full precision: Q R (K R)^T == Q K^T
    assert np.allclose((qf @ Rexact) @ (kf @ Rexact).T, qf @ kf.T, rtol=0, atol=1e-10)
    # the binary32 rotation agrees to binary32 rounding
    qr, kr = orc.hadamard_fp32(q).astype(np.float64), orc.hadamard_fp32(k).astype(np.float64)
    scale = np.linalg.norm(qf, axis=1)[:, None] * np.linalg.norm(kf, axis=1)[None, :]
    assert np.max(np.abs(qr @ kr.T - qf @ kf.T) / scale) < 1e-6
