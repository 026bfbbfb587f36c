"""Pins of the oracle's row-sum diagnostic ("MXAttention" section 5.5.2, Fig. 7 B):
a materialized P quantized in 32-key blocks, its row-sum error split into
zeroing, saturation, downward and upward rounding (reading D1).

* the four parts sum to the whole error, sum Q(P) - sum P, on random rows;
* a hand-worked 32-element block under UOS and under the OCP floor rule
  (the OCP scale saturates the block maximum 0.95 at 6 * 2^-3, UOS maps it
  to 4 * 2^-2 exactly as section 4 argues);
* closed forms of uniform rows: 1/128 is a power of two and quantizes
  exactly; 1/96 normalizes to 16/3 and rounds up to 6 in every block;
* the quantization itself is the oracle's pinned block quantizer
  (rotate_quantize_qk without rotation) on the same values.
"""
import numpy as np
import torch


def test_parts_sum_to_the_error(orc):
    rng = np.random.default_rng(31)
    for rule in (orc.UOS, orc.OCP, orc.TFS):
        P = np.exp(rng.standard_normal((40, 300)) * 3.0)
        P[:, 250:] = 0.0
        P /= P.sum(1, keepdims=True)
        r = orc.rowsum_parts(P, rule)
        assert np.allclose(r[:, 0] - P.sum(1), r[:, 1:].sum(1), rtol=0, atol=1e-13)
        assert np.all(r[:, 1] <= 0) and np.all(r[:, 2] <= 0) and np.all(r[:, 3] <= 0) and np.all(r[:, 4] >= 0)


def test_hand_worked_block_uos_and_ocp(orc):
    P = np.zeros((1, 32))
    P[0, :5] = [0.95, 0.2, 0.04, 0.011, 0.001]
    # UOS: e = ceil(log2(0.95 / 7.25)) = -2, scale 1/4: 3.8 -> 4, 0.8 -> 1, 0.16, 0.044, 0.004 -> 0
    u = orc.rowsum_parts(P, orc.UOS)[0]
    assert np.allclose(u, [1.25, -0.052, 0.0, 0.0, 0.10], rtol=0, atol=1e-15)
    # OCP: e = floor(log2 0.95) - 2 = -3, scale 1/8: 7.6 -> 6 (saturation), 1.6 -> 1.5, 0.32 -> 0.5, 0.088, 0.008 -> 0
    o = orc.rowsum_parts(P, orc.OCP)[0]
    assert np.allclose(o, [1.0, -0.012, -0.2, -0.0125, 0.0225], rtol=0, atol=1e-15)


def test_uniform_rows_closed_forms(orc):
    r = orc.rowsum_parts(np.full((1, 128), 1.0 / 128), orc.UOS)[0]
    assert np.array_equal(r, [1.0, 0.0, 0.0, 0.0, 0.0])
    # 1/96: e = ceil(log2(1/96 / 7.25)) = -9, normalized 512/96 = 16/3 in (5, 6] -> 6
    r = orc.rowsum_parts(np.full((1, 96), 1.0 / 96), orc.UOS)[0]
    assert np.allclose(r, [1.125, 0.0, 0.0, 0.0, 0.125], rtol=0, atol=1e-15)


def test_quantization_is_the_block_quantizer(orc):
    """The diagnostic's Q(P) is the oracle's block quantizer: on bf16-exact P, the
    dequantized Q/K quantizer output (no rotation) sums to the same row sums."""
    rng = np.random.default_rng(32)
    P = np.exp(rng.standard_normal((6, 128)) * 2.0)
    P /= P.sum(1, keepdims=True)
    bits = torch.from_numpy(P.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    Pb = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    codes, scales = orc.rotate_quantize_qk(bits, rotate=False)
    deq = orc.dequant_qk(codes, scales)
    r = orc.rowsum_parts(Pb, orc.UOS)
    assert np.allclose(r[:, 0], deq.sum(1), rtol=0, atol=1e-15)
