"""Pins of the oracle's NVFP4 comparison format (no GPU).

The pages fix what NVFP4 is ("MXAttention" section 1: E2M1 values in
16-element blocks, an E4M3 block scale and a tensor-level scale) and what the
NVFP4 baseline does (section 5.2: Q, K, V and P~ quantized for the two
products, no smoothing, no softmax-path scaling). The oracle's readings N1-N6
fill in the rest. These tests pin it against:
  * torch's float8_e4m3fn conversion (a library routine) for the E4M3 grid
    and its round-to-nearest-even below the saturation point;
  * properties the format forces: the block maximum maps to the E2M1 maximum
    6, the tensor maximum's block takes the largest scale 448, representable
    inputs round-trip exactly, all-zero input gives zero codes and scales;
  * the V blocking (tokens) against the Q/K blocking (channels) by transpose;
  * forward identities: V == 1 gives O == 1 under PNQ and not under direct
    placement, the row maximum's P^ closed form, plain softmax attention when
    P~ is not quantized, and no future leakage in causal mode.
"""
import numpy as np
import pytest
import torch


def _bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def _bf16_vals(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)


def test_e4m3_decode_matches_torch(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for c in range(127):
        assert orc.e4m3_value(c) == ref[c], c
    assert orc.e4m3_value(126) == 448.0 and orc.e4m3_value(1) == 2.0 ** -9 and orc.e4m3_value(0x38) == 1.0


def test_e4m3_rounding_matches_torch_below_saturation(orc):
    vals = np.array([orc.e4m3_value(c) for c in range(127)])
    mids = (vals[:-1] + vals[1:]) / 2
    pts = [np.float32(0.0)]
    for m in mids:
        m32 = np.float32(m)
        pts += [m32, np.nextafter(m32, np.float32(0)), np.nextafter(m32, np.float32(np.inf))]
    pts += list(vals.astype(np.float32))
    rng = np.random.default_rng(3)
    pts += list((rng.random(3000) * 463.0).astype(np.float32))
    pts += list(np.exp2(rng.uniform(-14, 8.8, 3000)).astype(np.float32))
    pts = np.array([p for p in pts if p < 464.0], dtype=np.float32)
    ref = torch.from_numpy(pts).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_code(float(p)) for p in pts])
    assert np.array_equal(got, ref)
    # N1: at or above 448 saturate to the largest finite value
    for v in (448.0, 463.9, 464.0, 479.0, 480.0, 1e6, float("inf")):
        assert orc.e4m3_code(v) == 126


def _tensor(seed, shape, spread=4.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape) * np.exp2(rng.uniform(-spread, spread, shape[:-1] + (1,)))
    return _bf16_bits(x)


def test_nvfp4_block_max_maps_to_six_and_amax_block_to_448(orc):
    xb = _tensor(1, (2, 300, 128))
    codes, scales, et = orc.nvfp4_quantize_qk(xb)
    x = _bf16_vals(xb)
    amax = np.abs(x).max()
    assert np.float32(et) == np.float32(2688.0) / np.float32(amax)
    xa = np.abs(x).reshape(2, 300, 8, 16)
    cm = (codes & 7).reshape(2, 300, 8, 16)
    arg = xa.argmax(-1)
    top = np.take_along_axis(cm, arg[..., None], -1)[..., 0]
    normal = scales >= 8           # E4M3 normal scales: at most 1/16 relative rounding
    assert normal.sum() > 0.9 * scales.size
    assert np.all(top[normal] == 7), "block maximum must take the E2M1 maximum 6"
    # the block holding the tensor maximum has the largest scale
    i = np.unravel_index(np.abs(x).argmax(), x.shape)
    assert scales[i[0], i[1], i[2] // 16] == 126


def test_nvfp4_representable_input_round_trips(orc):
    rng = np.random.default_rng(7)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    k = 5
    et = 2.0 ** k                  # amax = 2688 / 2^k makes e_t a power of two
    rows = 64
    g = grid[rng.integers(0, 8, (rows, 8, 16))] * rng.choice([-1, 1], (rows, 8, 16))
    g[:, :, 0] = 6.0               # every block's maximum is 6 S
    sc = rng.integers(40, 127, (rows, 8))
    sc[0, 0] = 126                 # one block at S = 448 holds the tensor maximum 2688 / e_t
    S = np.array([orc.e4m3_value(int(c)) for c in sc.reshape(-1)]).reshape(rows, 8, 1)
    x = (g * S / et).reshape(rows, 128)
    xb = _bf16_bits(x)
    assert np.array_equal(_bf16_vals(xb), x)   # exactly representable
    codes, scales, e_t = orc.nvfp4_quantize_qk(xb)
    assert e_t == et
    assert np.array_equal(scales, sc)
    deq = orc.nvfp4_dequant_qk(codes, scales, e_t)
    assert np.array_equal(deq, x)


def test_nvfp4_all_zero(orc):
    z = np.zeros((1, 40, 128), dtype=np.uint16)
    c, s, et = orc.nvfp4_quantize_qk(z)
    assert et == 1.0 and not c.any() and not s.any()
    c, s, et = orc.nvfp4_quantize_v(z)
    assert et == 1.0 and not c.any() and not s.any()


def test_nvfp4_v_blocks_are_token_blocks(orc):
    """V with N = 128 tokens equals the Q/K quantizer applied to V transposed (channel rows of 128 tokens)."""
    vb = _tensor(11, (3, 128, 128), spread=2.0)
    vc, vs, et = orc.nvfp4_quantize_v(vb)
    tc, ts, et2 = orc.nvfp4_quantize_qk(np.ascontiguousarray(np.transpose(vb, (0, 2, 1))))
    assert et == et2
    assert np.array_equal(vc, np.transpose(tc, (0, 2, 1)))
    assert np.array_equal(vs, ts)


def _fwd_inputs(orc, seed, BH, N, v_ones=False):
    rng = np.random.default_rng(seed)
    q = _bf16_bits(rng.standard_normal((BH, N, 128)) * 2)
    k = _bf16_bits(rng.standard_normal((BH, N, 128)) * 2)
    v = _bf16_bits(np.ones((BH, N, 128)) if v_ones else rng.standard_normal((BH, N, 128)))
    qc, qs, qe = orc.nvfp4_quantize_qk(q)
    kc, ks, ke = orc.nvfp4_quantize_qk(k)
    vc, vs, ve = orc.nvfp4_quantize_v(v)
    return (q, k, v), (qc, qs, qe, kc, ks, ke, vc, vs, ve)


def test_nvfp4_forward_v_ones(orc):
    (q, k, v), ops = _fwd_inputs(orc, 2, 1, 300, v_ones=True)
    rows = np.array([[0, i] for i in range(0, 300, 7)])
    pnq = orc.forward_nvfp4(*ops, rows, placement=orc.PNQ)
    assert np.all(pnq["out"] == 1.0)
    direct = orc.forward_nvfp4(*ops, rows, placement=orc.DIRECT)
    assert np.abs(direct["out"] - 1.0).max() > 1e-3
    # causal, PNQ: still exactly 1 (the diagonal block's bf16 V is 1 too)
    c = orc.forward_nvfp4(*ops, rows, vraw_u16=v, causal=True, placement=orc.PNQ)
    assert np.all(c["out"] == 1.0)


def test_nvfp4_row_max_phat_closed_form(orc):
    """The row-maximum key has P~ = 1: scale E4M3(fl32(1/6)) = 0.171875, code 6 -> P^ = 1.03125."""
    _, ops = _fwd_inputs(orc, 4, 1, 128)
    rows = np.array([[0, i] for i in range(0, 128, 5)])
    r = orc.forward_nvfp4(*ops, rows, want_phat=True)
    assert orc.e4m3_value(orc.e4m3_code(float(np.float32(1 / 6)))) == 0.171875
    assert np.all(r["phat"].max(axis=1) == 1.03125)


def test_nvfp4_forward_without_p_quantization_is_softmax_attention(orc):
    (q, k, v), ops = _fwd_inputs(orc, 5, 2, 200)
    qc, qs, qe, kc, ks, ke, vc, vs, ve = ops
    Q = orc.nvfp4_dequant_qk(qc, qs, qe)
    K = orc.nvfp4_dequant_qk(kc, ks, ke)
    V = orc.nvfp4_dequant_v(vc, vs, ve)
    rows = np.array([[b, i] for b in range(2) for i in (0, 1, 99, 127, 128, 199)])
    r = orc.forward_nvfp4(*ops, rows, quant_p=False, placement=orc.DIRECT)
    for t, (b, i) in enumerate(rows):
        s = K[b] @ Q[b, i] / np.sqrt(128)
        p = np.exp(s - s.max())
        ref = p @ V[b] / p.sum()
        assert np.abs(r["out"][t] - ref).max() <= 1e-12 * np.abs(ref).max()


def test_nvfp4_causal_no_future_leakage(orc):
    """Perturbing every token after i leaves row i bit-identical. The tensor-level scale is a function of the
    whole tensor (a sequence-global statistic), so the test holds each tensor's maximum at token 0; the block
    quantizers and the causal loop must not leak anything else."""
    (q, k, v), _ = _fwd_inputs(orc, 6, 1, 160)
    for t in (q, k, v):
        t[0, 0, 0] = _bf16_bits(np.array([16.0 * np.abs(_bf16_vals(t)).max()]))[0]
    rng = np.random.default_rng(9)

    def run(q, k, v, rows):
        qc, qs, qe = orc.nvfp4_quantize_qk(q)
        kc, ks, ke = orc.nvfp4_quantize_qk(k)
        vc, vs, ve = orc.nvfp4_quantize_v(v)
        return orc.forward_nvfp4(qc, qs, qe, kc, ks, ke, vc, vs, ve, rows, vraw_u16=v, causal=True)["out"]

    for i in (0, 7, 15, 16, 40, 130):
        rows = np.array([[0, i]])
        base = run(q, k, v, rows)
        q2, k2, v2 = q.copy(), k.copy(), v.copy()
        for t in (q2, k2, v2):
            t[0, i + 1:] = _bf16_bits(rng.standard_normal((160 - i - 1, 128)) * 3.0)
        assert np.array_equal(run(q2, k2, v2, rows), base), i


def test_nvfp4_causal_diagonal_is_the_own_16_token_block(orc):
    """Causal, P~ not quantized: softmax attention over keys <= i where the keys of the query's own 16-token
    block use the bf16 V rows and every other key uses V^ (reading N5). Rows with i % 32 >= 16 tell a 16-token
    diagonal block from a 32-token one."""
    (q, k, v), ops = _fwd_inputs(orc, 8, 1, 200)
    qc, qs, qe, kc, ks, ke, vc, vs, ve = ops
    Q = orc.nvfp4_dequant_qk(qc, qs, qe)[0]
    K = orc.nvfp4_dequant_qk(kc, ks, ke)[0]
    V = orc.nvfp4_dequant_v(vc, vs, ve)[0]
    Vb = _bf16_vals(v)[0]
    tok = [3, 16, 20, 31, 47, 50, 63, 127, 130, 150, 199]
    rows = np.array([[0, i] for i in tok])
    r = orc.forward_nvfp4(*ops, rows, vraw_u16=v, causal=True, quant_p=False, placement=orc.DIRECT)
    for t, i in enumerate(tok):
        s = K[:i + 1] @ Q[i] / np.sqrt(128)
        p = np.exp(s - s.max())
        Vm = V[:i + 1].copy()
        b0 = (i // 16) * 16
        Vm[b0:i + 1] = Vb[b0:i + 1]
        ref = p @ Vm / p.sum()
        assert np.abs(r["out"][t] - ref).max() <= 1e-12 * np.abs(ref).max(), i


@pytest.mark.parametrize("causal,placement", [(False, 1), (True, 1), (False, 0), (True, 0)])
def test_nvfp4_replay_of_own_phat_is_identical(orc, causal, placement):
    """Replay mode: feeding the loop its own P^ reproduces its output bit for bit, so a kernel's dumped P^
    replayed through it isolates accumulation differences from P^ decisions."""
    (q, k, v), ops = _fwd_inputs(orc, 12, 1, 300)
    rows = np.array([[0, i] for i in range(0, 300, 3)])
    own = orc.forward_nvfp4(*ops, rows, vraw_u16=v, causal=causal, placement=placement, want_phat=True)
    rep = orc.forward_nvfp4(*ops, rows, vraw_u16=v, causal=causal, placement=placement, phat_in=own["phat"])
    assert np.array_equal(rep["out"], own["out"]) and np.array_equal(rep["ell"], own["ell"])
    # and a different P^ changes the output (the replay input is used)
    alt = own["phat"].copy()
    alt[:, 0] *= 0.5
    assert not np.array_equal(orc.forward_nvfp4(*ops, rows, vraw_u16=v, causal=causal, placement=placement,
                                                phat_in=alt)["out"], own["out"])
