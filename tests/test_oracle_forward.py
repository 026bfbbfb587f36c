"""Pins of the oracle's online-softmax forward ("MXAttention" Algorithm 2).

* quantization off, the recurrence equals softmax attention, Eq. (1)-(8)
* one key tile: O = P^ V / sum(P^) with P^ = Q*(exp(S - rowmax)), Eq. (44)-(45)
* Lemma 2 / Eq. (99)-(105): l and O equal the beta-weighted sums of the
  per-tile P^, recomputed here from prefix maxima without the recurrence
* Proposition 1, Eq. (51): induced PNQ weights sum to one
* Appendix J, Eq. (118): l >= 1
* V == 1 gives O == 1 under PNQ; under the direct placement of Eq. (16)-(17)
  it does not (Eq. (110), negative control)
* causal: perturbing tokens > i leaves row i bit-identical (MatX note); without
  the diagonal-block rule a perturbation inside the query's own V block leaks
"""
import numpy as np
import pytest
import torch

D = 128


def _softmax_attn(q, K, V, causal_tok=None):
    S = q @ K.T / np.sqrt(D)
    if causal_tok is not None:
        mask = np.arange(K.shape[0])[None, :] > np.asarray(causal_tok)[:, None]
        S = np.where(mask, -np.inf, S)
    S = S - S.max(axis=1, keepdims=True)
    P = np.exp(S)
    return (P / P.sum(axis=1, keepdims=True)) @ V


def _quant_block(orc, x):
    """Algorithm 1 on a 1-D block using the oracle's pinned scalar pieces."""
    M = np.abs(x).max()
    if M == 0:
        return np.zeros_like(x)
    e = orc.scale_exponent(M, orc.UOS)
    codes = orc.e2m1_code(x / 2.0 ** e)
    return np.array([orc.e2m1_value(int(c)) for c in codes]) * 2.0 ** e


@pytest.mark.parametrize("bc", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_unquantized_recurrence_equals_softmax(orc, bc, causal):
    rng = np.random.default_rng(10 + bc)
    N = 300
    K, V = rng.standard_normal((N, D)), rng.standard_normal((N, D))
    tok = np.array([0, 5, 31, 32, 127, 128, 200, 299])
    q = rng.standard_normal((len(tok), D)) * 2
    res = orc.online_softmax(q, tok, K, V, causal=causal, quant_p=False, bc=bc)
    ref = _softmax_attn(q, K, V, tok if causal else None)
    assert np.max(np.abs(res["out"] - ref)) < 1e-12


def test_one_tile_closed_form(orc):
    rng = np.random.default_rng(11)
    N = 100
    K, V = rng.standard_normal((N, D)), rng.standard_normal((N, D))
    q = rng.standard_normal((6, D)) * 3
    res = orc.online_softmax(q, np.zeros(6, dtype=np.int64), K, V, quant_p=True)
    S = q @ K.T / np.sqrt(D)
    for r in range(6):
        Pt = np.concatenate([np.exp(S[r] - S[r].max()), np.zeros(128 - N)])
        Ph = np.concatenate([_quant_block(orc, Pt[b:b + 32]) for b in range(0, 128, 32)])[:N]
        ref = Ph @ V / Ph.sum()
        assert np.allclose(res["out"][r], ref, rtol=0, atol=1e-13)
        assert abs(res["ell"][r] - Ph.sum()) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_lemma2_prop1_from_prefix_maxima(orc, causal):
    rng = np.random.default_rng(12)
    N, bc = 700, 128
    K, V = rng.standard_normal((N, D)), rng.standard_normal((N, D))
    # make the running max move across tiles: the row maximum sits in a late tile
    tok = np.array([650, 699, 300, 129])
    q = rng.standard_normal((len(tok), D)) * 2
    K[600] = q[0] * 0.5
    res = orc.online_softmax(q, tok, K, V, causal=causal, quant_p=True, want_phat=True)
    S = q @ K.T / np.sqrt(D)
    ntiles = (N + bc - 1) // bc
    for r, i in enumerate(tok):
        nt = i // bc + 1 if causal else ntiles
        valid = np.arange(ntiles * bc) < N
        if causal:
            valid &= np.arange(ntiles * bc) <= i
        Srow = np.full(ntiles * bc, -np.inf)
        Srow[:N] = S[r]
        Srow[~valid] = -np.inf
        m_prefix = np.maximum.accumulate([Srow[j * bc:(j + 1) * bc].max() for j in range(nt)])
        phat_ref = np.zeros(ntiles * bc)
        for j in range(nt):
            Pt = np.where(valid[j * bc:(j + 1) * bc], np.exp(Srow[j * bc:(j + 1) * bc] - m_prefix[j]), 0.0)
            phat_ref[j * bc:(j + 1) * bc] = np.concatenate([_quant_block(orc, Pt[b:b + 32]) for b in range(0, bc, 32)])
        assert np.array_equal(res["phat"][r], phat_ref)
        assert np.allclose(res["mhist"][r, :nt], m_prefix, rtol=0, atol=1e-12)
        beta = np.exp(m_prefix - m_prefix[-1])                           # Eq. (99)
        eff = np.concatenate([beta[j] * phat_ref[j * bc:(j + 1) * bc] for j in range(nt)])  # Eq. (103)-(104)
        ell = eff.sum()                                                   # Eq. (102)
        assert abs(res["ell"][r] - ell) <= 1e-13 * ell
        Vp = np.zeros((ntiles * bc, D))
        Vp[:N] = V
        assert np.allclose(res["out"][r] * res["ell"][r], eff[:nt * bc] @ Vp[:nt * bc], rtol=1e-12, atol=1e-12)
        P_pnq = eff / res["ell"][r]                                       # Eq. (50)
        assert abs(P_pnq.sum() - 1.0) < 1e-14                             # Eq. (51)
        assert res["ell"][r] >= 1.0                                       # Eq. (118)


def test_ell_at_least_one_many_rows(orc):
    rng = np.random.default_rng(13)
    for scale in [0.1, 1.0, 10.0, 100.0]:
        N = 400
        K, V = rng.standard_normal((N, D)), rng.standard_normal((N, D))
        q = rng.standard_normal((16, D)) * scale
        res = orc.online_softmax(q, np.zeros(16, dtype=np.int64), K, V, quant_p=True)
        assert np.all(res["ell"] >= 1.0)


def test_v_ones_pnq_exact_and_direct_not(orc):
    rng = np.random.default_rng(14)
    N = 512
    K = rng.standard_normal((N, D))
    V = np.ones((N, D))
    q = rng.standard_normal((32, D)) * 0.5  # diffuse rows: many P~ entries are rounded
    tok = np.zeros(32, dtype=np.int64)
    pnq = orc.online_softmax(q, tok, K, V, quant_p=True, placement=orc.PNQ)
    assert np.all(pnq["out"] == 1.0)
    direct = orc.online_softmax(q, tok, K, V, quant_p=True, placement=orc.DIRECT)
    rowsum = direct["out"][:, 0]
    assert np.max(np.abs(rowsum - 1.0)) > 1e-3   # Eq. (110): row sums differ from one


def _bits(x):
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _pipeline(orc, q16, k16, v16, rows, vraw=None, causal=1):
    qc, qs = orc.rotate_quantize_qk(q16)
    kc, ks = orc.rotate_quantize_qk(k16)
    vc, vs = orc.quantize_v(v16)
    return orc.forward(qc, qs, kc, ks, vc, vs, rows, vraw_u16=v16 if vraw is None else vraw, causal=causal)


@pytest.mark.parametrize("mode", [1, 2])
def test_causal_no_future_leakage(orc, mode):
    rng = np.random.default_rng(15)
    N = 300
    q = rng.standard_normal((1, N, D)) * 2
    k = rng.standard_normal((1, N, D)) * 2
    v = rng.standard_normal((1, N, D))
    rows = np.array([[0, i] for i in [0, 3, 31, 33, 100, 127, 128, 170, 255, 299]])
    base = _pipeline(orc, _bits(q), _bits(k), _bits(v), rows, causal=mode)["out"]
    for r, (_, i) in enumerate(rows):
        q2, k2, v2 = q.copy(), k.copy(), v.copy()
        fut = slice(i + 1, N)
        q2[0, fut] = rng.standard_normal((N - i - 1, D)) * 50
        k2[0, fut] = rng.standard_normal((N - i - 1, D)) * 50
        v2[0, fut] = rng.standard_normal((N - i - 1, D)) * 50
        pert = _pipeline(orc, _bits(q2), _bits(k2), _bits(v2), rows[r:r + 1], causal=mode)["out"]
        assert np.array_equal(pert[0], base[r]), f"row {i} changed"


def test_causal_leak_without_diagonal_rule(orc):
    """Negative control: feeding the quantized V on the diagonal block lets a
    later token of the same 32-token V block reach row i."""
    rng = np.random.default_rng(16)
    N = 64
    q = rng.standard_normal((1, N, D))
    k = rng.standard_normal((1, N, D))
    v = rng.standard_normal((1, N, D))
    i = 40
    rows = np.array([[0, i]])
    vc, vs = orc.quantize_v(_bits(v))
    deq = orc.dequant_v(vc, vs)

    def run(vv):
        vc2, vs2 = orc.quantize_v(_bits(vv))
        deq2 = orc.dequant_v(vc2, vs2)
        qc, qs = orc.rotate_quantize_qk(_bits(q))
        kc, ks = orc.rotate_quantize_qk(_bits(k))
        return orc.forward(qc, qs, kc, ks, vc2, vs2, rows, vraw_u16=_bits(deq2), causal=True)["out"]

    v2 = v.copy()
    v2[0, 45, :] = 1000.0  # token 45 > 40, same 32-token block [32, 64)
    assert not np.array_equal(run(v), run(v2))


def test_causal_prefix_requantization_reduces_to_the_block_quantizer(orc):
    """causal = 2 re-quantizes the query's own 32-token V block over tokens b0..i.
    For the last token of a block (and the last token of a ragged final block)
    that prefix is the whole block, so the row equals the plain V^ path (the
    leaky one) bit for bit; for an earlier row it differs."""
    rng = np.random.default_rng(18)
    N = 200  # last block 192..199 is ragged
    Q, K, V = (rng.standard_normal((1, N, D)) for _ in range(3))
    q16, k16, v16 = _bits(Q), _bits(K), _bits(V)
    qc, qs = orc.rotate_quantize_qk(q16)
    kc, ks = orc.rotate_quantize_qk(k16)
    vc, vs = orc.quantize_v(v16)
    Qd, Kd, Vd = orc.dequant_qk(qc, qs)[0], orc.dequant_qk(kc, ks)[0], orc.dequant_v(vc, vs)[0]
    Vraw = v16.astype(np.uint32)[0]
    Vraw = (Vraw << 16).view(np.float32).astype(np.float64)
    for i in (31, 63, 127, 199):
        pre = orc.online_softmax(Qd[i][None], [i], Kd, Vd, Vraw, causal=2)["out"]
        leaky = orc.online_softmax(Qd[i][None], [i], Kd, Vd, Vd, causal=1)["out"]
        assert np.array_equal(pre, leaky), i
    i = 70
    pre = orc.online_softmax(Qd[i][None], [i], Kd, Vd, Vraw, causal=2)["out"]
    leaky = orc.online_softmax(Qd[i][None], [i], Kd, Vd, Vd, causal=1)["out"]
    assert not np.array_equal(pre, leaky)


def test_forward_on_codes_matches_real_valued_core(orc):
    rng = np.random.default_rng(17)
    BH, N = 2, 260
    q16, k16, v16 = (_bits(rng.standard_normal((BH, N, D))) for _ in range(3))
    qc, qs = orc.rotate_quantize_qk(q16)
    kc, ks = orc.rotate_quantize_qk(k16)
    vc, vs = orc.quantize_v(v16)
    rows = np.array([[1, 0], [1, 259], [0, 17]])
    res = orc.forward(qc, qs, kc, ks, vc, vs, rows)
    Q, Kd, Vd = orc.dequant_qk(qc, qs), orc.dequant_qk(kc, ks), orc.dequant_v(vc, vs)
    for r, (bh, i) in enumerate(rows):
        ref = orc.online_softmax(Q[bh, i][None], [i], Kd[bh], Vd[bh], quant_p=True)
        assert np.array_equal(res["out"][r], ref["out"][0])


# ------------------------------------------------------------ Eq. (1) oracle
def _bf16(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _bf16_vals(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 33, 129, 300])
def test_sdpa_is_softmax_attention(orc, causal, N):
    """orc.sdpa is Eq. (1) of section 2: softmax(QK^T / sqrt(d)) V on the bf16
    inputs, keys j <= i only when causal. Compared with a numpy evaluation of
    the same formula on every row of a ragged N, causal and not."""
    rng = np.random.default_rng(100 + N)
    BH = 2
    q = _bf16(rng.standard_normal((BH, N, D)) * 2)
    k = _bf16(rng.standard_normal((BH, N, D)))
    v = _bf16(rng.standard_normal((BH, N, D)))
    rows = np.array([[b, i] for b in range(BH) for i in range(N)], dtype=np.int64)
    got = orc.sdpa(q, k, v, rows, causal=causal)
    for b in range(BH):
        Q, K, V = _bf16_vals(q[b]), _bf16_vals(k[b]), _bf16_vals(v[b])
        ref = _softmax_attn(Q, K, V, np.arange(N) if causal else None)
        assert np.max(np.abs(got[b * N:(b + 1) * N] - ref)) < 1e-12


def test_sdpa_closed_forms(orc):
    """Two closed forms of Eq. (1) that fail on a wrong 1/sqrt(d) or a shifted
    causal mask: (i) equal keys give uniform weights, so row i of a causal
    pass is the mean of V rows 0..i and of a full pass the mean of all rows;
    (ii) with two keys whose scores differ by exactly sqrt(d) * ln 2 the
    softmax weights are 2/3 and 1/3."""
    N = 40
    rng = np.random.default_rng(7)
    q = _bf16(rng.standard_normal((1, N, D)))
    k = _bf16(np.tile(rng.standard_normal((1, 1, D)), (1, N, 1)))
    v = _bf16(rng.integers(-8, 9, (1, N, D)).astype(np.float32))
    rows = np.array([[0, i] for i in range(N)], dtype=np.int64)
    V = _bf16_vals(v[0])
    causal = orc.sdpa(q, k, v, rows, causal=True)
    full = orc.sdpa(q, k, v, rows, causal=False)
    for i in range(N):
        assert np.allclose(causal[i], V[: i + 1].mean(axis=0), rtol=0, atol=1e-12)
        assert np.allclose(full[i], V.mean(axis=0), rtol=0, atol=1e-12)
    # q . k0 - q . k1 = sqrt(128) ln 2 needs non-bf16 values; scale instead: q = e_0,
    # k0 = a e_0, k1 = 0 with a = sqrt(128) ln 2 rounded to bf16, weights e^s / (e^s + 1)
    a = float(_bf16_vals(_bf16(np.array([np.sqrt(D) * np.log(2.0)])))[0])
    qq = np.zeros((1, 2, D)); qq[0, :, 0] = 1.0
    kk = np.zeros((1, 2, D)); kk[0, 0, 0] = a
    vv = np.zeros((1, 2, D)); vv[0, 0, :] = 3.0; vv[0, 1, :] = -6.0
    out = orc.sdpa(_bf16(qq), _bf16(kk), _bf16(vv), np.array([[0, 1]]), causal=False)
    w0 = np.exp(a / np.sqrt(D)) / (np.exp(a / np.sqrt(D)) + 1.0)
    assert abs(w0 - 2.0 / 3.0) < 1e-2
    assert np.allclose(out[0], 3.0 * w0 - 6.0 * (1.0 - w0), rtol=0, atol=1e-12)
    # row 0 of a causal pass sees only key 0
    out0 = orc.sdpa(_bf16(qq), _bf16(kk), _bf16(vv), np.array([[0, 0]]), causal=True)
    assert np.allclose(out0[0], 3.0, rtol=0, atol=0)


def _vhat(orc, vc, vs):
    """Dequantized V^ [BH, N, 128] from the oracle's codes [BH, N, 128] and E8M0 scales [BH, 128, nblk]."""
    e2 = np.array([orc.e2m1_value(c) for c in range(16)])
    N = vc.shape[1]
    sc = np.exp2(vs.astype(np.float64) - 127.0)  # [BH, 128, nblk]
    blk = np.arange(N) // 32
    return e2[vc] * np.transpose(sc[:, :, blk], (0, 2, 1))


@pytest.mark.parametrize("causal", [0, 1])
def test_uniform_scores_give_block_means(orc, causal):
    """Degenerate case: Q = 0 makes every score 0, so m = 0 and P~ = 1 in every
    block; the UOS scale of a block whose maximum is 1 is 2^-2 and 1 / 2^-2 = 4
    is an E2M1 grid point, so P^ = 1 exactly (Eq. 44) and l counts the visible
    keys (Eq. 47). O is then the plain mean of the visible V^ rows (Eq. 48);
    in causal mode the query's own 32-token block contributes its bf16 V rows
    instead (the diagonal-block reading)."""
    rng = np.random.default_rng(31)
    N = 300
    q = np.zeros((1, N, D))
    k = rng.standard_normal((1, N, D)) * 3
    v = rng.standard_normal((1, N, D))
    q16, k16, v16 = _bits(q), _bits(k), _bits(v)
    rows = np.array([[0, i] for i in range(N)])
    out = _pipeline(orc, q16, k16, v16, rows, causal=causal)
    vc, vs = orc.quantize_v(v16)
    vhat = _vhat(orc, vc, vs)[0]
    vraw = _bf16_vals(v16)[0]
    for i in range(N):
        if not causal:
            want, ell = vhat.mean(axis=0), N
        else:
            d0 = 32 * (i // 32)
            want = (vhat[:d0].sum(axis=0) + vraw[d0:i + 1].sum(axis=0)) / (i + 1)
            ell = i + 1
        assert np.allclose(out["out"][i], want, rtol=0, atol=1e-12 * np.abs(vraw).max())
        assert out["ell"][i] == ell
