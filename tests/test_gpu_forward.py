"""GPU parity of the attention forward kernels (through the C ABI) against the oracle.

MXFP4 path ("MXAttention" Algorithm 2 with PNQ): the oracle quantizes the same
bf16 inputs on its own and runs the float64 recurrence with Bc = 128. Gates:
  * max |O_gpu - O_oracle| <= 2e-3 * RMS(O_oracle) over the compared rows;
  * fewer than 0.1 % of P^ entries differ (compared on the dumped P^ tiles);
  * causal: perturbing tokens > i leaves GPU row i bit-identical (MatX note);
  * V == 1 gives O == 1 (Proposition 1 through the kernel's own l).
BF16 path (Eqs. 1-8): within the bound set by bf16 rounding of P (see
test_bf16_forward_vs_exact_softmax). The bounded-wait failure path is
exercised through the test hook of the C ABI.
"""
import math

import numpy as np
import pytest
import torch

import _layouts as L
from mxfp4_precision_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_REL_RMS = 2e-3
MAX_FLIP_RATE = 1e-3


@pytest.fixture(scope="module")
def mx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mxfp4_precision_attention_gb300 as m

    m.load()
    return m


def _gpu_mx(mx, q, k, v, causal=False, dump=False):
    B, H, N, _ = q.shape
    qc, qs = mx.mxattn_rotate_quantize_qk(q)
    kc, ks = mx.mxattn_rotate_quantize_qk(k)
    vc, vs = mx.mxattn_quantize_v(v)
    if dump:
        out, pc, ps = mx.mxattn_forward_dump_phat(qc, qs, kc, ks, vc, vs, v, B, H, N, causal=causal)
        mx.mxattn_check()
        return out, pc, ps
    out = mx.mxattn_forward(qc, qs, kc, ks, vc, vs, v, B, H, N, causal=causal)
    mx.mxattn_check()
    return out


def _oracle(orc, q, k, v, rows, causal=False, heads=None, want_phat=False):
    """Oracle forward for rows [(bh, i)]; only the listed heads are copied and quantized."""
    B, H, N, _ = q.shape
    heads = sorted(set(int(r[0]) for r in rows)) if heads is None else list(heads)
    remap = {h: i for i, h in enumerate(heads)}
    idx = torch.tensor(heads, device=q.device)
    qb, kb, vb = (W.as_u16(t.reshape(B * H, N, 128).index_select(0, idx)) for t in (q, k, v))
    qc, qs = orc.rotate_quantize_qk(qb)
    kc, ks = orc.rotate_quantize_qk(kb)
    vc, vs = orc.quantize_v(vb)
    rr = np.array([[remap[int(b)], int(i)] for b, i in rows], dtype=np.int64)
    return orc.forward(qc, qs, kc, ks, vc, vs, rr, vraw_u16=vb, causal=causal, want_phat=want_phat)


def _gate(gpu_rows, ora_rows, what):
    err = np.abs(gpu_rows - ora_rows).max()
    rms = math.sqrt(np.mean(ora_rows ** 2))
    print(f"{what}: max|err| = {err:.3e}, RMS(oracle) = {rms:.3e}, ratio = {err / rms:.3e}")
    assert err <= TOL_REL_RMS * rms, f"{what}: max|err| {err:.3e} > {TOL_REL_RMS} * RMS {rms:.3e}"


def _flip_rate(orc, pc, ps, ora_phat, rows, N, causal):
    vals = np.array([orc.e2m1_value(c) for c in range(16)])
    pcn, psn = pc.cpu().numpy(), ps.cpu().numpy()
    gp = L.phat_values(pcn[rows[:, 0], rows[:, 1]], psn[rows[:, 0], rows[:, 1]], vals)
    keys = np.arange(gp.shape[1])[None, :]
    valid = np.broadcast_to(keys < N, gp.shape)
    if causal:
        valid = valid & (keys <= rows[:, 1:2])
    diff = (gp != ora_phat) & valid
    return diff.sum() / valid.sum(), diff.sum()


def _all_rows(BH, N):
    return np.array([[b, i] for b in range(BH) for i in range(N)], dtype=np.int64)


@pytest.mark.parametrize("case", ["tiny_outlier_512", "diffuse_1000", "causal_700"])
def test_forward_all_rows_and_phat(mx, orc, case):
    if case == "tiny_outlier_512":
        q, k, v = W.generate(W.WORKLOADS["tiny_outlier_512"], device="cuda")
        causal = False
    elif case == "diffuse_1000":
        q, k, v = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=2, N=1000)
        causal = False
    else:
        q, k, v = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=2, N=700, seed=9)
        causal = True
    B, H, N, _ = q.shape
    out, pc, ps = _gpu_mx(mx, q, k, v, causal=causal, dump=True)
    rows = _all_rows(B * H, N)
    ref = _oracle(orc, q, k, v, rows, causal=causal, want_phat=True)
    g = out.reshape(B * H, N, 128).cpu().numpy().astype(np.float64)[rows[:, 0], rows[:, 1]]
    rate, nflip = _flip_rate(orc, pc, ps, ref["phat"], rows, N, causal)
    print(f"{case}: P^ flip rate {rate:.2e} ({nflip} entries)")
    assert rate < MAX_FLIP_RATE
    _gate(g, ref["out"], case)


@pytest.mark.parametrize("direction", ["rising", "falling"])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_rising_maxima_rescale_every_tile(mx, orc, causal, direction):
    """Scores that grow along the keys (K_j = s_j * u + noise, Q_i = u + noise, s_j
    increasing): every key tile raises every row's running maximum, so each
    softmax warp rescales O and l in TMEM on every tile (Eqs. 3-5) and every
    P^ is taken relative to a new m. Falling scores are the opposite case: the
    maximum is set in the first tile and no later tile rescales. All rows and
    every P^ entry against the oracle; N = 900 (eight tiles, the last ragged)."""
    B, H, N = 1, 2, 900
    g = torch.Generator().manual_seed(53)
    u = torch.randn(B, H, 1, 128, generator=g)
    s = torch.linspace(0.0, 1.0, N).reshape(1, 1, N, 1)
    if direction == "falling":
        s = 1.0 - s
    q = (u + 0.1 * torch.randn(B, H, N, 128, generator=g)).to(torch.bfloat16).cuda()
    k = (s * u + 0.1 * torch.randn(B, H, N, 128, generator=g)).to(torch.bfloat16).cuda()
    v = torch.randn(B, H, N, 128, generator=g).to(torch.bfloat16).cuda()
    out, pc, ps = _gpu_mx(mx, q, k, v, causal=causal, dump=True)
    rows = _all_rows(B * H, N)
    ref = _oracle(orc, q, k, v, rows, causal=causal, want_phat=True)
    got = out.reshape(B * H, N, 128).cpu().numpy().astype(np.float64)[rows[:, 0], rows[:, 1]]
    rate, nflip = _flip_rate(orc, pc, ps, ref["phat"], rows, N, causal)
    print(f"{direction} maxima causal={causal}: P^ flip rate {rate:.2e} ({nflip} entries)")
    assert rate < MAX_FLIP_RATE
    _gate(got, ref["out"], f"{direction} maxima causal={causal}")


def test_forward_lognormal_sampled(mx, orc):
    w = W.WORKLOADS["lognormal_4096"]
    q, k, v = W.generate(w, device="cuda")
    rng = np.random.default_rng(5)
    heads = [0, 11, 23]
    rows = np.array([[h, i] for h in heads for i in np.concatenate([rng.integers(0, w.N, 60), [0, w.N - 1]])])
    out = _gpu_mx(mx, q, k, v).reshape(w.B * w.H, w.N, 128)
    ref = _oracle(orc, q, k, v, rows, heads=heads)
    g = out.cpu().numpy().astype(np.float64)[rows[:, 0], rows[:, 1]]
    _gate(g, ref["out"], "lognormal_4096 sampled")


@pytest.mark.parametrize("name,nrows", [("wan_32760", 48), ("hunyuan_118800", 12), ("causal_lm_8192", 64)])
def test_forward_full_size_sampled(mx, orc, name, nrows):
    w = W.WORKLOADS[name]
    q, k, v = W.generate(w, device="cuda")
    out = _gpu_mx(mx, q, k, v, causal=w.causal).reshape(w.B * w.H, w.N, 128)
    rng = np.random.default_rng(7)
    BH = w.B * w.H
    heads = sorted(set([0, BH - 1, int(rng.integers(0, BH))]))
    per = max(1, nrows // len(heads))
    rows = []
    for h in heads:
        rows += [[h, int(i)] for i in rng.integers(0, w.N, per)]
        rows += [[h, w.N - 1], [h, (w.N - 1) // 128 * 128]]  # ragged last tile
    rows = np.array(rows, dtype=np.int64)
    ridx = torch.tensor(rows[:, 0] * w.N + rows[:, 1], device="cuda")
    g = out.reshape(-1, 128).index_select(0, ridx).cpu().numpy().astype(np.float64)
    ref = _oracle(orc, q, k, v, rows, causal=w.causal, heads=heads)
    del q, k, v, out
    torch.cuda.empty_cache()
    _gate(g, ref["out"], f"{name} sampled")


@pytest.mark.parametrize("name,nrows", [("wan_32760", 40), ("hunyuan_118800", 16)])
def test_phat_flip_rate_full_length(mx, orc, name, nrows):
    """The P^ gate at the full sequence length of the outlier workloads: one head of
    the workload's recipe (x20 outlier channels, near-one-hot rows) at its full N,
    every P^ tile of the sampled rows dumped and compared entry by entry with the
    oracle's P^ (PNQ, Eqs. 44-48), and those rows' outputs within the tolerance.
    The dump is the production kernel plus stores: its output must equal the
    plain forward's bit for bit."""
    w = W.WORKLOADS[name]
    q, k, v = W.generate(w, device="cuda", H=1)
    B, H, N = 1, 1, w.N
    out, pc, ps = _gpu_mx(mx, q, k, v, causal=w.causal, dump=True)
    plain = _gpu_mx(mx, q, k, v, causal=w.causal)
    assert torch.equal(out, plain)
    rng = np.random.default_rng(17)
    tok = np.concatenate([rng.integers(0, N, nrows - 4), [0, 127, N - 1, (N - 1) // 128 * 128]])
    rows = np.array([[0, int(i)] for i in tok], dtype=np.int64)
    ridx = torch.tensor(rows[:, 1], device="cuda")
    pcr = pc.reshape(N, -1).index_select(0, ridx).cpu().numpy()
    psr = ps.reshape(N, -1).index_select(0, ridx).cpu().numpy()
    g = out.reshape(N, 128).index_select(0, ridx).cpu().numpy().astype(np.float64)
    del pc, ps, out, plain
    torch.cuda.empty_cache()
    ref = _oracle(orc, q, k, v, rows, causal=w.causal, want_phat=True)
    vals = np.array([orc.e2m1_value(c) for c in range(16)])
    gp = L.phat_values(pcr, psr, vals)
    valid = np.broadcast_to(np.arange(gp.shape[1])[None, :] < N, gp.shape)
    diff = (gp != ref["phat"]) & valid
    rate = diff.sum() / valid.sum()
    print(f"{name} full length: P^ flip rate {rate:.2e} ({diff.sum()} of {valid.sum()} entries)")
    assert rate < MAX_FLIP_RATE
    _gate(g, ref["out"], f"{name} full length, dumped rows")


def test_causal_no_future_leakage_gpu(mx):
    q, k, v = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=2, N=600, seed=31)
    base = _gpu_mx(mx, q, k, v, causal=True).clone()
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    for i in [0, 5, 31, 32, 63, 100, 127, 128, 200, 255, 256, 383, 450, 599]:
        q2, k2, v2 = q.clone(), k.clone(), v.clone()
        n = 600 - i - 1
        if n > 0:
            for t in (q2, k2, v2):
                t[:, :, i + 1:] = (torch.randn((1, 2, n, 128), generator=g, device="cuda") * 30).to(torch.bfloat16)
        out = _gpu_mx(mx, q2, k2, v2, causal=True)
        assert torch.equal(out[:, :, i], base[:, :, i]), f"row {i} changed"
        # the earlier rows as well
        assert torch.equal(out[:, :, : i + 1], base[:, :, : i + 1])


def test_v_ones_gives_ones(mx):
    q, k, _ = W.generate(W.WORKLOADS["tiny_outlier_512"], device="cuda", N=777)
    v = torch.ones_like(q)
    for causal in (False, True):
        out = _gpu_mx(mx, q, k, v, causal=causal)
        assert torch.max(torch.abs(out - 1.0)).item() <= 1e-6


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_scores_give_block_means(mx, orc, causal):
    """Degenerate case (Q = 0: every score 0, P~ = 1, P^ = 1 exactly, l = visible
    keys): O is the mean of the visible V^ rows, with the query's own 32-token
    block on its bf16 V rows in causal mode. The reference is that closed form
    over the oracle's V^, not a replay of the kernel; N is ragged."""
    B, H, N = 1, 2, 1000
    _, k, v = W.generate(W.WORKLOADS["lognormal_4096"], device="cuda", B=B, H=H, N=N, seed=41)
    q = torch.zeros_like(k)
    out = _gpu_mx(mx, q, k, v, causal=causal).reshape(B * H, N, 128).cpu().numpy().astype(np.float64)
    v16 = W.as_u16(v.reshape(B * H, N, 128))
    vc, vs = orc.quantize_v(v16)
    e2 = np.array([orc.e2m1_value(c) for c in range(16)])
    blk = np.arange(N) // 32
    vhat = e2[vc] * np.transpose(np.exp2(vs.astype(np.float64) - 127.0)[:, :, blk], (0, 2, 1))
    vraw = v.reshape(B * H, N, 128).float().cpu().numpy().astype(np.float64)
    if causal:
        csum = np.cumsum(vhat, axis=1)
        want = np.empty_like(vhat)
        for i in range(N):
            d0 = 32 * (i // 32)
            off = csum[:, d0 - 1] if d0 > 0 else 0.0
            want[:, i] = (off + vraw[:, d0:i + 1].sum(axis=1)) / (i + 1)
    else:
        want = np.broadcast_to(vhat.mean(axis=1, keepdims=True), vhat.shape)
    err = np.abs(out - want).max()
    print(f"uniform scores causal={causal}: max|O - mean| {err:.3e} (max|V| {np.abs(vraw).max():.3f})")
    assert err <= 1e-5 * np.abs(vraw).max()


def test_ell_consistency_direct_vs_dump(mx, orc):
    """l_i >= 1 (Appendix J) through the kernel: rows whose max entry sits in
    any tile keep an exact 1 in P^; the dumped P^ shows it."""
    q, k, v = W.generate(W.WORKLOADS["tiny_outlier_512"], device="cuda", N=300)
    _, pc, ps = _gpu_mx(mx, q, k, v, dump=True)
    vals = np.array([orc.e2m1_value(c) for c in range(16)])
    P = L.phat_values(pc.cpu().numpy().reshape(-1, pc.shape[-1]), ps.cpu().numpy().reshape(-1, ps.shape[-1]), vals)
    assert np.all(np.any(P == 1.0, axis=1))


def _bf16_host(x):
    return (x.float().cpu().numpy()).astype(np.float64)


@pytest.mark.parametrize("shape,causal", [((1, 2, 512), False), ((1, 3, 1000), True), ((1, 2, 4096), False)])
def test_bf16_forward_vs_exact_softmax(mx, orc, shape, causal):
    """BF16 path against fp64 softmax attention (Eq. 1). Each weight carries one
    bf16 rounding of P (relative 2^-9) and the fp32 products are exact, so
    |O - O_ref| <= 2 * 2^-9 * max|V| bounds the error."""
    B, H, N = shape
    q, k, v = W.generate(W.WORKLOADS["lognormal_4096"], device="cuda", B=B, H=H, N=N, seed=N)
    out = mx.mxattn_forward_bf16(q, k, v, causal=causal)
    mx.mxattn_check()
    rng = np.random.default_rng(1)
    rows = np.array([[b, int(i)] for b in range(B * H) for i in np.concatenate([rng.integers(0, N, 40), [0, N - 1]])])
    ref = orc.sdpa(W.as_u16(q).reshape(B * H, N, 128), W.as_u16(k).reshape(B * H, N, 128),
                   W.as_u16(v).reshape(B * H, N, 128), rows, causal=causal)
    g = out.reshape(B * H, N, 128).cpu().numpy().astype(np.float64)[rows[:, 0], rows[:, 1]]
    vmax = float(torch.max(torch.abs(v.float())).item())
    err = np.abs(g - ref).max()
    print(f"bf16 {shape} causal={causal}: max|err| {err:.3e}, bound {2 * 2 ** -9 * vmax:.3e}")
    assert err <= 2 * 2 ** -9 * vmax + 1e-5


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_forward_full_length(mx, orc, causal):
    """BF16 path over a full Wan-length key loop (one head, N = 32760: 256 key
    tiles, the ragged last one 120 keys long) with the outlier recipe, on
    sampled rows against fp64 softmax attention. Same bound as above."""
    N = 32760
    q, k, v = W.generate(W.WORKLOADS["wan_32760"], device="cuda", B=1, H=1, N=N)
    out = mx.mxattn_forward_bf16(q, k, v, causal=causal)
    mx.mxattn_check()
    rng = np.random.default_rng(5)
    rows = np.array([[0, int(i)] for i in np.concatenate([rng.integers(0, N, 40), [0, 127, 128, N - 121, N - 1]])])
    ref = orc.sdpa(W.as_u16(q).reshape(1, N, 128), W.as_u16(k).reshape(1, N, 128), W.as_u16(v).reshape(1, N, 128),
                   rows, causal=causal)
    g = out.reshape(1, N, 128)[0, torch.as_tensor(rows[:, 1], device=out.device)].cpu().numpy().astype(np.float64)
    vmax = float(torch.max(torch.abs(v.float())).item())
    err = np.abs(g - ref).max()
    assert err <= 2 * 2 ** -9 * vmax + 1e-5, (err, 2 * 2 ** -9 * vmax)


def test_mxfp4_error_vs_unquantized_reported(mx, orc):
    """Error of the MXFP4 path against fp64 unquantized attention: reported, not gated."""
    q, k, v = W.generate(W.WORKLOADS["tiny_outlier_512"], device="cuda")
    out = _gpu_mx(mx, q, k, v).reshape(2, 512, 128).cpu().numpy().astype(np.float64)
    rows = _all_rows(2, 512)
    ref = orc.sdpa(W.as_u16(q).reshape(2, 512, 128), W.as_u16(k).reshape(2, 512, 128),
                   W.as_u16(v).reshape(2, 512, 128), rows)
    g = out[rows[:, 0], rows[:, 1]]
    rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
    print(f"MXFP4 vs unquantized fp64 attention: relative L2 error {rel:.3e}")
    assert np.isfinite(rel)


def test_bounded_wait_timeout_reports_and_recovers(mx):
    q, k, v = W.generate(W.WORKLOADS["tiny_outlier_512"], device="cuda", N=256)
    good = _gpu_mx(mx, q, k, v).clone()
    qc, qs = mx.mxattn_rotate_quantize_qk(q)
    kc, ks = mx.mxattn_rotate_quantize_qk(k)
    vc, vs = mx.mxattn_quantize_v(v)
    mx.mxattn_check()
    mx.mxattn_set_debug_flags(1)
    try:
        mx.mxattn_forward(qc, qs, kc, ks, vc, vs, v, 1, 2, 256)
        with pytest.raises(mx.MxattnError) as ei:
            mx.mxattn_check()
        assert ei.value.status == 4
        mx.mxattn_forward_bf16(q, k, v)
        with pytest.raises(mx.MxattnError):
            mx.mxattn_check()
    finally:
        mx.mxattn_set_debug_flags(0)
    # the context is still usable and results are unchanged
    again = _gpu_mx(mx, q, k, v)
    assert torch.equal(again, good)


def test_host_entry_point_matches_device_path(mx):
    q, k, v = W.generate(W.WORKLOADS["tiny_outlier_512"], device="cuda", N=333)
    dev = _gpu_mx(mx, q, k, v, causal=True)
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    outh = torch.empty(q.shape, dtype=torch.float32).pin_memory()
    ws = torch.empty(mx.mxattn_workspace_bytes(1, 2, 333), dtype=torch.uint8, device="cuda")
    mx.mxattn_attention_host(qh, kh, vh, True, outh, ws)
    assert torch.equal(outh, dev.cpu())


@pytest.mark.parametrize("causal", [False, True])
def test_device_convenience_call_matches_device_path(mx, causal):
    """mxattn_attention (one quantizer launch, then the forward) gives the
    output of the separate single-tensor quantizers and the forward, bit for bit."""
    q, k, v = W.generate(W.WORKLOADS["tiny_outlier_512"], device="cuda", N=333)
    assert torch.equal(mx.mxattn_attention(q, k, v, causal=causal), _gpu_mx(mx, q, k, v, causal=causal))


@pytest.mark.parametrize("causal", [False, True])
def test_host_entry_point_pipelined_chunks(mx, causal):
    """21 heads of 32760 tokens (25 MB of input per head) run as 12 chunks
    (one head in the first and in the last, two in each of the others) whose
    copies overlap the kernels; two calls in a row (the internal streams and
    events are reused) give the device path's output bit for bit."""
    q, k, v = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=3, H=7, N=32760, seed=17)
    dev = _gpu_mx(mx, q, k, v, causal=causal).cpu()
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    ws = torch.empty(mx.mxattn_workspace_bytes(3, 7, 32760), dtype=torch.uint8, device="cuda")
    for _ in range(2):
        outh = torch.full(q.shape, float("nan"), dtype=torch.float32).pin_memory()
        mx.mxattn_attention_host(qh, kh, vh, causal, outh, ws)
        assert torch.equal(outh, dev)


def test_empty_problem(mx):
    z = torch.empty((1, 2, 0, 128), dtype=torch.bfloat16, device="cuda")
    c, s = mx.mxattn_rotate_quantize_qk(z)
    assert c.numel() == 0 and s.numel() == 0
    out = mx.mxattn_forward_bf16(z, z, z)
    assert out.shape == (1, 2, 0, 128)


@pytest.mark.parametrize("N", [1, 2, 31, 127, 128, 129, 255, 256, 257])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_tiny_and_ragged_lengths(mx, orc, N, causal):
    """Every row against the oracle where the tiling has edge cases: one key, a single partial tile,
    exactly one tile (no second query tile in the CTA), one row past a tile, odd tile counts."""
    q, k, v = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=3, N=N, seed=100 + N)
    B, H, _, _ = q.shape
    g = _gpu_mx(mx, q, k, v, causal=causal).reshape(B * H, N, 128).cpu().numpy().astype(np.float64)
    ref = _oracle(orc, q, k, v, _all_rows(B * H, N), causal=causal)["out"].reshape(B * H, N, 128)
    _gate(g.reshape(-1, 128), ref.reshape(-1, 128), f"N={N} causal={causal}")


def test_maximum_heads(mx, orc):
    """B*H = 65535, the largest the ABI accepts (one grid row per head): quantizers and forward against the oracle
    on sampled rows of the first, last and a middle head."""
    B, H, N = 5, 13107, 130
    g = torch.Generator(device="cuda").manual_seed(3)
    q, k, v = (torch.randn((B, H, N, 128), generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    out = _gpu_mx(mx, q, k, v, causal=True).reshape(B * H, N, 128)
    heads = [0, 32767, B * H - 1]
    rows = np.array([[h, i] for h in heads for i in (0, 1, 64, 127, 128, 129)], dtype=np.int64)
    ridx = torch.tensor(rows[:, 0] * N + rows[:, 1], device="cuda")
    gr = out.reshape(-1, 128).index_select(0, ridx).cpu().numpy().astype(np.float64)
    ref = _oracle(orc, q, k, v, rows, causal=True, heads=heads)
    del q, k, v, out
    torch.cuda.empty_cache()
    _gate(gr, ref["out"], "B*H = 65535")


def test_long_sequence_single_head(mx, orc):
    """N = 2^20 keys in one head (8192 key tiles per CTA), non-causal, sampled rows against the oracle."""
    N = 1 << 20
    g = torch.Generator(device="cuda").manual_seed(4)
    q, k, v = (torch.randn((1, 1, N, 128), generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    out = _gpu_mx(mx, q, k, v).reshape(N, 128)
    rows = np.array([[0, i] for i in (0, 1, 4095, 524288, N - 2, N - 1)], dtype=np.int64)
    gr = out.index_select(0, torch.tensor(rows[:, 1], device="cuda")).cpu().numpy().astype(np.float64)
    ref = _oracle(orc, q, k, v, rows)
    del q, k, v, out
    torch.cuda.empty_cache()
    _gate(gr, ref["out"], "N = 2^20")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 333, 1000])
def test_bf16_output_is_the_rounded_fp32_output(mx, N, causal):
    """mxattn_forward_out_bf16 writes exactly the fp32 output rounded to the
    nearest bf16 (ties to even), rows < N only."""
    q, k, v = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=3, N=N, seed=200 + N)
    qc, qs, kc, ks, vc, vs = mx.mxattn_quantize_qkv(q, k, v)
    o32 = mx.mxattn_forward(qc, qs, kc, ks, vc, vs, v, 1, 3, N, causal=causal)
    o16 = mx.mxattn_forward(qc, qs, kc, ks, vc, vs, v, 1, 3, N, causal=causal, out_dtype=torch.bfloat16)
    mx.mxattn_check()
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o16, o32.to(torch.bfloat16))


def test_bf16_output_full_length(mx):
    w = W.WORKLOADS["wan_32760"]
    q, k, v = W.generate(w, device="cuda", H=4)
    qc, qs, kc, ks, vc, vs = mx.mxattn_quantize_qkv(q, k, v)
    o32 = mx.mxattn_forward(qc, qs, kc, ks, vc, vs, v, 1, 4, w.N)
    o16 = torch.full(o32.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    mx.mxattn_forward(qc, qs, kc, ks, vc, vs, v, 1, 4, w.N, out=o16, out_dtype=torch.bfloat16)
    mx.mxattn_check()
    assert torch.equal(o16, o32.to(torch.bfloat16))


def test_binding_rejects_short_device_buffers(mx):
    """Buffers smaller than the layouts of B, H, N raise before any launch."""
    q, k, v = W.generate(W.WORKLOADS["tiny_outlier_512"], device="cuda", N=300)
    qc, qs, kc, ks, vc, vs = mx.mxattn_quantize_qkv(q, k, v)
    with pytest.raises(ValueError, match="k_codes"):
        mx.mxattn_forward(qc, qs, kc[:-1], ks, vc, vs, v, 1, 2, 300)
    with pytest.raises(ValueError, match="v_bf16"):
        mx.mxattn_forward(qc, qs, kc, ks, vc, vs, None, 1, 2, 300, causal=True)
    with pytest.raises(ValueError, match="out"):
        mx.mxattn_forward(qc, qs, kc, ks, vc, vs, v, 1, 2, 300, out=torch.empty((1, 2, 299, 128), device="cuda"))
    with pytest.raises(ValueError, match="dtype"):
        mx.mxattn_forward(qc, qs, kc, ks, vc, vs, v, 1, 2, 300, out=torch.empty((1, 2, 300, 128), device="cuda"),
                          out_dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="scales"):
        mx.mxattn_rotate_quantize_qk(q, scales=qs[:10])
    with pytest.raises(ValueError, match="v_codes"):
        mx.mxattn_quantize_qkv(q, k, v, out=(qc, qs, kc, ks, vc[:5], vs))
    mx.mxattn_check()


@pytest.mark.parametrize("causal", [False, True])
def test_cuda_graph_capture_and_replay(mx, causal):
    """The two-launch step (one quantizer launch, the forward) captures into a
    CUDA graph; replays give the eager output bit for bit, and recompute after
    the inputs are overwritten in place."""
    q, k, v = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=3, N=1000, seed=41)
    ref = mx.mxattn_attention(q, k, v, causal=causal)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        mx.mxattn_attention(q, k, v, causal=causal, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = mx.mxattn_attention(q, k, v, causal=causal)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    q2, k2, v2 = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=3, N=1000, seed=42)
    q.copy_(q2)
    k.copy_(k2)
    v.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, mx.mxattn_attention(q2, k2, v2, causal=causal))
    mx.mxattn_check()


@pytest.mark.parametrize("nq,nk,causal", [(300, 200, False), (200, 300, False), (300, 200, True), (200, 333, True),
                                          (129, 1, False), (1, 257, True), (513, 384, True)])
def test_bf16_forward_query_and_key_lengths_differ(mx, nq, nk, causal):
    """BF16 path with Nq != Nk against float64 softmax attention (Eq. 1) on the
    same bf16 inputs; causal keeps key j for query i iff j <= i. Bound as in
    the equal-length test: one bf16 rounding of each P entry."""
    w = W.WORKLOADS["lognormal_4096"]
    q = W.generate(w, device="cuda", B=1, H=2, N=nq, seed=nq)[0]
    _, k, v = W.generate(w, device="cuda", B=1, H=2, N=nk, seed=nk + 7)
    out = mx.mxattn_forward_bf16(q, k, v, causal=causal)
    mx.mxattn_check()
    assert out.shape == (1, 2, nq, 128)
    qd, kd, vd = (t.double().cpu() for t in (q, k, v))
    s = qd @ kd.transpose(-1, -2) / 128 ** 0.5
    if causal:
        s = s.masked_fill(torch.arange(nk)[None, :] > torch.arange(nq)[:, None], float("-inf"))
    ref = torch.softmax(s, -1) @ vd
    err = (out.double().cpu() - ref).abs().max().item()
    bound = 2 * 2 ** -9 * vd.abs().max().item()
    assert err <= bound, (err, bound)
