"""GPU parity of the NVFP4 comparison path against the oracle, through the C ABI.

NVFP4 as "MXAttention" describes it (section 1: 16-element blocks, E4M3 block
scales, a tensor-level scale) and its direct baseline (section 5.2: Q, K, V and
P~ quantized, no smoothing, no softmax-path scaling), with the oracle's
readings N1-N6:
  * quantizers: the tensor maximum, every E2M1 code and every E4M3 scale byte
    equal the oracle's (bit-exact; ragged N, special values);
  * forward: every P^ entry the kernel dumps is compared with the oracle's
    (< 0.1 % may differ: E4M3 has eight scale boundaries per octave where
    E8M0 has one, so a P~ maximum within rounding of a boundary can take the
    neighbouring scale), and the oracle replays every row with the kernel's
    own P^: max |O_gpu - O_replay| <= 2e-3 * RMS on every row of small cases
    (ragged N, causal and not, direct and PNQ placement). Sampled rows at the
    Wan size against the oracle's own loop; V == 1 gives O == 1 under PNQ.
"""
import math

import numpy as np
import pytest
import torch

import _layouts as L
from mxfp4_precision_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mxfp4_precision_attention_gb300 as m

    m.load()
    return m


def _nv_qk(mx, orc, x):
    B, H, N, _ = x.shape
    codes, scales, amax = mx.mxattn_nvfp4_quantize_qk(x)
    mx.mxattn_check()
    oc, os_, oet = orc.nvfp4_quantize_qk(W.as_u16(x).reshape(B * H, N, 128))
    assert np.float32(2688.0) / np.float32(amax.item()) == np.float32(oet)
    gc = L.qk_codes_logical(codes.cpu().numpy(), B * H, N)
    gs = L.nv_qk_scales_logical(scales.cpu().numpy(), B * H, N)
    assert np.array_equal(gc, oc), f"code mismatches: {(gc != oc).sum()}"
    assert np.array_equal(gs, os_), f"scale mismatches: {(gs != os_).sum()}"
    return codes, scales, amax


def _nv_v(mx, orc, v):
    B, H, N, _ = v.shape
    codes, scales, amax = mx.mxattn_nvfp4_quantize_v(v)
    mx.mxattn_check()
    oc, os_, oet = orc.nvfp4_quantize_v(W.as_u16(v).reshape(B * H, N, 128))
    assert np.float32(2688.0) / np.float32(amax.item()) == np.float32(oet)
    gc = L.v_codes_logical(codes.cpu().numpy(), B * H, N)
    gs = L.nv_v_scales_logical(scales.cpu().numpy(), B * H, N)
    assert np.array_equal(gc, oc), f"code mismatches: {(gc != oc).sum()}"
    assert np.array_equal(gs, os_), f"scale mismatches: {(gs != os_).sum()}"
    return codes, scales, amax


@pytest.mark.parametrize("N", [1, 15, 16, 17, 100, 128, 129, 300, 1000])
def test_nvfp4_quantizers_bitexact(mx, orc, N):
    q, k, v = W.generate(W.WORKLOADS["lognormal_4096"], device="cuda", N=N, H=3, seed=N + 1)
    _nv_qk(mx, orc, q)
    _nv_qk(mx, orc, k)
    _nv_v(mx, orc, v)


def test_nvfp4_quantizers_special_values(mx, orc):
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    x = torch.randn((1, 2, 384, 128), generator=g, device="cuda")
    x[0, 0, 0] = 0.0
    x[0, 0, 1, 16:32] = 0.0
    x[0, 0, 2] *= 1e-6                  # tiny blocks: E4M3 subnormal and zero scales
    x[0, 0, 3] *= 1e-12
    x[0, 0, 4] = -1e-39
    x[0, 1, 5, 7] = 3.0e4               # the tensor maximum
    x[0, 1, 64:80, 9] = 0.0
    x[0, 1, 80:96, 9] = 1e-9
    xb = x.to(torch.bfloat16).contiguous()
    _nv_qk(mx, orc, xb)
    _nv_v(mx, orc, xb)
    z = torch.zeros((1, 1, 200, 128), dtype=torch.bfloat16, device="cuda")
    c, s, a = mx.mxattn_nvfp4_quantize_qk(z)
    assert a.item() == 0.0 and not c.any() and not s.any()


TOL_REL_RMS = 2e-3


def _to_logical(mx, B, H, N, qt, kt, vt):
    BH = B * H
    qc = L.qk_codes_logical(qt[0].cpu().numpy(), BH, N)
    qs = L.nv_qk_scales_logical(qt[1].cpu().numpy(), BH, N)
    kc = L.qk_codes_logical(kt[0].cpu().numpy(), BH, N)
    ks = L.nv_qk_scales_logical(kt[1].cpu().numpy(), BH, N)
    vc = L.v_codes_logical(vt[0].cpu().numpy(), BH, N)
    vs = L.nv_v_scales_logical(vt[1].cpu().numpy(), BH, N)
    et = [float(np.float32(2688.0) / np.float32(t[2].item())) for t in (qt, kt, vt)]
    return qc, qs, et[0], kc, ks, et[1], vc, vs, et[2]


def _gpu_nv(mx, q, k, v, causal, placement):
    B, H, N, _ = q.shape
    qt, kt, vt = mx.mxattn_nvfp4_quantize_qk(q), mx.mxattn_nvfp4_quantize_qk(k), mx.mxattn_nvfp4_quantize_v(v)
    out = mx.mxattn_nvfp4_forward(qt, kt, vt, v, B, H, N, causal=causal, placement=placement)
    mx.mxattn_check()
    return out, (qt, kt, vt)


MAX_FLIP_RATE = 1e-3


def _nv_parity(mx, orc, q, k, v, causal, placement, what):
    """Kernel vs oracle: the P^ entries compared one by one, then every row replayed with the kernel's P^."""
    B, H, N, _ = q.shape
    qt, kt, vt = mx.mxattn_nvfp4_quantize_qk(q), mx.mxattn_nvfp4_quantize_qk(k), mx.mxattn_nvfp4_quantize_v(v)
    out, pc, ps = mx.mxattn_nvfp4_forward_dump_phat(qt, kt, vt, v, B, H, N, causal=causal, placement=placement)
    mx.mxattn_check()
    g = out.reshape(B * H, N, 128).cpu().numpy().astype(np.float64)
    qb, kb, vb = (W.as_u16(t).reshape(B * H, N, 128) for t in (q, k, v))
    oq, ok_, ov = orc.nvfp4_quantize_qk(qb), orc.nvfp4_quantize_qk(kb), orc.nvfp4_quantize_v(vb)
    rows = np.array([[b, i] for b in range(B * H) for i in range(N)], dtype=np.int64)
    own = orc.forward_nvfp4(*oq, *ok_, *ov, rows, vraw_u16=vb, causal=causal, placement=placement, want_phat=True)
    e2 = np.array([orc.e2m1_value(c) for c in range(16)])
    e4 = np.array([orc.e4m3_value(c) if c < 127 else np.nan for c in range(256)])
    gp = L.nv_phat_values(pc.cpu().numpy()[rows[:, 0], rows[:, 1]], ps.cpu().numpy()[rows[:, 0], rows[:, 1]], e2, e4)
    keys = np.arange(gp.shape[1])[None, :]
    valid = np.broadcast_to(keys < N, gp.shape)
    if causal:
        valid = valid & (keys <= rows[:, 1:2])
    diff = (gp != own["phat"]) & valid
    rate = diff.sum() / valid.sum()
    rep = orc.forward_nvfp4(*oq, *ok_, *ov, rows, vraw_u16=vb, causal=causal, placement=placement,
                            phat_in=np.where(valid, gp, 0.0))
    ref = rep["out"].reshape(B * H, N, 128)
    rms = math.sqrt(np.mean(ref ** 2))
    err = np.abs(g - ref).max()
    own_err = np.abs(g - own["out"].reshape(B * H, N, 128)).max()
    print(f"{what}: P^ flips {rate:.2e} ({diff.sum()}), max|O - replay| {err / rms:.3e} RMS, "
          f"max|O - oracle| {own_err / rms:.3e} RMS")
    assert rate < MAX_FLIP_RATE
    assert err <= TOL_REL_RMS * rms


@pytest.mark.parametrize("placement", [1, 0])
@pytest.mark.parametrize("causal", [False, True])
def test_nvfp4_forward_all_rows(mx, orc, causal, placement):
    if causal:
        q, k, v = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=2, N=700, seed=19)
    else:
        q, k, v = W.generate(W.WORKLOADS["tiny_outlier_512"], device="cuda", N=300)
    _nv_parity(mx, orc, q, k, v, causal, placement, f"nvfp4 causal={causal} placement={placement}")


def test_nvfp4_forward_v_ones_pnq(mx):
    q, k, _ = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=2, N=600, seed=23)
    v = torch.ones_like(q)
    for causal in (False, True):
        pnq, _ = _gpu_nv(mx, q, k, v, causal, 0)
        assert (pnq - 1.0).abs().max().item() <= 1e-5
        direct, _ = _gpu_nv(mx, q, k, v, causal, 1)
        assert (direct - 1.0).abs().max().item() > 1e-3


@pytest.mark.parametrize("name,nrows", [("wan_32760", 48), ("causal_lm_8192", 64)])
def test_nvfp4_forward_full_size_sampled(mx, orc, name, nrows):
    """At the benchmark sizes: the oracle's loop on the GPU-quantized operands (the quantizers are pinned
    bit-exact above; the tensor maxima are checked against torch here), on sampled rows."""
    w = W.WORKLOADS[name]
    q, k, v = W.generate(w, device="cuda")
    out, (qt, kt, vt) = _gpu_nv(mx, q, k, v, w.causal, 1)
    for t, x in ((qt, q), (kt, k), (vt, v)):
        assert t[2].item() == x.abs().max().float().item()
    BH, N = w.B * w.H, w.N
    rng = np.random.default_rng(11)
    heads = sorted(set([0, BH - 1, int(rng.integers(0, BH))]))
    per = max(1, nrows // len(heads))
    rows = []
    for h in heads:
        rows += [[h, int(i)] for i in rng.integers(0, N, per)]
        rows += [[h, N - 1], [h, (N - 1) // 128 * 128]]
    rows = np.array(rows, dtype=np.int64)
    g = out.reshape(BH * N, 128).index_select(0, torch.tensor(rows[:, 0] * N + rows[:, 1], device="cuda"))
    g = g.cpu().numpy().astype(np.float64)
    # the listed heads only, in the oracle's logical layouts
    idx = torch.tensor(heads, device="cuda")
    sub = lambda t, per_head: t.reshape(BH, -1).index_select(0, idx).reshape(-1)
    nh = len(heads)
    qt_s = (sub(qt[0], 1), sub(qt[1], 1), qt[2])
    kt_s = (sub(kt[0], 1), sub(kt[1], 1), kt[2])
    vt_s = (sub(vt[0], 1), sub(vt[1], 1), vt[2])
    ops = _to_logical(mx, 1, nh, N, qt_s, kt_s, vt_s)
    vraw = W.as_u16(v.reshape(BH, N, 128).index_select(0, idx))
    remap = {h: i for i, h in enumerate(heads)}
    rr = np.array([[remap[int(b)], int(i)] for b, i in rows], dtype=np.int64)
    ref = orc.forward_nvfp4(*ops, rr, vraw_u16=vraw, causal=w.causal, placement=1)["out"]
    del q, k, v, out
    torch.cuda.empty_cache()
    err = np.abs(g - ref).max()
    rms = math.sqrt(np.mean(ref ** 2))
    print(f"{name} nvfp4 sampled: max|err| {err:.3e}, ratio {err / rms:.3e}")
    assert err <= TOL_REL_RMS * rms


@pytest.mark.parametrize("causal", [False, True])
def test_nvfp4_forward_all_rows_past_two_ring_wraps(mx, orc, causal):
    """Nine key tiles (N = 1100): the 4-stage V ring wraps twice. The NVFP4 kernel keeps
    one buffer of V^ scales in TMEM and reloads it once the previous tile's products are
    complete, which it learns from that tile's ring release; every row against the oracle."""
    q, k, v = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=1, N=1100, seed=23)
    _nv_parity(mx, orc, q, k, v, causal, 1, f"nvfp4 N=1100 causal={causal}")


@pytest.mark.parametrize("N", [1, 17, 128, 129, 257])
@pytest.mark.parametrize("causal", [False, True])
def test_nvfp4_forward_tiny_and_ragged_lengths(mx, orc, N, causal):
    q, k, v = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=2, N=N, seed=200 + N)
    _nv_parity(mx, orc, q, k, v, causal, 1, f"nvfp4 N={N} causal={causal}")
