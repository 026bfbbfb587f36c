"""GPU parity of the ablation variants ("MXAttention" section 5.4, Table 3)
against the oracle, through the C ABI.

Switches: the block scale rule of every quantizer (UOS, Eq. 13; OCP floor,
Eq. 11; TFS ceil, Eq. 14; ceil with a swept Q_max, section 5.5.1), the fixed
Hadamard rotation on or off, and where l comes from (PNQ, Eq. 47, or direct
placement, Eqs. 16-17).
  * quantizers: every code and scale byte equals the oracle's;
  * forward: max |O_gpu - O_oracle| <= 2e-3 * RMS(O_oracle) on every row of
    small cases (ragged N, causal and not), for the rows of Table 3 and TFS;
  * row-sum control (Proposition 1 vs Eq. 110): with V == 1, PNQ gives
    O == 1 while direct placement gives rows that are not 1, as the oracle
    does.
"""
import math

import numpy as np
import pytest
import torch

import _layouts as L
from mxfp4_precision_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_REL_RMS = 2e-3

# (name, rule of Q/K/V/P~, rotate, placement, Q_max of the ceil rule) -- Table 3
# top to bottom, then TFS and two points of the section 5.5.1 Q_max sweep
CONFIGS = [
    ("full", 0, True, 0, 7.25),
    ("no_uos", 1, True, 0, 7.25),
    ("no_uos_no_pnq", 1, True, 1, 7.25),
    ("ocp_direct", 1, False, 1, 7.25),
    ("tfs_pnq", 2, True, 0, 7.25),
    ("ceil_6.8", 3, True, 0, 6.8),
    ("ceil_8", 3, True, 0, 8.0),
]


@pytest.fixture(scope="module")
def mx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mxfp4_precision_attention_gb300 as m

    m.load()
    return m


@pytest.mark.parametrize("rule", [0, 1, 2])
@pytest.mark.parametrize("rotate", [True, False])
def test_quantize_qk_rules(mx, orc, rule, rotate):
    q, _, _ = W.generate(W.WORKLOADS["lognormal_4096"], device="cuda", H=3, N=1000)
    B, H, N, _ = q.shape
    codes, scales = mx.mxattn_quantize_qk_ex(q, rule=rule, rotate=rotate)
    torch.cuda.synchronize()
    gc = L.qk_codes_logical(codes.cpu().numpy(), B * H, N)
    gs_all = L.tiles_logical(scales.cpu().numpy(), B * H, N)
    assert np.all(gs_all[:, N:] == 127)
    oc, os_ = orc.rotate_quantize_qk(W.as_u16(q).reshape(B * H, N, 128), rule=rule, rotate=rotate)
    assert np.array_equal(gc, oc), f"code mismatches: {(gc != oc).sum()}"
    assert np.array_equal(gs_all[:, :N], os_), f"scale mismatches: {(gs_all[:, :N] != os_).sum()}"


@pytest.mark.parametrize("rule", [0, 1, 2])
def test_quantize_v_rules(mx, orc, rule):
    _, _, v = W.generate(W.WORKLOADS["lognormal_4096"], device="cuda", H=3, N=1000)
    B, H, N, _ = v.shape
    codes, scales = mx.mxattn_quantize_v_ex(v, rule=rule)
    torch.cuda.synchronize()
    gc = L.v_codes_logical(codes.cpu().numpy(), B * H, N)
    gs = L.v_scales_logical(scales.cpu().numpy(), B * H, N)
    oc, os_ = orc.quantize_v(W.as_u16(v).reshape(B * H, N, 128), rule=rule)
    assert np.array_equal(gc, oc), f"code mismatches: {(gc != oc).sum()}"
    assert np.array_equal(gs, os_), f"scale mismatches: {(gs != os_).sum()}"


@pytest.mark.parametrize("qmax", [6.05, 7.2, 7.3, 8.0])
def test_quantizers_ceil_rule_any_qmax(mx, orc, qmax):
    """Section 5.5.1's swept Q_max: codes and scales bit-exact for Q/K (rotated) and V."""
    q, _, v = W.generate(W.WORKLOADS["lognormal_4096"], device="cuda", H=3, N=1000, seed=4)
    B, H, N, _ = q.shape
    codes, scales = mx.mxattn_quantize_qk_ex(q, rule=3, qmax=qmax)
    vcodes, vscales = mx.mxattn_quantize_v_ex(v, rule=3, qmax=qmax)
    torch.cuda.synchronize()
    oc, os_ = orc.rotate_quantize_qk(W.as_u16(q).reshape(B * H, N, 128), rule=3, q=qmax)
    assert np.array_equal(L.qk_codes_logical(codes.cpu().numpy(), B * H, N), oc)
    assert np.array_equal(L.qk_scales_logical(scales.cpu().numpy(), B * H, N), os_)
    ovc, ovs = orc.quantize_v(W.as_u16(v).reshape(B * H, N, 128), rule=3, q=qmax)
    assert np.array_equal(L.v_codes_logical(vcodes.cpu().numpy(), B * H, N), ovc)
    assert np.array_equal(L.v_scales_logical(vscales.cpu().numpy(), B * H, N), ovs)


def _run_gpu(mx, q, k, v, rule, rotate, placement, causal, qmax=7.25):
    B, H, N, _ = q.shape
    qc, qs = mx.mxattn_quantize_qk_ex(q, rule=rule, rotate=rotate, qmax=qmax)
    kc, ks = mx.mxattn_quantize_qk_ex(k, rule=rule, rotate=rotate, qmax=qmax)
    vc, vs = mx.mxattn_quantize_v_ex(v, rule=rule, qmax=qmax)
    out = mx.mxattn_forward_ex(qc, qs, kc, ks, vc, vs, v, B, H, N, causal=causal, p_rule=rule, placement=placement,
                               p_qmax=qmax)
    mx.mxattn_check()
    return out.reshape(B * H, N, 128).cpu().numpy().astype(np.float64)


def _run_oracle(orc, q, k, v, rule, rotate, placement, causal, qmax=7.25):
    B, H, N, _ = q.shape
    qb, kb, vb = (W.as_u16(t).reshape(B * H, N, 128) for t in (q, k, v))
    qc, qs = orc.rotate_quantize_qk(qb, rule=rule, rotate=rotate, q=qmax)
    kc, ks = orc.rotate_quantize_qk(kb, rule=rule, rotate=rotate, q=qmax)
    vc, vs = orc.quantize_v(vb, rule=rule, q=qmax)
    rows = np.array([[b, i] for b in range(B * H) for i in range(N)], dtype=np.int64)
    ref = orc.forward(qc, qs, kc, ks, vc, vs, rows, vraw_u16=vb, causal=causal, placement=placement, p_rule=rule,
                      p_q=qmax)
    return ref["out"].reshape(B * H, N, 128)


@pytest.mark.parametrize("name,rule,rotate,placement,qmax", CONFIGS)
@pytest.mark.parametrize("causal", [False, True])
def test_forward_variants_all_rows(mx, orc, name, rule, rotate, placement, qmax, causal):
    if causal:
        q, k, v = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=2, N=700, seed=13)
    else:
        q, k, v = W.generate(W.WORKLOADS["tiny_outlier_512"], device="cuda", N=300)
    g = _run_gpu(mx, q, k, v, rule, rotate, placement, causal, qmax)
    o = _run_oracle(orc, q, k, v, rule, rotate, placement, causal, qmax)
    err = np.abs(g - o).max()
    rms = math.sqrt(np.mean(o ** 2))
    print(f"{name} causal={causal}: max|err| = {err:.3e}, RMS = {rms:.3e}, ratio = {err / rms:.3e}")
    assert err <= TOL_REL_RMS * rms


def test_default_switches_equal_plain_entry_points(mx):
    """UOS + rotation + PNQ through the variant calls is the plain path, bit for bit."""
    q, k, v = W.generate(W.WORKLOADS["lognormal_4096"], device="cuda", H=2, N=1000)
    B, H, N, _ = q.shape
    a = _run_gpu(mx, q, k, v, 0, True, 0, False)
    qc, qs = mx.mxattn_rotate_quantize_qk(q)
    kc, ks = mx.mxattn_rotate_quantize_qk(k)
    vc, vs = mx.mxattn_quantize_v(v)
    b = mx.mxattn_forward(qc, qs, kc, ks, vc, vs, v, B, H, N).reshape(B * H, N, 128).cpu().numpy()
    assert np.array_equal(a, b.astype(np.float64))


@pytest.mark.parametrize("causal", [False, True])
def test_rowsum_control_v_ones(mx, orc, causal):
    """V == 1: PNQ rows are exactly normalized (Proposition 1); direct placement rows
    are not (Eq. 110), on the GPU and on the oracle alike."""
    q, k, _ = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=2, N=600, seed=21)
    v = torch.ones_like(q)
    pnq = _run_gpu(mx, q, k, v, 0, True, 0, causal)
    direct = _run_gpu(mx, q, k, v, 0, True, 1, causal)
    assert np.abs(pnq - 1.0).max() <= 1e-5
    dev_gpu = np.abs(direct - 1.0).max()
    dev_ora = np.abs(_run_oracle(orc, q, k, v, 0, True, 1, causal) - 1.0).max()
    print(f"direct placement, V == 1: max |O - 1| gpu {dev_gpu:.3e}, oracle {dev_ora:.3e}")
    assert dev_gpu > 1e-3 and dev_ora > 1e-3



@pytest.mark.parametrize("rule,placement", [(0, 0), (1, 1)])
def test_causal_prefix_mode_all_rows(mx, orc, rule, placement):
    """causal = 2: the query's own V block re-quantized over its prefix (the other
    reading of the MatX note's fix), against the oracle on every row."""
    q, k, v = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=2, N=700, seed=23)
    B, H, N, _ = q.shape
    g = _run_gpu(mx, q, k, v, rule, True, placement, 2)
    o = _run_oracle(orc, q, k, v, rule, True, placement, 2)
    err = np.abs(g - o).max()
    rms = math.sqrt(np.mean(o ** 2))
    print(f"prefix causal rule={rule} placement={placement}: max|err| = {err:.3e}, ratio = {err / rms:.3e}")
    assert err <= TOL_REL_RMS * rms
    # and it is not the bf16-diagonal reading
    assert not np.array_equal(g, _run_gpu(mx, q, k, v, rule, True, placement, 1))


def test_causal_prefix_mode_no_future_leakage(mx):
    """Perturbing every token after i leaves GPU row i bit-identical under causal = 2."""
    q, k, v = W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=1, N=300, seed=29)
    base = _run_gpu(mx, q, k, v, 0, True, 0, 2)
    g = torch.Generator(device="cpu").manual_seed(31)
    for i in (0, 5, 31, 40, 127, 128, 200, 299):
        q2, k2, v2 = q.clone(), k.clone(), v.clone()
        n = 300 - i - 1
        if n > 0:
            for t in (q2, k2, v2):
                t[0, 0, i + 1:] = (torch.randn(n, 128, generator=g) * 40).to(t.dtype).to(t.device)
        pert = _run_gpu(mx, q2, k2, v2, 0, True, 0, 2)
        assert np.array_equal(pert[0, i], base[0, i]), f"row {i} changed"


@pytest.mark.parametrize("name", ["causal_lm_8192", "wan_32760"])
def test_rowsum_diagnostic_matches_oracle(mx, orc, name):
    """bench.py --accuracy's row-sum diagnostic (section 5.5.2, Fig. 7 B), computed
    on the GPU through the library's quantizer, against the oracle's
    rowsum_parts on the same bf16 rows: row sum and the zeroing / saturation /
    downward / upward rounding parts, per row, under UOS and the OCP rule."""
    import bench
    from mxfp4_precision_attention_gb300 import workloads as W

    P, Pb = bench.materialized_p(W, W.WORKLOADS[name], 24)
    Pr = Pb.double().cpu().numpy()
    for rule in (orc.UOS, orc.OCP):
        g = bench.rowsum_parts_gpu(mx, Pb, rule).cpu().numpy()
        ref = orc.rowsum_parts(Pr, rule)
        assert np.allclose(g, ref, rtol=1e-12, atol=1e-12), np.abs(g - ref).max()
        assert np.allclose(g[:, 0] - Pr.sum(1), g[:, 1:].sum(1), rtol=0, atol=1e-12)
