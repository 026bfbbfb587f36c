"""GPU parity of the MXFP4 quantizers (C-ABI kernels) against the oracle.

Bit-exact: every E2M1 code and every E8M0 scale byte of Q, K (rotated) and V
must equal the oracle's ("MXAttention" Algorithm 1 and the quantization steps of Algorithm 2, section 4.3).
Small workloads are compared in full; the full-size workloads on sampled
tokens (Q/K) and sampled 128-token windows plus the ragged tail (V), in the
launch configuration the benchmark times.
"""
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


def _bits(t):
    return W.as_u16(t)


def _check_qk(mx, orc, x, token_idx=None):
    B, H, N, _ = x.shape
    BH = B * H
    codes, scales = mx.mxattn_rotate_quantize_qk(x)
    torch.cuda.synchronize()
    gc = L.qk_codes_logical(codes.cpu().numpy(), BH, N)
    gs_all = L.tiles_logical(scales.cpu().numpy(), BH, N)
    gs = gs_all[:, :N]
    # padded scale slots hold 127
    assert np.all(gs_all[:, N:] == 127)
    xb = _bits(x).reshape(BH, N, 128)
    if token_idx is None:
        oc, os_ = orc.rotate_quantize_qk(xb)
        assert np.array_equal(gc, oc), f"code mismatches: {(gc != oc).sum()}"
        assert np.array_equal(gs, os_), f"scale mismatches: {(gs != os_).sum()}"
    else:
        bh, n = token_idx
        oc, os_ = orc.rotate_quantize_qk(xb[bh, n])
        assert np.array_equal(gc[bh, n], oc), f"code mismatches: {(gc[bh, n] != oc).sum()}"
        assert np.array_equal(gs[bh, n], os_)


def _check_v(mx, orc, v, windows=None):
    B, H, N, _ = v.shape
    BH = B * H
    codes, scales = mx.mxattn_quantize_v(v)
    torch.cuda.synchronize()
    gc = L.v_codes_logical(codes.cpu().numpy(), BH, N)
    gsl = L.v_scales_logical(scales.cpu().numpy(), BH, N)
    vb = _bits(v).reshape(BH, N, 128)
    npad = ((N + 31) // 32) * 32
    raw = codes.cpu().numpy().reshape(BH, 128, npad // 2)
    if N % 32:
        # tokens past N in the last block are zero codes
        tail = L.unpack_nibbles(raw)[:, :, N:]
        assert np.all(tail == 0)
    if windows is None:
        oc, os_ = orc.quantize_v(vb)
        assert np.array_equal(gc, oc), f"code mismatches: {(gc != oc).sum()}"
        assert np.array_equal(gsl, os_), f"scale mismatches: {(gsl != os_).sum()}"
    else:
        for bh, t0, t1 in windows:
            assert t0 % 128 == 0
            oc, os_ = orc.quantize_v(vb[bh:bh + 1, t0:t1])
            assert np.array_equal(gc[bh, t0:t1], oc[0])
            assert np.array_equal(gsl[bh, :, t0 // 32:(t1 + 31) // 32], os_[0])


@pytest.mark.parametrize("name", ["tiny_outlier_512", "lognormal_4096"])
def test_quantizers_bitexact_full(mx, orc, name):
    q, k, v = W.generate(W.WORKLOADS[name], device="cuda")
    _check_qk(mx, orc, q)
    _check_qk(mx, orc, k)
    _check_v(mx, orc, v)


@pytest.mark.parametrize("N", [1, 31, 32, 100, 127, 128, 129, 300, 1000])
def test_quantizers_ragged_lengths(mx, orc, N):
    q, k, v = W.generate(W.WORKLOADS["tiny_outlier_512"], device="cuda", N=N, H=3, seed=N)
    _check_qk(mx, orc, q)
    _check_v(mx, orc, v)


def test_quantizers_special_values(mx, orc):
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    N = 384
    x = torch.randn((1, 2, N, 128), generator=g, device="cuda")
    x[0, 0, 0] = 0.0                              # all-zero token
    x[0, 0, 1, 32:64] = 0.0                       # all-zero block (V: zero channel block below)
    x[0, 0, 2] *= 1e30                            # huge magnitudes
    x[0, 0, 3] *= 1e-30                           # tiny magnitudes
    x[0, 0, 4] = -1e-39                           # bf16 subnormals, negative
    x[0, 0, 5, :] = -0.0                          # negative zeros
    x[0, 1, 6, 7] = 3.0e4                         # one spike
    x[0, 1, 7] = torch.linspace(-7.25, 7.25, 128, device="cuda")  # UOS boundary values
    x[0, 1, 64:96, 5] = 0.0                       # a zero V block in channel 5
    x[0, 1, 96:128, 9] = -1e-38
    xb = x.to(torch.bfloat16).contiguous()
    _check_qk(mx, orc, xb)
    _check_v(mx, orc, xb)


@pytest.mark.parametrize("name", ["wan_32760", "hunyuan_118800", "causal_lm_8192"])
def test_quantizers_full_size_sampled(mx, orc, name):
    w = W.WORKLOADS[name]
    q, k, v = W.generate(w, device="cuda")
    BH, N = w.B * w.H, w.N
    rng = np.random.default_rng(123)
    bh = rng.integers(0, BH, 3000)
    n = rng.integers(0, N, 3000)
    bh = np.concatenate([bh, np.arange(BH), np.arange(BH)])
    n = np.concatenate([n, np.full(BH, N - 1), np.zeros(BH, dtype=np.int64)])
    _check_qk(mx, orc, q, (bh, n))
    _check_qk(mx, orc, k, (bh, n))
    last = (N - 1) // 128 * 128
    windows = [(int(b), int(rng.integers(0, N // 128)) * 128, 0) for b in rng.integers(0, BH, 6)]
    windows = [(b, t0, t0 + 128) for b, t0, _ in windows] + [(BH - 1, last, N), (0, last, N)]
    _check_v(mx, orc, v, windows)
    del q, k, v
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,H,N", [(1, 1, 1), (1, 3, 31), (2, 3, 129), (1, 5, 300), (3, 7, 1000), (1, 2, 4096)])
def test_quantize_qkv_one_launch_equals_single_calls(mx, B, H, N):
    """Section 5.6's fused preprocessing: one launch writes exactly the bytes of the three single-tensor calls
    (ragged N, one to hundreds of interleaved tiles)."""
    q, k, v = W.generate(W.WORKLOADS["lognormal_4096"], device="cuda", B=B, H=H, N=N, seed=N + H)
    fused = mx.mxattn_quantize_qkv(q, k, v)
    single = (*mx.mxattn_rotate_quantize_qk(q), *mx.mxattn_rotate_quantize_qk(k), *mx.mxattn_quantize_v(v))
    mx.mxattn_check()
    for name, a, b in zip(("q_codes", "q_scales", "k_codes", "k_scales", "v_codes", "v_scales"), fused, single):
        assert torch.equal(a, b), name


def test_quantize_qkv_vs_oracle(mx, orc):
    q, k, v = W.generate(W.WORKLOADS["tiny_outlier_512"], device="cuda", N=333, H=3, seed=5)
    B, H, N, _ = q.shape
    qc, qs, kc, ks, vc, vs = (t.cpu().numpy() for t in mx.mxattn_quantize_qkv(q, k, v))
    mx.mxattn_check()
    for x, c, s_ in ((q, qc, qs), (k, kc, ks)):
        oc, os_ = orc.rotate_quantize_qk(_bits(x).reshape(B * H, N, 128))
        assert np.array_equal(L.qk_codes_logical(c, B * H, N), oc)
        assert np.array_equal(L.qk_scales_logical(s_, B * H, N), os_)
    oc, os_ = orc.quantize_v(_bits(v).reshape(B * H, N, 128))
    assert np.array_equal(L.v_codes_logical(vc, B * H, N), oc)
    assert np.array_equal(L.v_scales_logical(vs, B * H, N), os_)


def test_quantize_qkv_full_size_equals_single_calls(mx):
    """At the Wan-shaped size the benchmark times: the one-launch bytes equal the single calls' bytes (which the
    sampled oracle test above pins)."""
    w = W.WORKLOADS["wan_32760"]
    q, k, v = W.generate(w, device="cuda")
    fused = mx.mxattn_quantize_qkv(q, k, v)
    single = (*mx.mxattn_rotate_quantize_qk(q), *mx.mxattn_rotate_quantize_qk(k), *mx.mxattn_quantize_v(v))
    mx.mxattn_check()
    for a, b in zip(fused, single):
        assert torch.equal(a, b)
    del q, k, v, fused, single
    torch.cuda.empty_cache()
