"""GPU parity of the NVFP4 comparison path against the oracle, through the C ABI.

NVFP4 as "MXAttention" describes it (section 1: 16-element blocks, E4M3 block
scales, a tensor-level scale) and its direct baseline (section 5.2: Q, K, V and
P~ quantized, no smoothing, no softmax-path scaling), with the oracle's
readings N1-N6:
  * quantizers: the tensor maximum, every E2M1 code and every E4M3 scale byte
    equal the oracle's (bit-exact; ragged N, special values);
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
