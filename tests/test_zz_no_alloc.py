"""mxattn_attention_noalloc: the whole forward for callers that cannot allocate
device memory (for example an op behind a plugin interface that is handed only
its input and output buffers). It keeps its quantized intermediates in one
fixed device array of the library instead of caller-provided buffers.

Checked through the C ABI against the existing entry points
(mxattn_rotate_quantize_qk, mxattn_quantize_v, mxattn_forward with caller
buffers) on two calls in a row with different inputs (the shared array keeps
the previous call's contents, so stale data would show). Both paths run the
same deterministic kernels on the same bytes, so the outputs must be equal
bit for bit (a stricter check than the oracle tolerance, which the test also
states). This file is collected last.
"""
import math

import numpy as np
import pytest
import torch

from mxfp4_precision_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_REL_RMS = 2e-3


@pytest.fixture(scope="module")
def mx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mxfp4_precision_attention_gb300 as m

    m.load()
    return m


def _existing_path(mx, q, k, v, causal):
    B, H, N, _ = q.shape
    qc, qs = mx.mxattn_rotate_quantize_qk(q)
    kc, ks = mx.mxattn_rotate_quantize_qk(k)
    vc, vs = mx.mxattn_quantize_v(v)
    out = mx.mxattn_forward(qc, qs, kc, ks, vc, vs, v, B, H, N, causal=causal)
    mx.mxattn_check()
    return out


def _close(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    rms = math.sqrt(float(np.mean(b ** 2)))
    return float(np.abs(a - b).max()) <= TOL_REL_RMS * rms


def test_noalloc_matches_existing_entry_points_twice(mx):
    cases = [
        (W.generate(W.WORKLOADS["lognormal_4096"], device="cuda", H=4, N=4096), False),
        (W.generate(W.WORKLOADS["causal_lm_8192"], device="cuda", B=1, H=3, N=1000, seed=11), True),
    ]
    for (q, k, v), causal in cases:
        ref = _existing_path(mx, q, k, v, causal)
        out = torch.full_like(ref, float("nan"))
        mx.mxattn_attention_noalloc(q, k, v, causal, out)
        mx.mxattn_check()
        assert _close(out, ref)
        assert torch.equal(out, ref)


def test_noalloc_rejects_problems_beyond_its_scratch(mx):
    limit = mx.mxattn_attention_noalloc_max_scratch_bytes()
    assert limit == 32 << 20
    lib = mx.load()
    # NULL pointers: the size check rejects the problem first, and should that
    # order ever change, the NULL check still returns before any launch
    st = lib.mxattn_attention_noalloc(None, None, None, 1, 64, 32768, 128, 0, None, None)
    assert st == 2
    assert b"scratch" in lib.mxattn_last_error()
