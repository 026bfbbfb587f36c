"""The C-ABI library builds for sm_103a, loads, exports every symbol that
include/mxattn.h declares, and rejects invalid arguments on the host before
touching the GPU (so these run on a CPU-only machine)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxattn.h")


@pytest.fixture(scope="module")
def lib():
    import mxfp4_precision_attention_gb300 as mx

    return mx.load()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mxattn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_entry_points():
    names = _declared()
    for required in ["mxattn_rotate_quantize_qk", "mxattn_quantize_v", "mxattn_forward", "mxattn_forward_bf16",
                     "mxattn_check", "mxattn_last_error"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from mxfp4_precision_attention_gb300 import build

    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\b(mxattn_[a-z0-9_]+)\b", out))
    for name in _declared():
        assert name in exported, name
        assert hasattr(lib, name)
    # nothing else leaks out under the mxattn_ prefix
    assert exported == set(_declared())


def test_size_queries(lib):
    assert lib.mxattn_qk_codes_bytes(1, 2, 512) == 2 * 512 * 64
    assert lib.mxattn_qk_scales_bytes(1, 2, 512) == 2 * 4 * 512
    assert lib.mxattn_qk_scales_bytes(1, 1, 129) == 2 * 512
    assert lib.mxattn_v_codes_bytes(1, 1, 100) == 128 * 128 // 2
    assert lib.mxattn_v_codes_bytes(1, 40, 32760) == 40 * 128 * 32768 // 2
    assert lib.mxattn_v_scales_bytes(4, 32, 8192) == 128 * 64 * 512
    assert lib.mxattn_qk_codes_bytes(-1, 1, 1) == 0


def _err(lib):
    return lib.mxattn_last_error().decode()


def test_invalid_arguments_rejected_on_host(lib):
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: validation fails first
    odd = ctypes.c_void_p(0x10008)
    # unsupported head dim
    assert lib.mxattn_rotate_quantize_qk(fake, 1, 1, 128, 64, fake, fake, None) == 2
    assert "128" in _err(lib)
    # null pointers
    assert lib.mxattn_rotate_quantize_qk(None, 1, 1, 128, 128, fake, fake, None) == 1
    assert lib.mxattn_quantize_v(fake, 1, 1, 128, 128, None, fake, None) == 1
    # misaligned
    assert lib.mxattn_quantize_v(odd, 1, 1, 128, 128, fake, fake, None) == 1
    assert "aligned" in _err(lib)
    # negative sizes, too many heads
    assert lib.mxattn_forward_bf16(fake, fake, fake, 1, -1, 128, 128, 128, 0, fake, None) == 1
    assert lib.mxattn_forward_bf16(fake, fake, fake, 300, 300, 128, 128, 128, 0, fake, None) == 2
    assert lib.mxattn_forward_bf16(fake, fake, fake, 1, 1, 128, -1, 128, 0, fake, None) == 1
    assert lib.mxattn_forward_bf16(fake, fake, fake, 1, 1, 128, 0, 128, 0, fake, None) == 1
    assert "Nk=0" in _err(lib)
    # overlapping outputs
    a = ctypes.c_void_p(0x100000)
    assert lib.mxattn_rotate_quantize_qk(a, 1, 1, 128, 128, ctypes.c_void_p(0x100000 + 4096), fake, None) == 1
    # single-launch Q/K/V quantizer: misaligned, overlapping outputs, output over an input
    big9 = [ctypes.c_void_p(0x1000000 * (i + 1)) for i in range(9)]
    assert lib.mxattn_quantize_qkv(*big9[:3], 1, 1, 128, 128, *big9[3:8], odd, None) == 1
    assert "aligned" in _err(lib)
    assert lib.mxattn_quantize_qkv(*big9[:3], 1, 1, 128, 128, *big9[3:8], big9[7], None) == 1
    assert "overlap" in _err(lib)
    assert lib.mxattn_quantize_qkv(*big9[:3], 1, 1, 128, 128, big9[1], *big9[4:9], None) == 1
    assert lib.mxattn_quantize_qkv(*big9[:3], 1, 1, 128, 64, *big9[3:9], None) == 2
    # causal needs the bf16 V
    big = [ctypes.c_void_p(0x1000000 * (i + 1)) for i in range(8)]
    assert lib.mxattn_forward(*big[:6], None, 1, 1, 128, 128, 1, big[6], None) == 1
    assert "v_bf16" in _err(lib)
    assert lib.mxattn_forward(*big[:6], None, 1, 1, 128, 128, 2, big[6], None) == 1
    assert lib.mxattn_forward_out_bf16(*big[:6], big[7], 1, 1, 128, 128, 2, big[6], None) == 1
    assert lib.mxattn_forward_out_bf16(*big[:6], None, 1, 1, 128, 128, 1, big[6], None) == 1
    # dump needs both buffers
    assert lib.mxattn_forward_dump_phat(*big[:6], None, 1, 1, 128, 128, 0, big[6], big[7], None, None) == 1
    # host entry: workspace too small / misaligned
    assert lib.mxattn_attention_host(fake, fake, fake, 1, 1, 128, 128, 0, fake, big[0], 16, None) == 1
    assert lib.mxattn_attention_host(fake, fake, fake, 1, 1, 128, 128, 0, fake, ctypes.c_void_p(0x1000010),
                                     1 << 30, None) == 1
    # tensor-core rate probe: iteration count out of range, misaligned accumulator buffer
    assert lib.mxattn_mxf4_mma_rate(0, 256, None, None, None) == 1
    assert lib.mxattn_mxf4_mma_rate((1 << 27) + 1, 256, None, None, None) == 1
    assert "iters" in _err(lib)
    assert lib.mxattn_mxf4_mma_rate(10, 192, None, None, None) == 1
    assert lib.mxattn_mxf4_mma_rate(10, 256, ctypes.c_void_p(0x10002), None, None) == 1


def test_empty_problem_is_a_no_op(lib):
    # N = 0 or B*H = 0: OK and nothing launched (no CUDA call is made)
    assert lib.mxattn_rotate_quantize_qk(None, 1, 1, 0, 128, None, None, None) == 0
    assert lib.mxattn_quantize_v(None, 0, 4, 100, 128, None, None, None) == 0
    assert lib.mxattn_forward(None, None, None, None, None, None, None, 1, 1, 0, 128, 1, None, None) == 0
    assert lib.mxattn_forward_bf16(None, None, None, 1, 0, 10, 10, 128, 0, None, None) == 0
    assert lib.mxattn_forward_bf16(None, None, None, 1, 1, 0, 10, 128, 0, None, None) == 0
    assert lib.mxattn_quantize_qkv(None, None, None, 1, 1, 0, 128, None, None, None, None, None, None, None) == 0


def test_variant_switches_rejected_on_host(lib):
    """Out-of-range rule / rotate / placement switches of the ablation entry points."""
    big = [ctypes.c_void_p(0x1000000 * (i + 1)) for i in range(8)]
    assert lib.mxattn_quantize_qk_ex(big[0], 1, 1, 128, 128, 4, 7.25, 1, big[1], big[2], None) == 1
    assert "rule" in _err(lib)
    assert lib.mxattn_quantize_qk_ex(big[0], 1, 1, 128, 128, 3, 8.5, 1, big[1], big[2], None) == 1
    assert "qmax" in _err(lib)
    assert lib.mxattn_quantize_qk_ex(big[0], 1, 1, 128, 128, 3, 4.0, 1, big[1], big[2], None) == 1
    assert lib.mxattn_quantize_qk_ex(big[0], 1, 1, 128, 128, 0, 7.25, 2, big[1], big[2], None) == 1
    assert "rotate" in _err(lib)
    assert lib.mxattn_quantize_v_ex(big[0], 1, 1, 128, 128, -1, 7.25, big[1], big[2], None) == 1
    assert lib.mxattn_quantize_v_ex(big[0], 1, 1, 128, 128, 3, float("nan"), big[1], big[2], None) == 1
    assert lib.mxattn_forward_ex(*big[:6], None, 1, 1, 128, 128, 0, 4, 7.25, 0, big[6], None) == 1
    assert "p_rule" in _err(lib)
    assert lib.mxattn_forward_ex(*big[:6], None, 1, 1, 128, 128, 0, 0, 7.25, 2, big[6], None) == 1
    assert "placement" in _err(lib)
    # causal = 2 (prefix re-quantized diagonal block) exists only in mxattn_forward_ex
    assert lib.mxattn_forward(*big[:6], big[7], 1, 1, 128, 128, 2, big[6], None) == 1
    assert "causal" in _err(lib)
    assert lib.mxattn_forward_ex(*big[:6], big[7], 1, 1, 128, 128, 3, 0, 7.25, 0, big[6], None) == 1
    # empty problems stay no-ops through the variant calls too
    assert lib.mxattn_quantize_qk_ex(None, 1, 1, 0, 128, 1, 7.25, 0, None, None, None) == 0


def test_binding_rejects_wrong_buffers_before_any_launch():
    """The Python binding checks caller-supplied buffers (device, dtype, size)
    before calling into the library; CPU tensors where device buffers belong
    are refused here, on a machine without a GPU."""
    import torch

    import mxfp4_precision_attention_gb300 as mx

    u8 = torch.zeros(64, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA"):
        mx.mxattn_forward(u8, u8, u8, u8, u8, u8, None, 1, 1, 128)
    with pytest.raises(ValueError, match="CUDA"):
        mx.mxattn_mxf4_mma_rate(10, out=torch.zeros(128 * 256))
    q = torch.zeros((1, 1, 128, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="out_host"):
        mx.mxattn_attention_host(q, q, q, False, torch.zeros((1, 1, 128, 128), dtype=torch.float16), u8)
    with pytest.raises(ValueError, match="k_host"):
        mx.mxattn_attention_host(q, q.float(), q, False, torch.zeros((1, 1, 128, 128)), u8)
