"""Python binding of libmxattn, the sm_103a MXAttention forward (include/mxattn.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libmxattn.so``. The functions carry the names of the C entry
points, take PyTorch CUDA tensors (PyTorch provides device memory and the
current stream) and raise ``MxattnError`` when the library returns an error.
There is no CPU fallback: if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = [
    "MxattnError", "load", "mxattn_rotate_quantize_qk", "mxattn_quantize_v", "mxattn_quantize_qkv", "mxattn_forward",
    "mxattn_forward_dump_phat", "mxattn_forward_bf16", "mxattn_attention_host", "mxattn_workspace_bytes",
    "mxattn_check", "mxattn_set_debug_flags", "mxattn_attention", "qk_layout_sizes", "v_layout_sizes",
    "mxattn_attention_noalloc", "mxattn_attention_noalloc_max_scratch_bytes", "mxattn_nvfp4_quantize_qk",
    "mxattn_nvfp4_quantize_v", "mxattn_nvfp4_forward",
    "mxattn_nvfp4_forward_dump_phat",
]

D = 128
_lock = threading.Lock()
_lib = None

STATUS = {0: "MXATTN_OK", 1: "MXATTN_ERR_INVALID_ARG", 2: "MXATTN_ERR_UNSUPPORTED", 3: "MXATTN_ERR_CUDA",
          4: "MXATTN_ERR_TIMEOUT"}


class MxattnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the in-tree libmxattn.so."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise OSError(f"libmxattn.so not found at {path}; run mxfp4_precision_attention_gb300/build.py")
        lib = ctypes.CDLL(path)
        P, I64, I, U32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_size_t
        for name in ("mxattn_qk_codes_bytes", "mxattn_qk_scales_bytes", "mxattn_v_codes_bytes",
                     "mxattn_v_scales_bytes", "mxattn_workspace_bytes"):
            getattr(lib, name).argtypes = [I64, I64, I64]
            getattr(lib, name).restype = SZ
        lib.mxattn_rotate_quantize_qk.argtypes = [P, I64, I64, I64, I64, P, P, P]
        lib.mxattn_quantize_v.argtypes = [P, I64, I64, I64, I64, P, P, P]
        lib.mxattn_quantize_qkv.argtypes = [P, P, P, I64, I64, I64, I64, P, P, P, P, P, P, P]
        lib.mxattn_nvfp4_scales_bytes.argtypes = [I64, I64, I64]
        lib.mxattn_nvfp4_scales_bytes.restype = SZ
        lib.mxattn_nvfp4_quantize_qk.argtypes = [P, I64, I64, I64, I64, P, P, P, P]
        lib.mxattn_nvfp4_quantize_v.argtypes = [P, I64, I64, I64, I64, P, P, P, P]
        lib.mxattn_nvfp4_forward.argtypes = [P, P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, I, I, P, P]
        lib.mxattn_nvfp4_forward_dump_phat.argtypes = [P, P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, I, I, P, P,
                                                       P, P]
        lib.mxattn_forward.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I64, I, P, P]
        lib.mxattn_forward_dump_phat.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I64, I, P, P, P, P]
        lib.mxattn_forward_out_bf16.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I64, I, P, P]
        lib.mxattn_forward_bf16.argtypes = [P, P, P, I64, I64, I64, I64, I64, I, P, P]
        Dbl = ctypes.c_double
        lib.mxattn_quantize_qk_ex.argtypes = [P, I64, I64, I64, I64, I, Dbl, I, P, P, P]
        lib.mxattn_quantize_v_ex.argtypes = [P, I64, I64, I64, I64, I, Dbl, P, P, P]
        lib.mxattn_forward_ex.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I64, I, I, Dbl, I, P, P]
        lib.mxattn_attention_host.argtypes = [P, P, P, I64, I64, I64, I64, I, P, P, SZ, P]
        lib.mxattn_attention_noalloc.argtypes = [P, P, P, I64, I64, I64, I64, I, P, P]
        lib.mxattn_attention_noalloc.restype = I
        lib.mxattn_attention_noalloc_max_scratch_bytes.argtypes = []
        lib.mxattn_attention_noalloc_max_scratch_bytes.restype = SZ
        lib.mxattn_check.argtypes = [P]
        lib.mxattn_mxf4_mma_rate.argtypes = [I64, I, P, ctypes.POINTER(Dbl), P]
        lib.mxattn_set_debug_flags.argtypes = [U32]
        lib.mxattn_set_debug_flags.restype = None
        lib.mxattn_last_error.restype = ctypes.c_char_p
        for name in ("mxattn_rotate_quantize_qk", "mxattn_quantize_v", "mxattn_forward", "mxattn_forward_dump_phat",
                     "mxattn_forward_bf16", "mxattn_attention_host", "mxattn_check", "mxattn_quantize_qk_ex",
                     "mxattn_quantize_v_ex", "mxattn_forward_ex", "mxattn_mxf4_mma_rate",
                     "mxattn_forward_out_bf16"):
            getattr(lib, name).restype = I
        _lib = lib
        return lib


def _raise(st: int):
    if st != 0:
        raise MxattnError(st, (load().mxattn_last_error() or b"").decode())


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def _shape(x: torch.Tensor):
    if x.dim() != 4:
        raise ValueError("expected a [B, H, N, D] tensor")
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("expected a contiguous bf16 CUDA tensor")
    return x.shape


def _buf(t, nbytes: int, name: str, device=None, dtype=None) -> None:
    """A caller-supplied device buffer: a contiguous CUDA tensor on `device`, of
    `dtype` if given, holding at least `nbytes` bytes. Checked before any launch,
    so a wrong buffer raises here instead of reaching a kernel."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, not {t.dtype}")
    if t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes, {nbytes} needed")


def _elems(B: int, H: int, N: int) -> int:
    return max(B, 0) * max(H, 0) * max(N, 0) * D


def _check_mx_operands(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, v_bf16, B, H, N, causal,
                       scales_bytes=None):
    """The forward's quantized operands (and the bf16 V if given or needed) against B, H, N."""
    _buf(q_codes, 0, "q_codes")
    dev = q_codes.device
    nc, ns = qk_layout_sizes(B, H, N)
    vc, vs = v_layout_sizes(B, H, N)
    if scales_bytes is not None:
        ns = vs = scales_bytes
    for t, n, name in ((q_codes, nc, "q_codes"), (q_scales, ns, "q_scales"), (k_codes, nc, "k_codes"),
                       (k_scales, ns, "k_scales"), (v_codes, vc, "v_codes"), (v_scales, vs, "v_scales")):
        _buf(t, n, name, dev)
    if causal or v_bf16 is not None:
        _buf(v_bf16, 2 * _elems(B, H, N), "v_bf16", dev, torch.bfloat16)
    return dev


def _out(out, B, H, N, dtype, dev):
    if out is None:
        return torch.empty((max(B, 0), max(H, 0), max(N, 0), D), dtype=dtype, device=dev)
    _buf(out, _elems(B, H, N) * torch.empty(0, dtype=dtype).element_size(), "out", dev, dtype)
    return out


def qk_layout_sizes(B: int, H: int, N: int) -> tuple[int, int]:
    lib = load()
    return int(lib.mxattn_qk_codes_bytes(B, H, N)), int(lib.mxattn_qk_scales_bytes(B, H, N))


def v_layout_sizes(B: int, H: int, N: int) -> tuple[int, int]:
    lib = load()
    return int(lib.mxattn_v_codes_bytes(B, H, N)), int(lib.mxattn_v_scales_bytes(B, H, N))


def mxattn_rotate_quantize_qk(x: torch.Tensor, codes: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                              stream=None):
    """Hadamard rotation + UOS MXFP4 quantization of Q or K. Returns (codes, scales) uint8 tensors."""
    B, H, N, Dx = _shape(x)
    nc, ns = qk_layout_sizes(B, H, N)
    codes = torch.empty(nc, dtype=torch.uint8, device=x.device) if codes is None else codes
    scales = torch.empty(ns, dtype=torch.uint8, device=x.device) if scales is None else scales
    _buf(codes, nc, "codes", x.device)
    _buf(scales, ns, "scales", x.device)
    _raise(load().mxattn_rotate_quantize_qk(_ptr(x), B, H, N, Dx, _ptr(codes), _ptr(scales), _stream(stream)))
    return codes, scales


def mxattn_quantize_v(v: torch.Tensor, codes: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                      stream=None):
    """UOS MXFP4 quantization of V in 32-token blocks. Returns (codes, scales) uint8 tensors."""
    B, H, N, Dx = _shape(v)
    nc, ns = v_layout_sizes(B, H, N)
    codes = torch.empty(nc, dtype=torch.uint8, device=v.device) if codes is None else codes
    scales = torch.empty(ns, dtype=torch.uint8, device=v.device) if scales is None else scales
    _buf(codes, nc, "codes", v.device)
    _buf(scales, ns, "scales", v.device)
    _raise(load().mxattn_quantize_v(_ptr(v), B, H, N, Dx, _ptr(codes), _ptr(scales), _stream(stream)))
    return codes, scales


def mxattn_quantize_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out=None, stream=None):
    """Q and K rotated and quantized, V quantized, in one launch. Returns
    (q_codes, q_scales, k_codes, k_scales, v_codes, v_scales), the same bytes
    the three single-tensor calls write; `out` may supply those six buffers."""
    B, H, N, Dx = _shape(q)
    if _shape(k) != (B, H, N, Dx) or _shape(v) != (B, H, N, Dx):
        raise ValueError("q, k and v must have the same shape")
    if out is None:
        nc, ns = qk_layout_sizes(B, H, N)
        vc, vs = v_layout_sizes(B, H, N)
        out = tuple(torch.empty(n, dtype=torch.uint8, device=q.device) for n in (nc, ns, nc, ns, vc, vs))
    if len(out) != 6:
        raise ValueError("out must hold six buffers")
    nc, ns = qk_layout_sizes(B, H, N)
    vc, vs = v_layout_sizes(B, H, N)
    for t, n, name in zip(out, (nc, ns, nc, ns, vc, vs), ("q_codes", "q_scales", "k_codes", "k_scales", "v_codes",
                                                          "v_scales")):
        _buf(t, n, name, q.device)
    _raise(load().mxattn_quantize_qkv(_ptr(q), _ptr(k), _ptr(v), B, H, N, Dx, *(_ptr(t) for t in out),
                                      _stream(stream)))
    return tuple(out)


def mxattn_nvfp4_quantize_qk(x: torch.Tensor, stream=None):
    """NVFP4 Q/K quantization (no rotation). Returns (codes, scales, amax): uint8, uint8, fp32 [1]."""
    B, H, N, Dx = _shape(x)
    codes = torch.empty(qk_layout_sizes(B, H, N)[0], dtype=torch.uint8, device=x.device)
    scales = torch.empty(int(load().mxattn_nvfp4_scales_bytes(B, H, N)), dtype=torch.uint8, device=x.device)
    amax = torch.empty(1, dtype=torch.float32, device=x.device)
    _raise(load().mxattn_nvfp4_quantize_qk(_ptr(x), B, H, N, Dx, _ptr(codes), _ptr(scales), _ptr(amax),
                                           _stream(stream)))
    return codes, scales, amax


def mxattn_nvfp4_quantize_v(v: torch.Tensor, stream=None):
    """NVFP4 V quantization (16-token blocks). Returns (codes, scales, amax)."""
    B, H, N, Dx = _shape(v)
    codes = torch.empty(v_layout_sizes(B, H, N)[0], dtype=torch.uint8, device=v.device)
    scales = torch.empty(int(load().mxattn_nvfp4_scales_bytes(B, H, N)), dtype=torch.uint8, device=v.device)
    amax = torch.empty(1, dtype=torch.float32, device=v.device)
    _raise(load().mxattn_nvfp4_quantize_v(_ptr(v), B, H, N, Dx, _ptr(codes), _ptr(scales), _ptr(amax),
                                          _stream(stream)))
    return codes, scales, amax


def mxattn_nvfp4_forward(q, k, v, v_bf16, B: int, H: int, N: int, causal: bool = False, placement: int = 1,
                         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """NVFP4 forward; q, k, v are the (codes, scales, amax) triples of the NVFP4 quantizers.
    placement 1 (direct, the baseline) or 0 (PNQ). Returns fp32 [B, H, N, 128]."""
    sb = int(load().mxattn_nvfp4_scales_bytes(B, H, N))
    dev = _check_mx_operands(q[0], q[1], k[0], k[1], v[0], v[1], v_bf16, B, H, N, causal, scales_bytes=sb)
    for t, name in ((q[2], "q amax"), (k[2], "k amax"), (v[2], "v amax")):
        _buf(t, 4, name, dev, torch.float32)
    out = _out(out, B, H, N, torch.float32, dev)
    _raise(load().mxattn_nvfp4_forward(_ptr(q[0]), _ptr(q[1]), _ptr(q[2]), _ptr(k[0]), _ptr(k[1]), _ptr(k[2]),
                                       _ptr(v[0]), _ptr(v[1]), _ptr(v[2]), _ptr(v_bf16), B, H, N, D, int(causal),
                                       int(placement), _ptr(out), _stream(stream)))
    return out


def mxattn_nvfp4_forward_dump_phat(q, k, v, v_bf16, B: int, H: int, N: int, causal: bool = False,
                                   placement: int = 1, stream=None):
    """mxattn_nvfp4_forward plus every P^ tile: returns (out, phat_codes [B*H, N, NT*64],
    phat_scales [B*H, N, NT*8])."""
    sb = int(load().mxattn_nvfp4_scales_bytes(B, H, N))
    dev = _check_mx_operands(q[0], q[1], k[0], k[1], v[0], v[1], v_bf16, B, H, N, causal, scales_bytes=sb)
    for t, name in ((q[2], "q amax"), (k[2], "k amax"), (v[2], "v amax")):
        _buf(t, 4, name, dev, torch.float32)
    nt = (N + 127) // 128
    out = torch.empty((B, H, N, D), dtype=torch.float32, device=dev)
    pc = torch.zeros((B * H, N, nt * 64), dtype=torch.uint8, device=dev)
    ps = torch.zeros((B * H, N, nt * 8), dtype=torch.uint8, device=dev)
    _raise(load().mxattn_nvfp4_forward_dump_phat(_ptr(q[0]), _ptr(q[1]), _ptr(q[2]), _ptr(k[0]), _ptr(k[1]),
                                                 _ptr(k[2]), _ptr(v[0]), _ptr(v[1]), _ptr(v[2]), _ptr(v_bf16), B, H,
                                                 N, D, int(causal), int(placement), _ptr(out), _ptr(pc), _ptr(ps),
                                                 _stream(stream)))
    return out, pc, ps


def mxattn_forward(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, v_bf16, B: int, H: int, N: int,
                   causal: bool = False, out: torch.Tensor | None = None, stream=None,
                   out_dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """MXFP4 attention forward with PNQ on quantized operands. Returns [B, H, N, 128]
    in `out_dtype`: float32, or bfloat16 (the float32 result rounded to nearest even)."""
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
    dev = _check_mx_operands(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, v_bf16, B, H, N, causal)
    out = _out(out, B, H, N, out_dtype, dev)
    fn = load().mxattn_forward if out_dtype == torch.float32 else load().mxattn_forward_out_bf16
    _raise(fn(_ptr(q_codes), _ptr(q_scales), _ptr(k_codes), _ptr(k_scales), _ptr(v_codes),
              _ptr(v_scales), _ptr(v_bf16), B, H, N, D, int(causal), _ptr(out), _stream(stream)))
    return out


def mxattn_forward_dump_phat(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, v_bf16, B: int, H: int, N: int,
                             causal: bool = False, stream=None):
    """Diagnostic forward that also returns every P^ tile (codes [B*H, N, NT*64], scales [B*H, N, NT*4])."""
    dev = _check_mx_operands(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, v_bf16, B, H, N, causal)
    NT = (N + 127) // 128
    out = torch.empty((B, H, N, D), dtype=torch.float32, device=dev)
    pc = torch.zeros((B * H, N, NT * 64), dtype=torch.uint8, device=dev)
    ps = torch.zeros((B * H, N, NT * 4), dtype=torch.uint8, device=dev)
    _raise(load().mxattn_forward_dump_phat(_ptr(q_codes), _ptr(q_scales), _ptr(k_codes), _ptr(k_scales),
                                           _ptr(v_codes), _ptr(v_scales), _ptr(v_bf16), B, H, N, D, int(causal),
                                           _ptr(out), _ptr(pc), _ptr(ps), _stream(stream)))
    return out, pc, ps


# Ablation switches (include/mxattn.h: mxattn_scale_rule, mxattn_placement)
RULE_UOS, RULE_OCP, RULE_TFS, RULE_CEIL = 0, 1, 2, 3
PLACE_PNQ, PLACE_DIRECT = 0, 1


def mxattn_quantize_qk_ex(x: torch.Tensor, rule: int = RULE_UOS, rotate: bool = True, qmax: float = 7.25,
                          codes: torch.Tensor | None = None, scales: torch.Tensor | None = None, stream=None):
    """Q/K quantization with a chosen scale rule (qmax for RULE_CEIL) and optional rotation.
    Returns (codes, scales)."""
    B, H, N, Dx = _shape(x)
    nc, ns = qk_layout_sizes(B, H, N)
    codes = torch.empty(nc, dtype=torch.uint8, device=x.device) if codes is None else codes
    scales = torch.empty(ns, dtype=torch.uint8, device=x.device) if scales is None else scales
    _buf(codes, nc, "codes", x.device)
    _buf(scales, ns, "scales", x.device)
    _raise(load().mxattn_quantize_qk_ex(_ptr(x), B, H, N, Dx, int(rule), float(qmax), int(bool(rotate)),
                                        _ptr(codes), _ptr(scales), _stream(stream)))
    return codes, scales


def mxattn_quantize_v_ex(v: torch.Tensor, rule: int = RULE_UOS, qmax: float = 7.25, codes: torch.Tensor | None = None,
                         scales: torch.Tensor | None = None, stream=None):
    """V quantization with a chosen scale rule (qmax for RULE_CEIL). Returns (codes, scales)."""
    B, H, N, Dx = _shape(v)
    nc, ns = v_layout_sizes(B, H, N)
    codes = torch.empty(nc, dtype=torch.uint8, device=v.device) if codes is None else codes
    scales = torch.empty(ns, dtype=torch.uint8, device=v.device) if scales is None else scales
    _buf(codes, nc, "codes", v.device)
    _buf(scales, ns, "scales", v.device)
    _raise(load().mxattn_quantize_v_ex(_ptr(v), B, H, N, Dx, int(rule), float(qmax), _ptr(codes), _ptr(scales),
                                       _stream(stream)))
    return codes, scales


def mxattn_forward_ex(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, v_bf16, B: int, H: int, N: int,
                      causal: bool = False, p_rule: int = RULE_UOS, placement: int = PLACE_PNQ,
                      p_qmax: float = 7.25, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Forward with the P~ scale rule and the l placement as switches. Returns fp32 [B, H, N, 128]."""
    dev = _check_mx_operands(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, v_bf16, B, H, N, causal)
    out = _out(out, B, H, N, torch.float32, dev)
    _raise(load().mxattn_forward_ex(_ptr(q_codes), _ptr(q_scales), _ptr(k_codes), _ptr(k_scales), _ptr(v_codes),
                                    _ptr(v_scales), _ptr(v_bf16), B, H, N, D, int(causal), int(p_rule),
                                    float(p_qmax), int(placement), _ptr(out), _stream(stream)))
    return out


def mxattn_forward_bf16(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                        out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """BF16 tcgen05 attention forward (comparison path): q [B, H, Nq, 128], k and v
    [B, H, Nk, 128]; causal means key j is visible to query i iff j <= i.
    Returns fp32 [B, H, Nq, 128]."""
    B, H, Nq, Dx = _shape(q)
    Nk = _shape(k)[2]
    if _shape(k) != (B, H, Nk, Dx) or _shape(v) != (B, H, Nk, Dx):
        raise ValueError("k and v must be [B, H, Nk, D] with q's B, H and D")
    out = _out(out, B, H, Nq, torch.float32, q.device)
    _raise(load().mxattn_forward_bf16(_ptr(q), _ptr(k), _ptr(v), B, H, Nq, Nk, Dx, int(causal), _ptr(out),
                                      _stream(stream)))
    return out


def mxattn_workspace_bytes(B: int, H: int, N: int) -> int:
    return int(load().mxattn_workspace_bytes(B, H, N))


def mxattn_attention_host(q_host: torch.Tensor, k_host: torch.Tensor, v_host: torch.Tensor, causal: bool,
                          out_host: torch.Tensor, workspace: torch.Tensor, stream=None) -> torch.Tensor:
    """Whole forward from host (preferably pinned) bf16 tensors into a host fp32 tensor."""
    if q_host.dim() != 4:
        raise ValueError("expected [B, H, N, D] host tensors")
    B, H, N, Dx = q_host.shape
    for t, dt, name in ((q_host, torch.bfloat16, "q_host"), (k_host, torch.bfloat16, "k_host"),
                        (v_host, torch.bfloat16, "v_host"), (out_host, torch.float32, "out_host")):
        if t.is_cuda or not t.is_contiguous() or t.dtype != dt or tuple(t.shape) != (B, H, N, Dx):
            raise ValueError(f"{name} must be a contiguous CPU {dt} tensor of shape {(B, H, N, Dx)}")
    _buf(workspace, 0, "workspace")
    _raise(load().mxattn_attention_host(_ptr(q_host), _ptr(k_host), _ptr(v_host), B, H, N, Dx, int(causal),
                                        _ptr(out_host), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream)))
    return out_host


def mxattn_attention_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool, out: torch.Tensor,
                             stream=None) -> torch.Tensor:
    """Whole forward using the library's fixed device scratch (no allocation by the library or here)."""
    B, H, N, Dx = _shape(q)
    if _shape(k) != (B, H, N, Dx) or _shape(v) != (B, H, N, Dx):
        raise ValueError("q, k and v must have the same shape")
    if q.device.index != torch.cuda.current_device():
        raise ValueError(f"q is on {q.device} but the current device is cuda:{torch.cuda.current_device()}; "
                         "the library's scratch and launches belong to the current device")
    _buf(k, 0, "k", q.device)
    _buf(v, 0, "v", q.device)
    _buf(out, 4 * _elems(B, H, N), "out", q.device, torch.float32)
    _raise(load().mxattn_attention_noalloc(_ptr(q), _ptr(k), _ptr(v), B, H, N, Dx, int(causal), _ptr(out),
                                           _stream(stream)))
    return out


def mxattn_attention_noalloc_max_scratch_bytes() -> int:
    return int(load().mxattn_attention_noalloc_max_scratch_bytes())


def mxattn_check(stream=None) -> None:
    """Synchronize and raise MxattnError if a kernel reported an expired bounded wait."""
    _raise(load().mxattn_check(_stream(stream)))


def mxattn_mxf4_mma_rate(iters: int, n: int = 256, out: torch.Tensor | None = None, stream=None) -> float:
    """Launch the tensor-core rate probe (one CTA per SM, `iters` pairs of
    M128 Nn K64 kind::mxf4 MMAs each, n = 128 or 256) and return the launch's
    FLOP count. `out`, a device float32 [128, n], receives CTA 0's accumulator."""
    if out is not None:
        _buf(out, 4 * 128 * n, "out", dtype=torch.float32)
    flops = ctypes.c_double(0.0)
    _raise(load().mxattn_mxf4_mma_rate(int(iters), int(n), _ptr(out) if out is not None else None,
                                       ctypes.byref(flops), _stream(stream)))
    return flops.value


def mxattn_set_debug_flags(flags: int) -> None:
    load().mxattn_set_debug_flags(int(flags))


def mxattn_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False, stream=None):
    """The whole hot path on device tensors: rotate+quantize Q and K and quantize V
    (one launch), then the forward."""
    B, H, N, _ = _shape(q)
    qc, qs, kc, ks, vc, vs = mxattn_quantize_qkv(q, k, v, stream=stream)
    return mxattn_forward(qc, qs, kc, ks, vc, vs, v, B, H, N, causal=causal, stream=stream)
