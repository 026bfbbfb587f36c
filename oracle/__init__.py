"""MXAttention CPU oracle -- TEST INFRASTRUCTURE ONLY.

A plain float64 restatement of the MXAttention forward pass ("MXAttention:
Data-Free Optimal Scaling and Pre-Normalization Quantization for MXFP4
Attention", arXiv 2607.24377, Algorithms 1 and 2, Eqs. 1-18 and 44-52, with the
causal constraint of the MatX note "leaky quantization"). Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import it;
the product path never does. It shares no code with the CUDA kernels.

The arithmetic lives in ``mxattn_oracle.c`` (compiled on first use with gcc,
``-ffp-contract=off`` so that the binary32 Hadamard stage is evaluated exactly
as written). This module only marshals numpy arrays.

All layouts here are *logical*: codes one per byte, scales as biased E8M0
bytes (e + 127), Q/K scales ``[rows, 4]``, V codes ``[BH, N, 128]`` token-major
and V scales ``[BH, 128, ceil(N/32)]``.

Scale rules: 0 = UOS (ceil, Q_max = 7.25), 1 = OCP floor, 2 = TFS (ceil, 6),
3 = ceil with a given Q_max q in (4, 8] (the Q_max sweep of section 5.5.1).

NVFP4 comparison format (section 1 and the NVFP4 baseline of section 5.2):
16-element blocks, E4M3 block scales and a per-tensor encode factor
e_t = 2688 / amax (readings N1-N6 in ``mxattn_oracle.c``). NVFP4 Q/K scales
are ``[rows, 8]``, V scales ``[BH, 128, ceil(N/16)]`` (E4M3 bytes).

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against values and identities the pages fix (see the header of each test).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxattn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

UOS, OCP, TFS, CEIL_Q = 0, 1, 2, 3
PNQ, DIRECT = 0, 1
D = 128
BLOCK = 32
BC = 128


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (OpenMP if available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:6] + ["-fopenmp"] + base[6:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            lib.orc_e2m1_value.argtypes = [I]
            lib.orc_e2m1_value.restype = ctypes.c_double
            lib.orc_e2m1_code.argtypes = [ctypes.c_double]
            lib.orc_e2m1_code.restype = I
            lib.orc_scale_exponent.argtypes = [ctypes.c_double, I]
            lib.orc_scale_exponent.restype = I
            lib.orc_scale_exponent_q.argtypes = [ctypes.c_double, I, ctypes.c_double]
            lib.orc_scale_exponent_q.restype = I
            lib.orc_uos_qmax.argtypes = []
            lib.orc_uos_qmax.restype = ctypes.c_double
            lib.orc_hadamard_fp32.argtypes = [P, P]
            Dbl = ctypes.c_double
            lib.orc_rotate_quantize_qk.argtypes = [P, I64, I, Dbl, I, P, P]
            lib.orc_quantize_v.argtypes = [P, I64, I64, I, Dbl, P, P]
            lib.orc_online_softmax.argtypes = [P, P, I64, P, P, P, I64, I, I, I, I, Dbl, I, P, P, P, P]
            lib.orc_forward.argtypes = [P, P, P, P, P, P, P, I64, I64, I, I, I, Dbl, I, I, P, I64, P, P, P, P]
            lib.orc_forward.restype = I
            lib.orc_sdpa.argtypes = [P, P, P, I64, I64, I, P, I64, P]
            lib.orc_rowsum_parts.argtypes = [P, I64, I64, I, Dbl, P]
            lib.orc_e4m3_value.argtypes = [I]
            lib.orc_e4m3_value.restype = ctypes.c_double
            lib.orc_e4m3_code.argtypes = [ctypes.c_double]
            lib.orc_e4m3_code.restype = I
            lib.orc_nvfp4_encode.argtypes = [ctypes.c_float]
            lib.orc_nvfp4_encode.restype = ctypes.c_float
            lib.orc_nvfp4_quantize_qk.argtypes = [P, I64, P, P, P]
            lib.orc_nvfp4_quantize_v.argtypes = [P, I64, I64, P, P, P]
            F32 = ctypes.c_float
            lib.orc_forward_nvfp4.argtypes = [P, P, F32, P, P, F32, P, P, F32, P, I64, I64, I, I, I, P, I64, P, P, P,
                                              P, P]
            lib.orc_forward_nvfp4.restype = I
            lib.orc_num_threads.restype = I
            _lib = lib
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().orc_num_threads())


def uos_qmax() -> float:
    return float(_load().orc_uos_qmax())


def e2m1_value(code: int) -> float:
    return float(_load().orc_e2m1_value(int(code)))


def e2m1_code(v) -> np.ndarray:
    """Elementwise E2M1 code (round to nearest, ties to even, saturate at 6)."""
    lib = _load()
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    flat_in, flat_out = v.reshape(-1), out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = lib.orc_e2m1_code(float(flat_in[i]))
    return out


def scale_exponent(M: float, rule: int = UOS, q: float = 7.25) -> int:
    """Block scale exponent of a maximum M > 0 under `rule` (q is used by CEIL_Q)."""
    return int(_load().orc_scale_exponent_q(float(M), int(rule), float(q)))


def hadamard_fp32(x_u16: np.ndarray) -> np.ndarray:
    """Binary32 rotation of bf16 rows ``[..., 128]`` (given as uint16 bit patterns)."""
    lib = _load()
    x = _c(x_u16, np.uint16).reshape(-1, D)
    y = np.empty(x.shape, dtype=np.float32)
    for r in range(x.shape[0]):
        lib.orc_hadamard_fp32(_p(x[r]), _p(y[r]))
    return y.reshape(np.shape(x_u16))


def rotate_quantize_qk(x_u16: np.ndarray, rule: int = UOS, rotate: bool = True, q: float = 7.25):
    """Algorithm 2 (section 4.3), the rotation and Q/K quantization steps. ``x_u16``: bf16 bits ``[..., 128]``.

    Returns (codes ``[..., 128]`` uint8, scales ``[..., 4]`` uint8)."""
    lib = _load()
    x = _c(x_u16, np.uint16).reshape(-1, D)
    rows = x.shape[0]
    codes = np.empty((rows, D), dtype=np.uint8)
    scales = np.empty((rows, D // BLOCK), dtype=np.uint8)
    lib.orc_rotate_quantize_qk(_p(x), rows, int(rule), float(q), int(bool(rotate)), _p(codes), _p(scales))
    lead = np.shape(x_u16)[:-1]
    return codes.reshape(*lead, D), scales.reshape(*lead, D // BLOCK)


def quantize_v(v_u16: np.ndarray, rule: int = UOS, q: float = 7.25):
    """Algorithm 2 (section 4.3), the V quantization step, on ``[BH, N, 128]`` bf16 bits.

    Returns (codes ``[BH, N, 128]``, scales ``[BH, 128, ceil(N/32)]``)."""
    lib = _load()
    v = _c(v_u16, np.uint16)
    BH, N, _ = v.shape
    nblk = (N + BLOCK - 1) // BLOCK
    codes = np.empty((BH, N, D), dtype=np.uint8)
    scales = np.empty((BH, D, nblk), dtype=np.uint8)
    lib.orc_quantize_v(_p(v), BH, N, int(rule), float(q), _p(codes), _p(scales))
    return codes, scales


def online_softmax(q_rows, row_tok, K, V, Vraw=None, *, causal=False, quant_p=True, placement=PNQ,
                   p_rule=UOS, p_q=7.25, bc=BC, want_phat=False):
    """Algorithm 2 (section 4.3), the tiled online-softmax loop (Eqs. 2-8, 44-48), on real-valued inputs (float64).

    ``q_rows``: ``[R, 128]``; ``row_tok``: token index of each row; ``K, V``:
    ``[N, 128]``. Returns dict with ``out``, ``ell`` and optionally ``phat``
    ``[R, ntiles*bc]`` and ``mhist`` ``[R, ntiles]``."""
    lib = _load()
    q = _c(q_rows, np.float64).reshape(-1, D)
    tok = _c(row_tok, np.int64).reshape(-1)
    K = _c(K, np.float64)
    V = _c(V, np.float64)
    Vr = None if Vraw is None else _c(Vraw, np.float64)
    N = K.shape[0]
    R = q.shape[0]
    ntiles = (N + bc - 1) // bc
    out = np.empty((R, D))
    ell = np.empty(R)
    phat = np.zeros((R, ntiles * bc)) if want_phat else None
    mhist = np.full((R, ntiles), np.nan) if want_phat else None
    lib.orc_online_softmax(_p(q), _p(tok), R, _p(K), _p(V), _p(Vr), N, int(causal), int(quant_p),
                           int(placement), int(p_rule), float(p_q), int(bc), _p(out), _p(ell), _p(phat), _p(mhist))
    res = {"out": out, "ell": ell}
    if want_phat:
        res["phat"] = phat
        res["mhist"] = mhist
    return res


def forward(qc, qs, kc, ks, vc, vs, rows, *, vraw_u16=None, causal=False, placement=PNQ, p_rule=UOS,
            p_q=7.25, quant_p=True, bc=BC, want_phat=False):
    """Alg. 2 on quantized tensors in the oracle's logical layouts.

    ``rows``: ``[R, 2]`` int array of (bh, token). Returns dict as
    :func:`online_softmax`."""
    lib = _load()
    qc = _c(qc, np.uint8)
    qs = _c(qs, np.uint8)
    kc = _c(kc, np.uint8)
    ks = _c(ks, np.uint8)
    vc = _c(vc, np.uint8)
    vs = _c(vs, np.uint8)
    BH, N, _ = qc.shape
    vr = None if vraw_u16 is None else _c(vraw_u16, np.uint16)
    if causal and vr is None:
        raise ValueError("causal forward needs the unquantized V (vraw_u16)")
    rows = _c(rows, np.int64).reshape(-1, 2)
    R = rows.shape[0]
    ntiles = (N + bc - 1) // bc
    out = np.empty((R, D))
    ell = np.empty(R)
    phat = np.zeros((R, ntiles * bc)) if want_phat else None
    mhist = np.full((R, ntiles), np.nan) if want_phat else None
    rc = lib.orc_forward(_p(qc), _p(qs), _p(kc), _p(ks), _p(vc), _p(vs), _p(vr), BH, N, int(causal),
                         int(placement), int(p_rule), float(p_q), int(quant_p), int(bc), _p(rows), R, _p(out), _p(ell),
                         _p(phat), _p(mhist))
    if rc != 0:
        raise RuntimeError(f"orc_forward failed with code {rc}")
    res = {"out": out, "ell": ell}
    if want_phat:
        res["phat"] = phat
        res["mhist"] = mhist
    return res


def sdpa(q_u16, k_u16, v_u16, rows, *, causal=False):
    """Unquantized float64 attention, Eq. 1, on bf16 ``[BH, N, 128]`` inputs."""
    lib = _load()
    q = _c(q_u16, np.uint16)
    k = _c(k_u16, np.uint16)
    v = _c(v_u16, np.uint16)
    BH, N, _ = q.shape
    rows = _c(rows, np.int64).reshape(-1, 2)
    out = np.empty((rows.shape[0], D))
    lib.orc_sdpa(_p(q), _p(k), _p(v), BH, N, int(causal), _p(rows), rows.shape[0], _p(out))
    return out


def rowsum_parts(P, rule: int = UOS, q: float = 7.25) -> np.ndarray:
    """Row-sum diagnostic of section 5.5.2 (Fig. 7 B; reading D1 in mxattn_oracle.c):
    each row of the nonnegative ``P [R, N]`` quantized in 32-key blocks under
    ``rule``. Returns ``[R, 5]``: sum Q(P), then the zeroing, saturation,
    downward- and upward-rounding parts of sum(Q(P) - P)."""
    lib = _load()
    P = _c(P, np.float64)
    R, N = P.shape
    out = np.empty((R, 5))
    lib.orc_rowsum_parts(_p(P), R, N, int(rule), float(q), _p(out))
    return out


def dequant_qk(codes, scales):
    """Logical Q/K codes+scales -> float64 values ``[..., 128]``."""
    vals = np.array([e2m1_value(c) for c in range(16)])
    x = vals[np.asarray(codes)]
    s = np.repeat(np.asarray(scales, dtype=np.int64), BLOCK, axis=-1)
    return np.ldexp(x, s - 127)


def dequant_v(codes, scales):
    """Logical V codes ``[BH, N, 128]`` + scales ``[BH, 128, nblk]`` -> float64 ``[BH, N, 128]``."""
    vals = np.array([e2m1_value(c) for c in range(16)])
    x = vals[np.asarray(codes)]
    N = x.shape[1]
    s = np.repeat(np.asarray(scales, dtype=np.int64), BLOCK, axis=-1)[:, :, :N]  # [BH,128,N]
    return np.ldexp(x, np.transpose(s, (0, 2, 1)) - 127)


# ----------------------------------------------------------------- NVFP4

def e4m3_value(code: int) -> float:
    """Value of a finite nonnegative E4M3 code (0..126)."""
    return float(_load().orc_e4m3_value(int(code)))


def e4m3_code(v: float) -> int:
    """Nearest finite E4M3 code to v >= 0, ties to even, saturating at 448 (reading N1)."""
    return int(_load().orc_e4m3_code(float(v)))


def nvfp4_encode(amax: float) -> float:
    """Tensor encode factor e_t = fl32(2688 / amax), 1 for an all-zero tensor (N3)."""
    return float(_load().orc_nvfp4_encode(float(amax)))


def nvfp4_quantize_qk(x_u16: np.ndarray):
    """NVFP4 Q/K quantization (no rotation, N6) of bf16 bits ``[..., 128]`` as one tensor.

    Returns (codes ``[..., 128]``, scales ``[..., 8]`` E4M3 bytes, e_t)."""
    lib = _load()
    x = _c(x_u16, np.uint16).reshape(-1, D)
    rows = x.shape[0]
    codes = np.empty((rows, D), dtype=np.uint8)
    scales = np.empty((rows, D // 16), dtype=np.uint8)
    et = np.zeros(1, dtype=np.float32)
    lib.orc_nvfp4_quantize_qk(_p(x), rows, _p(codes), _p(scales), _p(et))
    lead = np.shape(x_u16)[:-1]
    return codes.reshape(*lead, D), scales.reshape(*lead, D // 16), float(et[0])


def nvfp4_quantize_v(v_u16: np.ndarray):
    """NVFP4 V quantization of ``[BH, N, 128]`` bf16 bits in 16-token blocks.

    Returns (codes ``[BH, N, 128]``, scales ``[BH, 128, ceil(N/16)]``, e_t)."""
    lib = _load()
    v = _c(v_u16, np.uint16)
    BH, N, _ = v.shape
    nblk = (N + 15) // 16
    codes = np.empty((BH, N, D), dtype=np.uint8)
    scales = np.empty((BH, D, nblk), dtype=np.uint8)
    et = np.zeros(1, dtype=np.float32)
    lib.orc_nvfp4_quantize_v(_p(v), BH, N, _p(codes), _p(scales), _p(et))
    return codes, scales, float(et[0])


def forward_nvfp4(qc, qs, q_et, kc, ks, k_et, vc, vs, v_et, rows, *, vraw_u16=None, causal=False,
                  placement=DIRECT, quant_p=True, want_phat=False, phat_in=None):
    """The attention loop on NVFP4 operands (logical layouts as returned above).

    P~ is quantized as NVFP4 (16-key blocks, e_t = 1). ``placement``: DIRECT
    (l from P~, the baseline's reading) or PNQ. ``phat_in`` ``[R, ntiles*128]``:
    replay those P^ values instead of computing them. Returns dict as :func:`forward`."""
    lib = _load()
    qc, qs, kc, ks, vc, vs = (_c(a, np.uint8) for a in (qc, qs, kc, ks, vc, vs))
    BH, N, _ = qc.shape
    vr = None if vraw_u16 is None else _c(vraw_u16, np.uint16)
    if causal and vr is None:
        raise ValueError("causal forward needs the unquantized V (vraw_u16)")
    rows = _c(rows, np.int64).reshape(-1, 2)
    R = rows.shape[0]
    ntiles = (N + BC - 1) // BC
    out = np.empty((R, D))
    ell = np.empty(R)
    phat = np.zeros((R, ntiles * BC)) if want_phat else None
    mhist = np.full((R, ntiles), np.nan) if want_phat else None
    if phat_in is not None:
        phat_in = _c(phat_in, np.float64).reshape(R, ntiles * BC)
    rc = lib.orc_forward_nvfp4(_p(qc), _p(qs), float(q_et), _p(kc), _p(ks), float(k_et), _p(vc), _p(vs),
                               float(v_et), _p(vr), BH, N, int(bool(causal)), int(placement), int(quant_p),
                               _p(rows), R, _p(out), _p(ell), _p(phat), _p(mhist),
                               _p(phat_in))
    if rc != 0:
        raise RuntimeError(f"orc_forward_nvfp4 failed with code {rc}")
    res = {"out": out, "ell": ell}
    if want_phat:
        res["phat"] = phat
        res["mhist"] = mhist
    return res


def nvfp4_dequant_qk(codes, scales, e_t):
    """Logical NVFP4 Q/K codes + scales -> float64 ``[..., 128]``."""
    vals = np.array([e2m1_value(c) for c in range(16)])
    svals = np.array([e4m3_value(c) if c < 127 else np.nan for c in range(256)])
    x = vals[np.asarray(codes)]
    s = np.repeat(svals[np.asarray(scales)], 16, axis=-1)
    return x * s / e_t


def nvfp4_dequant_v(codes, scales, e_t):
    """Logical NVFP4 V codes ``[BH, N, 128]`` + scales ``[BH, 128, nblk]`` -> float64 ``[BH, N, 128]``."""
    vals = np.array([e2m1_value(c) for c in range(16)])
    svals = np.array([e4m3_value(c) if c < 127 else np.nan for c in range(256)])
    x = vals[np.asarray(codes)]
    N = x.shape[1]
    s = np.repeat(svals[np.asarray(scales)], 16, axis=-1)[:, :, :N]
    return x * np.transpose(s, (0, 2, 1)) / e_t
