"""Index maps from the library's physical quantized layouts (include/mxattn.h)
to the oracle's logical layouts. Pure numpy; no arithmetic of the method."""
from __future__ import annotations

import numpy as np

D = 128


def nt(N: int) -> int:
    return (N + 127) // 128


def unpack_nibbles(b: np.ndarray) -> np.ndarray:
    """[..., n] bytes -> [..., 2n] codes, element 2j from the low nibble of byte j."""
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return out


def atom_index() -> np.ndarray:
    """[128 rows, 4 blocks] -> byte offset inside a 512-byte scale atom."""
    r = np.arange(128)[:, None]
    k = np.arange(4)[None, :]
    return (r % 32) * 16 + (r // 32) * 4 + k


def tiles_logical(scales: np.ndarray, BH: int, N: int) -> np.ndarray:
    """[BH*NT*512] bytes -> [BH, NT*128 rows, 4 blocks]."""
    s = np.asarray(scales, dtype=np.uint8).reshape(BH, nt(N), 512)
    g = s[:, :, atom_index()]  # [BH, NT, 128, 4]
    return g.reshape(BH, nt(N) * 128, 4)


def qk_codes_logical(codes: np.ndarray, BH: int, N: int) -> np.ndarray:
    return unpack_nibbles(np.asarray(codes, dtype=np.uint8).reshape(BH, N, 64))


def qk_scales_logical(scales: np.ndarray, BH: int, N: int) -> np.ndarray:
    return tiles_logical(scales, BH, N)[:, :N, :]


def v_codes_logical(codes: np.ndarray, BH: int, N: int) -> np.ndarray:
    npad = ((N + 31) // 32) * 32
    c = unpack_nibbles(np.asarray(codes, dtype=np.uint8).reshape(BH, D, npad // 2))  # [BH, 128, Npad]
    return np.ascontiguousarray(np.transpose(c, (0, 2, 1))[:, :N, :])


def v_scales_logical(scales: np.ndarray, BH: int, N: int) -> np.ndarray:
    """-> [BH, 128 channels, ceil(N/32) token blocks]."""
    t = tiles_logical(scales, BH, N).reshape(BH, nt(N), 128, 4)  # rows = channels
    g = np.transpose(t, (0, 2, 1, 3)).reshape(BH, 128, nt(N) * 4)
    return g[:, :, : (N + 31) // 32]


def phat_values(codes: np.ndarray, scales: np.ndarray, e2m1_values: np.ndarray) -> np.ndarray:
    """Dumped P^ tiles ([R, NT*64] codes, [R, NT*4] scales) -> dequantized [R, NT*128]."""
    c = unpack_nibbles(np.asarray(codes, dtype=np.uint8))
    s = np.repeat(np.asarray(scales, dtype=np.int64), 32, axis=-1)
    return np.ldexp(e2m1_values[c], s - 127)


def nv_tiles_logical(scales: np.ndarray, BH: int, N: int) -> np.ndarray:
    """NVFP4 scales [BH*NT*1024] bytes (two atoms per tile, atom kk = blocks 4kk..4kk+3)
    -> [BH, NT*128 rows, 8 blocks]."""
    s = np.asarray(scales, dtype=np.uint8).reshape(BH, nt(N), 2, 512)
    g = s[:, :, :, atom_index()]  # [BH, NT, 2, 128, 4]
    g = np.transpose(g, (0, 1, 3, 2, 4)).reshape(BH, nt(N), 128, 8)
    return g.reshape(BH, nt(N) * 128, 8)


def nv_qk_scales_logical(scales: np.ndarray, BH: int, N: int) -> np.ndarray:
    return nv_tiles_logical(scales, BH, N)[:, :N, :]


def nv_v_scales_logical(scales: np.ndarray, BH: int, N: int) -> np.ndarray:
    """-> [BH, 128 channels, ceil(N/16) token blocks]."""
    t = nv_tiles_logical(scales, BH, N).reshape(BH, nt(N), 128, 8)  # rows = channels
    g = np.transpose(t, (0, 2, 1, 3)).reshape(BH, 128, nt(N) * 8)
    return g[:, :, : (N + 15) // 16]


def nv_phat_values(codes: np.ndarray, scales: np.ndarray, e2m1_values: np.ndarray,
                   e4m3_values: np.ndarray) -> np.ndarray:
    """Dumped NVFP4 P^ tiles ([R, NT*64] codes, [R, NT*8] E4M3 scales) -> dequantized [R, NT*128]."""
    c = unpack_nibbles(np.asarray(codes, dtype=np.uint8))
    s = np.repeat(e4m3_values[np.asarray(scales, dtype=np.int64)], 16, axis=-1)
    return e2m1_values[c] * s
