"""GAAC oracle: ctypes access to the scalar C statement of the codec and of
fp64 decode attention (``gaac_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library and never imports it.

Source: "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference on
Personal Devices", sections 3.1-3.3 and Appendix D (see ``gaac_oracle.c``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gaac_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libgaac_oracle.so")
_lock = threading.Lock()
_lib = None

KIND_K, KIND_V = 0, 1
D, BLOCK, TILE = 128, 64, 8192
OFF_CODE, OFF_TAG, OFF_DIR, OFF_ESC = 8192, 11264, 11520, 11536
ESC_CAP = 496
SLOT_BYTES = 12032


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (plain C11, -O2)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if force or not fresh:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int, ctypes.c_int64
            L.gaac_ref_storage_index.argtypes = [i32, i32, i32]
            L.gaac_ref_storage_index.restype = i32
            L.gaac_ref_best_window.argtypes = [P, i32]
            L.gaac_ref_best_window.restype = i32
            L.gaac_ref_calibrate.argtypes = [P, i64, i64, i32, P, P]
            L.gaac_ref_calibrate.restype = None
            L.gaac_ref_encode_tile.argtypes = [P, i32, P, P, P, P, i32]
            L.gaac_ref_encode_tile.restype = i32
            L.gaac_ref_encode_open_tile.argtypes = [P, i32, i32, P, P, P, i32]
            L.gaac_ref_encode_open_tile.restype = i32
            L.gaac_ref_nested_slot_bytes.argtypes = []
            L.gaac_ref_nested_slot_bytes.restype = i32
            L.gaac_ref_nested_calibrate.argtypes = [P, i64, i64, i32, P]
            L.gaac_ref_nested_calibrate.restype = None
            L.gaac_ref_nested_encode_tile.argtypes = [P, i32, P, P, P, P, P]
            L.gaac_ref_nested_encode_tile.restype = i32
            L.gaac_ref_nested_decode_tile.argtypes = [P, i32, P, P, P, P]
            L.gaac_ref_nested_decode_tile.restype = i32
            L.gaac_ref_decode_tile.argtypes = [P, i32, P, P, i32, P]
            L.gaac_ref_decode_tile.restype = i32
            L.gaac_ref_mode_counts.argtypes = [P, P]
            L.gaac_ref_mode_counts.restype = None
            L.gaac_ref_raw_tile.argtypes = [P, i32, P]
            L.gaac_ref_raw_tile.restype = None
            L.gaac_ref_unraw_tile.argtypes = [P, i32, P]
            L.gaac_ref_unraw_tile.restype = None
            L.gaac_ref_escape_bytes_of_mode.argtypes = [i32]
            L.gaac_ref_escape_bytes_of_mode.restype = i32
            L.gaac_ref_attention.argtypes = [P, P, P, i64, i64, i32, i32, ctypes.c_double, P, P, P]
            L.gaac_ref_attention.restype = None
            L.gaac_ref_attention_d.argtypes = [P, P, P, i64, i64, i32, i32, i32, ctypes.c_double, P, P, P]
            L.gaac_ref_attention_d.restype = None
            L.gaac_ref_fp8_slot_bytes.argtypes = [i32]
            L.gaac_ref_fp8_slot_bytes.restype = i32
            L.gaac_ref_fp8_calibrate.argtypes = [P, i64, i64, i32, i32, P, P]
            L.gaac_ref_fp8_calibrate.restype = i32
            L.gaac_ref_fp8_encode_tile.argtypes = [P, i32, i32, P, P, P, P, i32]
            L.gaac_ref_fp8_encode_tile.restype = i32
            L.gaac_ref_fp8_decode_tile.argtypes = [P, i32, i32, P, P, i32, P]
            L.gaac_ref_fp8_decode_tile.restype = i32
            L.gaac_ref_fp8_mode_counts.argtypes = [P, i32, P]
            L.gaac_ref_fp8_mode_counts.restype = None
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.uint16))


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.uint8))


def storage_index(kind: int, t: int, c: int) -> int:
    return lib().gaac_ref_storage_index(kind, t, c)


def best_window(hist, width: int) -> int:
    h = np.ascontiguousarray(np.asarray(hist, dtype=np.uint64))
    assert h.shape == (256,)
    return lib().gaac_ref_best_window(_ptr(h), width)


def calibrate(x) -> tuple[np.ndarray, np.ndarray]:
    """x: uint16 [n_tok][n_heads][128] BF16 bits -> (base3, base4) uint8 [n_heads][128]."""
    x = _u16(x)
    n_tok, n_heads, d = x.shape
    assert d == D
    b3 = np.zeros((n_heads, D), np.uint8)
    b4 = np.zeros((n_heads, D), np.uint8)
    lib().gaac_ref_calibrate(_ptr(x), n_tok, n_heads * D, n_heads, _ptr(b3), _ptr(b4))
    return b3, b4


FULL_ESC = 8 * 1024  # every group raw: the largest escape stream a tile can have


def encode_tile(tile, kind: int, base3, base4, forced=None, esc_cap: int = ESC_CAP):
    """Encode a [64][128] BF16 tile.  Returns (image uint8 [11536+esc_cap], esc_len);
    esc_len (escape bytes, the directory not counted) is -1 when the escape
    stream would exceed esc_cap."""
    tile = _u16(tile).reshape(BLOCK, D)
    b3, b4 = _u8(base3).reshape(D), _u8(base4).reshape(D)
    img = np.zeros(OFF_ESC + esc_cap, np.uint8)
    fp = 0
    if forced is not None:
        forced = _u8(forced).reshape(1024)
        fp = _ptr(forced)
    esc = lib().gaac_ref_encode_tile(_ptr(tile), kind, _ptr(b3), _ptr(b4), fp, _ptr(img), esc_cap)
    return img, esc


def encode_open_tile(tile, n_tok: int, kind: int, base3, base4, esc_cap: int = ESC_CAP):
    """Encode the first n_tok (1..64) tokens of a [64][128] BF16 tile as an open slot image: the
    tokens past n_tok are absent (no part in a group's mode; all their fields zero).  Returns
    (image uint8 [11536+esc_cap], esc_len), esc_len -1 when the escape stream exceeds esc_cap."""
    tile = _u16(tile).reshape(BLOCK, D)
    b3, b4 = _u8(base3).reshape(D), _u8(base4).reshape(D)
    img = np.zeros(OFF_ESC + esc_cap, np.uint8)
    esc = lib().gaac_ref_encode_open_tile(_ptr(tile), int(n_tok), kind, _ptr(b3), _ptr(b4), _ptr(img), esc_cap)
    if esc == -2:
        raise ValueError("n_tok must be in [1, 64]")
    return img, esc


def decode_tile(img, kind: int, base3, base4, esc_limit: int | None = None):
    """Decode a slot image.  Returns (tile uint16 [64][128], status) where status is the
    escape byte count consumed (>= 0) or a negative error."""
    img = _u8(img)
    if esc_limit is None:
        esc_limit = img.size - OFF_ESC
    b3, b4 = _u8(base3).reshape(D), _u8(base4).reshape(D)
    out = np.zeros((BLOCK, D), np.uint16)
    st = lib().gaac_ref_decode_tile(_ptr(img), kind, _ptr(b3), _ptr(b4), esc_limit, _ptr(out))
    return out, st


def mode_counts(img) -> np.ndarray:
    img = _u8(img)
    out = np.zeros(4, np.int64)
    lib().gaac_ref_mode_counts(_ptr(img), _ptr(out))
    return out


def raw_tile(tile, kind: int) -> np.ndarray:
    tile = _u16(tile).reshape(BLOCK, D)
    out = np.zeros(TILE, np.uint16)
    lib().gaac_ref_raw_tile(_ptr(tile), kind, _ptr(out))
    return out


def unraw_tile(raw, kind: int) -> np.ndarray:
    raw = _u16(raw).reshape(TILE)
    out = np.zeros((BLOCK, D), np.uint16)
    lib().gaac_ref_unraw_tile(_ptr(raw), kind, _ptr(out))
    return out


def escape_bytes_of_mode(mode: int) -> int:
    return lib().gaac_ref_escape_bytes_of_mode(mode)


def attention(q, k, v, scale: float):
    """fp64 decode attention of one sequence.
    q: uint16 [Hq][d]; k, v: uint16 [T][Hkv][d] (BF16 bits), d = 128 or 256.
    Returns (out float64 [Hq][d], flags int32 [Hq])."""
    q = _u16(q)
    k = _u16(k)
    v = _u16(v)
    Hq, d = q.shape
    T, Hkv, dk = k.shape
    assert dk == d and d in (128, 256) and v.shape == k.shape and Hq % Hkv == 0
    out = np.zeros((Hq, d), np.float64)
    flags = np.zeros(Hq, np.int32)
    scratch = np.zeros(max(T, 1), np.float64)
    lib().gaac_ref_attention_d(_ptr(q), _ptr(k), _ptr(v), Hkv * d, T, Hq, Hkv, d, float(scale), _ptr(out),
                               _ptr(flags), _ptr(scratch))
    return out, flags


# ---------------------------------------------------------------- FP8 variant
FP8_E4M3, FP8_E5M2 = 0, 1
FP8_OFF_ESC = {FP8_E4M3: 7440, FP8_E5M2: 6416}


def fp8_slot_bytes(fmt: int) -> int:
    return lib().gaac_ref_fp8_slot_bytes(fmt)


def fp8_calibrate(x, fmt: int) -> tuple[np.ndarray, np.ndarray]:
    """x: uint8 [n_tok][n_heads][128] FP8 bits -> (base3, base4) uint8 [n_heads][128]."""
    x = _u8(x)
    n_tok, n_heads, d = x.shape
    assert d == D
    b3 = np.zeros((n_heads, D), np.uint8)
    b4 = np.zeros((n_heads, D), np.uint8)
    assert lib().gaac_ref_fp8_calibrate(_ptr(x), n_tok, n_heads * D, n_heads, fmt, _ptr(b3), _ptr(b4)) == 0
    return b3, b4


def fp8_encode_tile(tile, kind: int, fmt: int, base3, base4, forced=None, esc_cap: int = ESC_CAP):
    """Encode a [64][128] FP8 tile.  Returns (image uint8 [off_esc + esc_cap], esc_len); esc_len is -1
    when the escape area would exceed esc_cap."""
    tile = _u8(tile).reshape(BLOCK, D)
    b3, b4 = _u8(base3).reshape(D), _u8(base4).reshape(D)
    img = np.zeros(FP8_OFF_ESC[fmt] + esc_cap, np.uint8)
    fp = 0
    if forced is not None:
        forced = _u8(forced).reshape(1024)
        fp = _ptr(forced)
    esc = lib().gaac_ref_fp8_encode_tile(_ptr(tile), kind, fmt, _ptr(b3), _ptr(b4), fp, _ptr(img), esc_cap)
    return img, esc


def fp8_decode_tile(img, kind: int, fmt: int, base3, base4, esc_limit: int | None = None):
    img = _u8(img)
    if esc_limit is None:
        esc_limit = img.size - FP8_OFF_ESC[fmt]
    b3, b4 = _u8(base3).reshape(D), _u8(base4).reshape(D)
    out = np.zeros((BLOCK, D), np.uint8)
    st = lib().gaac_ref_fp8_decode_tile(_ptr(img), kind, fmt, _ptr(b3), _ptr(b4), esc_limit, _ptr(out))
    return out, st


def fp8_mode_counts(img, fmt: int) -> np.ndarray:
    img = _u8(img)
    out = np.zeros(4, np.int64)
    lib().gaac_ref_fp8_mode_counts(_ptr(img), fmt, _ptr(out))
    return out


# ---- nested 2-bit mode: the ablation format of the GAAC page's section 4.7.2 (Table 4)
NESTED_OFF_ESC = 11552


def nested_slot_bytes() -> int:
    return lib().gaac_ref_nested_slot_bytes()


def nested_calibrate(x) -> np.ndarray:
    """x: uint16 [n_tok][n_heads][128] BF16 bits -> base2 uint8 [n_heads][128] (best 4-window)."""
    x = _u16(x)
    n_tok, n_heads, d = x.shape
    assert d == D
    b2 = np.zeros((n_heads, D), np.uint8)
    lib().gaac_ref_nested_calibrate(_ptr(x), n_tok, n_heads * D, n_heads, _ptr(b2))
    return b2


def nested_encode_tile(tile, kind: int, base2, base3, base4):
    """[64][128] BF16 tile -> (image uint8 [nested_slot_bytes()], esc_len, code_bits); esc_len -1 when
    the escape stream exceeds 496 bytes."""
    tile = _u16(tile).reshape(BLOCK, D)
    b2, b3, b4 = (_u8(b).reshape(D) for b in (base2, base3, base4))
    img = np.zeros(nested_slot_bytes(), np.uint8)
    bits = ctypes.c_int(0)
    esc = lib().gaac_ref_nested_encode_tile(_ptr(tile), kind, _ptr(b2), _ptr(b3), _ptr(b4), _ptr(img),
                                            ctypes.addressof(bits))
    return img, esc, bits.value


def nested_decode_tile(img, kind: int, base2, base3, base4):
    img = _u8(img)
    b2, b3, b4 = (_u8(b).reshape(D) for b in (base2, base3, base4))
    out = np.zeros((BLOCK, D), np.uint16)
    st = lib().gaac_ref_nested_decode_tile(_ptr(img), kind, _ptr(b2), _ptr(b3), _ptr(b4), _ptr(out))
    return out, st
