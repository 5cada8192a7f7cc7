"""Python binding of the GAAC compressed-KV decode-attention library.

Thin marshalling over the C ABI declared in ``include/gaac.h`` (ctypes): every
function below passes torch device pointers, sizes and the current CUDA stream
to the library and raises on a nonzero status.  All computation happens in the
library's CUDA kernels; there is no CPU fallback.  If ``libgaac.so`` has not been
built, the first call raises.

Method: "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference on
Personal Devices" (sections 3.1-3.3).  Tile format v3 is described in gaac.h.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

HEAD_DIM = 128
BLOCK = 64
TILE_ELEMS = 8192
SLOT_BYTES = 12032
ESC_CAPACITY = 496
RAW_TILE_BYTES = 16384
MAX_GQA = 8

OK, EINVAL, EPOOL, EFORMAT, ECUDA, ETIMEOUT = range(6)
MODE_SLOT, MODE_RAW, MODE_NONE = 0, 1, 255
OPEN_COMPRESSED = 1  # flag of encode_blocks / append: keep the open block compressed in its slot

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgaac.so")
_lock = threading.Lock()
_lib = None


class GaacError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {strerror(status) if _lib is not None else status} (status {status})")


class gaac_pools(ctypes.Structure):
    _fields_ = [
        ("slot_pool", ctypes.c_void_p),
        ("n_slots", ctypes.c_int64),
        ("raw_pool", ctypes.c_void_p),
        ("n_raw", ctypes.c_int64),
        ("raw_free", ctypes.c_void_p),
        ("n_raw_free", ctypes.c_int64),
        ("raw_cursor", ctypes.c_void_p),
    ]


STATS_FIELDS = ("groups0", "groups1", "groups2", "groups3", "escape_bytes", "slot_tiles", "raw_tiles", "tail_tiles")


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it was not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"GAAC CUDA library not found at {LIB_PATH}; build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
            L = ctypes.CDLL(LIB_PATH)
            P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
            L.gaac_strerror.argtypes = [i32]
            L.gaac_strerror.restype = ctypes.c_char_p
            L.gaac_format_version.argtypes = []
            L.gaac_format_version.restype = i32
            L.gaac_calibrate.argtypes = [P, i64, i64, i32, P, P, P, P]
            L.gaac_calibrate.restype = i32
            L.gaac_encode_blocks.argtypes = [P, P, i64, i64, i64, P, i32, i32, i32, P, P, P, P, P, P, P, P]
            L.gaac_encode_blocks.restype = i32
            L.gaac_append.argtypes = [P, P, P, i32, i32, i32, P, P, P, P, P, P, P, P]
            L.gaac_append.restype = i32
            L.gaac_encode_blocks_ex.argtypes = [P, P, i64, i64, i64, P, i32, i32, i32, P, P, P, P, P, P,
                                                ctypes.c_uint, P, P]
            L.gaac_encode_blocks_ex.restype = i32
            L.gaac_append_ex.argtypes = [P, P, P, i32, i32, i32, P, P, P, P, P, P, ctypes.c_uint, P, P]
            L.gaac_append_ex.restype = i32
            L.gaac_attention_workspace.argtypes = [i32, i32, i32, i32]
            L.gaac_attention_workspace.restype = sz
            L.gaac_attention_auto_splits.argtypes = [i32, i32, i32]
            L.gaac_attention_auto_splits.restype = i32
            L.gaac_decode_attention.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, ctypes.c_float, i32, P, P, sz,
                                                P, P]
            L.gaac_decode_attention.restype = i32
            L.gaac_decode_attention_bf16.argtypes = [P, i32, i32, i32, i32, P, P, P, ctypes.c_float, i32, P, P, sz,
                                                     P, P]
            L.gaac_decode_attention_bf16.restype = i32
            L.gaac_decode_attention_hd256.argtypes = L.gaac_decode_attention.argtypes
            L.gaac_decode_attention_hd256.restype = i32
            L.gaac_decompress.argtypes = [P, P, i32, i32, i32, P, P, P, P, P, i64, i64, i64, P, P]
            L.gaac_decode_attention_noalloc.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, ctypes.c_float, i32, P,
                                                        P, P]
            L.gaac_decode_attention_noalloc.restype = i32
            L.gaac_decompress.restype = i32
            L.gaac_encode_tiles.argtypes = [P, i64, P, P, i32, P, P, P, P, P, P, P]
            L.gaac_encode_tiles.restype = i32
            L.gaac_decode_tiles.argtypes = [P, P, i64, P, P, i32, P, P, P, P, P]
            L.gaac_decode_tiles.restype = i32
            L.gaac_nested_calibrate.argtypes = [P, i64, i64, i32, P, P, P]
            L.gaac_nested_calibrate.restype = i32
            L.gaac_nested_encode_tiles.argtypes = [P, i64, P, P, i32, P, P, P, P, P, P, P]
            L.gaac_nested_encode_tiles.restype = i32
            L.gaac_nested_decode_tiles.argtypes = [P, P, i64, P, P, i32, P, P, P, P, P, P]
            L.gaac_nested_decode_tiles.restype = i32
            L.gaac_fp8_slot_bytes.argtypes = [i32]
            L.gaac_fp8_slot_bytes.restype = i32
            L.gaac_fp8_calibrate.argtypes = [P, i64, i64, i32, i32, P, P, P, P]
            L.gaac_fp8_calibrate.restype = i32
            L.gaac_fp8_encode_tiles.argtypes = [P, i64, i32, P, P, i32, P, P, P, P, P, P, P]
            L.gaac_fp8_encode_tiles.restype = i32
            L.gaac_fp8_decompress_tiles.argtypes = [P, P, i64, i32, P, P, i32, P, P, P, P, P]
            L.gaac_fp8_decompress_tiles.restype = i32
            _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().gaac_strerror(status).decode()


def format_version() -> int:
    return lib().gaac_format_version()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _check(fn: str, status: int):
    if status != OK:
        raise GaacError(fn, status)


def _cuda(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


class Pools:
    """Caller-owned storage of one layer's compressed cache.

    slot_pool: uint8 [n_slots, 12032]; raw_pool: int16 [n_raw, 8192] (BF16 bits);
    raw_free: optional int32 list of free raw-tile indices (None = 0..n_raw-1);
    raw_cursor: int32 [1] device counter of popped raw tiles."""

    def __init__(self, n_slots: int, n_raw: int, device="cuda", raw_free: torch.Tensor | None = None):
        self.slot_pool = torch.zeros((max(n_slots, 1), SLOT_BYTES), dtype=torch.uint8, device=device)
        self.raw_pool = torch.zeros((max(n_raw, 1), TILE_ELEMS), dtype=torch.int16, device=device)
        self.n_slots, self.n_raw = n_slots, n_raw
        self.raw_free = raw_free
        self.raw_cursor = torch.zeros(1, dtype=torch.int32, device=device)

    def c(self) -> gaac_pools:
        n_free = self.raw_free.numel() if self.raw_free is not None else self.n_raw
        return gaac_pools(self.slot_pool.data_ptr(), self.n_slots, self.raw_pool.data_ptr(), self.n_raw,
                          _ptr(self.raw_free), n_free, self.raw_cursor.data_ptr())


def new_table(batch: int, max_blocks: int, n_kv_heads: int, device="cuda") -> torch.Tensor:
    """Slot table of one layer: int64 [batch, max_blocks, n_kv_heads, 2], one gaac_entry per element
    (bits 0-31 index, 32-47 esc_len, 48-55 mode, 56-63 n_tok)."""
    t = torch.zeros((batch, max_blocks, n_kv_heads, 2), dtype=torch.int64, device=device)
    t.fill_(MODE_NONE << 48)
    return t


def entry_fields(table: torch.Tensor):
    """(index, esc_len, mode, n_tok) tensors of a table."""
    return table & 0xFFFFFFFF, (table >> 32) & 0xFFFF, (table >> 48) & 0xFF, (table >> 56) & 0xFF


def new_stats(device="cuda") -> torch.Tensor:
    return torch.zeros(len(STATS_FIELDS), dtype=torch.int64, device=device)


def stats_dict(stats: torch.Tensor) -> dict:
    return dict(zip(STATS_FIELDS, stats.tolist()))


def _kv_strides(x: torch.Tensor, name: str):
    if x.dtype not in (torch.bfloat16, torch.int16) or x.dim() != 4 or x.shape[-1] != HEAD_DIM:
        raise ValueError(f"{name} must be a [batch, tokens, kv_heads, 128] BF16 tensor")
    if x.stride(3) != 1 or x.stride(2) != HEAD_DIM:
        raise ValueError(f"{name}: heads and channels must be contiguous")
    return x.stride(0), x.stride(1)


def calibrate(x: torch.Tensor, base3: torch.Tensor, base4: torch.Tensor, status: torch.Tensor | None = None,
              stream=None) -> None:
    """x: BF16 [n_tok, kv_heads, 128] (token stride free); writes uint8 base3/base4 [kv_heads, 128]."""
    _cuda(x, "x")
    if x.dim() != 3 or x.shape[-1] != HEAD_DIM or x.stride(2) != 1 or x.stride(1) != HEAD_DIM:
        raise ValueError("x must be [n_tok, kv_heads, 128] with contiguous heads and channels")
    _check("gaac_calibrate", lib().gaac_calibrate(x.data_ptr(), x.shape[0], x.stride(0), x.shape[1], base3.data_ptr(),
                                                   base4.data_ptr(), _ptr(status), _stream(stream)))


def encode_blocks(k, v, seq_lens, max_blocks, base3, base4, table, slot_ids, pools: Pools, stats=None, status=None,
                  stream=None, open_compressed: bool = False) -> None:
    """Prefill encode of a layer.  k, v: BF16 [batch, tokens, kv_heads, 128]; seq_lens int32 [batch];
    base3/base4 uint8 [2, kv_heads, 128]; table from new_table(); slot_ids int32 shaped like the table,
    or None to store every block as a raw BF16 tile (the uncompressed baseline).  open_compressed keeps
    each sequence's incomplete last block in its slot (GAAC_OPEN_COMPRESSED)."""
    for t, n in ((k, "k"), (v, "v"), (seq_lens, "seq_lens"), (table, "table")):
        _cuda(t, n)
    ss, ts = _kv_strides(k, "k")
    if _kv_strides(v, "v") != (ss, ts):
        raise ValueError("k and v must share strides")
    pc = pools.c()
    _check("gaac_encode_blocks_ex", lib().gaac_encode_blocks_ex(
        k.data_ptr(), v.data_ptr(), ss, ts, min(k.shape[1], v.shape[1]), seq_lens.data_ptr(), k.shape[0], k.shape[2],
        max_blocks,
        base3.data_ptr(), base4.data_ptr(), table.data_ptr(), _ptr(slot_ids), ctypes.byref(pc), _ptr(stats),
        OPEN_COMPRESSED if open_compressed else 0, _ptr(status), _stream(stream)))


def append(k_new, v_new, seq_lens, max_blocks, base3, base4, table, slot_ids, pools: Pools, stats=None,
           status=None, stream=None, open_compressed: bool = False) -> None:
    """Append one token per sequence.  k_new, v_new: BF16 [batch, kv_heads, 128]; slot_ids shaped like the
    table (the slot a block is sealed into, or kept open in with open_compressed), or None for a cache of
    raw tiles only (full tails stay raw); seq_lens is incremented."""
    pc = pools.c()
    _check("gaac_append_ex", lib().gaac_append_ex(
        k_new.data_ptr(), v_new.data_ptr(), seq_lens.data_ptr(), k_new.shape[0], k_new.shape[1], max_blocks,
        base3.data_ptr(), base4.data_ptr(), table.data_ptr(), _ptr(slot_ids), ctypes.byref(pc),
        _ptr(stats), OPEN_COMPRESSED if open_compressed else 0, _ptr(status), _stream(stream)))


def attention_workspace(batch: int, n_kv_heads: int, max_blocks: int, n_splits: int = 0) -> int:
    return lib().gaac_attention_workspace(batch, n_kv_heads, max_blocks, n_splits)


def auto_splits(batch: int, n_kv_heads: int, max_blocks: int) -> int:
    return lib().gaac_attention_auto_splits(batch, n_kv_heads, max_blocks)


def decode_attention(q, seq_lens, table, pools: Pools, base3, base4, scale: float, out, workspace, n_splits: int = 0,
                     status=None, stream=None) -> None:
    """q: BF16 [batch, q_heads, 128]; out: fp32 [batch, q_heads, 128]; workspace: uint8 device buffer."""
    batch, hq = q.shape[0], q.shape[1]
    max_blocks, hkv = table.shape[1], table.shape[2]
    pc = pools.c()
    _check("gaac_decode_attention", lib().gaac_decode_attention(
        q.data_ptr(), batch, hq, hkv, max_blocks, seq_lens.data_ptr(), table.data_ptr(), ctypes.byref(pc),
        base3.data_ptr(), base4.data_ptr(), float(scale), n_splits, out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)))


def decode_attention_bf16(q, seq_lens, table, pools: Pools, scale: float, out, workspace, n_splits: int = 0,
                          status=None, stream=None) -> None:
    """decode_attention over an uncompressed BF16 cache (every entry a raw tile): the same kernel specialised
    to raw tiles, with no decode path."""
    batch, hq = q.shape[0], q.shape[1]
    max_blocks, hkv = table.shape[1], table.shape[2]
    pc = pools.c()
    _check("gaac_decode_attention_bf16", lib().gaac_decode_attention_bf16(
        q.data_ptr(), batch, hq, hkv, max_blocks, seq_lens.data_ptr(), table.data_ptr(), ctypes.byref(pc),
        float(scale), n_splits, out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream)))


def decompress(table, seq_lens, pools: Pools, base3, base4, k_out, v_out, status=None, stream=None) -> None:
    """Rebuild BF16 k_out/v_out [batch, tokens, kv_heads, 128] for tokens < seq_lens."""
    ss, ts = _kv_strides(k_out, "k_out")
    if _kv_strides(v_out, "v_out") != (ss, ts):
        raise ValueError("k_out and v_out must share strides")
    pc = pools.c()
    _check("gaac_decompress", lib().gaac_decompress(
        table.data_ptr(), seq_lens.data_ptr(), table.shape[0], table.shape[2], table.shape[1], ctypes.byref(pc),
        base3.data_ptr(), base4.data_ptr(), k_out.data_ptr(), v_out.data_ptr(), ss, ts,
        min(k_out.shape[1], v_out.shape[1]), _ptr(status), _stream(stream)))


STATIC_SCRATCH_BYTES = 4 << 20


def decode_attention_noalloc(q, seq_lens, table, pools: Pools, base3, base4, scale: float, out, n_splits: int = 0,
                             status=None, stream=None) -> None:
    """decode_attention without a workspace: for callers that cannot allocate device memory at call time.
    The split partials use the library's own fixed scratch array (STATIC_SCRATCH_BYTES per device), so
    calls must not overlap on the GPU, and the first call on a device must come before any stream capture."""
    batch, hq = q.shape[0], q.shape[1]
    max_blocks, hkv = table.shape[1], table.shape[2]
    pc = pools.c()
    _check("gaac_decode_attention_noalloc", lib().gaac_decode_attention_noalloc(
        q.data_ptr(), batch, hq, hkv, max_blocks, seq_lens.data_ptr(), table.data_ptr(), ctypes.byref(pc),
        base3.data_ptr(), base4.data_ptr(), float(scale), n_splits, out.data_ptr(), _ptr(status), _stream(stream)))


# ---------------------------------------------------------------- FP8 variant of the codec
FP8_E4M3, FP8_E5M2 = 0, 1
FP8_NO_SLOT = 0xFFFF  # esc_len of a tile that stays FP8


def fp8_slot_bytes(fmt: int) -> int:
    return lib().gaac_fp8_slot_bytes(fmt)


def fp8_calibrate(x: torch.Tensor, fmt: int, base3: torch.Tensor, base4: torch.Tensor, status=None,
                  stream=None) -> None:
    """x: uint8 FP8 bits [n_tok, kv_heads, 128] (token stride free); writes uint8 base3/base4 [kv_heads, 128]."""
    _cuda(x, "x")
    if x.dtype != torch.uint8 or x.dim() != 3 or x.shape[-1] != HEAD_DIM or x.stride(2) != 1 or x.stride(1) != HEAD_DIM:
        raise ValueError("x must be uint8 [n_tok, kv_heads, 128] with contiguous heads and channels")
    _check("gaac_fp8_calibrate", lib().gaac_fp8_calibrate(x.data_ptr(), x.shape[0], x.stride(0), x.shape[1], fmt,
                                                           base3.data_ptr(), base4.data_ptr(), _ptr(status),
                                                           _stream(stream)))


def _tile_batch(tiles, slots, esc_len, tile_kind, tile_row, bases, elem_bytes: int, slot_bytes: int) -> int:
    """Checks a tile batch's tensors (device, contiguity, shapes, element sizes) and returns n."""
    n = tiles.shape[0] if tiles.dim() == 3 else -1
    for t, name in ((tiles, "tiles"), (slots, "slots"), (esc_len, "esc_len"), (tile_kind, "tile_kind"),
                    (tile_row, "tile_row"), *((b, "base") for b in bases)):
        _cuda(t, name)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if tiles.dim() != 3 or tuple(tiles.shape[1:]) != (BLOCK, HEAD_DIM) or tiles.element_size() != elem_bytes:
        raise ValueError(f"tiles must be [n, {BLOCK}, {HEAD_DIM}] of {elem_bytes}-byte elements")
    if tuple(slots.shape) != (n, slot_bytes) or slots.element_size() != 1:
        raise ValueError(f"slots must be uint8 [n, {slot_bytes}]")
    if esc_len.numel() != n or esc_len.element_size() != 2:
        raise ValueError("esc_len must hold n 16-bit values")
    if tile_kind.numel() != n or tile_kind.element_size() != 1 or tile_row.numel() != n or tile_row.dtype != torch.int32:
        raise ValueError("tile_kind must be uint8 [n] and tile_row int32 [n]")
    for b in bases:
        if b.dim() != 2 or b.shape[1] != HEAD_DIM or b.element_size() != 1 or b.shape[0] != bases[0].shape[0]:
            raise ValueError("bases must be uint8 [rows, 128], all with the same rows")
    return n


def fp8_encode_tiles(tiles, fmt: int, tile_kind, tile_row, base3, base4, slots, esc_len, stats=None, status=None,
                     stream=None) -> None:
    """tiles: uint8 [n, 64, 128]; tile_kind: uint8 [n] (0 K, 1 V); tile_row: int32 [n] (row of base3/base4
    [rows, 128]); slots: uint8 [n, fp8_slot_bytes(fmt)]; esc_len: int16 [n] (0xFFFF = stays FP8)."""
    n = _tile_batch(tiles, slots, esc_len, tile_kind, tile_row, (base3, base4), 1, fp8_slot_bytes(fmt))
    _check("gaac_fp8_encode_tiles", lib().gaac_fp8_encode_tiles(
        tiles.data_ptr(), n, fmt, tile_kind.data_ptr(), tile_row.data_ptr(), base3.shape[0], base3.data_ptr(),
        base4.data_ptr(), slots.data_ptr(), esc_len.data_ptr(), _ptr(stats), _ptr(status), _stream(stream)))


def fp8_decompress_tiles(slots, esc_len, fmt: int, tile_kind, tile_row, base3, base4, tiles, status=None,
                         stream=None) -> None:
    n = _tile_batch(tiles, slots, esc_len, tile_kind, tile_row, (base3, base4), 1, fp8_slot_bytes(fmt))
    _check("gaac_fp8_decompress_tiles", lib().gaac_fp8_decompress_tiles(
        slots.data_ptr(), esc_len.data_ptr(), n, fmt, tile_kind.data_ptr(), tile_row.data_ptr(), base3.shape[0],
        base3.data_ptr(), base4.data_ptr(), tiles.data_ptr(), _ptr(status), _stream(stream)))


def encode_tiles(tiles, tile_kind, tile_row, base3, base4, slots, esc_len, stats=None, status=None,
                 stream=None) -> None:
    """Format v3 tile batch.  tiles: BF16 [n, 64, 128] token-major; tile_kind: uint8 [n] (0 K, 1 V);
    tile_row: int32 [n] (row of base3/base4 [rows, 128]); slots: uint8 [n, SLOT_BYTES]; esc_len: int16 [n]
    (0xFFFF: does not fit, slot untouched)."""
    n = _tile_batch(tiles, slots, esc_len, tile_kind, tile_row, (base3, base4), 2, SLOT_BYTES)
    _check("gaac_encode_tiles", lib().gaac_encode_tiles(
        tiles.data_ptr(), n, tile_kind.data_ptr(), tile_row.data_ptr(), base3.shape[0],
        base3.data_ptr(), base4.data_ptr(), slots.data_ptr(), esc_len.data_ptr(), _ptr(stats), _ptr(status),
        _stream(stream)))


def decode_tiles(slots, esc_len, tile_kind, tile_row, base3, base4, tiles, status=None, stream=None) -> None:
    n = _tile_batch(tiles, slots, esc_len, tile_kind, tile_row, (base3, base4), 2, SLOT_BYTES)
    _check("gaac_decode_tiles", lib().gaac_decode_tiles(
        slots.data_ptr(), esc_len.data_ptr(), n, tile_kind.data_ptr(), tile_row.data_ptr(),
        base3.shape[0], base3.data_ptr(), base4.data_ptr(), tiles.data_ptr(), _ptr(status), _stream(stream)))


NESTED_SLOT_BYTES = 12048


def nested_calibrate(x: torch.Tensor, base2: torch.Tensor, status=None, stream=None) -> None:
    """x: BF16 [n_tok, kv_heads, 128] -> base2 uint8 [kv_heads, 128] (best 4-exponent window)."""
    _cuda(x, "x")
    if x.dim() != 3 or x.shape[-1] != HEAD_DIM or x.stride(2) != 1 or x.stride(1) != HEAD_DIM:
        raise ValueError("x must be [n_tok, kv_heads, 128] with contiguous heads and channels")
    _check("gaac_nested_calibrate", lib().gaac_nested_calibrate(x.data_ptr(), x.shape[0], x.stride(0), x.shape[1],
                                                                 base2.data_ptr(), _ptr(status), _stream(stream)))


def nested_encode_tiles(tiles, tile_kind, tile_row, base2, base3, base4, slots, esc_len, status=None,
                        stream=None) -> None:
    """Nested 2-bit-mode ablation format; arguments as encode_tiles, slots [n, NESTED_SLOT_BYTES]."""
    n = _tile_batch(tiles, slots, esc_len, tile_kind, tile_row, (base2, base3, base4), 2, NESTED_SLOT_BYTES)
    _check("gaac_nested_encode_tiles", lib().gaac_nested_encode_tiles(
        tiles.data_ptr(), n, tile_kind.data_ptr(), tile_row.data_ptr(), base3.shape[0],
        base2.data_ptr(), base3.data_ptr(), base4.data_ptr(), slots.data_ptr(), esc_len.data_ptr(), _ptr(status),
        _stream(stream)))


def nested_decode_tiles(slots, esc_len, tile_kind, tile_row, base2, base3, base4, tiles, status=None,
                        stream=None) -> None:
    n = _tile_batch(tiles, slots, esc_len, tile_kind, tile_row, (base2, base3, base4), 2, NESTED_SLOT_BYTES)
    _check("gaac_nested_decode_tiles", lib().gaac_nested_decode_tiles(
        slots.data_ptr(), esc_len.data_ptr(), n, tile_kind.data_ptr(), tile_row.data_ptr(),
        base3.shape[0], base2.data_ptr(), base3.data_ptr(), base4.data_ptr(), tiles.data_ptr(), _ptr(status),
        _stream(stream)))


def decode_attention_hd256(q, seq_lens, table, pools: Pools, base3, base4, scale: float, out, workspace,
                           n_splits: int = 0, status=None, stream=None) -> None:
    """Attention over 256-channel heads stored as two 128-channel half-heads: q BF16 [batch, n_q_heads, 256],
    table [batch, max_blocks, 2 * n_kv_heads, 2], base3/base4 [2, 2 * n_kv_heads, 128], out fp32
    [batch, n_q_heads, 256]; workspace >= attention_workspace(batch, 2 * n_kv_heads, max_blocks, n_splits)."""
    B, Hq, d = q.shape
    if d != 256 or out.shape != (B, Hq, 256):
        raise ValueError("q and out must be [batch, n_q_heads, 256]")
    n_kv = table.shape[2] // 2
    pc = pools.c()
    _check("gaac_decode_attention_hd256", lib().gaac_decode_attention_hd256(
        q.data_ptr(), B, Hq, n_kv, table.shape[1], seq_lens.data_ptr(), table.data_ptr(), ctypes.byref(pc),
        base3.data_ptr(), base4.data_ptr(), float(scale), n_splits, out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)))
