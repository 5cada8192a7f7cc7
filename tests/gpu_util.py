"""Helpers shared by the GPU parity tests: build a cache with the CUDA library,
then compare it with the oracle on the same input bits.

The oracle never sees anything the CUDA path produced except the values under
test; its inputs are the seeded BF16 bits copied back from the device."""
from __future__ import annotations

import numpy as np
import torch

import gaac_workloads as W
import oracle as O
from lossless_compressed_kv_gaac_gb300 import MODE_NONE, MODE_RAW, MODE_SLOT
from lossless_compressed_kv_gaac_gb300.cache import LayerCache

TOL = 2e-3  # max relative error (row-normwise) of decode attention against the fp64 oracle


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def build(k, v, lens, n_calib=512, max_blocks=None, slot_ids=None, n_slots=None, n_raw=None, raw=False):
    B, T, H, _ = k.shape
    max_blocks = max_blocks or (T + 63) // 64
    c = LayerCache(B, H, max_blocks, device=k.device, slot_ids=slot_ids, n_slots=n_slots, n_raw=n_raw)
    nc = min(n_calib, T)
    c.calibrate(k[0, :nc], v[0, :nc])
    c.encode(k, v, lens, raw=raw)
    torch.cuda.synchronize()
    return c


def oracle_bases(k, v, n_calib=512):
    nc = min(n_calib, k.shape[1])
    b3k, b4k = O.calibrate(u16(k[0, :nc]))
    b3v, b4v = O.calibrate(u16(v[0, :nc]))
    return np.stack([b3k, b3v]), np.stack([b4k, b4v])


def logical_tile(x_np, b, blk, h, nv):
    tile = np.zeros((64, 128), np.uint16)
    tile[:nv] = x_np[b, blk * 64: blk * 64 + nv, h]
    return tile


def check_tiles(c: LayerCache, k, v, lens, tiles=None, b3=None, b4=None, raw_all=False, open_compressed=False):
    """Every (or the listed) tile of the cache equals the oracle's encoding of the input bits.
    tiles: iterable of (b, blk, h, kind).  open_compressed: open blocks are expected in their slots
    (the oracle's open-tile image) unless that overflows.  Returns counts of slot / raw tiles checked."""
    kn, vn = u16(k), u16(v)
    lens_np = lens.cpu().numpy()
    if b3 is None:
        b3, b4 = oracle_bases(k, v)
    idx, esc, mode, ntok = (x.cpu().numpy() for x in c.fields())
    slots = c.pools.slot_pool.cpu().numpy()
    raws = c.pools.raw_pool.cpu().numpy().view(np.uint16)
    if tiles is None:
        tiles = [(b, blk, h, kind) for b in range(c.batch) for blk in range(c.max_blocks)
                 for h in range(c.n_kv_heads) for kind in (0, 1)]
    n = {"slot": 0, "raw": 0, "none": 0}
    for b, blk, h, kind in tiles:
        nv = int(min(64, max(0, lens_np[b] - blk * 64)))
        m = mode[b, blk, h, kind]
        if nv == 0:
            assert m == MODE_NONE, (b, blk, h, kind, m)
            n["none"] += 1
            continue
        tile = logical_tile(kn if kind == 0 else vn, b, blk, h, nv)
        if (nv == 64 or open_compressed) and not raw_all:
            img, e = O.encode_open_tile(tile, nv, kind, b3[kind, h], b4[kind, h])
            if e >= 0:
                assert m == MODE_SLOT, (b, blk, h, kind, m)
                assert esc[b, blk, h, kind] == e and ntok[b, blk, h, kind] == nv
                got = slots[idx[b, blk, h, kind]]
                if not np.array_equal(got, img):
                    bad = np.nonzero(got != img)[0]
                    raise AssertionError(f"tile {(b, blk, h, kind)}: {bad.size} bytes differ, first at {bad[:8]}")
                n["slot"] += 1
                continue
        assert m == MODE_RAW, (b, blk, h, kind, m, nv)
        assert ntok[b, blk, h, kind] == nv
        np.testing.assert_array_equal(raws[idx[b, blk, h, kind]], O.raw_tile(tile, kind))
        n["raw"] += 1
    return n


def rel_err_rows(out: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Row-normwise error max_c |o - ref| / max_c |ref| per (b, h)."""
    num = np.abs(out - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    return np.where(den > 0, num / np.where(den > 0, den, 1), num)


ELEM_FLOOR = 1e-3  # element-wise error: |o - ref| / max(|ref|, ELEM_FLOOR * max_c |ref|) of the row
# Bar of the element-wise error, a secondary metric reported beside the row-normwise one: elements near
# the floor carry the row's absolute error over a denominator 1,000 times smaller than the row's maximum.
ELEM_TOL = 2e-2


def rel_err_elems(out: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Element-wise relative error per (b, h): max_c |o - ref| / max(|ref_c|, ELEM_FLOOR * max_c |ref|).
    Without a floor it is unbounded where an output element is near zero."""
    den = np.maximum(np.abs(ref), ELEM_FLOOR * np.abs(ref).max(axis=-1, keepdims=True))
    q = np.abs(out - ref) / np.where(den > 0, den, 1)
    q = np.where(den > 0, q, np.abs(out - ref))
    return q.max(axis=-1)


def oracle_attention(q, k, v, lens, scale, seqs=None):
    """fp64 oracle output [B, Hq, d] and flags [B, Hq] for the listed sequences (d = 128 or 256)."""
    qn, kn, vn = u16(q), u16(k), u16(v)
    lens_np = lens.cpu().numpy()
    B, Hq = q.shape[0], q.shape[1]
    ref = np.zeros((B, Hq, q.shape[-1]))
    flags = np.zeros((B, Hq), np.int32)
    for b in (range(B) if seqs is None else seqs):
        L = int(lens_np[b])
        ref[b], flags[b] = O.attention(qn[b], kn[b, :L], vn[b, :L], scale)
    return ref, flags


# Every check_attention call of the session, for the terminal summary (tests/conftest.py).
RECORD: list = []


class AttnCheck(tuple):
    """(worst row-normwise error, rows compared, rows flagged, worst element-wise error)."""

    def __new__(cls, worst, compared, flagged, worst_elem):
        return super().__new__(cls, (worst, compared, flagged, worst_elem))

    worst = property(lambda s: s[0])
    compared = property(lambda s: s[1])
    flagged = property(lambda s: s[2])
    worst_elem = property(lambda s: s[3])


def check_attention(out, q, k, v, lens, scale, seqs=None, tol=TOL, allow_flagged=False):
    """Kernel output against the fp64 oracle on every (sequence, q head) row of the listed sequences
    (all by default).  Rows the oracle flags as outside the fp32 range are not held to `tol`; unless
    allow_flagged, there must be none, so that every row is compared."""
    ref, flags = oracle_attention(q, k, v, lens, scale, seqs)
    o = out.double().cpu().numpy()
    rows = list(range(q.shape[0])) if seqs is None else list(seqs)
    err = rel_err_rows(o[rows], ref[rows])
    elem = rel_err_elems(o[rows], ref[rows])
    ok = flags[rows] == 0
    n_flag = int((~ok).sum())
    assert allow_flagged or n_flag == 0, f"{n_flag} rows flagged outside the fp32 range"
    assert np.isfinite(o[rows][ok]).all()
    worst = float(err[ok].max()) if ok.any() else 0.0
    worst_elem = float(elem[ok].max()) if ok.any() else 0.0
    assert worst <= tol, f"max relative error {worst:.3e} > {tol}"
    assert worst_elem <= ELEM_TOL, f"element-wise error {worst_elem:.3e} > {ELEM_TOL}"
    res = AttnCheck(worst, int(ok.sum()), n_flag, worst_elem)
    RECORD.append(res)
    return res


def lens_tensor(vals, device="cuda"):
    return torch.tensor(vals, dtype=torch.int32, device=device)


def kv(config, layer, B, T, H, adversarial=0.0, device="cuda"):
    return W.make_kv(config, layer, B, T, H, device=device, adversarial=adversarial)
