"""Pins of the oracle's open-tile encoding (the last block kept in its slot while decode tokens arrive,
"GAAC: Lossless KV Compression ..." section 3.3 and Figure 3; the layout is format v3's).

Reading: an element of a token not yet present is absent.  It takes no part in its group's mode, and
every field it owns is zero (mantissa, the sign bit it lends inside its aligned group of four, code,
escape bit, raw exponent byte).  Pinned by:
  * the full-tile encoder (itself pinned by the hand-derived golden images): the open image of the first
    n tokens equals the full encoding of a tile whose absent elements are filled with values that
    reproduce those zeros (sign and mantissa 0; exponent base3, base4 or 0 according to the mode of the
    group's present elements);
  * losslessness on the present tokens, a hand-derived one-token image, the monotone escape length, and
    n = 64 giving the sealed bytes.
"""
import numpy as np
import pytest

import gaac_workloads as W

NS = [1, 2, 7, 8, 9, 10, 15, 16, 17, 31, 40, 63, 64]


def _tile_and_bases(orc, seed, kind):
    k, v = W.make_kv(seed, 0, 1, 256, 1)
    x = W.bits(k if kind == 0 else v).numpy().view(np.uint16)[0, :, 0]  # [256][128]
    b3, b4 = orc.calibrate(x[:128, None, :])
    return x[128:192].copy(), b3[0], b4[0]


def _fill_absent(orc, tile, n, kind, b3, b4):
    """A full tile whose encoding must equal the open image of tile's first n tokens."""
    idx = np.array([[orc.storage_index(kind, t, c) for c in range(128)] for t in range(64)])
    tok = np.empty(8192, np.int64)
    ch = np.empty(8192, np.int64)
    tok[idx.reshape(-1)] = np.repeat(np.arange(64), 128)
    ch[idx.reshape(-1)] = np.tile(np.arange(128), 64)
    e = (tile[tok, ch] >> 7) & 0xFF
    pres = tok < n
    o3 = e.astype(np.int64) - b3[ch].astype(np.int64)
    o4 = e.astype(np.int64) - b4[ch].astype(np.int64)
    fit3 = ((~pres) | ((o3 >= 0) & (o3 <= 7))).reshape(1024, 8).all(axis=1)
    fit4 = ((~pres) | ((o4 >= 0) & (o4 <= 15))).reshape(1024, 8).all(axis=1)
    fill_e = np.where(np.repeat(fit3, 8), b3[ch], np.where(np.repeat(fit4, 8), b4[ch], 0)).astype(np.int64)
    out = tile.copy()
    absent = ~pres
    out[tok[absent], ch[absent]] = (fill_e[absent] << 7).astype(np.uint16)
    return out


@pytest.mark.parametrize("kind", [0, 1])
def test_open_image_equals_full_encoding_of_filled_tile(orc, kind):
    tile, b3, b4 = _tile_and_bases(orc, 5, kind)
    # widen a few groups so that 4-bit and raw groups straddle the open boundary
    tile[9, 3] = (tile[9, 3] & 0x807F) | ((int(b4[3]) + 12) << 7)
    tile[9, 40] = (tile[9, 40] & 0x807F) | (((int(b4[40]) + 40) & 0xFF) << 7)
    tile[1, 7] = (tile[1, 7] & 0x807F) | (((int(b4[7]) + 30) & 0xFF) << 7)
    for n in NS:
        img, esc = orc.encode_open_tile(tile, n, kind, b3, b4)
        ref, resc = orc.encode_tile(_fill_absent(orc, tile, n, kind, b3, b4), kind, b3, b4)
        assert esc == resc, n
        np.testing.assert_array_equal(img, ref, err_msg=f"n={n}")


@pytest.mark.parametrize("kind", [0, 1])
def test_open_image_lossless_monotone_and_sealed(orc, kind):
    tile, b3, b4 = _tile_and_bases(orc, 6, kind)
    last = -1
    for n in range(1, 65):
        img, esc = orc.encode_open_tile(tile, n, kind, b3, b4)
        assert esc >= last  # modes only widen as elements arrive
        last = esc
        back, st = orc.decode_tile(img, kind, b3, b4)
        assert st == esc
        np.testing.assert_array_equal(back[:n], tile[:n])
    full, fesc = orc.encode_tile(tile, kind, b3, b4)
    assert fesc == last
    np.testing.assert_array_equal(img, full)


def test_open_image_one_token_by_hand(orc):
    """K tile, n = 1, base3 = 120 and base4 = 112 on every channel.  Token 0 holds channel c with
    exponent 120 + c % 8 and mantissa c, the sign set on channel 5; channel 9's exponent is 113 (outside
    the 3-bit window), so group 1 (channels 8..15) is 4-bit: offsets from base4 are 8 + j except 1 for
    element 1, codes j, escape byte 0b11111101.  Tokens 1..63 hold data but are absent."""
    b3 = np.full(128, 120, np.uint8)
    b4 = np.full(128, 112, np.uint8)
    tile = np.full((64, 128), 0xBF80, np.uint16)  # absent tokens: -1.0 everywhere
    for c in range(128):
        tile[0, c] = ((120 + c % 8) << 7) | (c & 0x7F)
    tile[0, 5] |= 0x8000
    tile[0, 9] = (113 << 7) | 9
    img, esc = orc.encode_open_tile(tile, 1, 0, b3, b4)
    assert esc == 1
    exp = np.zeros_like(img)
    exp[:128] = np.arange(128)
    exp[6] |= 0x80  # byte s carries the sign of element 4(s/4) + (s+3)%4: element 5's sign sits in byte 6
    # code plane: every group of token 0 has codes 0..7 in element order (group 1: 0, 1, 2, ..., 7 as
    # well); unit u's words are plane words u, 256+u and 512+u, unit 0..3 = token 0
    for u in range(4):
        for h in range(2):
            w0 = 0
            w2 = 0
            for L in range(4):
                c0, c1, c2, c3 = L, 4 + L, L, 4 + L  # element 16h + {L, 4+L, 8+L, 12+L}: codes (j % 8)
                w0 |= (c0 | (c1 << 3) | ((c3 & 3) << 6)) << (8 * L)
                w2 |= ((c2 << (3 * h)) | (((c3 >> 2) & 1) << (6 + h))) << (8 * L)
            exp[8192 + 4 * (h * 256 + u): 8192 + 4 * (h * 256 + u) + 4] = np.frombuffer(np.uint32(w0).tobytes(), np.uint8)
            cur = int.from_bytes(exp[8192 + 4 * (512 + u): 8192 + 4 * (512 + u) + 4].tobytes(), "little")
            exp[8192 + 4 * (512 + u): 8192 + 4 * (512 + u) + 4] = np.frombuffer(np.uint32(cur | w2).tobytes(),
                                                                                  np.uint8)
    exp[11264] = 0b0100  # group 1 is 4-bit (tag 1 in bits 2-3 of the first tag byte)
    exp[11520:11536] = np.tile(np.array([1, 0], np.uint8), 8)  # every directory entry counts that one group
    exp[11536] = 0b11111101
    np.testing.assert_array_equal(img, exp)


def test_open_tile_argument_range(orc):
    t = np.zeros((64, 128), np.uint16)
    z = np.zeros(128, np.uint8)
    for n in (0, 65):
        with pytest.raises(ValueError):
            orc.encode_open_tile(t, n, 0, z, z)
