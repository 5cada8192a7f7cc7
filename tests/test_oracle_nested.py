"""Pins of the oracle's nested 2-bit-mode ablation format (GAAC page, section 4.7.2 and Table 4: a 2-bit
mode nested inside the 3-bit one).  The format keeps format v3's sign|mantissa plane, tags and escape
area, and replaces the fixed 3-bit code planes with a code stream of 16 bits per 2-bit group, 24 per
3-bit or 4-bit group and none per raw group.  Pinned by a hand-derived image, losslessness on the
synthetic layer and on random tiles, and the measured ratio gain against format v3 on the same tiles."""
import numpy as np
import pytest

import gaac_workloads as W


def _dir_entry(n4, nraw, bits):
    return n4 | (nraw << 9) | (bits << 16)


def test_nested_image_by_hand(orc):
    """K tile, bases 112 (2-bit), 110 (3-bit), 100 (4-bit) on every channel; sign and mantissa 0.
    Token 0: group 0 exponents 112 + (0,1,2,3,3,2,1,0) (2-bit), group 1 110 + (7,...,0) (3-bit),
    group 2 108..115 (4-bit, offsets 8..15 from 100), group 3 1,2,3,4,250..253 (raw); every other
    element 112 (2-bit, code 0)."""
    b2 = np.full(128, 112, np.uint8)
    b3 = np.full(128, 110, np.uint8)
    b4 = np.full(128, 100, np.uint8)
    e = np.full((64, 128), 112, np.int64)
    e[0, 0:8] = 112 + np.array([0, 1, 2, 3, 3, 2, 1, 0])
    e[0, 8:16] = 110 + np.arange(7, -1, -1)
    e[0, 16:24] = 108 + np.arange(8)
    e[0, 24:32] = [1, 2, 3, 4, 250, 251, 252, 253]
    tile = (e << 7).astype(np.uint16)
    img, esc, bits = orc.nested_encode_tile(tile, 0, b2, b3, b4)
    assert esc == 9 and bits == 16 + 24 + 24 + 1020 * 16 == 16384
    exp = np.zeros(orc.nested_slot_bytes(), np.uint8)
    exp[8192:8200] = [0xE4, 0x1B, 0x77, 0x39, 0x05, 0x88, 0xC6, 0xFA]  # groups 0-2; the rest of the stream is 0
    exp[11264] = 0x93  # tags 3, 0, 1, 2
    exp[11265:11520] = 0xFF  # every other group 2-bit
    for w in range(8):
        exp[11520 + 4 * w: 11524 + 4 * w] = np.frombuffer(np.uint32(_dir_entry(1, 1, 2048 * (w + 1))).tobytes(),
                                                          np.uint8)
    exp[11552:11561] = [0xFF, 1, 2, 3, 4, 250, 251, 252, 253]
    np.testing.assert_array_equal(img, exp)
    back, st = orc.nested_decode_tile(img, 0, b2, b3, b4)
    assert st == 9
    np.testing.assert_array_equal(back, tile)


def test_nested_lossless_and_gain_on_synthetic_layer(orc):
    """Every tile of a synthetic layer (K and V, 4 kv-heads, 1024 tokens) round-trips; the code stream
    has 16 bits per 2-bit group and 24 per 3-bit or 4-bit group; and the payload gain over format v3 on
    the same tiles is the page's +2.3% (within sampling: 1.5% to 3.5%)."""
    T, H = 1024, 4
    k, v = W.make_kv(1, 0, 1, T + 512, H)
    v3_bytes = n_bytes = 0
    for x, kind in ((k, 0), (v, 1)):
        xb = W.bits(x).numpy().view(np.uint16)[0]
        b3, b4 = orc.calibrate(xb[:512])
        b2 = orc.nested_calibrate(xb[:512])
        for h in range(H):
            for blk in range(8, (T + 512) // 64):
                tile = xb[blk * 64:(blk + 1) * 64, h]
                img, esc, bits = orc.nested_encode_tile(tile, kind, b2[h], b3[h], b4[h])
                assert esc >= 0
                tags = np.unpackbits(img[11264:11520], bitorder="little").reshape(1024, 2)
                modes = tags[:, 0] | (tags[:, 1] << 1)
                counts = np.bincount(modes, minlength=4)
                assert bits == 16 * counts[3] + 24 * (counts[0] + counts[1])
                assert esc == counts[1] + 8 * counts[2]
                back, st = orc.nested_decode_tile(img, kind, b2[h], b3[h], b4[h])
                assert st == esc
                np.testing.assert_array_equal(back, tile)
                _, e3 = orc.encode_tile(tile, kind, b3[h], b4[h])
                v3_bytes += 11536 + e3
                n_bytes += 8192 + (bits + 7) // 8 + 256 + 32 + esc
    gain = v3_bytes / n_bytes - 1
    assert 0.015 < gain < 0.035, gain


def test_nested_random_tiles_round_trip(orc):
    rng = np.random.default_rng(21)
    for i in range(20):
        b2 = rng.integers(100, 130, 128).astype(np.uint8)
        b3 = (b2.astype(np.int64) - rng.integers(0, 5, 128)).astype(np.uint8)
        b4 = (b3.astype(np.int64) - rng.integers(0, 9, 128)).astype(np.uint8)
        e = b2[None, :].astype(np.int64) + rng.integers(-10, 12, (64, 128)) * (rng.random((64, 128)) < 0.05)
        tile = ((rng.integers(0, 2, (64, 128)) << 15) | (np.clip(e, 0, 254) << 7) | rng.integers(0, 128, (64, 128)))
        tile = tile.astype(np.uint16)
        for kind in (0, 1):
            img, esc, bits = orc.nested_encode_tile(tile, kind, b2, b3, b4)
            if esc < 0:
                continue
            back, st = orc.nested_decode_tile(img, kind, b2, b3, b4)
            assert st == esc
            np.testing.assert_array_equal(back, tile)


def test_nested_directory_checked(orc):
    b = np.full(128, 120, np.uint8)
    tile = np.full((64, 128), 120 << 7, np.uint16)
    img, esc, bits = orc.nested_encode_tile(tile, 1, b, b, b)
    assert esc == 0 and bits == 16 * 1024
    img[11520] ^= 1
    _, st = orc.nested_decode_tile(img, 1, b, b, b)
    assert st == -3
