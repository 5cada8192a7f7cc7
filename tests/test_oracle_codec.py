"""Pins of the oracle codec against facts that do not come from the oracle.

Method: "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference on
Personal Devices", section 3.1 (lossless: sign and mantissa verbatim, exponent
coded with per-channel windows of 8 and 16, groups of eight widened as a whole)
and Appendix D (3-bit codes, 2-bit tags, escape bytes).

  * losslessness, exhaustively: all 65,536 BF16 patterns, both tile kinds, a
    sweep of window bases including the edges
  * the byte layout: hand-derived golden images (tests/golden)
  * the mode rule: brute force over every forced mode, validity judged by
    round trip alone; the encoder must pick the cheapest valid mode
  * the stream size: closed form sum of {0,1,8} bytes per group mode
  * the aggregate statistics: the Gaussian prediction of mode shares on the
    synthetic key distribution
"""
import json
import os

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
FULL_CAP = 8 * 1024  # every group raw: the largest escape stream a tile can have


def _bases(rng, kind):
    """Edge and random per-channel window bases (base3 <= 248, base4 <= 240)."""
    out = []
    edges3 = [0, 1, 120, 121, 122, 123, 124, 125, 126, 127, 240, 248]
    edges4 = [0, 1, 112, 116, 120, 124, 127, 240, 240, 240, 240, 240]
    for b3, b4 in zip(edges3, edges4):
        out.append((np.full(128, b3, np.uint8), np.full(128, b4, np.uint8)))
    for _ in range(16):
        out.append((rng.integers(0, 249, 128).astype(np.uint8), rng.integers(0, 241, 128).astype(np.uint8)))
    return out


@pytest.mark.parametrize("kind", [0, 1])
def test_exhaustive_roundtrip_all_bf16_patterns(orc, kind):
    """decode(encode(x)) == x for every one of the 65,536 BF16 bit patterns."""
    rng = np.random.default_rng(1234 + kind)
    patterns = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    arrangements = [patterns, rng.permutation(patterns)]
    seen_modes = np.zeros(4, np.int64)
    for b3, b4 in _bases(rng, kind):
        for arr in arrangements:
            for i in range(8):
                tile = arr[i * 8192:(i + 1) * 8192].reshape(64, 128)
                if kind == 1 and arr is patterns:  # consecutive patterns along the V storage order
                    tile = orc.unraw_tile(arr[i * 8192:(i + 1) * 8192], kind)
                img, esc = orc.encode_tile(tile, kind, b3, b4, esc_cap=FULL_CAP)
                assert esc >= 0
                dec, st = orc.decode_tile(img, kind, b3, b4, esc_limit=esc)
                assert st == esc
                np.testing.assert_array_equal(dec, tile)
                seen_modes += orc.mode_counts(img)
    assert seen_modes[0] > 0 and seen_modes[1] > 0 and seen_modes[2] > 0 and seen_modes[3] == 0


def _golden_tile(case):
    tile = np.full((64, 128), case["default_bits"], np.uint16)
    for t, c, b in case["elements"]:
        tile[t, c] = b
    return tile


def test_golden_format_examples(orc):
    cases = json.load(open(os.path.join(HERE, "golden", "format_v3_examples.json")))["cases"]
    for case in cases:
        tile = _golden_tile(case)
        b3 = np.full(128, case["base3"], np.uint8)
        b4 = np.full(128, case["base4"], np.uint8)
        img, esc = orc.encode_tile(tile, case["kind"], b3, b4)
        assert img.size == 12032
        assert esc == case["expect_esc_len"], case["name"]
        for lo, hi, val in case["expect_ranges"]:
            assert (img[lo:hi] == val).all(), (case["name"], lo, hi, val)
        for off, val in case["expect_bytes"]:
            assert img[off] == val, (case["name"], off, hex(img[off]), hex(val))
        dec, st = orc.decode_tile(img, case["kind"], b3, b4, esc)
        assert st == esc
        np.testing.assert_array_equal(dec, tile)


# V operand order (format v3), worked out by hand: (t, c) -> s
V_ORDER_PINS = [
    ((0, 0), 0),      # unit 0, element 0
    ((0, 8), 1),      # channel g+8 of the same 16-channel block: r bit 0
    ((1, 0), 2),      # the next token of the pair: r bit 1
    ((8, 0), 4),      # token + 8: r bit 2
    ((0, 16), 8),     # next 16-channel block: the next group of the unit
    ((2, 0), 32),     # next token pair: the next unit (lane q)
    ((0, 1), 128),    # next channel: unit + 4 (lane g)
    ((0, 64), 1024),  # upper 64 channels: the next eighth
    ((16, 0), 2048),  # next quarter of the tokens: two eighths on
    ((5, 3), 450),
    ((63, 127), 8191),
]


def _v_tc(s):
    """Inverse of the V operand order, restated from the format rule."""
    u, j = divmod(s, 32)
    eighth, lane = divmod(u, 32)
    w, h = divmod(eighth, 2)
    g, q = divmod(lane, 4)
    i, r = divmod(j, 8)
    return 16 * w + 8 * (r >> 2) + 2 * q + ((r >> 1) & 1), 16 * (4 * h + i) + 8 * (r & 1) + g


def test_storage_order_pins(orc):
    """K tiles are token-major; V tiles follow the operand order of format v3."""
    assert orc.storage_index(0, 5, 3) == 5 * 128 + 3
    for (t, c), s in V_ORDER_PINS:
        assert orc.storage_index(1, t, c) == s, (t, c)
        assert _v_tc(s) == (t, c)
    tile = np.arange(8192, dtype=np.uint16).reshape(64, 128)
    np.testing.assert_array_equal(orc.raw_tile(tile, 0), tile.reshape(-1))
    rv = orc.raw_tile(tile, 1)
    expect = np.array([tile[_v_tc(s)] for s in range(8192)], np.uint16)
    np.testing.assert_array_equal(rv, expect)
    assert sorted(rv.tolist()) == list(range(8192))  # a permutation
    np.testing.assert_array_equal(orc.unraw_tile(rv, 1), tile)


def test_v_units_are_operand_fragments(orc):
    """Each V unit 32*(2w+h) + 4g + q holds, for the 16-channel blocks 4h..4h+3,
    channels 16m+g and 16m+g+8 at tokens 16w + 2q + {0, 1, 8, 9}: one lane's
    share of a 16 x 16 (channels x tokens) operand tile."""
    for u in range(256):
        eighth, lane = divmod(u, 32)
        w, h = divmod(eighth, 2)
        g, q = divmod(lane, 4)
        want = {(16 * w + 2 * q + dt, 16 * m + g + dc) for m in range(4 * h, 4 * h + 4) for dt in (0, 1, 8, 9)
                for dc in (0, 8)}
        got = {(t, c) for t in range(64) for c in range(128) if orc.storage_index(1, t, c) // 32 == u}
        assert got == want, u


def _near_edge_exponents(rng, b3, b4, n):
    """Exponents mostly inside the 8-window, some on the 16-window's and the
    8-window's edges, a few far outside, so that all three modes occur."""
    inside3 = b3 + rng.integers(0, 8, n)
    edges = rng.choice(np.array([b3 - 1, b3 + 8, b4, b4 + 1, b4 + 14, b4 + 15, b4 - 1, b4 + 16]), n)
    far = rng.choice(np.array([0, 1, 254, 255, b3 + 40, b4 - 30]), n)
    u = rng.random(n)
    e = np.where(u < 0.85, inside3, np.where(u < 0.97, edges, far))
    return np.clip(e, 0, 255)


@pytest.mark.parametrize("kind", [0, 1])
def test_mode_minimality_brute_force(orc, kind):
    """Every group's mode must be the cheapest one that round-trips.

    For each candidate mode m in {3-bit, 4-bit, raw} the whole tile is encoded
    with every group forced to m; a group is valid under m when decoding that
    image reproduces its eight values.  Nothing about the mode rule is assumed.
    """
    rng = np.random.default_rng(77 + kind)
    for trial in range(6):
        b3 = rng.integers(100, 140, 128).astype(np.uint8)
        b4 = np.clip(b3.astype(int) - rng.integers(0, 9, 128), 0, 240).astype(np.uint8)
        # per-element exponent near its channel's windows
        ch = np.arange(128)
        e = np.stack([_near_edge_exponents(rng, int(b3[c]), int(b4[c]), 64) for c in ch], axis=1)
        sm = rng.integers(0, 256, (64, 128))
        tile = (((sm & 0x80) << 8) | (e.astype(np.int64) << 7) | (sm & 0x7F)).astype(np.uint16)
        # group g of storage order holds elements 8g..8g+7
        order = np.array([[orc.storage_index(kind, t, c) for c in range(128)] for t in range(64)])
        seq = np.empty(8192, np.uint16)
        seq[order.reshape(-1)] = tile.reshape(-1)
        valid = np.zeros((3, 1024), bool)
        for m in range(3):
            forced = np.full(1024, m, np.uint8)
            img, esc = orc.encode_tile(tile, kind, b3, b4, forced=forced, esc_cap=FULL_CAP)
            assert esc == 1024 * [0, 1, 8][m]
            dec, st = orc.decode_tile(img, kind, b3, b4, esc)
            dseq = np.empty(8192, np.uint16)
            dseq[order.reshape(-1)] = dec.reshape(-1)
            valid[m] = (dseq.reshape(1024, 8) == seq.reshape(1024, 8)).all(axis=1)
        assert valid[2].all(), "raw mode must always round-trip"
        cheapest = np.argmax(valid, axis=0)  # first valid mode in cost order 3-bit < 4-bit < raw
        img, esc = orc.encode_tile(tile, kind, b3, b4, esc_cap=FULL_CAP)
        tags = np.array([(img[11264 + g // 4] >> (2 * (g % 4))) & 3 for g in range(1024)])
        np.testing.assert_array_equal(tags, cheapest)
        assert (np.bincount(cheapest, minlength=3) > 0).all(), "the trial must exercise every mode"
        # closed form of the stream size
        counts = orc.mode_counts(img)
        assert esc == counts[1] * 1 + counts[2] * 8


def test_capacity_overflow_reported(orc):
    """A tile whose escape stream exceeds the 496-byte area is reported (-1): it must stay BF16."""
    rng = np.random.default_rng(5)
    tile = rng.integers(0, 65536, (64, 128)).astype(np.uint16)
    b3 = np.full(128, 124, np.uint8)
    b4 = np.full(128, 120, np.uint8)
    img, esc = orc.encode_tile(tile, 0, b3, b4)
    assert esc == -1
    img, esc = orc.encode_tile(tile, 0, b3, b4, esc_cap=FULL_CAP)
    assert esc > 496


def test_capacity_edge(orc):
    """496 escape bytes fit, 497 do not: 496 4-bit groups fill the area exactly, and so do
    62 raw groups (8 bytes each); one more 4-bit group next to them overflows."""
    b3 = np.full(128, 124, np.uint8)
    b4 = np.full(128, 120, np.uint8)
    tile = np.full((64, 128), 16256, np.uint16)  # 1.0: exponent 127, 3-bit mode
    flat = tile.reshape(-1)  # K storage order is token-major = logical order
    for n_wide, expect in ((496, 496), (497, -1)):
        t = flat.copy()
        t[8 * np.arange(n_wide)] = 135 << 7  # exponent 135: outside [124,131], inside [120,135]
        img, esc = orc.encode_tile(t.reshape(64, 128), 0, b3, b4)
        assert esc == expect
    for n_wide, expect in ((0, 496), (1, -1)):
        t = flat.copy()
        t[8 * np.arange(62)] = 200 << 7  # exponent 200: outside both windows, the group is raw
        t[8 * (62 + np.arange(n_wide))] = 135 << 7
        img, esc = orc.encode_tile(t.reshape(64, 128), 0, b3, b4)
        assert esc == expect
        if esc > 0:
            dec, st = orc.decode_tile(img, 0, b3, b4, esc)
            assert st == esc
            np.testing.assert_array_equal(dec, t.reshape(64, 128))


def _tags(img):
    return np.array([(int(img[11264 + g // 4]) >> (2 * (g % 4))) & 3 for g in range(1024)])


@pytest.mark.parametrize("kind", [0, 1])
def test_escape_directory_is_the_eighth_prefix(orc, kind):
    """Directory entry w = (4-bit groups of [0, 128(w+1))) + 512 * (raw groups there), counted
    from the tag plane; the escape area holds one byte per 4-bit group, then 8 per raw group."""
    rng = np.random.default_rng(77 + kind)
    for trial in range(6):
        b3 = rng.integers(100, 130, 128).astype(np.uint8)
        b4 = (b3.astype(int) - rng.integers(0, 8, 128)).clip(0, 240).astype(np.uint8)
        e = b3[None, :].astype(int) + rng.integers(-3, 12, (64, 128))
        e = np.where(rng.random((64, 128)) < 0.002, rng.integers(0, 255, (64, 128)), e).clip(0, 254)
        tile = ((rng.integers(0, 2, (64, 128)) << 15) | (e << 7) | rng.integers(0, 128, (64, 128))).astype(np.uint16)
        img, esc = orc.encode_tile(tile, kind, b3, b4, esc_cap=FULL_CAP)
        assert esc >= 0
        tags = _tags(img).reshape(8, 128)
        n4 = np.cumsum((tags == 1).sum(axis=1))
        nr = np.cumsum((tags == 2).sum(axis=1))
        got = img[11520:11536].view("<u2")
        np.testing.assert_array_equal(got, (n4 % 512) + 512 * (nr % 128))
        assert n4[7] + 8 * nr[7] == esc
        dec, st = orc.decode_tile(img, kind, b3, b4, esc_limit=esc)
        assert st == esc
        np.testing.assert_array_equal(dec, tile)


def test_corrupt_directory_rejected(orc):
    tile = np.full((64, 128), 16256, np.uint16)
    tile[20, 0] = 135 << 7  # one 4-bit group in eighth 2 (tokens 16-23)
    b3 = np.full(128, 124, np.uint8)
    b4 = np.full(128, 120, np.uint8)
    img, esc = orc.encode_tile(tile, 0, b3, b4)
    assert esc == 1
    assert list(img[11520:11536]) == [0, 0, 0, 0, 1, 0, 1, 0, 1, 0, 1, 0, 1, 0, 1, 0]
    bad = img.copy()
    bad[11520] = 1  # claims eighth 0 holds one escape byte
    _, st = orc.decode_tile(bad, 0, b3, b4, esc)
    assert st == -3


def test_sign_rotation_pins(orc):
    """Byte s of the sign|mantissa plane carries the mantissa of element s and the sign of
    element 4(s/4) + (s+3)%4: a single negative element at s sets bit 7 of byte 4(s/4) + (s+1)%4."""
    b = np.full(128, 124, np.uint8)
    for kind in (0, 1):
        for s in (0, 1, 2, 3, 4101, 8191):
            tile = np.full((64, 128), 16256, np.uint16)
            t, c = (s // 128, s % 128) if kind == 0 else _v_tc(s)
            tile[t, c] = 0xBF80 | 0x2D  # -1.0 with mantissa 0x2D
            img, esc = orc.encode_tile(tile, kind, b, b)
            holder = 4 * (s // 4) + (s + 1) % 4
            expect = np.zeros(8192, np.uint8)
            expect[s] |= 0x2D
            expect[holder] |= 0x80
            np.testing.assert_array_equal(img[:8192], expect)


def test_reserved_tag_rejected(orc):
    tile = np.full((64, 128), 16256, np.uint16)
    b = np.full(128, 124, np.uint8)
    img, esc = orc.encode_tile(tile, 0, b, b)
    img[11264 + 10] |= 0x3  # group 40 -> tag 3
    _, st = orc.decode_tile(img, 0, b, b, 0)
    assert st == -1


def _window_prob(sigma, lo_e, width):
    """P(BF16(z*sigma) has an exponent in [lo_e, lo_e+width)), z ~ N(0,1).
    Round to nearest even moves |x| >= 2^k (1 - 2^-9) up to exponent k."""
    from scipy.stats import norm

    lo = 2.0 ** (lo_e - 127) * (1 - 2.0 ** -9)
    hi = 2.0 ** (lo_e + width - 127) * (1 - 2.0 ** -9)
    return 2.0 * (norm.cdf(hi / sigma) - norm.cdf(lo / sigma))


def test_mode_shares_match_gaussian_prediction(orc):
    """The measured 3-bit / 4-bit / raw shares on synthetic keys agree with the
    shares the Gaussian model of the keys predicts for the calibrated windows."""
    pytest.importorskip("scipy")
    import gaac_workloads as W

    T, H = 2048, 8
    k, _ = W.make_kv(0, 0, 1, T, H)
    kb = W.bits(k).numpy().view(np.uint16)[0]
    sk, _ = W.channel_scales(0, 0, H)
    sk = sk.numpy().astype(np.float64)
    b3, b4 = orc.calibrate(kb[:512])
    counts = np.zeros(4)
    pred = np.zeros(3)
    n_groups = 0
    for h in range(H):
        p3 = np.array([_window_prob(sk[h, c], int(b3[h, c]), 8) for c in range(128)])
        p4 = np.array([_window_prob(sk[h, c], int(b4[h, c]), 16) for c in range(128)])
        lo = np.maximum(b3[h].astype(int), b4[h].astype(int))
        hi = np.minimum(b3[h].astype(int) + 8, b4[h].astype(int) + 16)
        p34 = np.array([_window_prob(sk[h, c], lo[c], hi[c] - lo[c]) if hi[c] > lo[c] else 0.0 for c in range(128)])
        # K groups: 8 consecutive channels of one token; channels independent
        for g in range(16):
            sl = slice(8 * g, 8 * g + 8)
            P3 = np.prod(p3[sl])
            P4 = np.prod(p4[sl])
            P34 = np.prod(p34[sl])
            pred += (T // 64) * 64 * np.array([P3, P4 - P34, 1 - P3 - (P4 - P34)])
        for blk in range(T // 64):
            img, esc = orc.encode_tile(kb[blk * 64:(blk + 1) * 64, h], 0, b3[h], b4[h], esc_cap=FULL_CAP)
            counts += orc.mode_counts(img)
            n_groups += 1024
    share = counts[:3] / n_groups
    pshare = pred / n_groups
    se = np.sqrt(pshare * (1 - pshare) / n_groups)
    assert share[0] > 0.8
    assert np.all(np.abs(share - pshare) < 6 * se + 2e-3), (share, pshare, se)
