"""GPU parity of the tile-batch codecs against the oracle: format v3 (gaac_encode_tiles /
gaac_decode_tiles) and the nested 2-bit-mode ablation format of the GAAC page's section 4.7.2
(gaac_nested_*).  Slot images and escape lengths must equal the oracle's byte for byte, decoding must
give the tiles back, and tiles whose escape stream does not fit must be reported and left untouched."""
import numpy as np
import pytest
import torch

import gaac_workloads as W
import lossless_compressed_kv_gaac_gb300 as G
import oracle as O

pytestmark = pytest.mark.gpu


def _tiles(x: torch.Tensor) -> torch.Tensor:
    """[T, H, 128] -> [H * (T/64), 64, 128] (head-major, then block)."""
    T, H, _ = x.shape
    return x.view(T // 64, 64, H, 128).permute(2, 0, 1, 3).reshape(-1, 64, 128).contiguous()


def _u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _batch(T=512, H=4, n_wild=3):
    k, v = W.make_kv(1, 0, 1, T + 256, H, device="cuda")
    kc, vc = k[0, :256], v[0, :256]
    tiles = torch.cat([_tiles(k[0, 256:]), _tiles(v[0, 256:])])
    nb = T // 64
    kinds = torch.cat([torch.zeros(H * nb), torch.ones(H * nb)]).to(torch.uint8)
    rows = torch.cat([torch.arange(H).repeat_interleave(nb), H + torch.arange(H).repeat_interleave(nb)]).int()
    rng = np.random.default_rng(3)
    wild = torch.from_numpy((rng.integers(0, 0x7F00, (n_wild, 64, 128)) | (rng.integers(0, 2, (n_wild, 64, 128)) << 15))
                            .astype(np.uint16).view(np.int16)).view(torch.bfloat16).cuda()
    tiles = torch.cat([tiles, wild]).contiguous()
    kinds = torch.cat([kinds, torch.tensor([0, 1, 0][:n_wild], dtype=torch.uint8)]).cuda()
    rows = torch.cat([rows, torch.tensor([0, H, 1][:n_wild], dtype=torch.int32)]).cuda()
    return kc, vc, tiles, kinds, rows


def test_v3_tile_batch_matches_oracle():
    kc, vc, tiles, kinds, rows = _batch()
    H = kc.shape[1]
    b3 = torch.zeros((2 * H, 128), dtype=torch.uint8, device="cuda")
    b4 = torch.zeros_like(b3)
    G.calibrate(kc, b3[:H], b4[:H])
    G.calibrate(vc, b3[H:], b4[H:])
    n = tiles.shape[0]
    slots = torch.zeros((n, G.SLOT_BYTES), dtype=torch.uint8, device="cuda")
    esc = torch.zeros(n, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.encode_tiles(tiles, kinds, rows, b3, b4, slots, esc, status=status)
    back = torch.zeros_like(tiles)
    G.decode_tiles(slots, esc, kinds, rows, b3, b4, back, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    tn, sn, en = _u16(tiles), slots.cpu().numpy(), esc.cpu().numpy().astype(np.int64) & 0xFFFF
    bn, b3n, b4n = _u16(back), b3.cpu().numpy(), b4.cpu().numpy()
    kn, rn = kinds.cpu().numpy(), rows.cpu().numpy()
    fitted = 0
    for i in range(n):
        img, e = O.encode_tile(tn[i], int(kn[i]), b3n[rn[i]], b4n[rn[i]])
        if e < 0:
            assert en[i] == 0xFFFF and not sn[i].any() and not bn[i].any(), i
            continue
        fitted += 1
        assert en[i] == e, i
        np.testing.assert_array_equal(sn[i], img, err_msg=f"tile {i}")
        np.testing.assert_array_equal(bn[i], tn[i])
    assert fitted == n - 3


def test_nested_codec_matches_oracle():
    kc, vc, tiles, kinds, rows = _batch()
    H = kc.shape[1]
    b2 = torch.zeros((2 * H, 128), dtype=torch.uint8, device="cuda")
    b3, b4 = torch.zeros_like(b2), torch.zeros_like(b2)
    G.calibrate(kc, b3[:H], b4[:H])
    G.calibrate(vc, b3[H:], b4[H:])
    G.nested_calibrate(kc, b2[:H])
    G.nested_calibrate(vc, b2[H:])
    ob2 = np.concatenate([O.nested_calibrate(_u16(kc)), O.nested_calibrate(_u16(vc))])
    np.testing.assert_array_equal(b2.cpu().numpy(), ob2)
    n = tiles.shape[0]
    slots = torch.zeros((n, G.NESTED_SLOT_BYTES), dtype=torch.uint8, device="cuda")
    esc = torch.zeros(n, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.nested_encode_tiles(tiles, kinds, rows, b2, b3, b4, slots, esc, status=status)
    back = torch.zeros_like(tiles)
    G.nested_decode_tiles(slots, esc, kinds, rows, b2, b3, b4, back, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    tn, sn, en = _u16(tiles), slots.cpu().numpy(), esc.cpu().numpy().astype(np.int64) & 0xFFFF
    bn = _u16(back)
    b2n, b3n, b4n = b2.cpu().numpy(), b3.cpu().numpy(), b4.cpu().numpy()
    kn, rn = kinds.cpu().numpy(), rows.cpu().numpy()
    fitted = n2 = 0
    for i in range(n):
        img, e, bits = O.nested_encode_tile(tn[i], int(kn[i]), b2n[rn[i]], b3n[rn[i]], b4n[rn[i]])
        if e < 0:
            assert en[i] == 0xFFFF and not sn[i].any() and not bn[i].any(), i
            continue
        fitted += 1
        assert en[i] == e, i
        np.testing.assert_array_equal(sn[i], img, err_msg=f"tile {i}")
        np.testing.assert_array_equal(bn[i], tn[i])
        n2 += bits < 24 * 1024
    assert fitted == n - 3 and n2 == fitted  # every synthetic tile has some 2-bit groups


def test_tile_batch_bad_row_reported():
    kc, vc, tiles, kinds, rows = _batch(T=128, H=1, n_wild=1)
    b = torch.full((2, 128), 120, dtype=torch.uint8, device="cuda")
    n = tiles.shape[0]
    bad = torch.full((n,), 7, dtype=torch.int32, device="cuda")
    for nested in (False, True):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        esc = torch.zeros(n, dtype=torch.int16, device="cuda")
        if nested:
            slots = torch.zeros((n, G.NESTED_SLOT_BYTES), dtype=torch.uint8, device="cuda")
            G.nested_encode_tiles(tiles, kinds, bad, b, b, b, slots, esc, status=status)
        else:
            slots = torch.zeros((n, G.SLOT_BYTES), dtype=torch.uint8, device="cuda")
            G.encode_tiles(tiles, kinds, bad, b, b, slots, esc, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == G.EINVAL
        assert ((esc.cpu().numpy().astype(np.int64) & 0xFFFF) == 0xFFFF).all()
        assert not slots.any().item()


def _wild_base_batch():
    """Base rows: all out of the calibrated ranges, random over [0, 255], random inside them, at their
    limits.  base4 lies 3-8 below base3, so a 4-bit window holds the 3-bit one and the three exponents
    below it.  Exponents are base3 plus an offset: in [0, 7] for 97.7% of elements, one or three below it
    (4-bit groups) for 2.1%, 40 away (raw groups) for 0.2%; sign and mantissa are random."""
    rng = np.random.default_rng(11)
    b3 = np.stack([rng.integers(249, 256, 128), rng.integers(0, 256, 128), rng.integers(8, 249, 128),
                   np.full(128, 248)])
    b4 = np.clip(b3 - rng.integers(3, 9, (4, 128)), 0, 255)
    b4[2] = np.minimum(b4[2], 240)
    b4[3] = 240
    tiles, kinds, rows = [], [], []
    for r in range(4):
        for kind in (0, 1):
            for _ in range(2):
                off = rng.choice([0, 1, 2, 3, 4, 5, 6, 7, -1, -3, 40, -40], (64, 128),
                                 p=[.2, .2, .15, .12, .1, .08, .072, .055, .012, .009, .001, .001])
                e = np.clip(b3[r][None, :] + off, 0, 255)
                x = (rng.integers(0, 2, (64, 128)) << 15) | (e << 7) | rng.integers(0, 128, (64, 128))
                tiles.append(x.astype(np.uint16))
                kinds.append(kind)
                rows.append(r)
    return np.stack(tiles), kinds, rows, b3.astype(np.uint8), b4.astype(np.uint8)


def test_v3_tile_batch_any_bases_match_oracle():
    """Bases anywhere in [0, 255] (calibration gives base3 <= 248 and base4 <= 240; the encoder decides a
    group's fit a word at a time only for those, element by element otherwise)."""
    tn, kinds, rows, b3, b4 = _wild_base_batch()
    n = tn.shape[0]
    t_dev = torch.from_numpy(tn.view(np.int16)).view(torch.bfloat16).cuda()
    k_dev = torch.tensor(kinds, dtype=torch.uint8, device="cuda")
    r_dev = torch.tensor(rows, dtype=torch.int32, device="cuda")
    b3d, b4d = torch.from_numpy(b3).cuda(), torch.from_numpy(b4).cuda()
    slots = torch.zeros((n, G.SLOT_BYTES), dtype=torch.uint8, device="cuda")
    esc = torch.zeros(n, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    G.encode_tiles(t_dev, k_dev, r_dev, b3d, b4d, slots, esc, status=status)
    back = torch.zeros_like(t_dev)
    G.decode_tiles(slots, esc, k_dev, r_dev, b3d, b4d, back, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sn, en, bn = slots.cpu().numpy(), esc.cpu().numpy().astype(np.int64) & 0xFFFF, _u16(back)
    for i in range(n):
        img, e = O.encode_tile(tn[i], kinds[i], b3[rows[i]], b4[rows[i]])
        assert e >= 0, i  # the batch is built to fit
        assert en[i] == e, i
        np.testing.assert_array_equal(sn[i], img, err_msg=f"tile {i}")
        np.testing.assert_array_equal(bn[i], tn[i])
