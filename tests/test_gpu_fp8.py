"""GPU parity of the FP8 variant of the codec (GAAC page, Appendix B) against the oracle.

Inputs are the seeded synthetic K/V of the workloads, converted to FP8 (E4M3
and E5M2) with torch's round-to-nearest casts, plus adversarial random bytes.
Calibration bases and slot images must match the oracle byte for byte, and
decoding must give the FP8 tiles back exactly."""
import numpy as np
import pytest
import torch

import gaac_workloads as W
import lossless_compressed_kv_gaac_gb300 as G
import oracle as O

pytestmark = pytest.mark.gpu

FP8_DTYPES = {G.FP8_E4M3: "float8_e4m3fn", G.FP8_E5M2: "float8_e5m2"}


def _fp8(x: torch.Tensor, fmt: int) -> torch.Tensor:
    return x.float().to(getattr(torch, FP8_DTYPES[fmt])).view(torch.uint8)


def _tiles(x: torch.Tensor) -> torch.Tensor:
    """[T, H, 128] uint8 -> [H * (T/64), 64, 128] (head-major, then block)."""
    T, H, _ = x.shape
    return x.view(T // 64, 64, H, 128).permute(2, 0, 1, 3).reshape(-1, 64, 128).contiguous()


def _run(tiles, kinds, rows, b3, b4, fmt):
    n = tiles.shape[0]
    slots = torch.zeros((n, G.fp8_slot_bytes(fmt)), dtype=torch.uint8, device="cuda")
    esc = torch.zeros(n, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stats = G.new_stats()
    G.fp8_encode_tiles(tiles, fmt, kinds, rows, b3, b4, slots, esc, stats=stats, status=status)
    back = torch.zeros_like(tiles)
    G.fp8_decompress_tiles(slots, esc, fmt, kinds, rows, b3, b4, back, status=status)
    torch.cuda.synchronize()
    return slots, esc.view(torch.int16).cpu().numpy().astype(np.int64) & 0xFFFF, back, int(status.item()), G.stats_dict(stats)


@pytest.mark.parametrize("fmt", [G.FP8_E4M3, G.FP8_E5M2])
def test_fp8_codec_matches_oracle(fmt):
    T, H = 512, 8
    k, v = W.make_kv(0, 0, 1, T, H, device="cuda")
    k8, v8 = _fp8(k[0], fmt), _fp8(v[0], fmt)
    b3 = torch.zeros((2 * H, 128), dtype=torch.uint8, device="cuda")
    b4 = torch.zeros_like(b3)
    G.fp8_calibrate(k8[:256], fmt, b3[:H], b4[:H])
    G.fp8_calibrate(v8[:256], fmt, b3[H:], b4[H:])
    ob3k, ob4k = O.fp8_calibrate(k8[:256].cpu().numpy(), fmt)
    ob3v, ob4v = O.fp8_calibrate(v8[:256].cpu().numpy(), fmt)
    np.testing.assert_array_equal(b3.cpu().numpy(), np.concatenate([ob3k, ob3v]))
    np.testing.assert_array_equal(b4.cpu().numpy(), np.concatenate([ob4k, ob4v]))
    tiles = torch.cat([_tiles(k8), _tiles(v8)])  # K tiles of heads 0..7, then V tiles
    nb = T // 64
    kinds = torch.cat([torch.zeros(H * nb, dtype=torch.uint8), torch.ones(H * nb, dtype=torch.uint8)]).cuda()
    rows = torch.cat([torch.arange(H).repeat_interleave(nb), H + torch.arange(H).repeat_interleave(nb)]).int().cuda()
    slots, esc, back, status, stats = _run(tiles, kinds, rows, b3, b4, fmt)
    assert status == 0
    torch.testing.assert_close(back, tiles, rtol=0, atol=0)
    tn, sn = tiles.cpu().numpy(), slots.cpu().numpy()
    kn, rn, b3n, b4n = kinds.cpu().numpy(), rows.cpu().numpy(), b3.cpu().numpy(), b4.cpu().numpy()
    fitted = 0
    for i in range(tn.shape[0]):
        img, oesc = O.fp8_encode_tile(tn[i], int(kn[i]), fmt, b3n[rn[i]], b4n[rn[i]])
        if oesc < 0:
            assert esc[i] == 0xFFFF, i
            continue
        fitted += 1
        assert esc[i] == oesc, i
        np.testing.assert_array_equal(sn[i], img, err_msg=f"tile {i}")
    assert fitted > 0
    assert stats["slot_tiles"] == fitted
    payload = sum(O.FP8_OFF_ESC[fmt] + int(e) for e in esc if e != 0xFFFF) + 8192 * (tn.shape[0] - fitted)
    assert tn.shape[0] * 8192 / payload > 1.0  # compression on the synthetic keys and values


@pytest.mark.parametrize("fmt", [G.FP8_E4M3, G.FP8_E5M2])
def test_fp8_random_bytes_overflow_and_edges(fmt):
    """Random bytes: most tiles overflow their escape area (esc_len 0xFFFF, slot untouched); a tile of
    one repeated value per channel always fits; bad rows are reported."""
    rng = np.random.default_rng(11 + fmt)
    n = 6
    tn = rng.integers(0, 256, (n, 64, 128)).astype(np.uint8)
    b3n = rng.integers(0, (16 if fmt == 0 else 32) - 7, (2, 128)).astype(np.uint8)
    b4n = np.zeros_like(b3n) if fmt == 0 else rng.integers(0, 17, (2, 128)).astype(np.uint8)
    mw = 3 if fmt == 0 else 2
    # tile 1 (V, row 1): every channel's exponent at its base3, so every group is 3-bit
    tn[1] = ((b3n[1].astype(np.int64) << mw) | (np.arange(128) & ((1 << mw) - 1)))[None, :].astype(np.uint8)
    tiles = torch.from_numpy(tn).cuda()
    b3, b4 = torch.from_numpy(b3n).cuda(), torch.from_numpy(b4n).cuda()
    kinds = torch.tensor([0, 1, 0, 1, 0, 1], dtype=torch.uint8, device="cuda")
    rows = torch.tensor([0, 1, 1, 0, 0, 1], dtype=torch.int32, device="cuda")
    slots, esc, back, status, _ = _run(tiles, kinds, rows, b3, b4, fmt)
    assert status == 0
    for i in range(n):
        img, oesc = O.fp8_encode_tile(tn[i], int(kinds[i]), fmt, b3[rows[i]].cpu().numpy(), b4[rows[i]].cpu().numpy())
        if oesc < 0:
            assert esc[i] == 0xFFFF
            assert (slots[i].cpu().numpy() == 0).all()  # not written
            assert (back[i].cpu().numpy() == 0).all()  # not decoded
        else:
            assert esc[i] == oesc
            np.testing.assert_array_equal(slots[i].cpu().numpy(), img)
            np.testing.assert_array_equal(back[i].cpu().numpy(), tn[i])
    assert esc[1] != 0xFFFF
    # a row past the bases is an argument error found by the kernel
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_rows = torch.full((n,), 5, dtype=torch.int32, device="cuda")
    e2 = torch.zeros(n, dtype=torch.int16, device="cuda")
    G.fp8_encode_tiles(tiles, fmt, kinds, bad_rows, b3, b4, torch.zeros_like(slots), e2, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == G.EINVAL
    assert ((e2.cpu().numpy().astype(np.int64) & 0xFFFF) == 0xFFFF).all()


@pytest.mark.parametrize("fmt", [G.FP8_E4M3, G.FP8_E5M2])
def test_fp8_out_of_range_bases_match_oracle(fmt):
    """A row with a base3 above 248 or a base4 above 240 (calibration never gives one) is encoded
    element by element; every tile, of those rows and of the others, must equal the oracle's."""
    T, H = 256, 4
    k, v = W.make_kv(0, 1, 1, T, H, device="cuda")
    k8, v8 = _fp8(k[0], fmt), _fp8(v[0], fmt)
    b3 = torch.zeros((2 * H, 128), dtype=torch.uint8, device="cuda")
    b4 = torch.zeros_like(b3)
    G.fp8_calibrate(k8, fmt, b3[:H], b4[:H])
    G.fp8_calibrate(v8, fmt, b3[H:], b4[H:])
    b3[0, 5] = 250  # K row 0
    b4[H + 1, 77] = 245  # V row 1
    tiles = torch.cat([_tiles(k8), _tiles(v8)])
    nb = T // 64
    kinds = torch.cat([torch.zeros(H * nb, dtype=torch.uint8), torch.ones(H * nb, dtype=torch.uint8)]).cuda()
    rows = torch.cat([torch.arange(H).repeat_interleave(nb), H + torch.arange(H).repeat_interleave(nb)]).int().cuda()
    slots, esc, back, status, _ = _run(tiles, kinds, rows, b3, b4, fmt)
    assert status == 0
    tn, sn, bn = tiles.cpu().numpy(), slots.cpu().numpy(), back.cpu().numpy()
    kn, rn, b3n, b4n = kinds.cpu().numpy(), rows.cpu().numpy(), b3.cpu().numpy(), b4.cpu().numpy()
    for i in range(tn.shape[0]):
        img, oesc = O.fp8_encode_tile(tn[i], int(kn[i]), fmt, b3n[rn[i]], b4n[rn[i]])
        if oesc < 0:
            assert esc[i] == 0xFFFF, i
            continue
        assert esc[i] == oesc, i
        np.testing.assert_array_equal(sn[i], img, err_msg=f"tile {i}")
        np.testing.assert_array_equal(bn[i], tn[i])
