"""CUDA path against the oracle, through the C ABI (marked gpu).

Bit-exact: calibration bases, slot images (byte for byte, per logical tile of
the table), raw tiles, decompression.  Attention: within 2e-3 max relative
error (row-normwise) of the fp64 oracle on every (sequence, q head) row; each
test asserts how many rows it compared (the oracle flags none of these inputs
as outside the fp32 range).

Method: "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference
on Personal Devices", sections 3.1 (codec), 3.2 (fused attention), 3.3 (slots,
raw fallback, BF16 tail).
"""
import numpy as np
import pytest
import torch

import gaac_workloads as W
import oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import lossless_compressed_kv_gaac_gb300 as G
    from lossless_compressed_kv_gaac_gb300.cache import LayerCache
    from tests import gpu_util as U


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    G.lib()


def _status(c):
    torch.cuda.synchronize()
    return int(c.status.item())


def test_calibrate_bit_exact():
    k, v = U.kv(0, 0, 1, 1024, 8)
    c = U.build(k, v, U.lens_tensor([1024]))
    b3, b4 = U.oracle_bases(k, v)
    np.testing.assert_array_equal(c.base3.cpu().numpy(), b3)
    np.testing.assert_array_equal(c.base4.cpu().numpy(), b4)
    # a flat histogram region and random bits
    rng = np.random.default_rng(0)
    x = torch.from_numpy(rng.integers(0, 65536, (777, 3, 128)).astype(np.int64).astype(np.int16)).cuda()
    g3 = torch.zeros(3, 128, dtype=torch.uint8, device="cuda")
    g4 = torch.zeros_like(g3)
    G.calibrate(x.view(torch.bfloat16), g3, g4)
    r3, r4 = O.calibrate(U.u16(x))
    np.testing.assert_array_equal(g3.cpu().numpy(), r3)
    np.testing.assert_array_equal(g4.cpu().numpy(), r4)


def test_config0_encode_decompress_attention():
    """Config 0: 1 layer, batch 1, 16q/8kv, T=4096, calibrate on 512 tokens, scale 1/sqrt(128)."""
    wl = W.WORKLOADS[0]
    k, v = U.kv(0, 0, 1, wl.seq_len, wl.n_kv_heads)
    lens = U.lens_tensor([wl.seq_len])
    c = U.build(k, v, lens)
    assert _status(c) == 0
    n = U.check_tiles(c, k, v, lens)
    assert n["slot"] > 0.95 * (64 * 8 * 2)
    kd, vd = c.decompress(wl.seq_len)
    assert torch.equal(kd.view(torch.int16), k.view(torch.int16))
    assert torch.equal(vd.view(torch.int16), v.view(torch.int16))
    q = W.make_q(0, 0, 1, wl.n_q_heads, device="cuda")
    out = c.attention(q, wl.scale)
    assert _status(c) == 0
    assert U.check_attention(out, q, k, v, lens, wl.scale).compared == wl.n_q_heads
    st = G.stats_dict(c.stats)
    assert st["groups0"] + st["groups1"] + st["groups2"] == 1024 * st["slot_tiles"]


def test_block_encoder_out_of_range_bases():
    """Bases above the calibrated ranges (base3 > 248 or base4 > 240; calibration never gives one) send a
    head's tiles down the block encoder's element-by-element fit: every tile of those heads and of the others
    must still equal the oracle's image, and the cache must decode and attend exactly as with calibrated
    bases.  Ragged lengths put open tails (raw) beside sealed tiles."""
    lens_v = [1024, 700, 65]
    B, T, H = len(lens_v), 1024, 4
    k, v = U.kv(0, 3, B, T, H)
    lens = U.lens_tensor(lens_v)
    c = LayerCache(B, H, T // 64, device=k.device)
    c.calibrate(k[0, :512], v[0, :512])
    c.base3[0, 0, 5] = 250  # K of head 0
    c.base4[1, 1, 77] = 245  # V of head 1
    c.base3[1, 3, 0] = 255  # V of head 3
    c.encode(k, v, lens)
    assert _status(c) == 0
    b3, b4 = c.base3.cpu().numpy(), c.base4.cpu().numpy()
    n = U.check_tiles(c, k, v, lens, b3=b3, b4=b4)
    assert n["slot"] > 0 and n["raw"] >= 2 * H * 2  # the two ragged sequences' open tails
    kd, vd = c.decompress(T)
    for b, L in enumerate(lens_v):
        assert torch.equal(kd[b, :L].view(torch.int16), k[b, :L].view(torch.int16))
        assert torch.equal(vd[b, :L].view(torch.int16), v[b, :L].view(torch.int16))
    q = W.make_q(0, 3, B, 16, device="cuda")
    out = c.attention(q, 1 / np.sqrt(128))
    assert _status(c) == 0
    assert U.check_attention(out, q, k, v, lens, 1 / np.sqrt(128)).compared == B * 16


@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8), (8, 8), (64, 8), (12, 4)])
def test_ragged_lengths_and_gqa(hq, hkv):
    lens_v = [0, 1, 63, 64, 65, 700, 1024, 333]
    B, T = len(lens_v), 1024
    k, v = U.kv(0, 1, B, T, hkv)
    lens = U.lens_tensor(lens_v)
    c = U.build(k, v, lens, n_calib=512)
    assert _status(c) == 0
    U.check_tiles(c, k, v, lens)
    kd, vd = c.decompress(T)
    for b, L in enumerate(lens_v):
        assert torch.equal(kd[b, :L].view(torch.int16), k[b, :L].view(torch.int16))
        assert torch.equal(vd[b, :L].view(torch.int16), v[b, :L].view(torch.int16))
    q = W.make_q(0, 1, B, hq, device="cuda")
    for n_splits in (1, 3, 0, 2):  # the last call reuses a workspace sized for more splits
        out = c.attention(q, 1 / np.sqrt(128), n_splits=n_splits)
        assert _status(c) == 0
        assert U.check_attention(out, q, k, v, lens, 1 / np.sqrt(128)).compared == B * hq
    assert out[0].abs().max().item() == 0.0  # empty sequence -> zeros


def test_all_raw_baseline_same_outputs():
    """The uncompressed baseline: every block stored raw, read by the compressed kernel's raw path and by
    the BF16 kernel (the same kernel without a decode path); both against the oracle, and the BF16 kernel
    on a compressed cache reports a format error."""
    k, v = U.kv(0, 2, 2, 2048, 8)
    lens = U.lens_tensor([2048, 1500])
    c = U.build(k, v, lens, raw=True)
    assert _status(c) == 0
    n = U.check_tiles(c, k, v, lens, raw_all=True)
    assert n["slot"] == 0
    q = W.make_q(0, 2, 2, 32, device="cuda")
    out = c.attention(q, 1 / np.sqrt(128))
    assert U.check_attention(out, q, k, v, lens, 1 / np.sqrt(128)).compared == 2 * 32
    cz = U.build(k, v, lens)
    outz = cz.attention(q, 1 / np.sqrt(128))
    torch.cuda.synchronize()
    assert (out - outz).abs().max().item() < 1e-5
    for n_splits in (1, 5, 0):
        ob = c.attention(q, 1 / np.sqrt(128), n_splits=n_splits, bf16=True)
        assert _status(c) == 0
        assert U.check_attention(ob, q, k, v, lens, 1 / np.sqrt(128)).compared == 2 * 32
    assert (ob - out).abs().max().item() < 1e-5  # the same values through the compressed kernel's raw path
    cz.attention(q, 1 / np.sqrt(128), bf16=True)
    assert _status(cz) == G.EFORMAT


@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8), (64, 8)])
def test_bf16_kernel_ragged_lengths(hq, hkv):
    """The BF16 kernel over ragged lengths (empty, one token, block edges, open tails) and GQA ratios."""
    lens_v = [0, 1, 63, 64, 65, 700, 1024, 333]
    B, T = len(lens_v), 1024
    k, v = U.kv(0, 9, B, T, hkv)
    lens = U.lens_tensor(lens_v)
    c = U.build(k, v, lens, raw=True)
    assert _status(c) == 0
    q = W.make_q(0, 9, B, hq, device="cuda")
    for n_splits in (1, 3, 0):
        out = c.attention(q, 1 / np.sqrt(128), n_splits=n_splits, bf16=True)
        assert _status(c) == 0
        assert U.check_attention(out, q, k, v, lens, 1 / np.sqrt(128)).compared == B * hq
    assert out[0].abs().max().item() == 0.0


def test_incremental_append_equals_one_shot():
    """Config 3 shape, small: prefill then appends; sealed tiles equal a one-shot encode of the final cache."""
    B, H, T0, steps = 3, 8, 200, 130
    T = T0 + steps
    k, v = U.kv(3, 0, B, T, H)
    max_blocks = (T + 63) // 64 + 1
    inc = LayerCache(B, H, max_blocks)
    inc.calibrate(k[0, :T0], v[0, :T0])
    inc.encode(k[:, :T0], v[:, :T0], U.lens_tensor([T0] * B))
    q = W.make_q(3, 0, B, 16, device="cuda")
    for s in range(steps):
        inc.append(k[:, T0 + s].contiguous(), v[:, T0 + s].contiguous())
        if s in (0, 55, 56, 57, steps - 1):
            out = inc.attention(q, 1 / np.sqrt(128))
            torch.cuda.synchronize()
            L = T0 + s + 1
            U.check_attention(out, q, k[:, :L], v[:, :L], U.lens_tensor([L] * B), 1 / np.sqrt(128))
    assert _status(inc) == 0
    assert inc.seq_lens.tolist() == [T] * B
    one = LayerCache(B, H, max_blocks)
    one.base3.copy_(inc.base3)
    one.base4.copy_(inc.base4)
    one.encode(k, v, U.lens_tensor([T] * B))
    torch.cuda.synchronize()
    b3, b4 = inc.base3.cpu().numpy(), inc.base4.cpu().numpy()
    U.check_tiles(inc, k, v, inc.seq_lens, b3=b3, b4=b4)
    U.check_tiles(one, k, v, one.seq_lens, b3=b3, b4=b4)
    kd, vd = inc.decompress(T)
    assert torch.equal(kd.view(torch.int16), k.view(torch.int16))
    assert torch.equal(vd.view(torch.int16), v.view(torch.int16))


def test_adversarial_small():
    """Config 4 shape, small: 10% random-bit tokens after 512 clean ones."""
    B, T, H = 2, 4096, 8
    k, v = U.kv(4, 0, B, T, H, adversarial=0.1)
    lens = U.lens_tensor([T, T - 100])
    c = U.build(k, v, lens)
    assert _status(c) == 0
    n = U.check_tiles(c, k, v, lens)
    assert n["raw"] > 0 and n["slot"] > 0
    kd, vd = c.decompress(T)
    assert torch.equal(kd[0].view(torch.int16), k[0].view(torch.int16))
    q = W.make_q(4, 0, B, 32, device="cuda")
    out = c.attention(q, 1 / np.sqrt(128))
    assert U.check_attention(out, q, k, v, lens, 1 / np.sqrt(128)).compared == B * 32


def test_paged_scattered_slots():
    """Config 2 shape, small: variable lengths, full blocks scattered over a shared slot pool."""
    B, H, maxT = 8, 8, 2048
    lens = W.make_lengths(2, B, 300, maxT, device="cuda")
    k, v = U.kv(2, 0, B, maxT, H)
    max_blocks = maxT // 64
    positions = B * max_blocks * H * 2
    pool = 2 * positions
    perm = W.slot_permutation(2, 0, pool, device="cuda")[:positions].to(torch.int32)
    slot_ids = perm.view(B, max_blocks, H, 2)
    c = U.build(k, v, lens, slot_ids=slot_ids, n_slots=pool)
    assert _status(c) == 0
    U.check_tiles(c, k, v, lens)
    q = W.make_q(2, 0, B, 16, device="cuda")
    out = c.attention(q, 1 / np.sqrt(128))
    U.check_attention(out, q, k, v, lens, 1 / np.sqrt(128))


def test_full_size_config1_layer():
    """Config 1 sizes, one layer: T=65536, 32q/8kv, in the bench's launch configuration (auto splits)."""
    T, H, Hq = 65536, 8, 32
    k, v = U.kv(1, 0, 1, T, H)
    lens = U.lens_tensor([T])
    c = U.build(k, v, lens)
    assert _status(c) == 0
    n = U.check_tiles(c, k, v, lens)  # all 16,384 tiles of the layer, byte for byte
    assert n["slot"] + n["raw"] == 1024 * H * 2
    kd, vd = c.decompress(T)
    assert torch.equal(kd.view(torch.int16), k.view(torch.int16))
    assert torch.equal(vd.view(torch.int16), v.view(torch.int16))
    q = W.make_q(1, 0, 1, Hq, device="cuda")
    out = c.attention(q, 1 / np.sqrt(128))
    assert _status(c) == 0
    assert U.check_attention(out, q, k, v, lens, 1 / np.sqrt(128)).compared == Hq


def test_full_size_config4():
    """Config 4 sizes: batch 4, T=131072, 10% random-bit tokens; attention on every row."""
    B, T, H, Hq = 4, 131072, 8, 32
    k, v = U.kv(4, 0, B, T, H, adversarial=0.1)
    lens = U.lens_tensor([T] * B)
    c = U.build(k, v, lens)
    assert _status(c) == 0
    rng = np.random.default_rng(4)
    tiles = [(int(rng.integers(0, B)), int(rng.integers(0, 2048)), int(rng.integers(0, H)), int(rng.integers(0, 2)))
             for _ in range(300)]
    n = U.check_tiles(c, k, v, lens, tiles=tiles)
    assert n["raw"] > 0
    kd, vd = c.decompress(T)
    assert torch.equal(kd.view(torch.int16), k.view(torch.int16))
    assert torch.equal(vd.view(torch.int16), v.view(torch.int16))
    del kd, vd
    q = W.make_q(4, 0, B, Hq, device="cuda")
    out = c.attention(q, 1 / np.sqrt(128))
    assert _status(c) == 0
    # every one of the 128 rows: the random-bit keys bring sum_c |q_c k_c| near 2^131, yet each logit is an
    # fp32 number and the kernel never scales a score before subtracting its running maximum
    assert U.check_attention(out, q, k, v, lens, 1 / np.sqrt(128)).compared == B * Hq


def test_device_errors_are_reported_not_faulted():
    k, v = U.kv(0, 3, 2, 512, 8)
    lens = U.lens_tensor([512, 300])
    c = U.build(k, v, lens)
    assert _status(c) == 0
    q = W.make_q(0, 3, 2, 16, device="cuda")
    good = c.attention(q, 0.1).clone()
    # a table entry with an unknown mode and one with an out-of-range index
    c.table[0, 2, 1, 0] = (7 << 48)
    c.table[1, 1, 3, 1] = (G.MODE_SLOT << 48) | (10 ** 9)
    c.status.zero_()
    out = c.attention(q, 0.1)
    assert _status(c) == G.EFORMAT
    assert torch.isfinite(out).all()
    # entry (0,2,1,K) feeds q heads 2,3 of sequence 0; entry (1,1,3,V) q heads 6,7 of sequence 1
    assert torch.equal(out[0, :2], good[0, :2]) and torch.equal(out[0, 4:], good[0, 4:])
    assert torch.equal(out[1, :6], good[1, :6]) and torch.equal(out[1, 8:], good[1, 8:])
    # raw pool exhaustion during encode
    c2 = LayerCache(2, 8, 8, n_raw=3)
    c2.calibrate(k[0], v[0])
    c2.encode(k, v, lens)
    assert _status(c2) == G.EPOOL
    # host-side validation
    with pytest.raises(G.GaacError):
        G.decode_attention(q, c.seq_lens, c.table, c.pools, c.base3, c.base4, 0.1, out, c.workspace()[:8])
    with pytest.raises(G.GaacError):
        G.decode_attention(W.make_q(0, 3, 2, 80, device="cuda"), c.seq_lens, c.table, c.pools, c.base3, c.base4,
                           0.1, torch.empty(2, 80, 128, device="cuda"), c.workspace())


def test_full_size_config2_paged():
    """Config 2 sizes, one layer: batch 32, lengths uniform in [4096, 32768], 16q/8kv, full blocks
    scattered over a shared slot pool by a seeded permutation."""
    B, H, Hq, maxT = 32, 8, 16, 32768
    lens = W.make_lengths(2, B, 4096, maxT, device="cuda")
    k, v = U.kv(2, 0, B, maxT, H)
    max_blocks = maxT // 64
    positions = B * max_blocks * H * 2
    perm = W.slot_permutation(2, 0, positions, device="cuda").to(torch.int32)
    c = U.build(k, v, lens, slot_ids=perm.view(B, max_blocks, H, 2), n_slots=positions)
    assert _status(c) == 0
    rng = np.random.default_rng(2)
    lens_np = lens.cpu().numpy()
    tiles = []
    for _ in range(300):
        b = int(rng.integers(0, B))
        tiles.append((b, int(rng.integers(0, (lens_np[b] + 63) // 64)), int(rng.integers(0, H)), int(rng.integers(0, 2))))
    U.check_tiles(c, k, v, lens, tiles=tiles)
    kd, vd = c.decompress(maxT)
    for b in range(B):
        L = int(lens_np[b])
        assert torch.equal(kd[b, :L].view(torch.int16), k[b, :L].view(torch.int16))
        assert torch.equal(vd[b, :L].view(torch.int16), v[b, :L].view(torch.int16))
    del kd, vd
    q = W.make_q(2, 0, B, Hq, device="cuda")
    out = c.attention(q, 1 / np.sqrt(128))
    assert _status(c) == 0
    assert U.check_attention(out, q, k, v, lens, 1 / np.sqrt(128)).compared == B * Hq  # all 32 sequences


def test_full_size_config3_incremental():
    """Config 3 sizes, one layer: batch 8, prefill 32768 tokens, then 256 decode steps that each append
    one token per sequence and attend; the final compressed bytes equal a one-shot encode of the cache."""
    B, H, Hq, T0, steps = 8, 8, 16, 32768, 256
    T = T0 + steps
    k, v = U.kv(3, 0, B, T, H)
    max_blocks = T // 64
    inc = LayerCache(B, H, max_blocks)
    inc.calibrate(k[0, :512], v[0, :512])
    inc.encode(k[:, :T0], v[:, :T0], U.lens_tensor([T0] * B))
    q = W.make_q(3, 0, B, Hq, device="cuda")
    for s in range(steps):
        inc.append(k[:, T0 + s].contiguous(), v[:, T0 + s].contiguous())
        out = inc.attention(q, 1 / np.sqrt(128))
        if s % 64 == 0 or s % 64 == 63:  # each block's first and sealing step, all 8 sequences
            torch.cuda.synchronize()
            L = T0 + s + 1
            r = U.check_attention(out, q, k[:, :L], v[:, :L], U.lens_tensor([L] * B), 1 / np.sqrt(128))
            assert r.compared == B * Hq
    assert _status(inc) == 0
    assert inc.seq_lens.tolist() == [T] * B
    one = LayerCache(B, H, max_blocks)
    one.base3.copy_(inc.base3)
    one.base4.copy_(inc.base4)
    one.encode(k, v, U.lens_tensor([T] * B))
    torch.cuda.synchronize()
    assert _status(one) == 0
    # compare every logical tile: same mode and escape length, same slot or raw bytes
    ia, ea, ma, na = inc.fields()
    ib, eb, mb, nb = one.fields()
    assert torch.equal(ma, mb) and torch.equal(ea, eb) and torch.equal(na, nb)
    slot = ma == G.MODE_SLOT
    assert bool(slot.all()), "every block of the final cache is full and compressible"
    sa = inc.pools.slot_pool[ia[slot].long()]
    sb = one.pools.slot_pool[ib[slot].long()]
    assert torch.equal(sa, sb)
    b3, b4 = inc.base3.cpu().numpy(), inc.base4.cpu().numpy()
    rng = np.random.default_rng(3)
    tiles = [(int(rng.integers(0, B)), int(rng.integers(0, max_blocks)), int(rng.integers(0, H)),
              int(rng.integers(0, 2))) for _ in range(100)]
    U.check_tiles(inc, k, v, inc.seq_lens, tiles=tiles, b3=b3, b4=b4)


@pytest.mark.parametrize("scale", [1 / np.sqrt(128), -1 / np.sqrt(128), 0.0])
def test_extreme_logits_and_scale_signs(scale):
    """Logits near the top of the fp32 range, and softmax scales of either sign or zero.  One token of
    sequence 0 has every key channel at 2^124 and q = 1 on every channel: its logit is 2^127.5 at
    scale 2^-3.5, an fp32 number although its raw dot product times the scale's 16 log2(e) would not
    be.  At a positive scale that token's weight is 1 and every other weight 0, so the output is its
    value row; at a negative scale its weight is 0; at scale 0 the output is the mean of the values."""
    B, T, H, Hq = 2, 1000, 8, 16
    k, v = U.kv(0, 5, B, T, H)
    k[0, 700] = 2.0 ** 124
    lens = U.lens_tensor([T, 777])
    c = U.build(k, v, lens)
    assert _status(c) == 0
    q = torch.ones(B, Hq, 128, dtype=torch.bfloat16, device="cuda")
    q[1] = W.make_q(0, 5, 1, Hq, device="cuda")[0]
    out = c.attention(q, scale)
    assert _status(c) == 0
    assert U.check_attention(out, q, k, v, lens, scale).compared == B * Hq
    if scale > 0:
        assert torch.equal(out[0], v[0, 700].float().repeat_interleave(Hq // H, dim=0))


@pytest.mark.parametrize("H", [8, 12])
def test_raw_cache_appends_stay_raw(H):
    """A cache of raw tiles only (the BF16 baseline) grows by appends whose full tails stay raw tiles; the
    BF16 kernel reads it.  H = 8 runs the single-launch append (a sequence's 16 CTAs as one cluster),
    H = 12 the two-kernel form (24 CTAs per sequence)."""
    B, T0, steps = 3, 200, 130
    T = T0 + steps
    k, v = U.kv(3, 1, B, T, H)
    c = LayerCache(B, H, (T + 63) // 64 + 1)
    c.calibrate(k[0, :T0], v[0, :T0])
    c.encode(k[:, :T0], v[:, :T0], U.lens_tensor([T0] * B), raw=True)
    q = W.make_q(3, 1, B, 2 * H, device="cuda")
    for s in range(steps):
        c.append(k[:, T0 + s].contiguous(), v[:, T0 + s].contiguous())
    assert _status(c) == 0
    assert c.seq_lens.tolist() == [T] * B
    n = U.check_tiles(c, k, v, c.seq_lens, raw_all=True)
    assert n["slot"] == 0 and n["raw"] == B * ((T + 63) // 64) * H * 2
    out = c.attention(q, 1 / np.sqrt(128), bf16=True)
    assert _status(c) == 0
    assert U.check_attention(out, q, k, v, c.seq_lens, 1 / np.sqrt(128)).compared == B * 2 * H


def test_corrupted_slot_images_are_reported():
    """Slot images that break the format are reported as GAAC_EFORMAT by the attention kernel, without a
    fault, and only the kv-head they belong to is affected: a reserved tag (tag 3) in a K tile, then an
    escape-directory entry that disagrees with the tags in a V tile."""
    k, v = U.kv(0, 4, 1, 512, 8)
    lens = U.lens_tensor([512])
    c = U.build(k, v, lens)
    q = W.make_q(0, 4, 1, 16, device="cuda")
    good = c.attention(q, 1 / np.sqrt(128)).clone()
    assert _status(c) == 0
    idx = c.fields()[0]
    pool = c.pools.slot_pool
    for (blk, h, kind, off, val) in ((2, 1, 0, 11264 + 40, 0x03), (5, 5, 1, 11520 + 2 * 3, 0x7F)):
        s = int(idx[0, blk, h, kind])
        saved = pool[s].clone()
        pool[s, off] = pool[s, off] | val
        c.status.zero_()
        out = c.attention(q, 1 / np.sqrt(128))
        assert _status(c) == G.EFORMAT
        assert torch.isfinite(out).all()
        others = [hq for hq in range(16) if hq // 2 != h]
        assert torch.equal(out[0, others], good[0, others])
        pool[s] = saved
