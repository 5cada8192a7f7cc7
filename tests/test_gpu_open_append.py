"""GPU parity of the token-granular compressed append: the open block kept in its slot from its first
token ("GAAC: Lossless KV Compression ...", section 3.3 and Figure 3 keep the last block open while
decode tokens arrive; the open-tile image is the oracle's encoding of the first n tokens with the later
ones absent).  After every append the open slot must equal the oracle's image byte for byte, sealed
blocks must equal a one-shot encode, attention must match the fp64 oracle, and decompression must give
the input back."""
import numpy as np
import pytest
import torch

import gaac_workloads as W
from lossless_compressed_kv_gaac_gb300 import EFORMAT, MODE_RAW, MODE_SLOT
from lossless_compressed_kv_gaac_gb300.cache import LayerCache

from . import gpu_util as U

pytestmark = pytest.mark.gpu

SCALE = 1 / np.sqrt(128)


def _status(c):
    return int(c.status.item())


def _open_tiles(c, lens):
    """(b, blk, h, kind) of every open (partial) block."""
    out = []
    for b, L in enumerate(lens):
        if L % 64:
            out += [(b, L // 64, h, kind) for h in range(c.n_kv_heads) for kind in (0, 1)]
    return out


def test_open_append_every_step_matches_oracle():
    B, H, T = 2, 2, 150
    k, v = U.kv(3, 0, B, T + 128, H)
    c = LayerCache(B, H, (T + 63) // 64, open_compressed=True)
    c.calibrate(k[0, :128], v[0, :128])
    k, v = k[:, 128:].contiguous(), v[:, 128:].contiguous()
    # a new table is empty (every entry GAAC_MODE_NONE, seq_lens 0): the first append opens block 0
    b3, b4 = c.base3.cpu().numpy(), c.base4.cpu().numpy()
    q = W.make_q(3, 0, B, 8, device="cuda")
    for s in range(T):
        c.append(k[:, s].contiguous(), v[:, s].contiguous())
        L = s + 1
        lens = U.lens_tensor([L] * B)
        torch.cuda.synchronize()
        if L % 64:
            n = U.check_tiles(c, k, v, lens, tiles=_open_tiles(c, [L] * B), b3=b3, b4=b4, open_compressed=True)
            assert n["slot"] == 2 * B * H, (L, n)
        if L in (1, 2, 9, 63, 64, 65, 100, T):
            out = c.attention(q, SCALE)
            torch.cuda.synchronize()
            U.check_attention(out, q, k[:, :L], v[:, :L], lens, SCALE)
    assert _status(c) == 0
    U.check_tiles(c, k, v, c.seq_lens, b3=b3, b4=b4, open_compressed=True)
    kd, vd = c.decompress(T)
    assert torch.equal(kd.view(torch.int16), k.view(torch.int16))
    assert torch.equal(vd.view(torch.int16), v.view(torch.int16))


def test_open_prefill_then_append_equals_one_shot():
    """Ragged prefill with open slots, then appends: every block, open or sealed, equals the same
    cache encoded at once from the final lengths."""
    H = 4
    lens0 = [1, 63, 64, 100, 130, 7]
    steps = 70
    B = len(lens0)
    T = max(lens0) + steps
    k, v = U.kv(3, 1, B, T, H)
    mb = (T + 63) // 64
    inc = LayerCache(B, H, mb, open_compressed=True)
    inc.calibrate(k[0, :64], v[0, :64])
    inc.encode(k, v, U.lens_tensor(lens0))
    torch.cuda.synchronize()
    b3, b4 = inc.base3.cpu().numpy(), inc.base4.cpu().numpy()
    n = U.check_tiles(inc, k, v, inc.seq_lens, b3=b3, b4=b4, open_compressed=True)
    assert n["slot"] > 0
    for s in range(steps):
        L = torch.tensor(lens0) + s
        kn = torch.stack([k[b, L[b]] for b in range(B)]).contiguous()
        vn = torch.stack([v[b, L[b]] for b in range(B)]).contiguous()
        inc.append(kn, vn)
    torch.cuda.synchronize()
    assert _status(inc) == 0
    final = [x + steps for x in lens0]
    assert inc.seq_lens.tolist() == final
    one = LayerCache(B, H, mb, open_compressed=True)
    one.base3.copy_(inc.base3)
    one.base4.copy_(inc.base4)
    one.encode(k, v, U.lens_tensor(final))
    torch.cuda.synchronize()
    U.check_tiles(inc, k, v, inc.seq_lens, b3=b3, b4=b4, open_compressed=True)
    U.check_tiles(one, k, v, one.seq_lens, b3=b3, b4=b4, open_compressed=True)
    i1, e1, m1, n1 = (x.cpu().numpy() for x in inc.fields())
    i2, e2, m2, n2 = (x.cpu().numpy() for x in one.fields())
    np.testing.assert_array_equal(m1, m2)
    np.testing.assert_array_equal(e1, e2)
    np.testing.assert_array_equal(n1, n2)
    s1, s2 = inc.pools.slot_pool.cpu().numpy(), one.pools.slot_pool.cpu().numpy()
    for pos in zip(*np.nonzero(m1 == MODE_SLOT)):
        np.testing.assert_array_equal(s1[i1[pos]], s2[i2[pos]])
    q = W.make_q(3, 1, B, 16, device="cuda")
    out = inc.attention(q, SCALE)
    torch.cuda.synchronize()
    U.check_attention(out, q, k, v, inc.seq_lens, SCALE)


def test_open_block_overflow_moves_to_raw():
    """Tokens whose exponents leave every window make the open block's escape stream outgrow the slot
    (K: 16 raw groups, 128 escape bytes, per token): from that token on the block is a raw tile holding
    its tokens so far, and it seals as RAW."""
    B, H = 1, 2
    k, v = U.kv(3, 2, B, 256, H)
    c = LayerCache(B, H, 4, open_compressed=True)
    c.calibrate(k[0, :128], v[0, :128])
    c.encode(k, v, U.lens_tensor([64]))  # block 0 sealed from the first 64 tokens
    rng = np.random.default_rng(7)
    # keys with random signs and mantissas and exponents spread over [90, 141): almost every group of eight
    # leaves its windows (raw), yet the scores stay finite
    shape = (B, 80, H, 128)
    bits = (rng.integers(0, 2, shape) << 15) | (rng.integers(90, 141, shape) << 7) | rng.integers(0, 128, shape)
    wild = torch.from_numpy(bits.astype(np.uint16).view(np.int16)).cuda().view(torch.bfloat16)
    k2, v2 = k.clone(), v.clone()
    for s in range(80):
        kn = wild[:, s] if s % 3 else k[:, 64 + s]  # two thirds of the tokens wild (keys only)
        k2[:, 64 + s] = kn
        c.append(kn.contiguous(), v[:, 64 + s].contiguous())
        torch.cuda.synchronize()
    assert _status(c) == 0
    b3, b4 = c.base3.cpu().numpy(), c.base4.cpu().numpy()
    n = U.check_tiles(c, k2, v, c.seq_lens, b3=b3, b4=b4, open_compressed=True)
    _, _, mode, ntok = (x.cpu().numpy() for x in c.fields())
    assert mode[0, 1, 0, 0] == MODE_RAW and ntok[0, 1, 0, 0] == 64  # K of block 1 overflowed and sealed raw
    assert mode[0, 1, 0, 1] == MODE_SLOT  # its values stayed compressed
    assert mode[0, 2, 0, 0] == MODE_RAW and ntok[0, 2, 0, 0] == 16  # K of the open block 2 overflowed too
    assert n["raw"] >= 2
    q = W.make_q(3, 2, B, 4, device="cuda")
    out = c.attention(q, SCALE)
    torch.cuda.synchronize()
    U.check_attention(out, q, k2[:, :144], v[:, :144], c.seq_lens, SCALE)
    kd, vd = c.decompress(144)
    assert torch.equal(kd.view(torch.int16), k2[:, :144].view(torch.int16))


def test_raw_tail_continues_under_open_flag():
    """A cache prefilled with BF16 tails keeps its raw tails when appended with the flag (hand-over of the
    raw tile at each seal), and its sealed blocks equal a one-shot encode."""
    B, H, T0, steps = 2, 2, 100, 90
    k, v = U.kv(3, 3, B, T0 + steps, H)
    c = LayerCache(B, H, 4)
    c.calibrate(k[0, :T0], v[0, :T0])
    c.encode(k[:, :T0], v[:, :T0], U.lens_tensor([T0] * B))
    c.open_compressed = True
    for s in range(steps):
        c.append(k[:, T0 + s].contiguous(), v[:, T0 + s].contiguous())
    torch.cuda.synchronize()
    assert _status(c) == 0
    b3, b4 = c.base3.cpu().numpy(), c.base4.cpu().numpy()
    n = U.check_tiles(c, k, v, c.seq_lens, b3=b3, b4=b4)
    assert n["raw"] == 2 * B * H  # the open block 2 (190 = 2*64 + 62) is a raw tail


def test_open_slot_entry_mismatch_reported():
    """An open slot whose entry does not match the sequence length is a format error; nothing is written."""
    B, H = 1, 1
    k, v = U.kv(3, 4, B, 64, H)
    c = LayerCache(B, H, 2, open_compressed=True)
    c.calibrate(k[0], v[0])
    c.encode(k, v, U.lens_tensor([10]))
    torch.cuda.synchronize()
    before = c.pools.slot_pool.clone()
    c.seq_lens.fill_(11)  # entry says 10 tokens
    c.append(k[:, 11].contiguous(), v[:, 11].contiguous())
    torch.cuda.synchronize()
    assert _status(c) == EFORMAT
    assert torch.equal(before, c.pools.slot_pool)
