"""GPU parity of decode attention over 256-channel heads, stored as two
128-channel half-heads (GAAC page, Appendix D), against the fp64 oracle over
the whole 256-channel heads.  Ragged lengths with open BF16 tails, GQA 4:1,
blocks spread over several splits."""
import numpy as np
import pytest
import torch

import gaac_workloads as W
import lossless_compressed_kv_gaac_gb300 as G
from lossless_compressed_kv_gaac_gb300.cache import LayerCache
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_splits", [0, 3])
def test_attention_hd256_matches_oracle(n_splits):
    B, Hkv, Hq = 2, 2, 8
    lens_list = [700, 1300]
    T = max(lens_list)
    k, v = W.make_kv(0, 7, B, T, 2 * Hkv, device="cuda")  # 2 * Hkv half-heads of 128 channels
    lens = U.lens_tensor(lens_list)
    c = U.build(k, v, lens)
    g = torch.Generator(device="cuda")
    g.manual_seed(256)
    q = torch.randn(B, Hq, 256, generator=g, device="cuda").to(torch.bfloat16)
    out = torch.full((B, Hq, 256), float("nan"), dtype=torch.float32, device="cuda")
    nkv = 2 * Hkv
    ws = torch.zeros(G.attention_workspace(B, nkv, c.max_blocks, n_splits), dtype=torch.uint8, device="cuda")
    G.decode_attention_hd256(q, c.seq_lens, c.table, c.pools, c.base3, c.base4, 1 / 16, out, ws, n_splits=n_splits,
                             status=c.status)
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0
    k256 = k.view(B, T, Hkv, 256)
    v256 = v.view(B, T, Hkv, 256)
    assert U.check_attention(out, q, k256, v256, lens, 1 / 16).compared == B * Hq
    # a second call reuses the workspace (the merge counters return to zero)
    out2 = torch.empty_like(out)
    G.decode_attention_hd256(q, c.seq_lens, c.table, c.pools, c.base3, c.base4, 1 / 16, out2, ws, n_splits=n_splits,
                             status=c.status)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_attention_hd256_rejects_bad_shapes():
    c = LayerCache(1, 4, 4)
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, 8, 128, device="cuda")
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        G.decode_attention_hd256(q, c.seq_lens, c.table, c.pools, c.base3, c.base4, 1 / 16, out, ws)


def test_attention_hd256_long_splits_reuse_mailboxes():
    """Few splits over a long sequence: each CTA of a cluster pair takes 64 blocks (about 21 per warp),
    so every warp reuses both of its score mailboxes many times; the result must still match the fp64
    oracle, and an open BF16 tail must be read too."""
    B, Hkv, Hq = 1, 2, 8
    T = 8192 + 37
    k, v = W.make_kv(0, 8, B, T, 2 * Hkv, device="cuda")
    lens = U.lens_tensor([T])
    c = U.build(k, v, lens)
    g = torch.Generator(device="cuda")
    g.manual_seed(257)
    q = torch.randn(B, Hq, 256, generator=g, device="cuda").to(torch.bfloat16)
    out = torch.empty((B, Hq, 256), dtype=torch.float32, device="cuda")
    ws = torch.zeros(G.attention_workspace(B, 2 * Hkv, c.max_blocks, 2), dtype=torch.uint8, device="cuda")
    G.decode_attention_hd256(q, c.seq_lens, c.table, c.pools, c.base3, c.base4, 1 / 16, out, ws, n_splits=2,
                             status=c.status)
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0
    assert U.check_attention(out, q, k.view(B, T, Hkv, 256), v.view(B, T, Hkv, 256), lens, 1 / 16).compared == B * Hq
