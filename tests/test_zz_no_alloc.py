"""The allocation-free decode attention entry point (gaac_decode_attention_noalloc).

It exists for callers that cannot allocate device memory when they call the
library (a serving loop with a frozen memory plan, a plugin whose host owns all
device memory): its split partials live in a fixed scratch array inside the
library instead of a caller workspace.  Checked here through the C ABI against
the workspace entry point, on two calls in a row (the second reuses the scratch
the first left behind).  Kept last in collection order."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import gaac_workloads as W
    import lossless_compressed_kv_gaac_gb300 as G
    from tests import gpu_util as U

    B, T, H, Hq = 3, 4096, 8, 32
    k, v = U.kv(0, 7, B, T, H)
    lens = U.lens_tensor([4096, 1000, 2500])
    c = U.build(k, v, lens)
    q = W.make_q(0, 7, B, Hq, device="cuda")
    scale = 1 / np.sqrt(128)
    ref = c.attention(q, scale)
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        G.decode_attention_noalloc(q, c.seq_lens, c.table, c.pools, c.base3, c.base4, scale, out, status=c.status)
        torch.cuda.synchronize()
        assert int(c.status.item()) == 0, f"call {call}"
        err = U.rel_err_rows(out.double().cpu().numpy(), ref.double().cpu().numpy())
        assert float(err.max()) <= U.TOL, f"call {call}: {err.max()}"
    # another split count still fits; with 7 splits sequence 1's 16 blocks leave split 6 empty, so the
    # merge folds in a partial with no tokens, read back from the shared array
    out = torch.full_like(ref, float("nan"))
    c.status.zero_()
    G.decode_attention_noalloc(q, c.seq_lens, c.table, c.pools, c.base3, c.base4, scale, out, n_splits=7,
                               status=c.status)
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0
    err = U.rel_err_rows(out.double().cpu().numpy(), ref.double().cpu().numpy())
    assert float(err.max()) <= U.TOL, f"7 splits: {err.max()}"
    # ... and one whose partials exceed the fixed scratch is refused before anything is enqueued
    need = G.attention_workspace(B, H, c.max_blocks, 64)
    assert need > G.STATIC_SCRATCH_BYTES
    with pytest.raises(G.GaacError) as e:
        G.decode_attention_noalloc(q, c.seq_lens, c.table, c.pools, c.base3, c.base4, scale, out, n_splits=64)
    assert e.value.status == G.EINVAL
    torch.cuda.synchronize()
