"""Positional drift of rotary keys (GAAC page, Appendix C and Table 8): windows
calibrated on a short prefix let the keys' escape bytes per tile grow along the
sequence, windows calibrated on the whole context keep them flat, and values
(not rotated) do not drift.  Synthetic rotary keys (base 1e6), GPU encoder,
escape lengths read from the slot table."""
import pytest
import torch

import gaac_workloads as W
import lossless_compressed_kv_gaac_gb300 as G
from lossless_compressed_kv_gaac_gb300.cache import LayerCache

pytestmark = pytest.mark.gpu


def _segments(n_cal, k, v, T, H, seg):
    c = LayerCache(1, H, T // 64, device="cuda", n_raw=2 * H * (T // 64) + 16)
    c.calibrate(k[0, :n_cal], v[0, :n_cal])
    c.encode(k, v, torch.tensor([T], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0
    _, esc, mode, _ = G.entry_fields(c.table)
    # an overflowing tile is stored raw: count it at the escape capacity
    e = torch.where(mode[0] == G.MODE_SLOT, esc[0], torch.full_like(esc[0], G.ESC_CAPACITY)).double()
    return [e[i * seg // 64:(i + 1) * seg // 64, :, kv].mean().item() for kv in (0, 1) for i in range(T // seg)]


def test_rope_drift_grows_with_short_calibration():
    T, H, seg = 16384, 4, 4096
    k, v = W.make_kv(1, 0, 1, T, H, device="cuda", rope_theta=1e6)
    n = T // seg
    short = _segments(1024, k, v, T, H, seg)
    full = _segments(T, k, v, T, H, seg)
    k_short, v_short, k_full, v_full = short[:n], short[n:], full[:n], full[n:]
    assert k_short[-1] > 1.5 * k_short[0], k_short  # keys drift away from short-prefix windows
    assert max(k_full) < 1.3 * min(k_full), k_full   # whole-context windows keep them flat
    assert max(v_short) < 1.3 * min(v_short), v_short  # values are not rotated
    assert k_full[-1] < k_short[-1]
