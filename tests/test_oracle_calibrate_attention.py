"""Pins of the oracle's calibration and fp64 attention.

Calibration ("GAAC: Lossless KV Compression ...", section 3.1 and section 4.7.1):
per head-channel windows of 8 and 16 exponents chosen from calibration data;
this build takes the window with the largest count, ties to the smallest base.
Pinned by an exhaustive window scan done with numpy and by hand-derived cases.

Attention (section 3.2: compressed blocks and the raw tail share one softmax):
softmax(scale * q.k) v in fp64.  Pinned by closed forms (T=1, equal keys, one
dominant logit, per-kv-head constants for the grouped-query mapping) and by an
independent numpy float64 softmax on small random cases.
"""
import numpy as np
import pytest


def test_best_window_exhaustive_scan(orc):
    rng = np.random.default_rng(3)
    for _ in range(200):
        hist = rng.integers(0, 50, 256) * (rng.random(256) < 0.3)
        for w in (8, 16):
            sums = np.convolve(hist, np.ones(w, dtype=np.int64), mode="valid")  # window sums at b=0..256-w
            assert sums.size == 257 - w
            assert orc.best_window(hist, w) == int(np.argmax(sums))  # argmax: first maximum


def test_best_window_ties_take_smallest_base(orc):
    assert orc.best_window(np.zeros(256), 8) == 0
    assert orc.best_window(np.ones(256), 16) == 0
    hist = np.zeros(256, np.int64)
    hist[[50, 150]] = 7  # two equal isolated peaks: window covering 50 starts at 43..50
    assert orc.best_window(hist, 8) == 43
    assert orc.best_window(hist, 16) == 35


def test_calibrate_hand_derived(orc):
    """Channel c of head h holds exponents spread uniformly over [a, a+5] with
    a = 100 + (c + h) % 20.  Every 8-window starting in [a-2, a] covers all six
    values (count = n_tok), so the smallest, a-2, wins; the 16-window: a-10."""
    n_tok, H = 384, 2
    x = np.zeros((n_tok, H, 128), np.uint16)
    for h in range(H):
        for c in range(128):
            a = 100 + (c + h) % 20
            e = a + (np.arange(n_tok) % 6)
            sign_mant = (np.arange(n_tok) * 37 + c) % 256
            x[:, h, c] = ((sign_mant & 0x80) << 8) | (e << 7) | (sign_mant & 0x7F)
    b3, b4 = orc.calibrate(x)
    for h in range(H):
        for c in range(128):
            a = 100 + (c + h) % 20
            assert b3[h, c] == a - 2
            assert b4[h, c] == a - 10


def _bf16_to_f64(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def _f32_to_bf16_bits(x):
    x = np.asarray(x, np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16  # round to nearest even
    return u.astype(np.uint16)


def _numpy_attention(q, k, v, scale):
    qf, kf, vf = _bf16_to_f64(q), _bf16_to_f64(k), _bf16_to_f64(v)
    Hq, Hkv = qf.shape[0], kf.shape[1]
    r = Hq // Hkv
    out = np.zeros((Hq, 128))
    for h in range(Hq):
        s = scale * (kf[:, h // r, :] @ qf[h])
        w = np.exp(s - s.max())
        out[h] = (w / w.sum()) @ vf[:, h // r, :]
    return out


@pytest.mark.parametrize("T,Hq,Hkv", [(1, 4, 2), (7, 8, 2), (100, 16, 8), (257, 32, 8)])
def test_attention_matches_numpy_float64(orc, T, Hq, Hkv):
    rng = np.random.default_rng(T)
    q = _f32_to_bf16_bits(rng.standard_normal((Hq, 128)))
    k = _f32_to_bf16_bits(rng.standard_normal((T, Hkv, 128)) * 2)
    v = _f32_to_bf16_bits(rng.standard_normal((T, Hkv, 128)))
    scale = 1 / np.sqrt(128)
    out, flags = orc.attention(q, k, v, scale)
    ref = _numpy_attention(q, k, v, scale)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    assert (flags == 0).all()


def test_attention_closed_forms(orc):
    rng = np.random.default_rng(9)
    Hq, Hkv = 8, 2
    q = _f32_to_bf16_bits(rng.standard_normal((Hq, 128)))
    # T = 1: the output is the single value row of the head's kv-head
    k = _f32_to_bf16_bits(rng.standard_normal((1, Hkv, 128)))
    v = _f32_to_bf16_bits(rng.standard_normal((1, Hkv, 128)))
    out, _ = orc.attention(q, k, v, 0.1)
    for h in range(Hq):
        np.testing.assert_array_equal(out[h], _bf16_to_f64(v[0, h // 4]))
    # equal keys: uniform weights, the mean of V
    T = 50
    k = np.repeat(_f32_to_bf16_bits(rng.standard_normal((1, Hkv, 128))), T, axis=0)
    v = _f32_to_bf16_bits(rng.standard_normal((T, Hkv, 128)))
    out, _ = orc.attention(q, k, v, 0.1)
    for h in range(Hq):
        np.testing.assert_allclose(out[h], _bf16_to_f64(v[:, h // 4]).mean(axis=0), rtol=0, atol=1e-14)
    # one dominant logit: that token's V row (others' weights underflow to 0)
    k = _f32_to_bf16_bits(rng.standard_normal((T, Hkv, 128)) * 0.01)
    qq = np.full((Hq, 128), 0x3F80, np.uint16)  # q = 1.0 everywhere
    k[17] = 0x4780  # 65536.0 on every channel of both kv-heads
    out, _ = orc.attention(qq, k, v, 1.0)
    for h in range(Hq):
        np.testing.assert_array_equal(out[h], _bf16_to_f64(v[17, h // 4]))
    # grouped-query mapping: q head h reads kv-head h // (Hq/Hkv)
    Hq, Hkv, T = 16, 8, 5
    v = np.zeros((T, Hkv, 128), np.uint16)
    for hk in range(Hkv):
        v[:, hk, :] = _f32_to_bf16_bits(np.float32(hk + 1))
    k = _f32_to_bf16_bits(rng.standard_normal((T, Hkv, 128)))
    q = _f32_to_bf16_bits(rng.standard_normal((Hq, 128)))
    out, _ = orc.attention(q, k, v, 0.3)
    for h in range(Hq):
        np.testing.assert_allclose(out[h], h // 2 + 1, rtol=1e-15)
    # empty sequence: zeros
    out, _ = orc.attention(q, k[:0], v[:0], 0.3)
    assert (out == 0).all()


def test_attention_range_flags(orc):
    Hq, Hkv, T = 4, 1, 3
    q = np.full((Hq, 128), 0x4080, np.uint16)  # 4.0
    k = np.full((T, Hkv, 128), 0x3F80, np.uint16)
    v = np.full((T, Hkv, 128), 0x3F80, np.uint16)
    _, flags = orc.attention(q, k, v, 0.1)
    assert (flags == 0).all()
    k[1, 0, :] = 0x7F00  # 2^127: sum_c |q k| = 128 * 4 * 2^127 >= 2^130
    _, flags = orc.attention(q, k, v, 0.1)
    assert (flags & 1).all()
    k[1, 0, :] = 0x3F80
    v[:, 0, 0] = 0x7F7F  # near the fp32 maximum, three tokens of equal weight
    _, flags = orc.attention(q, k, v, 0.1)
    assert (flags == 2).all()


def test_attention_range_flag_boundary(orc):
    """Bit 0 marks a row once |scale| * sum_c |q_c k_c| of some token passes the largest fp32 value, and
    not before: with q = 1 and one token's 128 keys at 2^124, the sum is 2^131 and the logit at scale
    2^-3.5 is 2^127.5 (representable, unflagged); at 2^125 the bound is 2^128.5 (flagged).  A negative
    scale has the same magnitudes.  The unflagged extreme row's output is that token's value row: its
    weight is 1 and every other weight underflows to 0 in fp64."""
    Hq, Hkv, T = 2, 1, 5
    q = np.full((Hq, 128), 0x3F80, np.uint16)  # 1.0
    k = np.full((T, Hkv, 128), 0x3F80, np.uint16)
    v = _f32_to_bf16_bits(np.arange(T * 128, dtype=np.float64).reshape(T, Hkv, 128) / 64.0)
    scale = 2.0 ** -3.5
    for s_ in (scale, -scale):
        k[3, 0, :] = 0x7D80  # 2^124
        out, flags = orc.attention(q, k, v, s_)
        assert (flags == 0).all()
        if s_ > 0:
            np.testing.assert_array_equal(out, np.broadcast_to(_bf16_to_f64(v[3, 0]), out.shape))
        k[3, 0, :] = 0x7E00  # 2^125
        _, flags = orc.attention(q, k, v, s_)
        assert (flags == 1).all()


def test_attention_on_decoded_cache_equals_original(orc):
    """Attention reads the decoded cache; by losslessness it must equal attention
    on the original cache exactly (this pins the codec-to-attention plumbing)."""
    import gaac_workloads as W

    T, Hkv, Hq = 256, 8, 16
    k, v = W.make_kv(0, 0, 1, T, Hkv)
    kb = W.bits(k).numpy().view(np.uint16)[0]
    vb = W.bits(v).numpy().view(np.uint16)[0]
    q = W.bits(W.make_q(0, 0, 1, Hq)).numpy().view(np.uint16)[0]
    b3k, b4k = orc.calibrate(kb[:128])
    b3v, b4v = orc.calibrate(vb[:128])
    kd = np.zeros_like(kb)
    vd = np.zeros_like(vb)
    for blk in range(T // 64):
        for h in range(Hkv):
            for kind, src, dst, b3, b4 in ((0, kb, kd, b3k, b4k), (1, vb, vd, b3v, b4v)):
                img, esc = orc.encode_tile(src[blk * 64:(blk + 1) * 64, h], kind, b3[h], b4[h])
                assert esc >= 0
                dst[blk * 64:(blk + 1) * 64, h], st = orc.decode_tile(img, kind, b3[h], b4[h], esc)
    o1, _ = orc.attention(q, kb, vb, 1 / np.sqrt(128))
    o2, _ = orc.attention(q, kd, vd, 1 / np.sqrt(128))
    np.testing.assert_array_equal(o1, o2)


def test_attention_256_dim_heads(orc):
    """A 256-dimensional head (stored as two 128-channel half-heads) attends over the whole head:
    its output equals float64 numpy, and with the second half of q zero its weights are those of
    the 128-dimensional attention on the first halves."""
    rng = np.random.default_rng(256)
    T, Hq, Hkv = 37, 4, 2
    q = _f32_to_bf16_bits(rng.normal(size=(Hq, 256)))
    k = _f32_to_bf16_bits(rng.normal(size=(T, Hkv, 256)))
    v = _f32_to_bf16_bits(rng.normal(size=(T, Hkv, 256)))
    out, _ = orc.attention(q, k, v, 1 / 16)
    qf, kf, vf = _bf16_to_f64(q), _bf16_to_f64(k), _bf16_to_f64(v)
    for h in range(Hq):
        s = kf[:, h // 2] @ qf[h] / 16
        w = np.exp(s - s.max())
        np.testing.assert_allclose(out[h], (w / w.sum()) @ vf[:, h // 2], rtol=1e-12, atol=1e-12)
    q0 = q.copy()
    q0[:, 128:] = 0
    out0, _ = orc.attention(q0, k, v, 1 / 16)
    lo, _ = orc.attention(q0[:, :128], k[:, :, :128], v[:, :, :128], 1 / 16)
    hi, _ = orc.attention(q0[:, :128], k[:, :, :128], v[:, :, 128:], 1 / 16)
    np.testing.assert_allclose(out0[:, :128], lo, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out0[:, 128:], hi, rtol=1e-12, atol=1e-12)
