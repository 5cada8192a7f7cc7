#!/usr/bin/env python3
"""Decode-step attention over a GAAC-compressed BF16 KV cache on GB300.

One step = decode attention for all 36 layers of a Qwen3-8B-shaped model
(32 query / 8 kv heads, head_dim 128, batch 1) at 65,536 cached tokens, read
from the resident compressed cache (block 64, calibration on the first 512
tokens), as in the GAAC page's section 4.4 setting (64K context, batch 1).

Prints one JSON line (rank 0).  Default: N=1, 20 timed steps after 5 warm-up.
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gaac|reference]
--impl reference times the CPU oracle (scalar C decode + fp64 attention) on a
bounded sample of the same workload, scaled to one step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/step & achieved HBM GB/s at 64K ctx; encode GB/s; ratio"
UNIT = "us/step"
WORKLOAD = "Qwen3-8B-shaped decode attention: 36 layers, batch 1, 32q/8kv, head_dim 128, T=65536, block 64"
CONFIG_ID = 1


# DRAM bytes (read + write) of one attn_split_kernel launch on this workload, from an
# ncu capture, valid only for the kernel source it was taken on (see profiles/).
NCU_TRAFFIC = {"kernel_sha": "0ca89dd882a14465", "bytes_per_launch": 195751680}


def code_digest(texts) -> str:
    """Hash of C++ sources with // comments, trailing blanks and empty lines removed, so that an edit
    of comments alone keeps it."""
    import hashlib
    import re

    h = hashlib.sha256()
    for t in texts:
        for line in t.splitlines():
            line = re.sub(r"//.*$", "", line).rstrip()
            if line:
                h.update(line.encode() + b"\n")
    return h.hexdigest()[:16]


def kernel_sha() -> str:
    """Digest of the attention kernel's code (attention.cu + common.cuh)."""
    return code_digest(open(os.path.join(ROOT, "lossless_compressed_kv_gaac_gb300", "csrc", f)).read()
                       for f in ("attention.cu", "common.cuh"))


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="gaac", choices=["gaac", "reference"])
    p.add_argument("--layers", type=int, default=36, help="layers per step (36 = the Qwen3-8B workload)")
    p.add_argument("--cpu-units", type=int, default=48, help="(layer, kv-head) units in the CPU oracle sample")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    p.add_argument("--no-side", action="store_true", help="skip the side workloads (configs 0, 2, 3, 4)")
    p.add_argument("--study", choices=["rope-drift"], default=None,
                   help="rope-drift: escape bytes per tile along 32K rotary keys for short and long calibration")
    p.add_argument("--timeline", action="store_true",
                   help="build the instrumented library and print the per-CTA timeline of one attention launch over "
                        "one layer of the workload (compressed, then BF16), instead of the benchmark")
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(x: float, device=None) -> float:
    """Max of x over the ranks of the default process group (x itself when there is none)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(ms_per_step_max: float, world: int) -> float:
    """µs per step of the whole job: N replicas each finish one step per ms_per_step_max."""
    return ms_per_step_max * 1e3 / world


# ---------------------------------------------------------------- clocks ----
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ workload -----
def build_layers(n_layers: int, device, raw: bool):
    """Compressed (or all-raw) caches of n_layers layers, plus the per-layer queries."""
    import torch

    import gaac_workloads as W
    from lossless_compressed_kv_gaac_gb300.cache import LayerCache

    wl = W.WORKLOADS[CONFIG_ID]
    T, H, Hq = wl.seq_len, wl.n_kv_heads, wl.n_q_heads
    caches, qs = [], []
    lens = torch.tensor([T], dtype=torch.int32, device=device)
    for layer in range(n_layers):
        k, v = W.make_kv(CONFIG_ID, layer, 1, T, H, device=device)
        c = LayerCache(1, H, T // 64, device=device, n_slots=0 if raw else None, n_raw=T // 64 * H * 2 if raw else 256)
        c.calibrate(k[0, :wl.n_calib], v[0, :wl.n_calib])
        c.encode(k, v, lens, raw=raw)
        caches.append(c)
        qs.append(W.make_q(CONFIG_ID, layer, 1, Hq, device=device))
        del k, v
    torch.cuda.synchronize()
    for c in caches:
        assert int(c.status.item()) == 0, "encode reported an error"
    return caches, qs


def algorithmic_bytes(cache) -> int:
    """Bytes the method must read for one attention launch over this layer: per slot tile the
    planes and the escape directory (11,536 B) plus its escape bytes, per raw tile 16,384 B,
    plus 8 B per table entry."""
    import torch

    _, esc, mode, _ = cache.fields()
    slot = mode == 0
    raw = mode == 1
    n = int(slot.sum().item()) * 11536 + int(esc[slot].sum().item()) + int(raw.sum().item()) * 16384
    n += int((slot | raw).sum().item()) * 8
    return n


def time_calls(fn, reps: int = 5, rounds: int = 3) -> float:
    """Device time of one call of fn (ms): `reps` back-to-back calls between two CUDA events on the
    current stream, min over rounds.  One more call is queued before the first event, so the device is
    busy while the host enqueues the timed calls and their launch overhead is not in the time."""
    import torch

    best = float("inf")
    for _ in range(rounds):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fn()
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1) / reps)
    return best


def time_graph(g, stream, steps: int):
    """Replays the graph `steps` times on `stream`; CUDA-event time on that stream (ms)."""
    import torch

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            g.replay()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end)


def fp8_codec(k, v, n_calib: int) -> dict:
    """FP8 variant of the codec on one layer's K and V cast to FP8 (round to nearest): payload ratio
    against the FP8 bytes (a tile that does not fit its slot counts as 8 KiB), encode and decode GB/s
    of FP8 bytes, round trip checked."""
    import torch

    import lossless_compressed_kv_gaac_gb300 as G

    T, H = k.shape[1], k.shape[2]
    nb = T // 64
    out = {}
    for fmt, name, dt in ((G.FP8_E4M3, "e4m3", torch.float8_e4m3fn), (G.FP8_E5M2, "e5m2", torch.float8_e5m2)):
        k8, v8 = k[0].float().to(dt).view(torch.uint8), v[0].float().to(dt).view(torch.uint8)
        b3 = torch.zeros((2 * H, 128), dtype=torch.uint8, device=k.device)
        b4 = torch.zeros_like(b3)
        G.fp8_calibrate(k8[:n_calib], fmt, b3[:H], b4[:H])
        G.fp8_calibrate(v8[:n_calib], fmt, b3[H:], b4[H:])
        tiles = torch.cat([x[: nb * 64].view(nb, 64, H, 128).permute(2, 0, 1, 3).reshape(-1, 64, 128) for x in (k8, v8)]).contiguous()
        n = tiles.shape[0]
        kinds = torch.cat([torch.zeros(H * nb), torch.ones(H * nb)]).to(torch.uint8).to(k.device)
        rows = torch.cat([torch.arange(H).repeat_interleave(nb), H + torch.arange(H).repeat_interleave(nb)]).int().to(k.device)
        slots = torch.empty((n, G.fp8_slot_bytes(fmt)), dtype=torch.uint8, device=k.device)
        esc = torch.empty(n, dtype=torch.int16, device=k.device)
        back = torch.empty_like(tiles)
        te = time_calls(lambda: G.fp8_encode_tiles(tiles, fmt, kinds, rows, b3, b4, slots, esc))
        td = time_calls(lambda: G.fp8_decompress_tiles(slots, esc, fmt, kinds, rows, b3, b4, back))
        torch.cuda.synchronize()
        e = esc.view(torch.int16).long() & 0xFFFF
        fits = e != 0xFFFF
        assert torch.equal(back[fits], tiles[fits])
        off_esc = G.fp8_slot_bytes(fmt) - 496
        payload = int((off_esc + e[fits]).sum().item()) + 8192 * int((~fits).sum().item())
        out[name] = {"payload_ratio": round(n * 8192 / payload, 4), "resident_ratio": round(8192 / G.fp8_slot_bytes(fmt), 4),
                     "tiles_kept_fp8": int((~fits).sum().item()), "encode_gbs": round(n * 8192 / (te * 1e-3) / 1e9, 1),
                     "decode_gbs": round(n * 8192 / (td * 1e-3) / 1e9, 1)}
    return out


def mode_ablation(k, v, n_calib: int) -> dict:
    """The GAAC page's nested 2-bit-mode ablation on one layer's tiles: format v3 and the nested format
    (a 2-bit mode and a variable-width code stream) encode the same K and V tiles; payload ratio of
    each (BF16 bytes / bytes a read of the tile needs) and the decode time of each tile-batch decoder
    (same launch shape: one CTA per tile, one thread per 32-element unit), round trips checked."""
    import torch

    import lossless_compressed_kv_gaac_gb300 as G

    T, H = k.shape[1], k.shape[2]
    nb = T // 64
    tiles = torch.cat([x[0, : nb * 64].view(nb, 64, H, 128).permute(2, 0, 1, 3).reshape(-1, 64, 128)
                       for x in (k, v)]).contiguous()
    n = tiles.shape[0]
    dev = k.device
    kinds = torch.cat([torch.zeros(H * nb), torch.ones(H * nb)]).to(torch.uint8).to(dev)
    rows = torch.cat([torch.arange(H).repeat_interleave(nb), H + torch.arange(H).repeat_interleave(nb)]).int().to(dev)
    b2, b3, b4 = (torch.zeros((2 * H, 128), dtype=torch.uint8, device=dev) for _ in range(3))
    for x, lo in ((k, 0), (v, H)):
        G.calibrate(x[0, :n_calib], b3[lo:lo + H], b4[lo:lo + H])
        G.nested_calibrate(x[0, :n_calib], b2[lo:lo + H])
    s3 = torch.empty((n, G.SLOT_BYTES), dtype=torch.uint8, device=dev)
    sn = torch.empty((n, G.NESTED_SLOT_BYTES), dtype=torch.uint8, device=dev)
    e3 = torch.empty(n, dtype=torch.int16, device=dev)
    en = torch.empty(n, dtype=torch.int16, device=dev)
    G.encode_tiles(tiles, kinds, rows, b3, b4, s3, e3)
    G.nested_encode_tiles(tiles, kinds, rows, b2, b3, b4, sn, en)
    c3 = time_calls(lambda: G.encode_tiles(tiles, kinds, rows, b3, b4, s3, e3))
    cn = time_calls(lambda: G.nested_encode_tiles(tiles, kinds, rows, b2, b3, b4, sn, en))
    back = torch.empty_like(tiles)
    d3 = time_calls(lambda: G.decode_tiles(s3, e3, kinds, rows, b3, b4, back))
    dn = time_calls(lambda: G.nested_decode_tiles(sn, en, kinds, rows, b2, b3, b4, back))
    torch.cuda.synchronize()
    assert torch.equal(back.view(torch.int16), tiles.view(torch.int16))
    G.decode_tiles(s3, e3, kinds, rows, b3, b4, back)
    torch.cuda.synchronize()
    assert torch.equal(back.view(torch.int16), tiles.view(torch.int16))
    e3l, enl = e3.long() & 0xFFFF, en.long() & 0xFFFF
    assert bool((e3l != 0xFFFF).all()) and bool((enl != 0xFFFF).all()), "a tile overflowed its escape area"
    d7 = sn[:, 11548:11552].long()
    bits = (d7[:, 0] | (d7[:, 1] << 8) | (d7[:, 2] << 16) | (d7[:, 3] << 24)) >> 16
    pay3 = int((11536 + e3l).sum().item())
    payn = int((8192 + (bits + 7) // 8 + 256 + 32 + enl).sum().item())
    raw = n * 16384
    return {"tiles": n, "payload_ratio_v3": round(raw / pay3, 4), "payload_ratio_nested": round(raw / payn, 4),
            "ratio_gain_pct": round(100 * (pay3 / payn - 1), 2),
            "decode_us_v3": round(d3 * 1e3, 1), "decode_us_nested": round(dn * 1e3, 1),
            "decode_time_ratio": round(dn / d3, 3),
            "encode_us_v3": round(c3 * 1e3, 1), "encode_us_nested": round(cn * 1e3, 1)}


def hd256_attention(device, n_calib: int) -> dict:
    """Decode attention over 256-channel heads (stored as two 128-channel half-heads): one layer of a
    Qwen3-family shape with head_dim 256, 16 q / 4 kv heads, T = 65,536, batch 1, the same synthetic
    value recipe; CUDA-event time per launch (10 launches after warm-up) and algorithmic GB/s."""
    import torch

    import gaac_workloads as W
    import lossless_compressed_kv_gaac_gb300 as G
    from lossless_compressed_kv_gaac_gb300.cache import LayerCache

    T, Hkv, Hq = 65536, 4, 16
    k, v = W.make_kv(CONFIG_ID, 0, 1, T, 2 * Hkv, device=device)  # 8 half-heads of 128 channels
    c = LayerCache(1, 2 * Hkv, T // 64, device=device, n_raw=256)
    c.calibrate(k[0, :n_calib], v[0, :n_calib])
    c.encode(k, v, torch.tensor([T], dtype=torch.int32, device=device))
    del k, v
    g = torch.Generator(device=device)
    g.manual_seed(256)
    q = torch.randn(1, Hq, 256, generator=g, device=device).to(torch.bfloat16)
    out = torch.empty((1, Hq, 256), dtype=torch.float32, device=device)
    ws = torch.zeros(G.attention_workspace(1, 2 * Hkv, c.max_blocks), dtype=torch.uint8, device=device)

    def launch():
        G.decode_attention_hd256(q, c.seq_lens, c.table, c.pools, c.base3, c.base4, 1 / 16, out, ws, status=c.status)

    for _ in range(3):
        launch()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(10):
        launch()
    e1.record()
    e1.synchronize()
    assert int(c.status.item()) == 0, "hd256 attention reported an error"
    us = e0.elapsed_time(e1) * 1e3 / 10
    alg = algorithmic_bytes(c)
    return {"workload": "one layer, head_dim 256 (two 128-channel half-heads), 16 q / 4 kv heads, T=65536, batch 1",
            "us_per_layer": round(us, 2), "algorithmic_bytes": alg, "compressed_gbs": round(alg / (us * 1e-6) / 1e9, 1)}


def graph_of(fn, stream):
    """fn() run once eagerly (kernel attributes set outside the capture), then captured in a CUDA graph.
    Synchronises first: the caches were built on the default stream, which `stream` does not wait for."""
    import torch

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def config_entry(name, launches, us_compressed, us_bf16, alg_bytes, raw_bytes, peak, **extra) -> dict:
    """One side config's figures: per-step times of both kernels and the compressed kernel's GB/s and
    roofline fraction (algorithmic bytes of the step / its time)."""
    d = {"workload": name, "launches_per_step": launches, "us_per_step": round(us_compressed, 2),
         "bf16_cache_us_per_step": round(us_bf16, 2), "speedup_vs_bf16_cache": round(us_bf16 / us_compressed, 3),
         "algorithmic_bytes_per_step": int(alg_bytes), "raw_bytes_per_step": int(raw_bytes),
         "hbm_gbs_compressed": round(alg_bytes / (us_compressed * 1e-6) / 1e9, 1),
         "equiv_uncompressed_gbs": round(raw_bytes / (us_compressed * 1e-6) / 1e9, 1),
         "frac": round(alg_bytes / (us_compressed * 1e-6) / 1e9 / peak, 4),
         "bf16_frac": round(raw_bytes / (us_bf16 * 1e-6) / 1e9 / peak, 4)}
    d.update(extra)
    return d


def raw_cache_bytes(cache) -> int:
    """Bytes the BF16 kernel reads for one launch: 16,384 per raw tile and 8 per table entry."""
    _, _, mode, _ = cache.fields()
    return int((mode == 1).sum().item()) * (16384 + 8)


def side_configs(device, stream, steps: int, peak: float) -> dict:
    """The other workloads, each with the compressed kernel and the BF16 kernel over an all-raw twin cache of
    the same data (CUDA graphs, CUDA-event time, caches larger than L2 except config 0):
      config 0: one layer, T = 4096 (L2-resident: launch latency only);
      config 2: paged batch 32, lengths uniform in [4096, 32768], slots scattered by a seeded permutation,
                28 launches per step cycling 4 distinct layers (1.7 GB compressed each);
      config 3: batch 8 after a 32,768-token prefill, 28 layers, each of 256 decode steps appends one token
                per sequence and layer and then attends (every step timed, seals included);
      config 4: batch 4, T = 131,072, 10% random-bit tokens (one layer, 8 launches per timing)."""
    import torch

    import gaac_workloads as W
    from lossless_compressed_kv_gaac_gb300.cache import LayerCache

    out = {}
    scale = W.WORKLOADS[0].scale

    def pair_caches(cfg, layer, B, T, H, lens, adversarial=0.0, paged=False, max_blocks=None):
        k, v = W.make_kv(cfg, layer, B, T, H, device=device, adversarial=adversarial)
        mb = max_blocks or (T + 63) // 64
        positions = B * mb * H * 2
        ids = W.slot_permutation(cfg, layer, positions, device=device).to(torch.int32).view(B, mb, H, 2) if paged else None
        c = LayerCache(B, H, mb, device=device, slot_ids=ids, n_slots=positions,
                       n_raw=(positions if adversarial > 0 else 4096) + B * H * 2)
        c.calibrate(k[0, :512], v[0, :512])
        c.encode(k, v, lens)
        r = LayerCache(B, H, mb, device=device, n_slots=0, n_raw=positions + B * H * 2)
        r.encode(k, v, lens, raw=True)
        del k, v
        return c, r

    def time_pair(cs, rs, qs, launches, reps):
        outs = [torch.empty(q.shape, dtype=torch.float32, device=device) for q in qs]
        res = []
        for caches, bf in ((cs, False), (rs, True)):
            def step():
                for i in range(launches):
                    caches[i % len(caches)].attention(qs[i % len(qs)], scale, out=outs[i % len(qs)], bf16=bf)
            g = graph_of(step, stream)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g.replay()
            res.append(time_graph(g, stream, reps) / reps * 1e3)
            for c in caches:
                assert int(c.status.item()) == 0, "attention reported an error"
        return res

    # ---- config 0: L2-resident single layer
    wl = W.WORKLOADS[0]
    lens = torch.tensor([wl.seq_len], dtype=torch.int32, device=device)
    c, r = pair_caches(0, 0, 1, wl.seq_len, wl.n_kv_heads, lens)
    q = W.make_q(0, 0, 1, wl.n_q_heads, device=device)
    uc, ub = time_pair([c], [r], [q], 1, max(steps, 20))
    out["config0"] = {"workload": wl.name, "us_per_launch": round(uc, 2), "bf16_cache_us_per_launch": round(ub, 2),
                      "note": "16.8 MB of raw K/V: L2-resident, so a latency figure, not a bandwidth one"}
    del c, r

    # ---- config 2: paged batch 32, 28 layers (4 distinct layers cycled)
    wl = W.WORKLOADS[2]
    lens = W.make_lengths(2, wl.batch, wl.min_len, wl.seq_len, device=device)
    cs, rs, qs = [], [], []
    for layer in range(4):
        c, r = pair_caches(2, layer, wl.batch, wl.seq_len, wl.n_kv_heads, lens, paged=True)
        cs.append(c)
        rs.append(r)
        qs.append(W.make_q(2, layer, wl.batch, wl.n_q_heads, device=device))
    uc, ub = time_pair(cs, rs, qs, wl.n_layers, steps)
    alg = sum(algorithmic_bytes(c) for c in cs) / 4 * wl.n_layers
    rawb = sum(raw_cache_bytes(r) for r in rs) / 4 * wl.n_layers
    out["config2"] = config_entry(wl.name, wl.n_layers, uc, ub, alg, rawb, peak,
                                  tokens=int(lens.sum().item()), distinct_layers=4,
                                  splits=cs[0].auto_splits())
    del cs, rs, qs
    torch.cuda.empty_cache()

    # ---- config 4: adversarial, one layer
    wl = W.WORKLOADS[4]
    lens = torch.tensor([wl.seq_len] * wl.batch, dtype=torch.int32, device=device)
    c, r = pair_caches(4, 0, wl.batch, wl.seq_len, wl.n_kv_heads, lens, adversarial=wl.adversarial)
    q = W.make_q(4, 0, wl.batch, wl.n_q_heads, device=device)
    uc, ub = time_pair([c], [r], [q], 8, steps)
    _, _, mode, _ = c.fields()
    raw_share = float((mode == 1).double().mean().item())
    out["config4"] = config_entry(wl.name, 1, uc / 8, ub / 8, algorithmic_bytes(c), raw_cache_bytes(r), peak,
                                  raw_tile_share=round(raw_share, 4), splits=c.auto_splits())
    del c, r
    torch.cuda.empty_cache()

    # ---- config 3: prefill 32768, then 256 steps of append + attention over 28 layers
    wl = W.WORKLOADS[3]
    B, H, T0, n_app = wl.batch, wl.n_kv_heads, wl.seq_len, wl.appends
    mb = (T0 + n_app + 63) // 64
    lens0 = torch.tensor([T0] * B, dtype=torch.int32, device=device)
    cs, rs, qs, news = [], [], [], []
    for layer in range(wl.n_layers):
        c, r = pair_caches(3, layer, B, T0, H, lens0, max_blocks=mb)
        cs.append(c)
        rs.append(r)
        qs.append(W.make_q(3, layer, B, wl.n_q_heads, device=device))
        kn, vn = W.make_kv(3, layer, B, n_app, H, device=device, token_offset=T0)
        news.append((kn, vn))
    stage_k = [torch.empty((B, H, 128), dtype=torch.bfloat16, device=device) for _ in range(wl.n_layers)]
    stage_v = [torch.empty_like(x) for x in stage_k]
    outs = [torch.empty((B, wl.n_q_heads, 128), dtype=torch.float32, device=device) for _ in range(wl.n_layers)]
    res = []
    for caches, bf in ((cs, False), (rs, True)):
        def step():
            for i, c in enumerate(caches):
                c.append(stage_k[i], stage_v[i])
                c.attention(qs[i], scale, out=outs[i], bf16=bf)
        g = graph_of(step, stream)  # the capture's eager run is step 0
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for i in range(wl.n_layers):
                stage_k[i].copy_(news[i][0][:, 0])
                stage_v[i].copy_(news[i][1][:, 0])
            torch.cuda.synchronize()
            e0.record(stream)
            for s_ in range(1, n_app):
                for i in range(wl.n_layers):  # the step's new tokens (from the projections in a model)
                    stage_k[i].copy_(news[i][0][:, s_])
                    stage_v[i].copy_(news[i][1][:, s_])
                g.replay()
            e1.record(stream)
        e1.synchronize()
        res.append(e0.elapsed_time(e1) * 1e3 / (n_app - 1))
        for c in caches:
            stv = int(c.status.item())
            assert stv == 0, f"config 3 ({'BF16' if bf else 'compressed'} cache): status {stv}"
            assert c.seq_lens.tolist() == [T0 + n_app] * B, f"config 3 lengths {c.seq_lens.tolist()}"
        del g
    alg = sum(algorithmic_bytes(c) for c in cs)  # at the end of the run (33,024 tokens)
    rawb = sum(raw_cache_bytes(r) for r in rs)
    out["config3"] = config_entry(wl.name + " (append + attention per step)", 2 * wl.n_layers, res[0], res[1], alg,
                                  rawb, peak, steps_timed=n_app - 1, splits=cs[0].auto_splits(),
                                  note="bytes and GB/s at the final length, 33,024 tokens")
    del cs, rs, qs, news
    torch.cuda.empty_cache()
    return out


def bf16_sdpa_step(n_layers: int, device, stream, steps: int) -> dict:
    """Context for the uncompressed path: torch's scaled_dot_product_attention (a library kernel) over a
    contiguous BF16 cache of the same workload (32 q / 8 kv heads with GQA, T = 65,536, batch 1), one call per
    layer, 36 calls per step captured in a CUDA graph.  Four distinct layers' caches are cycled (each 268 MB,
    larger than L2)."""
    import torch
    import torch.nn.functional as F

    import gaac_workloads as W

    wl = W.WORKLOADS[CONFIG_ID]
    T, H, Hq = wl.seq_len, wl.n_kv_heads, wl.n_q_heads
    kv = []
    for layer in range(4):
        k, v = W.make_kv(CONFIG_ID, layer, 1, T, H, device=device)
        kv.append((k.permute(0, 2, 1, 3).contiguous(), v.permute(0, 2, 1, 3).contiguous()))  # [1, H, T, 128]
        del k, v
    q = W.make_q(CONFIG_ID, 0, 1, Hq, device=device).view(1, Hq, 1, 128)
    out = torch.empty((1, Hq, 1, 128), dtype=torch.bfloat16, device=device)

    def step():
        for i in range(n_layers):
            k, v = kv[i % 4]
            out.copy_(F.scaled_dot_product_attention(q, k, v, scale=wl.scale, enable_gqa=True))

    try:
        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        time_graph(g, stream, 2)
        ms = time_graph(g, stream, steps) / steps
    except RuntimeError as e:  # a backend that cannot run this shape or be captured
        return {"unavailable": str(e).splitlines()[0][:160]}
    raw_bytes = 2 * T * H * 128 * 2 * n_layers
    return {"us_per_step": round(ms * 1e3, 2), "gbs": round(raw_bytes / (ms * 1e-3) / 1e9, 1),
            "kernel": "torch scaled_dot_product_attention, BF16 cache [1, 8, 65536, 128], enable_gqa"}


def append_cost(k, v, n_calib: int) -> dict:
    """Device time of one decode-token append (all kv-heads, K and V, one layer, batch 1) with the
    open block as a BF16 raw tail and with it kept compressed in its slot.  64 consecutive appends (a
    block opening, 62 in-block tokens and a seal) are captured in a CUDA graph and replayed; the
    time per append is the replay's CUDA-event time / 64.  Each append is one launch (the length
    advance is folded in)."""
    import torch

    from lossless_compressed_kv_gaac_gb300.cache import LayerCache

    H = k.shape[2]
    T0, reps = 1024, 4
    out = {"unit": "us per append", "tokens_per_replay": 64}
    stream = torch.cuda.Stream(k.device)
    kn = k[0, T0:T0 + 64].unsqueeze(1).contiguous()  # [64, 1, H, 128]
    vn = v[0, T0:T0 + 64].unsqueeze(1).contiguous()
    # one eager append on a throwaway cache first: the library settles its launch form (one launch, the
    # sequence's CTAs as a cluster) outside a capture, as a serving loop's first decode step would
    warm = LayerCache(1, H, T0 // 64 + 2, device=k.device)
    warm.calibrate(k[0, :n_calib], v[0, :n_calib])
    warm.encode(k[:, :T0], v[:, :T0], torch.tensor([T0], dtype=torch.int32, device=k.device))
    warm.append(kn[0], vn[0])
    torch.cuda.synchronize()
    del warm
    for name, open_c in (("raw_tail", False), ("open_compressed", True)):
        c = LayerCache(1, H, T0 // 64 + 64 * (reps + 2) // 64, device=k.device, open_compressed=open_c)
        c.calibrate(k[0, :n_calib], v[0, :n_calib])
        c.encode(k[:, :T0], v[:, :T0], torch.tensor([T0], dtype=torch.int32, device=k.device))
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(64):
                    c.append(kn[i], vn[i], stream=stream)
        torch.cuda.synchronize()
        times = []
        for r in range(reps):
            t = time_graph(g, stream, 1)
            if r:
                times.append(t)
        assert int(c.status.item()) == 0, "append reported an error"
        assert int(c.seq_lens.item()) == T0 + 64 * reps
        out[name] = round(min(times) * 1e3 / 64, 2)
    return out


def run_gaac(args):
    import torch

    import gaac_workloads as W
    import lossless_compressed_kv_gaac_gb300 as G

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)
    wl = W.WORKLOADS[CONFIG_ID]
    L = args.layers
    scale = wl.scale
    stream = torch.cuda.Stream(device)

    # ---- build the compressed cache of every layer (encode timed on layer 0)
    caches, qs = build_layers(L, device, raw=False)
    outs = [torch.empty((1, wl.n_q_heads, 128), dtype=torch.float32, device=device) for _ in range(L)]
    c0 = caches[0]
    k0, v0 = W.make_kv(CONFIG_ID, 0, 1, wl.seq_len, wl.n_kv_heads, device=device)
    lens = torch.tensor([wl.seq_len], dtype=torch.int32, device=device)
    enc_ms = time_calls(lambda: c0.encode(k0, v0, lens))
    raw_bytes_layer = 2 * wl.seq_len * wl.n_kv_heads * 128 * 2
    encode_gbs = raw_bytes_layer / (enc_ms * 1e-3) / 1e9
    kd = torch.empty_like(k0)
    vd = torch.empty_like(v0)
    dec_ms = time_calls(lambda: G.decompress(c0.table, c0.seq_lens, c0.pools, c0.base3, c0.base4, kd, vd))
    torch.cuda.synchronize()
    assert torch.equal(kd.view(torch.int16), k0.view(torch.int16)) and torch.equal(vd.view(torch.int16), v0.view(torch.int16))
    decompress_gbs = raw_bytes_layer / (dec_ms * 1e-3) / 1e9
    st = G.stats_dict(c0.stats)
    fp8 = fp8_codec(k0, v0, wl.n_calib)
    app = append_cost(k0, v0, wl.n_calib)
    abl = mode_ablation(k0, v0, wl.n_calib)
    del k0, v0, kd, vd
    hd256 = hd256_attention(device, wl.n_calib)
    alg = [algorithmic_bytes(c) for c in caches]
    alg_step = sum(alg)
    raw_step = raw_bytes_layer * L
    res = [c.resident_bytes() for c in caches]
    resident_step = sum(r["slot_bytes"] + r["raw_bytes"] + r["table_bytes"] for r in res)
    payload_ratio = raw_step / (alg_step - sum(r["table_bytes"] for r in res))
    resident_ratio = raw_step / resident_step

    # ---- one step: all layers, captured in a CUDA graph
    def step():
        for c, q, o in zip(caches, qs, outs):
            c.attention(q, scale, out=o)

    with torch.cuda.stream(stream):
        for _ in range(2):
            step()  # first calls set kernel attributes outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            g.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    clocks = ClockSampler(vis.split(",")[local] if vis else str(local))
    clocks.start()
    time.sleep(0.3)
    ms = time_graph(g, stream, args.steps)
    clk = clocks.stop()
    ms = reduce_max(ms, device)
    if world > 1:
        torch.distributed.barrier()
    for c in caches:
        assert int(c.status.item()) == 0
    ms_per_step = ms / args.steps

    # ---- per-launch duration of the attention call (one kernel; the split merge runs in its last CTAs),
    # eager launches timed one by one on the same stream (for the launch-level figure; the roofline
    # below uses the graph-timed region)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
    per_launch = []
    for rep in range(3):
        with torch.cuda.stream(stream):
            for (e0, e1), c, q, o in zip(ev, caches, qs, outs):
                e0.record(stream)
                c.attention(q, scale, out=o)
                e1.record(stream)
        stream.synchronize()
        per_launch.append(sum(e0.elapsed_time(e1) for e0, e1 in ev) / L)
    launch_ms = min(per_launch)
    alg_launch = alg_step / L
    region_launch_ms = ms_per_step / L  # average launch duration inside the timed graph replays
    achieved_gbs = alg_launch / (region_launch_ms * 1e-3) / 1e9

    # ---- uncompressed BF16 baseline: the BF16 kernel (the attention kernel specialised to raw tiles, no
    # decode path) over an all-raw cache of the same layers; also the compressed kernel's own raw path
    bf16_ms = raw_path_ms = None
    try:
        raw_caches, _ = build_layers(L, device, raw=True)

        def step_raw(bf16):
            for c, q, o in zip(raw_caches, qs, outs):
                c.attention(q, scale, out=o, bf16=bf16)

        times = {}
        for bf16 in (True, False):
            with torch.cuda.stream(stream):
                step_raw(bf16)
            torch.cuda.synchronize()
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2, stream=stream):
                step_raw(bf16)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g2.replay()
            times[bf16] = time_graph(g2, stream, args.steps) / args.steps
            del g2
        for c in raw_caches:
            assert int(c.status.item()) == 0, "BF16 attention reported an error"
        bf16_ms, raw_path_ms = times[True], times[False]
        del raw_caches
    except torch.cuda.OutOfMemoryError:
        bf16_ms = None
    torch.cuda.empty_cache()
    sdpa = bf16_sdpa_step(L, device, stream, args.steps)

    # ---- end to end through the public API: pinned host q in, host out back, every step
    q_host = torch.stack([q for q in qs]).cpu().pin_memory()
    out_host = torch.empty((L, 1, wl.n_q_heads, 128), dtype=torch.float32).pin_memory()
    q_dev = torch.empty_like(q_host, device=device)
    out_dev = torch.empty((L, 1, wl.n_q_heads, 128), dtype=torch.float32, device=device)

    def step_e2e():
        q_dev.copy_(q_host, non_blocking=True)
        for i, c in enumerate(caches):
            c.attention(q_dev[i], scale, out=out_dev[i])
        out_host.copy_(out_dev, non_blocking=True)

    with torch.cuda.stream(stream):
        step_e2e()
    torch.cuda.synchronize()
    g3 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g3, stream=stream):
        step_e2e()
    with torch.cuda.stream(stream):
        for _ in range(3):
            g3.replay()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            g3.replay()
            stream.synchronize()  # the host reads the result every step
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    e2e_ms = reduce_max(e2e_ms, device)

    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    side = None
    if not args.no_side:
        del g, g3
        side = side_configs(device, stream, args.steps, peaks.get("hbm_gbs") or 6800.0)
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or 6800.0
    traffic = NCU_TRAFFIC["bytes_per_launch"] if NCU_TRAFFIC["kernel_sha"] == kernel_sha() else None
    # BF16 kernel: per layer 16,384 raw tiles of 16 KiB plus 8 B per table entry
    bf16_bytes = L * (raw_bytes_layer + 2 * (wl.seq_len // 64) * wl.n_kv_heads * 8)

    result = {
        "metric": METRIC,
        "value": round(job_value(ms_per_step, world), 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; lognormal channel scales, 4 x20 outlier key channels per head)",
        "config": {"workload": WORKLOAD, "layers": L, "batch": 1, "seq_len": wl.seq_len, "q_heads": wl.n_q_heads,
                   "kv_heads": wl.n_kv_heads, "head_dim": 128, "block": 64, "calibration_tokens": wl.n_calib,
                   "l2": "inputs larger than L2 (%.2f GB compressed per step)" % (alg_step / 1e9),
                   "replicas": "each rank runs the whole workload" if world > 1 else "single GPU"},
        "hbm_gbs_compressed": round(alg_step / (ms_per_step * 1e-3) / 1e9, 1),
        "equiv_uncompressed_gbs": round(raw_step / (ms_per_step * 1e-3) / 1e9, 1),
        "bf16_cache_us_per_step": round(bf16_ms * 1e3, 2) if bf16_ms else None,
        "speedup_vs_bf16_cache": round(bf16_ms / ms_per_step, 3) if bf16_ms else None,
        "bf16_kernel": ({"us_per_step": round(bf16_ms * 1e3, 2), "gbs": round(bf16_bytes / (bf16_ms * 1e-3) / 1e9, 1),
                         "frac": round(bf16_bytes / (bf16_ms * 1e-3) / 1e9 / peak, 4),
                         "bytes_per_step": bf16_bytes,
                         "kernel": "attn_split_kernel<1, 1, true>: the attention kernel specialised to raw tiles "
                                   "(no decode path), all-raw BF16 cache of the same layers",
                         "raw_cache_through_compressed_kernel_us_per_step": round(raw_path_ms * 1e3, 2)}
                        if bf16_ms else None),
        "bf16_sdpa": sdpa,
        "encode_gbs": round(encode_gbs, 1),
        "decompress_gbs": round(decompress_gbs, 1),
        "fp8": fp8,
        "append": app,
        "mode_ablation": abl,
        "hd256": hd256,
        "configs": side,
        "ratio": {"payload": round(payload_ratio, 4), "resident": round(resident_ratio, 4),
                  "mode_shares": [round(st[f"groups{m}"] / max(1, 1024 * st["slot_tiles"]), 5) for m in range(3)]},
        "roofline": {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved_gbs / peak, 4), "traffic": traffic,
                     "kernel": "attn_split_kernel (decode + attention + split merge, one launch per layer)",
                     "peak_source": peak_src, "launch_us": round(region_launch_ms * 1e3, 2),
                     "eager_launch_us": round(launch_ms * 1e3, 2),
                     "algorithmic_bytes_per_launch": alg_launch},
        "clocks": clk,
        "e2e": {"value": round(job_value(e2e_ms, world), 2), "unit": UNIT, "h2d_bytes_per_step": q_host.numel() * 2,
                "d2h_bytes_per_step": out_host.numel() * 4},
        "gpu_launches": L * args.steps,
    }
    if rank == 0 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(args.cpu_units, L)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


# --------------------------------------------------------------- oracle ----
class OracleSample:
    """The oracle as it stands, on the host cores: scalar C tile decode plus fp64
    attention over one (layer, kv-head) unit of the workload (1,024 K and 1,024 V
    tiles decoded, 4 query heads over 65,536 tokens).  The unit's tiles are
    encoded by the oracle itself, untimed."""

    def __init__(self, unit_ids):
        import numpy as np

        import gaac_workloads as W
        import oracle as O

        wl = W.WORKLOADS[CONFIG_ID]
        self.T, self.H, self.r, self.scale = wl.seq_len, wl.n_kv_heads, wl.n_q_heads // wl.n_kv_heads, wl.scale
        self.units = []
        layer_data = {}
        for u in unit_ids:
            layer, h = u // self.H, u % self.H
            if layer not in layer_data:
                k, v = W.make_kv(CONFIG_ID, layer, 1, self.T, self.H)
                kn = W.bits(k).numpy().view(np.uint16)[0]
                vn = W.bits(v).numpy().view(np.uint16)[0]
                q = W.bits(W.make_q(CONFIG_ID, layer, 1, wl.n_q_heads)).numpy().view(np.uint16)[0]
                layer_data = {layer: (kn, vn, q, O.calibrate(kn[:512]), O.calibrate(vn[:512]))}
            kn, vn, q, (b3k, b4k), (b3v, b4v) = layer_data[layer]
            imgs = []
            for blk in range(self.T // 64):
                for kind, x, b3, b4 in ((0, kn, b3k, b4k), (1, vn, b3v, b4v)):
                    img, e = O.encode_tile(x[blk * 64:(blk + 1) * 64, h], kind, b3[h], b4[h])
                    imgs.append((kind, img, e, blk, b3[h].copy(), b4[h].copy()))
            self.units.append((imgs, q[h * self.r:(h + 1) * self.r].copy()))

    def run(self, u: int) -> float:
        """Seconds for unit u: decode its tiles, then fp64 attention."""
        import numpy as np

        import oracle as O

        imgs, q = self.units[u]
        kd = np.zeros((self.T, 1, 128), np.uint16)
        vd = np.zeros((self.T, 1, 128), np.uint16)
        t0 = time.perf_counter()
        for kind, img, e, blk, b3, b4 in imgs:
            tile, _ = O.decode_tile(img, kind, b3, b4, e)
            (kd if kind == 0 else vd)[blk * 64:(blk + 1) * 64, 0] = tile
        O.attention(q, kd, vd, self.scale)
        return time.perf_counter() - t0


def _oracle_units(unit_ids) -> list:
    """Pool task: build (untimed) and time the listed units in this process."""
    smp = OracleSample(unit_ids)
    return [smp.run(i) for i in range(len(unit_ids))]


def host_cores() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(16, n))


def oracle_pool_times(unit_lists) -> list:
    """Per-unit seconds of the oracle, the unit lists run concurrently in spawned processes (one per
    list; spawn, because this process has already initialised CUDA)."""
    import multiprocessing as mp

    if len(unit_lists) == 1:
        return _oracle_units(unit_lists[0])
    with mp.get_context("spawn").Pool(len(unit_lists)) as pool:
        return [t for ts in pool.map(_oracle_units, unit_lists) for t in ts]


def cpu_config0_single_thread() -> dict:
    """The oracle on one host thread over the whole config-0 workload (one layer, batch 1, 8 kv-heads,
    T = 4096, 16 query heads; seeded inputs drawn on the CPU): calibration, encode of its 1,024 tiles,
    decode of them, and fp64 attention over the decoded cache, each timed."""
    import numpy as np

    import gaac_workloads as W
    import oracle as O

    wl = W.WORKLOADS[0]
    T, H = wl.seq_len, wl.n_kv_heads
    k, v = W.make_kv(0, 0, 1, T, H)
    kn, vn = (W.bits(x).numpy().view(np.uint16)[0] for x in (k, v))
    q = W.bits(W.make_q(0, 0, 1, wl.n_q_heads)).numpy().view(np.uint16)[0]
    t0 = time.perf_counter()
    bases = (O.calibrate(kn[:wl.n_calib]), O.calibrate(vn[:wl.n_calib]))
    t1 = time.perf_counter()
    imgs = []
    for blk in range(T // 64):
        for h in range(H):
            for kind, x in ((0, kn), (1, vn)):
                b3, b4 = bases[kind]
                img, e = O.encode_tile(x[blk * 64:(blk + 1) * 64, h], kind, b3[h], b4[h])
                imgs.append((blk, h, kind, img, e))
    t2 = time.perf_counter()
    kd, vd = np.zeros_like(kn), np.zeros_like(vn)
    for blk, h, kind, img, e in imgs:
        b3, b4 = bases[kind]
        tile, _ = O.decode_tile(img, kind, b3[h], b4[h], e)
        (kd if kind == 0 else vd)[blk * 64:(blk + 1) * 64, h] = tile
    t3 = time.perf_counter()
    O.attention(q, kd, vd, wl.scale)
    t4 = time.perf_counter()
    assert np.array_equal(kd, kn) and np.array_equal(vd, vn)
    return {"workload": wl.name, "threads": 1, "calibrate_s": round(t1 - t0, 4), "encode_s": round(t2 - t1, 3),
            "decode_s": round(t3 - t2, 3), "attention_s": round(t4 - t3, 3),
            "decode_attention_us_per_step": round((t4 - t2) * 1e6, 1)}


def cpu_baseline(units: int, n_layers: int) -> dict:
    """Oracle throughput on the host cores: `units` (layer, kv-head) units spread over one process per core,
    all cores busy at once; a step is n_layers x 8 units shared by those cores."""
    cores = min(host_cores(), units)
    lists = [list(range(c, units, cores)) for c in range(cores)]
    t0 = time.perf_counter()
    times = oracle_pool_times(lists)
    wall = time.perf_counter() - t0
    H = 8
    step_us = statistics.mean(times) * n_layers * H / cores * 1e6
    return {"value": round(step_us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "extrapolated": {"units_timed": units, "units_per_step": n_layers * H,
                             "mean_s_per_unit_all_cores_busy": round(statistics.mean(times), 4)},
            "sample": f"sampled extrapolation: {units} (layer, kv-head) units of the workload timed, {cores} processes "
                      f"at once: per unit the oracle decodes 2x1024 tiles and runs fp64 attention for 4 query heads "
                      f"over 65536 tokens (mean {statistics.mean(times):.3f} s per unit with every core busy); the "
                      f"value is that mean x {n_layers * H} units per step / {cores} cores; {wall:.0f} s wall "
                      f"including the untimed encode",
            "config0_single_thread": cpu_config0_single_thread()}


_WORKER_SAMPLE = None


def _init_reference_worker(counter, n_units: int):
    """Pool initializer: this worker's own (layer, kv-head) unit, encoded once (untimed)."""
    global _WORKER_SAMPLE
    with counter.get_lock():
        uid = counter.value
        counter.value += 1
    _WORKER_SAMPLE = OracleSample([uid % n_units])


def _time_reference_worker(_) -> float:
    return _WORKER_SAMPLE.run(0)


def run_reference(args):
    """The oracle arm: one process per host core, each holding one (layer, kv-head) unit of the workload
    built once; a step runs every core's unit at once, scaled to a full step."""
    import multiprocessing as mp

    rank, world, _ = dist_env()
    if rank != 0:
        return
    cores = host_cores()
    H = 8
    ctx = mp.get_context("spawn")
    counter = ctx.Value("i", 0)
    steps_us, walls = [], []
    with ctx.Pool(cores, initializer=_init_reference_worker, initargs=(counter, args.layers * H)) as pool:
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            times = pool.map(_time_reference_worker, range(cores), chunksize=1)
            if i >= args.warmup:
                walls.append(time.perf_counter() - t0)
                steps_us.append(statistics.mean(times) * args.layers * H / cores * 1e6)
    v = statistics.median(steps_us)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(v / 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers": args.layers},
        "cpu_baseline": {"value": round(v, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "extrapolated": {"units_timed_per_step": cores, "units_per_step": args.layers * H,
                                          "wall_s_per_timed_step": round(statistics.median(walls), 3)},
                         "sample": f"sampled extrapolation: per step {cores} (layer, kv-head) units run at once, one "
                                   "process per core (decode 2x1024 tiles + fp64 attention, 4 heads x 65536 tokens); "
                                   f"the value is their mean time x {args.layers} layers x {H} kv-heads / {cores} "
                                   f"cores, so a timed step takes {statistics.median(walls):.2f} s of wall time and "
                                   "stands for the whole step"},
        "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def rope_drift_study() -> dict:
    """The positional-drift study of the GAAC page's Appendix C on synthetic rotary keys: a 32,768-token
    sequence (8 kv-heads, the Qwen3-8B-shaped workload's channel scales, rotary base 1e6) is encoded with
    windows calibrated on its first 2K, 8K or all 32K tokens; per 4,096-token segment it reports the mean
    escape bytes of the K and V tiles kept in slots and the share of tiles that fell back to BF16."""
    import torch

    import gaac_workloads as W
    import lossless_compressed_kv_gaac_gb300 as G
    from lossless_compressed_kv_gaac_gb300.cache import LayerCache

    T, H, seg = 32768, 8, 4096
    k, v = W.make_kv(CONFIG_ID, 0, 1, T, H, device="cuda", rope_theta=1e6)
    lens = torch.tensor([T], dtype=torch.int32, device="cuda")
    out = {"study": "rope-drift", "tokens": T, "kv_heads": H, "segment_tokens": seg, "rope_theta": 1e6, "calibration": {}}
    for n_cal in (2048, 8192, 32768):
        c = LayerCache(1, H, T // 64, device="cuda", n_raw=2 * H * (T // 64) + 16)
        c.calibrate(k[0, :n_cal], v[0, :n_cal])
        c.encode(k, v, lens)
        torch.cuda.synchronize()
        _, esc, mode, _ = G.entry_fields(c.table)
        esc, mode = esc[0].cpu(), mode[0].cpu()  # [blocks, heads, K|V]
        row = {}
        for kv, name in ((0, "k"), (1, "v")):
            e = esc[:, :, kv].view(T // seg, -1).double()
            m = mode[:, :, kv].view(T // seg, -1)
            slot = m == G.MODE_SLOT
            row[name + "_esc_bytes_per_slot_tile"] = [round(float(e[i][slot[i]].mean()), 1) if slot[i].any() else None
                                                       for i in range(T // seg)]
            row[name + "_raw_tile_share"] = [round(float((~slot[i]).double().mean()), 4) for i in range(T // seg)]
        out["calibration"][str(n_cal)] = row
    return out


def timeline_summary(raw, n_ctas: int, n_blocks: int, grid) -> dict:
    """Per-CTA timeline records (u64 ns: start, split_end, exit, merged, then issue/arrive/land/release per
    block) of one launch with grid (splits, kv-heads, batch), summarised in microseconds."""
    import numpy as np

    X, Y, Z = grid
    n = X * Y * Z
    rec = raw.reshape(n_ctas, -1)[:n].astype(np.float64)
    start, split_end, exit_, merged = rec[:, 0], rec[:, 1], rec[:, 2], rec[:, 3]
    issue, arrive, land, release = (rec[:, 4 + i * n_blocks: 4 + (i + 1) * n_blocks] for i in range(4))
    t0 = start.min()
    end = np.maximum(exit_, merged)
    used = land > 0
    q = lambda x, p: round(float(np.percentile(x, p)) / 1e3, 3) if x.size else None
    inflight = (land - issue)[used]
    waited = (land - arrive)[used]
    return {"ctas": n, "span_us": round((end.max() - t0) / 1e3, 2),
            "start_spread_us": round((start.max() - t0) / 1e3, 2),
            "split_work_us": {"min": round((split_end - start).min() / 1e3, 2),
                              "mean": round((split_end - start).mean() / 1e3, 2),
                              "max": round((split_end - start).max() / 1e3, 2)},
            "split_end_spread_us": round((split_end.max() - split_end.min()) / 1e3, 2),
            "merge_us": {"mean": round(float((merged - exit_)[merged > 0].mean()) / 1e3, 2),
                         "max": round(float((merged - exit_)[merged > 0].max()) / 1e3, 2)},
            "copy_issue_to_land_us": {"p10": q(inflight, 10), "p50": q(inflight, 50), "p90": q(inflight, 90)},
            "group_wait_for_data_us": {"p10": q(waited, 10), "p50": q(waited, 50), "p90": q(waited, 90)},
            "blocks_per_cta": round(float(used.sum(axis=1).mean()), 1),
            # split work per kv-head: the spread within a head (per-SM speed) against the spread of the
            # heads' means (per-head data)
            "split_work_by_head_us": {"head_means_min": round(float(((split_end - start).reshape(Z * Y, X).mean(1)).min()) / 1e3, 2),
                                      "head_means_max": round(float(((split_end - start).reshape(Z * Y, X).mean(1)).max()) / 1e3, 2),
                                      "within_head_spread_mean": round(float(np.ptp((split_end - start).reshape(Z * Y, X), axis=1).mean()) / 1e3, 2)},
            "smid_note": "CTA order x fastest: split, kv-head, sequence"}


def run_timeline() -> None:
    """One Qwen3-8B-shaped layer (T = 65,536) through the instrumented library: the per-CTA timeline of the
    third attention launch over the compressed cache and over the all-raw cache with the BF16 kernel."""
    import ctypes

    import numpy as np
    import torch

    import gaac_workloads as W
    import lossless_compressed_kv_gaac_gb300 as G
    from lossless_compressed_kv_gaac_gb300 import build as B

    G.LIB_PATH = B.build(timeline=True)
    L = G.lib()
    L.gaac_timeline_fetch.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p]
    cb, nc, nb = ctypes.c_size_t(), ctypes.c_int(), ctypes.c_int()
    L.gaac_timeline_fetch(None, 0, ctypes.byref(cb), ctypes.byref(nc), ctypes.byref(nb))
    dev = torch.device("cuda", 0)
    wl = W.WORKLOADS[CONFIG_ID]
    out = {"timeline": "one layer, T=65536, 32q/8kv, batch 1 (third launch)"}
    for name, raw in (("compressed", False), ("bf16", True)):
        caches, qs = build_layers(1, dev, raw=raw)
        c, q = caches[0], qs[0]
        for _ in range(3):
            o = c.attention(q, wl.scale, bf16=raw)
        torch.cuda.synchronize()
        assert int(c.status.item()) == 0
        buf = np.zeros(nc.value * cb.value // 8, np.uint64)
        G._check("gaac_timeline_fetch", L.gaac_timeline_fetch(buf.ctypes.data, buf.nbytes, None, None, None))
        ns = G.lib().gaac_attention_auto_splits(1, wl.n_kv_heads, c.max_blocks)
        out[name] = timeline_summary(buf, nc.value, nb.value, (ns, wl.n_kv_heads, 1))
        del caches, o
        torch.cuda.empty_cache()
    print(json.dumps(out))


def main():
    args = parse()
    if args.timeline:
        run_timeline()
        return
    if args.study == "rope-drift":
        print(json.dumps(rope_drift_study()))
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gaac(args)


if __name__ == "__main__":
    main()
