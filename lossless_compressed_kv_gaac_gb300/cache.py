"""One layer's GAAC compressed KV cache held in torch device memory.

Allocation and argument marshalling only: the calibration, encoding, append,
attention and decompression themselves run in the library's kernels.
"""
from __future__ import annotations

import torch

from . import (BLOCK, HEAD_DIM, Pools, append, attention_workspace, calibrate, decode_attention,
               decode_attention_bf16, decompress, encode_blocks, entry_fields, new_stats, new_table)


class LayerCache:
    """Slot table, pools, window bases and counters of one layer.

    slot_ids: int32 [batch, max_blocks, n_kv_heads, 2]: the slot each block is
    encoded (or sealed) into.  Default: a dense map (one slot per table position).
    n_raw: raw tiles available for tails and fallbacks (default: one per
    (sequence, kv-head, K|V) plus one per table position, i.e. never exhausted).
    open_compressed: keep each sequence's open block compressed in its slot
    (prefill and append), instead of as a BF16 tail.
    """

    def __init__(self, batch: int, n_kv_heads: int, max_blocks: int, device="cuda", slot_ids=None, n_slots=None,
                 n_raw=None, raw_free=None, open_compressed: bool = False):
        self.batch, self.n_kv_heads, self.max_blocks = batch, n_kv_heads, max_blocks
        self.open_compressed = open_compressed
        self.device = torch.device(device)
        positions = batch * max_blocks * n_kv_heads * 2
        if slot_ids is None:
            slot_ids = torch.arange(positions, dtype=torch.int32, device=device).view(batch, max_blocks, n_kv_heads, 2)
            n_slots = positions if n_slots is None else n_slots
        elif n_slots is None:
            n_slots = int(slot_ids.max().item()) + 1
        self.slot_ids = slot_ids.to(torch.int32).contiguous()
        if n_raw is None:
            n_raw = positions + batch * n_kv_heads * 2
        self.pools = Pools(n_slots, n_raw, device=device, raw_free=raw_free)
        self.table = new_table(batch, max_blocks, n_kv_heads, device=device)
        self.base3 = torch.zeros((2, n_kv_heads, HEAD_DIM), dtype=torch.uint8, device=device)
        self.base4 = torch.zeros((2, n_kv_heads, HEAD_DIM), dtype=torch.uint8, device=device)
        self.stats = new_stats(device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.seq_lens = torch.zeros(batch, dtype=torch.int32, device=device)
        self._ws = None
        self.all_raw = False  # encoded with raw=True: every block a raw tile, appends keep it so

    # -- building
    def calibrate(self, k_cal: torch.Tensor, v_cal: torch.Tensor, stream=None):
        """k_cal, v_cal: BF16 [n_tok, kv_heads, 128] calibration tokens."""
        calibrate(k_cal, self.base3[0], self.base4[0], self.status, stream)
        calibrate(v_cal, self.base3[1], self.base4[1], self.status, stream)

    def encode(self, k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor, stream=None, raw: bool = False):
        """Prefill: k, v BF16 [batch, tokens, kv_heads, 128]; seq_lens int32 [batch].
        raw=True stores every block as BF16 (the uncompressed baseline cache)."""
        self.seq_lens.copy_(seq_lens)
        self.all_raw = raw
        encode_blocks(k, v, self.seq_lens, self.max_blocks, self.base3, self.base4, self.table,
                      None if raw else self.slot_ids, self.pools, self.stats, self.status, stream,
                      open_compressed=self.open_compressed and not raw)

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """Decode step: one token per sequence, k_new/v_new BF16 [batch, kv_heads, 128]."""
        append(k_new, v_new, self.seq_lens, self.max_blocks, self.base3, self.base4, self.table,
               None if self.all_raw else self.slot_ids, self.pools, self.stats, self.status, stream,
               open_compressed=self.open_compressed)

    # -- reading
    def auto_splits(self) -> int:
        from . import auto_splits

        return auto_splits(self.batch, self.n_kv_heads, self.max_blocks)

    def workspace(self, n_splits: int = 0) -> torch.Tensor:
        need = attention_workspace(self.batch, self.n_kv_heads, self.max_blocks, n_splits)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=self.device)
        return self._ws

    def attention(self, q: torch.Tensor, scale: float, out: torch.Tensor | None = None, n_splits: int = 0,
                  stream=None, bf16: bool = False) -> torch.Tensor:
        """q: BF16 [batch, q_heads, 128] -> fp32 [batch, q_heads, 128].  bf16=True: the uncompressed BF16
        kernel (the cache must have been encoded with raw=True)."""
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        if bf16:
            decode_attention_bf16(q, self.seq_lens, self.table, self.pools, scale, out, self.workspace(n_splits),
                                  n_splits, self.status, stream)
        else:
            decode_attention(q, self.seq_lens, self.table, self.pools, self.base3, self.base4, scale, out,
                             self.workspace(n_splits), n_splits, self.status, stream)
        return out

    def decompress(self, n_tok: int | None = None, stream=None):
        """BF16 (k, v) [batch, n_tok, kv_heads, 128] rebuilt from the cache (tokens past a sequence: 0)."""
        n_tok = self.max_blocks * BLOCK if n_tok is None else n_tok
        shape = (self.batch, n_tok, self.n_kv_heads, HEAD_DIM)
        k = torch.zeros(shape, dtype=torch.bfloat16, device=self.device)
        v = torch.zeros(shape, dtype=torch.bfloat16, device=self.device)
        decompress(self.table, self.seq_lens, self.pools, self.base3, self.base4, k, v, self.status, stream)
        return k, v

    def fields(self):
        return entry_fields(self.table)

    def resident_bytes(self) -> dict:
        """Bytes held by the cache's blocks: slots, raw tiles, table entries."""
        _, _, mode, _ = entry_fields(self.table)
        n_slot = int((mode == 0).sum().item())
        n_raw = int((mode == 1).sum().item())
        return {"slot_tiles": n_slot, "raw_tiles": n_raw, "slot_bytes": n_slot * 12032, "raw_bytes": n_raw * 16384,
                "table_bytes": self.table.numel() * 8}
