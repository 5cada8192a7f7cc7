// Decompression of a GAAC layer cache back to BF16 (the block decode whose
// latency the GAAC page's section 4.3 / Figure 4 reports; used here for
// bit-exact checks and the decode-bandwidth measurement).
//
// One CTA of 256 threads per tile.  The slot image's used bytes are staged in
// shared memory with 16-byte asynchronous copies; thread u decodes code unit u
// (32 storage elements) from it with the same packed decoder the attention
// kernel uses; the tile is then assembled token-major in the same buffer and
// written out row by row.
#include <cuda_runtime.h>

#include "common.cuh"

namespace gaac {

constexpr int kDecThreads = 256;

struct DecompressArgs {
  const gaac_entry* table;
  const int32_t* seq_lens;
  int n_kv_heads, max_blocks;
  const uint8_t* slot_pool;
  int64_t n_slots;
  const uint16_t* raw_pool;
  int64_t n_raw;
  const uint8_t* base3;
  const uint8_t* base4;
  uint16_t* k_out;
  uint16_t* v_out;
  int64_t seq_stride, tok_stride, n_tok;
  int32_t* status;
};

// 16-byte asynchronous global -> shared copy.
__device__ __forceinline__ void cp_async16_dec(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// grid (2*n_kv_heads, max_blocks, batch): x = h*2 + kind.
__global__ void __launch_bounds__(kDecThreads, 8) decompress_kernel(DecompressArgs a) {
  // the slot image's used bytes, then (after a barrier) the token-major tile [t][c] with padded rows
  __shared__ alignas(16) uint16_t logical[kLogicalElems];
  uint8_t* simg = reinterpret_cast<uint8_t*>(logical);
  __shared__ int word_prefix[65];
  __shared__ uint32_t vbt[2][16][8];  // V: base words of the unit classes
  const int h = blockIdx.x >> 1, kind = blockIdx.x & 1;
  const int blk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, u = tid;
  const int len = a.seq_lens[b];
  if (len < 0 || len > a.max_blocks * kBlock) {
    if (tid == 0) report(a.status, GAAC_EINVAL);
    return;
  }
  if (len > a.n_tok && blk == 0 && tid == 0 && h == 0 && kind == 0) report(a.status, GAAC_EINVAL);
  const int lim = static_cast<int>(min(static_cast<int64_t>(len), a.n_tok));
  if (blk * kBlock >= lim) return;
  const int nv = min(kBlock, lim - blk * kBlock);
  const gaac_entry ent = a.table[((static_cast<size_t>(b) * a.max_blocks + blk) * a.n_kv_heads + h) * 2 + kind];
  const bool as_slot = ent.mode == GAAC_MODE_SLOT && static_cast<int64_t>(ent.index) < a.n_slots &&
                       ent.esc_len <= kEscCap;
  const bool as_raw = ent.mode == GAAC_MODE_RAW && static_cast<int64_t>(ent.index) < a.n_raw;
  if (!as_slot && !as_raw) {
    if (tid == 0) report(a.status, GAAC_EFORMAT);
    return;
  }
  uint32_t pairs[16];  // bf16x2 of storage elements 32u + 2m, +1
  if (as_raw) {
    const uint4* src = reinterpret_cast<const uint4*>(a.raw_pool + static_cast<size_t>(ent.index) * kTile + 32 * u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 w = src[i];
      pairs[4 * i] = w.x;
      pairs[4 * i + 1] = w.y;
      pairs[4 * i + 2] = w.z;
      pairs[4 * i + 3] = w.w;
    }
  } else {
    const uint8_t* slot = a.slot_pool + static_cast<size_t>(ent.index) * kSlot;
    const uint8_t* b3g = a.base3 + (kind * a.n_kv_heads + h) * kD;
    const uint8_t* b4g = a.base4 + (kind * a.n_kv_heads + h) * kD;
    // The image's used bytes move to shared memory as 16-byte asynchronous copies while the tag prefix and
    // the base table are built from global memory; the units then read the staged image.
    const int n16 = (kOffEsc + ent.esc_len + 15) >> 4;
    for (int q = tid; q < n16; q += kDecThreads) cp_async16_dec(simg + 16 * q, slot + 16 * q);
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (tid < 32) slot_word_prefix(slot, tid, word_prefix);
    if (kind == 1) fill_v_base_table(vbt, b3g, b4g, tid);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    const int cls = v_unit_class(u);
    const bool bad = kind == 0 ? decode_slot_unit(simg, 0, u, b3g, b4g, ent.esc_len, word_prefix, pairs)
                               : decode_slot_unit_w(simg, u, vbt[0][cls], vbt[1][cls], ent.esc_len, word_prefix, pairs);
    if (bad) report(a.status, GAAC_EFORMAT);
    __syncthreads();  // every unit has read the staged image
  }
  unit_to_logical(logical, kind, u, pairs);  // storage order -> token-major
  __syncthreads();
  uint16_t* dst = (kind == 0 ? a.k_out : a.v_out) + static_cast<int64_t>(b) * a.seq_stride +
                  static_cast<int64_t>(blk) * kBlock * a.tok_stride + h * kD;
  logical_to_global(logical, dst, a.tok_stride, nv, tid);
}

struct DecodeTilesArgs {
  const uint8_t* slots;
  const uint16_t* esc_len;
  const uint8_t* kind;
  const int32_t* row;
  int n_rows;
  const uint8_t* base3;
  const uint8_t* base4;
  uint16_t* tiles;
  int32_t* status;
};

// grid (n_tiles): one CTA rebuilds one slot image of the batch into its
// token-major tile (tiles whose esc_len is 0xFFFF are skipped).
__global__ void __launch_bounds__(kDecThreads, 8) decode_tiles_kernel(DecodeTilesArgs a) {
  __shared__ alignas(16) uint16_t logical[kLogicalElems];
  __shared__ int word_prefix[65];
  __shared__ uint32_t vbt[2][16][8];  // V: base words of the unit classes
  const int64_t i = blockIdx.x;
  const int tid = threadIdx.x;
  const int esc = a.esc_len[i];
  if (esc == 0xFFFF) return;
  const int kind = a.kind[i], r = a.row[i];
  if (kind > 1 || r < 0 || r >= a.n_rows || esc > kEscCap) {
    if (tid == 0) report(a.status, GAAC_EINVAL);
    return;
  }
  const uint8_t* slot = a.slots + i * kSlot;
  if (tid < 32) slot_word_prefix(slot, tid, word_prefix);
  if (kind == 1) fill_v_base_table(vbt, a.base3 + r * kD, a.base4 + r * kD, tid);
  __syncthreads();
  uint32_t pairs[16];
  const int cls = v_unit_class(tid);
  const bool bad = kind == 0 ? decode_slot_unit(slot, 0, tid, a.base3 + r * kD, a.base4 + r * kD, esc, word_prefix, pairs)
                             : decode_slot_unit_w(slot, tid, vbt[0][cls], vbt[1][cls], esc, word_prefix, pairs);
  if (bad) report(a.status, GAAC_EFORMAT);
  unit_to_logical(logical, kind, tid, pairs);
  __syncthreads();
  logical_to_global(logical, a.tiles + i * kTile, kD, kBlock, tid);
}

}  // namespace gaac

using namespace gaac;

extern "C" int gaac_decompress(const gaac_entry* table, const int32_t* seq_lens, int batch, int n_kv_heads,
                               int max_blocks, const gaac_pools* pools, const uint8_t* base3, const uint8_t* base4,
                               uint16_t* k_out, uint16_t* v_out, int64_t seq_stride, int64_t tok_stride,
                               int64_t n_tok, int32_t* d_status, void* stream) {
  if (table == nullptr || seq_lens == nullptr || pools == nullptr || pools->slot_pool == nullptr ||
      pools->raw_pool == nullptr || pools->n_slots < 0 || pools->n_raw < 0 || base3 == nullptr ||
      base4 == nullptr || k_out == nullptr || v_out == nullptr)
    return GAAC_EINVAL;
  const uint8_t* slot_pool = pools->slot_pool;
  const uint16_t* raw_pool = pools->raw_pool;
  if (batch <= 0 || batch > 65535 || n_kv_heads <= 0 || n_kv_heads > 1024 || max_blocks <= 0 || max_blocks > 65535)
    return GAAC_EINVAL;
  if (tok_stride < static_cast<int64_t>(n_kv_heads) * kD || (tok_stride & 7) || (seq_stride & 7) ||
      (reinterpret_cast<uintptr_t>(k_out) & 15u) || (reinterpret_cast<uintptr_t>(v_out) & 15u) ||
      (reinterpret_cast<uintptr_t>(slot_pool) & 15u) || (reinterpret_cast<uintptr_t>(raw_pool) & 15u) ||
      (reinterpret_cast<uintptr_t>(base3) & 15u) || (reinterpret_cast<uintptr_t>(base4) & 15u))
    return GAAC_EINVAL;
  if (n_tok < 0) return GAAC_EINVAL;
  DecompressArgs a{table, seq_lens, n_kv_heads, max_blocks, slot_pool, pools->n_slots, raw_pool, pools->n_raw,
                   base3, base4, k_out, v_out, seq_stride, tok_stride, n_tok, d_status};
  decompress_kernel<<<dim3(2 * n_kv_heads, max_blocks, batch), kDecThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}

extern "C" int gaac_decode_tiles(const uint8_t* slots, const uint16_t* esc_len, int64_t n_tiles,
                                 const uint8_t* tile_kind, const int32_t* tile_row, int n_rows, const uint8_t* base3,
                                 const uint8_t* base4, uint16_t* tiles, int32_t* d_status, void* stream) {
  if (slots == nullptr || esc_len == nullptr || tile_kind == nullptr || tile_row == nullptr || base3 == nullptr ||
      base4 == nullptr || tiles == nullptr || n_rows <= 0)
    return GAAC_EINVAL;
  if (n_tiles < 0 || n_tiles > 0x7FFFFFFF || (reinterpret_cast<uintptr_t>(tiles) & 15u) ||
      (reinterpret_cast<uintptr_t>(slots) & 15u) || (reinterpret_cast<uintptr_t>(base3) & 3u) ||
      (reinterpret_cast<uintptr_t>(base4) & 3u))
    return GAAC_EINVAL;
  if (n_tiles == 0) return GAAC_OK;
  DecodeTilesArgs a{slots, esc_len, tile_kind, tile_row, n_rows, base3, base4, tiles, d_status};
  decode_tiles_kernel<<<static_cast<unsigned>(n_tiles), kDecThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}
