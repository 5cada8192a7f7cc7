// Decompression of a GAAC layer cache back to BF16 (the block decode whose
// latency the GAAC page's section 4.3 / Figure 4 reports; used here for
// bit-exact checks and the decode-bandwidth measurement).
//
// One CTA of 256 threads per tile; thread u decodes code unit u (32 storage
// elements) with the same packed decoder the attention kernel uses, the tile
// is assembled token-major in shared memory and written out row by row.
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

// grid (2*n_kv_heads, max_blocks, batch): x = h*2 + kind.
__global__ void __launch_bounds__(kDecThreads) decompress_kernel(DecompressArgs a) {
  __shared__ alignas(16) uint16_t logical[kBlock * kD];  // [t][c]
  __shared__ int word_prefix[65];
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
    const uint32_t* tagw = reinterpret_cast<const uint32_t*>(slot + kOffTag);
    if (tid < 32) {  // exclusive prefixes of 4-bit and raw group counts over the 64 tag words (packed)
      const int c0 = n4_of(tagw[tid]) | (nraw_of(tagw[tid]) << 16);
      const int c1 = n4_of(tagw[tid + 32]) | (nraw_of(tagw[tid + 32]) << 16);
      int i0 = c0, i1 = c1;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v0 = __shfl_up_sync(0xFFFFFFFFu, i0, d), v1 = __shfl_up_sync(0xFFFFFFFFu, i1, d);
        if (tid >= d) {
          i0 += v0;
          i1 += v1;
        }
      }
      const int tot0 = __shfl_sync(0xFFFFFFFFu, i0, 31);
      word_prefix[tid] = i0 - c0;
      word_prefix[tid + 32] = tot0 + i1 - c1;
      if (tid == 31) word_prefix[64] = tot0 + i1;  // tile totals
    }
    __syncthreads();
    const uint32_t* cw = reinterpret_cast<const uint32_t*>(slot + kOffCode);
    const uint32_t W0 = cw[u], W1 = cw[256 + u], W2 = cw[512 + u];
    const uint32_t tagbyte = slot[kOffTag + u];
    const uint32_t tword = tagw[u >> 2];
    const uint32_t before = tword & ((1u << (8 * (u & 3))) - 1u);  // tags of the word's earlier units
    const int pre = word_prefix[u >> 2] + (n4_of(before) | (nraw_of(before) << 16));
    const int tot = word_prefix[64];
    const int tot4 = tot & 0xFFFF, totraw = tot >> 16;
    int o4 = pre & 0xFFFF, oraw = tot4 + 8 * (pre >> 16);
    // The escape directory must hold the counts at each eighth boundary and the totals.
    const uint16_t* dir = reinterpret_cast<const uint16_t*>(slot + kOffDir);
    bool bad = reserved_in(tagbyte);
    if ((u & (kDirUnits - 1)) == 0 && u > 0 &&
        dir[u / kDirUnits - 1] != (((pre & 0xFFFF) & 0x1FF) | (((pre >> 16) & 0x7F) << 9)))
      bad = true;
    if (u == 255 && (dir[7] != ((tot4 & 0x1FF) | ((totraw & 0x7F) << 9)) || tot4 + 8 * totraw != ent.esc_len))
      bad = true;
    const uint4* smp = reinterpret_cast<const uint4*>(slot + 32 * u);
    const uint4 s0 = smp[0], s1 = smp[1];
    uint32_t smw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // signs back to their own bytes (stored one byte up, cyclically)
      const uint32_t sg = smw[j] & 0x80808080u;
      smw[j] = (smw[j] & 0x7F7F7F7Fu) | ((sg >> 8) | (sg << 24));
    }
    const uint8_t* b3g = a.base3 + (kind * a.n_kv_heads + h) * kD;
    const uint8_t* b4g = a.base4 + (kind * a.n_kv_heads + h) * kD;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t b3[4], b4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (kind == 0) {  // K: element 4q+L of half hh is channel 32(u%4) + 16hh + 4q + L
          const int c = 32 * (u & 3) + 16 * hh + 4 * q;
          b3[q] = *reinterpret_cast<const uint32_t*>(b3g + c);
          b4[q] = *reinterpret_cast<const uint32_t*>(b4g + c);
        } else {  // V: element 4q+L of half hh is storage element 32u + 16hh + 4q + L
          b3[q] = b4[q] = 0u;
#pragma unroll
          for (int L = 0; L < 4; ++L) {
            const int c = v_channel_of(32 * u + 16 * hh + 4 * q + L);
            b3[q] |= static_cast<uint32_t>(b3g[c]) << (8 * L);
            b4[q] |= static_cast<uint32_t>(b4g[c]) << (8 * L);
          }
        }
      }
      uint32_t e[4];
      half_exponents_v3(hh == 0 ? W0 : W1, W2, hh, (tagbyte >> (4 * hh)) & 15u, b3, b4, slot, &o4, &oraw,
                        ent.esc_len, e, &bad);
#pragma unroll
      for (int q = 0; q < 4; ++q) join_bf16x4(smw[4 * hh + q], e[q], pairs[8 * hh + 2 * q], pairs[8 * hh + 2 * q + 1]);
    }
    if (bad) report(a.status, GAAC_EFORMAT);
  }
  // Storage order -> token-major.
  if (kind == 0) {
    uint4* d = reinterpret_cast<uint4*>(logical + 32 * u);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = make_uint4(pairs[4 * i], pairs[4 * i + 1], pairs[4 * i + 2], pairs[4 * i + 3]);
  } else {
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const int s0 = 32 * u + 2 * m;
      logical[v_token_of(s0) * kD + v_channel_of(s0)] = static_cast<uint16_t>(pairs[m] & 0xFFFFu);
      logical[v_token_of(s0 + 1) * kD + v_channel_of(s0 + 1)] = static_cast<uint16_t>(pairs[m] >> 16);
    }
  }
  __syncthreads();
  uint16_t* dst = (kind == 0 ? a.k_out : a.v_out) + static_cast<int64_t>(b) * a.seq_stride +
                  static_cast<int64_t>(blk) * kBlock * a.tok_stride + h * kD;
  const int t = tid >> 2, part = tid & 3;
  if (t < nv) {
    uint4* d = reinterpret_cast<uint4*>(dst + t * a.tok_stride + 32 * part);
    const uint4* s = reinterpret_cast<const uint4*>(logical + t * kD + 32 * part);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = s[i];
  }
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
