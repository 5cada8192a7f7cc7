// FP8 variant of the GAAC codec: calibration, tile encoder and decoder for
// E4M3 and E5M2 KV tiles.
//
// "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference on
// Personal Devices", Appendix B (Relation to FP8 KV): the same exponent coding
// applied to a cache already quantised to FP8, lossless with respect to the FP8
// values.  Section 3.1 gives the coding: windows of 8 and 16 exponents per
// head-channel, groups of eight in 3-bit / 4-bit / raw mode, sign and mantissa
// verbatim.  Layout: GAAC-FP8 tile format v1 (gaac.h) -- the format v3 storage
// order, groups, codes, tags, directory and escape area, with the sign and
// mantissa as 4-bit nibbles (E4M3) or 3-bit fields laid out like the code plane
// (E5M2), and the exponent windows inside the format's 16 or 32 exponents.
//
// One CTA of 256 threads per tile; thread u owns the 32-element code unit u.
#include <cuda_runtime.h>

#include "common.cuh"

namespace gaac {

struct Fp8Layout {
  int ew, mw, off_code, off_tag, off_dir, off_esc, slot;
};

__host__ __device__ inline bool fp8_layout(int fmt, Fp8Layout* L) {
  if (fmt == GAAC_FP8_E4M3) {
    *L = Fp8Layout{4, 3, 4096, 7168, 7424, 7440, 7936};
    return true;
  }
  if (fmt == GAAC_FP8_E5M2) {
    *L = Fp8Layout{5, 2, 3072, 6144, 6400, 6416, 6912};
    return true;
  }
  return false;
}

constexpr int kFp8Threads = 256;
constexpr int kFp8Stride = kD + 16;  // padded row of a staged FP8 tile: consecutive tokens 4 banks apart

// Calibration: one CTA per row of bases (kv-head), one thread per channel, a
// histogram of the format's 16 or 32 exponents per channel in shared memory.
__global__ void __launch_bounds__(kD) fp8_calibrate_kernel(const uint8_t* __restrict__ x, int64_t n_tok,
                                                           int64_t tok_stride, int ew, int mw,
                                                           uint8_t* __restrict__ base3, uint8_t* __restrict__ base4) {
  __shared__ uint32_t hist[32][kD];
  const int h = blockIdx.x, c = threadIdx.x;
  const int nb = 1 << ew;
  for (int b = 0; b < nb; ++b) hist[b][c] = 0u;
  const uint8_t* p = x + static_cast<int64_t>(h) * kD + c;
  for (int64_t t = 0; t < n_tok; ++t) hist[(p[t * tok_stride] >> mw) & (nb - 1)][c] += 1u;
  // strict '>' keeps the smallest base on ties
  uint32_t best3 = 0, best4 = 0;
  int arg3 = 0, arg4 = 0;
  for (int b = 0; b + 8 <= nb; ++b) {
    uint32_t s = 0;
    for (int i = 0; i < 8; ++i) s += hist[b + i][c];
    if (b == 0 || s > best3) {
      best3 = s;
      arg3 = b;
    }
  }
  for (int b = 0; b + 16 <= nb; ++b) {
    uint32_t s = 0;
    for (int i = 0; i < 16; ++i) s += hist[b + i][c];
    if (b == 0 || s > best4) {
      best4 = s;
      arg4 = b;
    }
  }
  base3[h * kD + c] = static_cast<uint8_t>(arg3);
  base4[h * kD + c] = static_cast<uint8_t>(arg4);
}

// Adds element j's 3-bit field v to the unit's three words (format v3's code-plane placement: element
// 16h + 4q + L in byte lane L of W[h] at bits 0-2 (q = 0) or 3-5 (q = 1), of W[2] at bits 3h.. (q = 2), or
// split as bits 6-7 of W[h] and bit 6+h of W[2] (q = 3)).
__device__ __forceinline__ void put_field3(uint32_t W[3], int j, uint32_t v) {
  const int h = j >> 4, jj = j & 15, L = jj & 3, q = jj >> 2;
  if (q == 0) W[h] |= v << (8 * L);
  if (q == 1) W[h] |= v << (8 * L + 3);
  if (q == 2) W[2] |= v << (8 * L + 3 * h);
  if (q == 3) {
    W[h] |= (v & 3u) << (8 * L + 6);
    W[2] |= ((v >> 2) & 1u) << (8 * L + 6 + h);
  }
}

// Adds the 3-bit fields of group gi (f0: elements 8gi..8gi+3, f1: 8gi+4..8gi+7, one field per byte lane)
// to the unit's three words in put_field3's placement: words 2gi and 2gi+1 are q = 2(gi%2) and q+1 of
// half gi/2.
__device__ __forceinline__ void place_fields3(uint32_t W[3], int gi, uint32_t f0, uint32_t f1) {
  const int h = gi >> 1;
  if ((gi & 1) == 0) {
    W[h] |= f0 | (f1 << 3);
  } else {
    W[2] |= (f0 << (3 * h)) | ((f1 & 0x04040404u) << (4 + h));
    W[h] |= (f1 & 0x03030303u) << 6;
  }
}

struct Fp8Args {
  const uint8_t* tiles;
  int64_t n_tiles;
  Fp8Layout L;
  const uint8_t* tile_kind;
  const int32_t* tile_row;
  int n_rows;
  const uint8_t* base3;
  const uint8_t* base4;
  uint8_t* slots;
  uint16_t* esc_len;
  gaac_stats* stats;
  int32_t* status;
};

// The group loop element by element (bases outside the calibrated ranges).  Rare, so kept out of line:
// the word-wide loop then gets the registers.
struct Fp8UnitCodes {
  uint32_t CW[3], SW[4], esc4, tagbyte;
  int n4, nraw, my_counts[3];
};

__device__ __noinline__ void fp8_groups_elementwise(const uint8_t* seq, int u, const Fp8Layout& L,
                                                    const uint32_t (*vtab)[16][8], int cls, Fp8UnitCodes* out) {
  const uint32_t emask = (1u << L.ew) - 1u, mmask = (1u << L.mw) - 1u;
  uint32_t CW[3] = {0u, 0u, 0u};
  uint32_t SW[4] = {0u, 0u, 0u, 0u};
  uint32_t esc4 = 0, tagbyte = 0;
  int n4 = 0, nraw = 0, my_counts[3] = {0, 0, 0};
#pragma unroll
  for (int gi = 0; gi < 4; ++gi) {
    uint32_t e[8];
    int b3[8], b4[8];
    bool fits3 = true, fits4 = true;
    const uint32_t b3q[2] = {vtab[0][cls][2 * gi], vtab[0][cls][2 * gi + 1]};  // four bases per word
    const uint32_t b4q[2] = {vtab[1][cls][2 * gi], vtab[1][cls][2 * gi + 1]};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int el = 8 * gi + j;
      const uint32_t x = seq[32 * u + el];
      e[j] = (x >> L.mw) & emask;
      const uint32_t smv = ((x >> 7) << L.mw) | (x & mmask);
      if (L.ew == 4)
        SW[el >> 3] |= smv << (4 * (el & 7));
      else
        put_field3(SW, el, smv);
      b3[j] = (b3q[j >> 2] >> (8 * (j & 3))) & 0xFFu;
      b4[j] = (b4q[j >> 2] >> (8 * (j & 3))) & 0xFFu;
      const int o3 = static_cast<int>(e[j]) - b3[j], o4 = static_cast<int>(e[j]) - b4[j];
      fits3 = fits3 && o3 >= 0 && o3 <= 7;
      fits4 = fits4 && o4 >= 0 && o4 <= 15;
    }
    const uint32_t mode = fits3 ? 0u : (fits4 ? 1u : 2u);
    tagbyte |= mode << (2 * gi);
    my_counts[mode] += 1;
    uint32_t eb = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t cd = 0;  // raw groups keep code 0: their exponents are escape bytes
      if (mode == 0u) {
        cd = (e[j] - static_cast<uint32_t>(b3[j])) & 7u;
      } else if (mode == 1u) {
        const uint32_t off = (e[j] - static_cast<uint32_t>(b4[j])) & 0xFFu;
        cd = off & 7u;
        eb |= ((off >> 3) & 1u) << j;
      }
      put_field3(CW, 8 * gi + j, cd);
    }
    if (mode == 1u) {
      esc4 |= eb << (8 * n4);
      n4 += 1;
    }
    if (mode == 2u) nraw += 1;
  }
#pragma unroll
  for (int i = 0; i < 3; ++i) out->CW[i] = CW[i];
#pragma unroll
  for (int i = 0; i < 4; ++i) out->SW[i] = SW[i];
  out->esc4 = esc4;
  out->tagbyte = tagbyte;
  out->n4 = n4;
  out->nraw = nraw;
#pragma unroll
  for (int i = 0; i < 3; ++i) out->my_counts[i] = my_counts[i];
}

__global__ void __launch_bounds__(kFp8Threads, 6) fp8_encode_kernel(Fp8Args a) {
  __shared__ alignas(16) uint8_t seq[kTile];  // the tile in storage order
  __shared__ uint32_t vtab[2][16][8];         // V: base3 / base4 words of the 16 unit classes
  __shared__ int warp_sums[kFp8Threads / 32];
  __shared__ int mode_counts[4];
  const int64_t tile = blockIdx.x;
  const int u = threadIdx.x, lane = u & 31, warp = u >> 5;
  const int kind = a.tile_kind[tile], row = a.tile_row[tile];
  if ((kind != 0 && kind != 1) || row < 0 || row >= a.n_rows) {
    if (u == 0) {
      a.esc_len[tile] = 0xFFFFu;
      report(a.status, GAAC_EINVAL);
    }
    return;
  }
  const Fp8Layout L = a.L;
  const uint8_t* src = a.tiles + tile * kTile;
  {  // stage: 32 bytes per thread, storage order
    const uint4* s4 = reinterpret_cast<const uint4*>(src + 32 * u);
    const uint4 x0 = s4[0], x1 = s4[1];
    if (kind == 0) {
      uint4* d = reinterpret_cast<uint4*>(seq + 32 * u);
      d[0] = x0;
      d[1] = x1;
    } else {
      // Storage elements 2m' and 2m'+1 are channels c and c+8 of one token, so the thread's 32 channels
      // 32p .. 32p+31 of token t form 16 byte pairs: channels 32p + 16m + j and + 8 (j < 8) at pair index
      // v_storage_index(t, 32p + 16m + j) / 2 = base + 64j + 4m.
      const int t = u >> 2, p = u & 3;
      const int base = 1024 * (t >> 4) + 512 * (p >> 1) + 16 * ((t >> 1) & 3) + 8 * (p & 1) + (t & 1) + 2 * ((t >> 3) & 1);
      uint16_t* sp = reinterpret_cast<uint16_t*>(seq) + base;
      const uint32_t lo[2][2] = {{x0.x, x0.y}, {x1.x, x1.y}};  // [m][j / 4]: channels 16m + j
      const uint32_t hi[2][2] = {{x0.z, x0.w}, {x1.z, x1.w}};  // the same + 8
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int j = 0; j < 8; ++j)
          sp[64 * j + 4 * m] = static_cast<uint16_t>(__byte_perm(lo[m][j >> 2], hi[m][j >> 2], 0x40 | (j & 3) | ((j & 3) << 4)));
    }
  }
  const uint8_t* b3g = a.base3 + static_cast<size_t>(row) * kD;
  const uint8_t* b4g = a.base4 + static_cast<size_t>(row) * kD;
  // Base words by unit class: V, the 16 classes of v_unit_class; K, class u % 4.
  if (kind == 1) {
    fill_v_base_table(vtab, b3g, b4g, u);
  } else if (u < 64) {
    const int which = u >> 5, c = (u >> 3) & 3, k = u & 7;
    vtab[which][c][k] = *reinterpret_cast<const uint32_t*>((which ? b4g : b3g) + 32 * c + 4 * k);
  }
  if (u < 4) mode_counts[u] = 0;
  // Bases above 248 (base3) or 240 (base4) take the element-by-element path (the word test below is exact
  // only up to those).
  bool odd_base = false;
  if (u < kD / 4) {
    const uint32_t w3 = reinterpret_cast<const uint32_t*>(b3g)[u], w4 = reinterpret_cast<const uint32_t*>(b4g)[u];
#pragma unroll
    for (int q = 0; q < 4; ++q) odd_base = odd_base || ((w3 >> (8 * q)) & 0xFFu) > 248u || ((w4 >> (8 * q)) & 0xFFu) > 240u;
  }
  const bool word_fit = __syncthreads_or(odd_base) == 0;
  const int cls = kind == 0 ? (u & 3) : v_unit_class(u);
  const uint32_t emask = (1u << L.ew) - 1u, mmask = (1u << L.mw) - 1u;
  uint32_t CW[3] = {0u, 0u, 0u};  // code-plane words, filled field by field
  uint32_t SW[4] = {0u, 0u, 0u, 0u};  // sign|mantissa: nibbles (E4M3) or 3-bit fields in SW[0..2] (E5M2)
  uint32_t esc4 = 0, tagbyte = 0;
  int n4 = 0, nraw = 0, my_counts[3] = {0, 0, 0};
  if (word_fit) {
    // Four elements per word (word k = elements 4k..4k+3 of the unit): exponent bytes E, offsets
    // D = E - base in one subtraction; a group fits the 3-bit (4-bit) mode iff no byte of D has a bit
    // above bit 2 (bit 3), exact for base3 <= 248 (base4 <= 240) as in the BF16 encoder.
    const uint4* s4 = reinterpret_cast<const uint4*>(seq + 32 * u);
    const uint4 q0 = s4[0], q1 = s4[1];
    const uint32_t x[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const uint32_t emw = emask * 0x01010101u, mmw = mmask * 0x01010101u, sgw = 0x01010101u << L.mw;
#pragma unroll
    for (int gi = 0; gi < 4; ++gi) {
      const uint32_t w0 = x[2 * gi], w1 = x[2 * gi + 1];
      const uint32_t E0 = (w0 >> L.mw) & emw, E1 = (w1 >> L.mw) & emw;
      // sign|mantissa fields: the sign (bit 7) to bit mw above the mantissa
      const uint32_t s0 = ((w0 >> (7 - L.mw)) & sgw) | (w0 & mmw), s1 = ((w1 >> (7 - L.mw)) & sgw) | (w1 & mmw);
      const uint32_t d3a = E0 - vtab[0][cls][2 * gi], d3b = E1 - vtab[0][cls][2 * gi + 1];
      const uint32_t d4a = E0 - vtab[1][cls][2 * gi], d4b = E1 - vtab[1][cls][2 * gi + 1];
      const bool fits3 = ((d3a | d3b) & 0xF8F8F8F8u) == 0u, fits4 = ((d4a | d4b) & 0xF0F0F0F0u) == 0u;
      const uint32_t mode = fits3 ? 0u : (fits4 ? 1u : 2u);
      tagbyte |= mode << (2 * gi);
      my_counts[mode] += 1;
      const uint32_t c0 = fits3 ? d3a : (fits4 ? (d4a & 0x07070707u) : 0u);
      const uint32_t c1 = fits3 ? d3b : (fits4 ? (d4b & 0x07070707u) : 0u);
      place_fields3(CW, gi, c0, c1);
      if (L.ew == 4) {  // nibbles, element 8gi + j in nibble j of SW[gi]
        const uint32_t n0 = (s0 & 0x000F000Fu) | ((s0 >> 4) & 0x00F000F0u);
        const uint32_t n1 = (s1 & 0x000F000Fu) | ((s1 >> 4) & 0x00F000F0u);
        SW[gi] = __byte_perm(n0, n1, 0x6420);
      } else {
        place_fields3(SW, gi, s0, s1);
      }
      if (mode == 1u) {
        const uint32_t eb = ((((d4a >> 3) & 0x01010101u) * 0x01020408u) >> 24) |
                            (((((d4b >> 3) & 0x01010101u) * 0x01020408u) >> 24) << 4);
        esc4 |= eb << (8 * n4);
        n4 += 1;
      }
      if (mode == 2u) nraw += 1;
    }
  } else {
    Fp8UnitCodes uc;
    fp8_groups_elementwise(seq, u, L, vtab, cls, &uc);
#pragma unroll
    for (int i = 0; i < 3; ++i) CW[i] = uc.CW[i];
#pragma unroll
    for (int i = 0; i < 4; ++i) SW[i] = uc.SW[i];
    esc4 = uc.esc4;
    tagbyte = uc.tagbyte;
    n4 = uc.n4;
    nraw = uc.nraw;
#pragma unroll
    for (int i = 0; i < 3; ++i) my_counts[i] = uc.my_counts[i];
  }
  // exclusive scans of the 4-bit and raw group counts (packed; each total is at most 1024)
  const int packed = n4 | (nraw << 16);
  int incl = packed;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kFp8Threads / 32; ++w) {
    const int s = warp_sums[w];
    if (w < warp) before += s;
    total += s;
  }
  const int excl = before + incl - packed;
  const int off4 = excl & 0xFFFF, offraw = excl >> 16, tot4 = total & 0xFFFF, totraw = total >> 16;
  const int esc = tot4 + 8 * totraw;
  if (esc > kEscCap) {  // CTA-uniform: the tile stays FP8
    if (u == 0) {
      a.esc_len[tile] = 0xFFFFu;
      if (a.stats != nullptr) atomicAdd(&a.stats->raw_tiles, 1ull);
    }
    return;
  }
  uint8_t* slot = a.slots + tile * L.slot;
  // sign|mantissa plane
  if (L.ew == 4) {  // nibble of element s in byte s/2 (low nibble for even s): 16 bytes per unit
    *reinterpret_cast<uint4*>(slot + 16 * u) = make_uint4(SW[0], SW[1], SW[2], SW[3]);
  } else {  // 3-bit fields laid out like the code plane, at offset 0
    uint32_t* sw = reinterpret_cast<uint32_t*>(slot);
    sw[u] = SW[0];
    sw[256 + u] = SW[1];
    sw[512 + u] = SW[2];
  }
  {
    uint32_t* cw = reinterpret_cast<uint32_t*>(slot + L.off_code);
    cw[u] = CW[0];
    cw[256 + u] = CW[1];
    cw[512 + u] = CW[2];
  }
  slot[L.off_tag + u] = static_cast<uint8_t>(tagbyte);
  uint8_t* escp = slot + L.off_esc;
  for (int k = 0; k < n4; ++k) escp[off4 + k] = static_cast<uint8_t>(esc4 >> (8 * k));
  if (nraw) {
    int r = tot4 + 8 * offraw;
#pragma unroll
    for (int gi = 0; gi < 4; ++gi) {
      if (((tagbyte >> (2 * gi)) & 3u) != 2u) continue;
#pragma unroll
      for (int j = 0; j < 8; ++j) escp[r + j] = static_cast<uint8_t>((seq[32 * u + 8 * gi + j] >> L.mw) & emask);
      r += 8;
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int at = 2 * u + i;
    if (at >= esc && at < kEscCap) escp[at] = 0;
  }
  if ((u & (kDirUnits - 1)) == kDirUnits - 1) {
    const int w = u / kDirUnits;
    const uint32_t entry = ((off4 + n4) & 0x1FF) | (((offraw + nraw) & 0x7F) << 9);
    slot[L.off_dir + 2 * w] = static_cast<uint8_t>(entry & 0xFFu);
    slot[L.off_dir + 2 * w + 1] = static_cast<uint8_t>(entry >> 8);
  }
  if (u == 0) a.esc_len[tile] = static_cast<uint16_t>(esc);
  if (a.stats != nullptr) {
#pragma unroll
    for (int m = 0; m < 3; ++m)
      if (my_counts[m]) atomicAdd(&mode_counts[m], my_counts[m]);
    __syncthreads();
    if (u == 0) {
#pragma unroll
      for (int m = 0; m < 3; ++m) atomicAdd(&a.stats->groups[m], static_cast<unsigned long long>(mode_counts[m]));
      atomicAdd(&a.stats->escape_bytes, static_cast<unsigned long long>(esc));
      atomicAdd(&a.stats->slot_tiles, 1ull);
    }
  }
}

__global__ void __launch_bounds__(kFp8Threads) fp8_decompress_kernel(Fp8Args a, uint8_t* __restrict__ out) {
  // the staged slot image, then (after a barrier) the token-major tile with padded rows
  __shared__ alignas(16) uint8_t logical[kBlock * kFp8Stride];
  static_assert(kBlock * kFp8Stride >= 7936, "the buffer holds the larger FP8 slot image");
  __shared__ uint32_t vtab[2][16][8];  // V: base3 / base4 words of the 16 unit classes
  __shared__ int word_prefix[65];
  const int64_t tile = blockIdx.x;
  const int u = threadIdx.x;
  const int kind = a.tile_kind[tile], row = a.tile_row[tile];
  const int esc_len = a.esc_len[tile];
  if (esc_len == 0xFFFF) return;  // kept as FP8 by the caller
  if ((kind != 0 && kind != 1) || row < 0 || row >= a.n_rows || esc_len > kEscCap) {
    if (u == 0) report(a.status, GAAC_EINVAL);
    return;
  }
  const Fp8Layout L = a.L;
  const uint8_t* gslot = a.slots + tile * L.slot;
  // The image's used bytes move to shared memory as 16-byte asynchronous copies, into the buffer that takes
  // the token-major tile later; the tag prefix and the V base table are built from global memory meanwhile.
  const int n16 = (L.off_esc + esc_len + 15) >> 4;
  for (int q = u; q < n16; q += kFp8Threads)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(logical + 16 * q)), "l"(gslot + 16 * q)
                 : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
  const uint32_t* tagw = reinterpret_cast<const uint32_t*>(gslot + L.off_tag);
  const uint8_t* b3g = a.base3 + static_cast<size_t>(row) * kD;
  const uint8_t* b4g = a.base4 + static_cast<size_t>(row) * kD;
  if (kind == 1) fill_v_base_table(vtab, b3g, b4g, u);
  if (u < 32) {  // exclusive prefixes of 4-bit and raw group counts over the 64 tag words (packed)
    const int c0 = n4_of(tagw[u]) | (nraw_of(tagw[u]) << 16);
    const int c1 = n4_of(tagw[u + 32]) | (nraw_of(tagw[u + 32]) << 16);
    int i0 = c0, i1 = c1;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v0 = __shfl_up_sync(0xFFFFFFFFu, i0, d), v1 = __shfl_up_sync(0xFFFFFFFFu, i1, d);
      if (u >= d) {
        i0 += v0;
        i1 += v1;
      }
    }
    const int tot0 = __shfl_sync(0xFFFFFFFFu, i0, 31);
    word_prefix[u] = i0 - c0;
    word_prefix[u + 32] = tot0 + i1 - c1;
    if (u == 31) word_prefix[64] = tot0 + i1;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();
  const uint8_t* slot = logical;  // the staged image
  const uint32_t tagbyte = slot[L.off_tag + u];
  const uint32_t before = reinterpret_cast<const uint32_t*>(slot + L.off_tag)[u >> 2] & ((1u << (8 * (u & 3))) - 1u);
  const int pre = word_prefix[u >> 2] + (n4_of(before) | (nraw_of(before) << 16));
  const int tot = word_prefix[64], tot4 = tot & 0xFFFF, totraw = tot >> 16;
  int o4 = pre & 0xFFFF, oraw = tot4 + 8 * (pre >> 16);
  const uint16_t* dir = reinterpret_cast<const uint16_t*>(slot + L.off_dir);
  bool bad = reserved_in(tagbyte);
  if ((u & (kDirUnits - 1)) == 0 && u > 0 &&
      dir[u / kDirUnits - 1] != static_cast<uint16_t>(((pre & 0xFFFF) & 0x1FF) | (((pre >> 16) & 0x7F) << 9)))
    bad = true;
  if (u == 255 && (dir[7] != static_cast<uint16_t>((tot4 & 0x1FF) | ((totraw & 0x7F) << 9)) ||
                   tot4 + 8 * totraw != esc_len))
    bad = true;
  uint32_t C[3], S[3] = {0u, 0u, 0u};
  const uint32_t* cw = reinterpret_cast<const uint32_t*>(slot + L.off_code);
  C[0] = cw[u];
  C[1] = cw[256 + u];
  C[2] = cw[512 + u];
  uint4 nib = make_uint4(0u, 0u, 0u, 0u);
  if (L.ew == 4) {
    nib = *reinterpret_cast<const uint4*>(slot + 16 * u);
  } else {
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(slot);
    S[0] = sw[u];
    S[1] = sw[256 + u];
    S[2] = sw[512 + u];
  }
  // Four elements per 32-bit word (byte lane L = element 4k + L of the unit), as in the BF16 decoder:
  // codes and E5M2 sign|mantissa fields come out of their three-word units by byte lanes, E4M3 nibbles by
  // two masks and a byte permute.
  uint32_t cq[8], sq[8];
  extract_codes(C[0], C[2], 0, &cq[0]);
  extract_codes(C[1], C[2], 1, &cq[4]);
  if (L.ew == 4) {
    const uint32_t nw[4] = {nib.x, nib.y, nib.z, nib.w};  // word i: elements 8i..8i+7, low nibble first
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = nw[i] & 0x0F0F0F0Fu, hi = (nw[i] >> 4) & 0x0F0F0F0Fu;
      sq[2 * i] = __byte_perm(lo, hi, 0x5140);
      sq[2 * i + 1] = __byte_perm(lo, hi, 0x7362);
    }
  } else {
    extract_codes(S[0], S[2], 0, &sq[0]);
    extract_codes(S[1], S[2], 1, &sq[4]);
  }
  uint32_t b3w[8], b4w[8];
  if (kind == 0) {
    unit_base_words(0, u, b3g, b3w);
    unit_base_words(0, u, b4g, b4w);
  } else {
    const int cls = v_unit_class(u);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      b3w[k] = vtab[0][cls][k];
      b4w[k] = vtab[1][cls][k];
    }
  }
  const uint32_t emask_w = ((1u << L.ew) - 1u) * 0x01010101u, mmask_w = ((1u << L.mw) - 1u) * 0x01010101u;
  uint32_t xw[8];
#pragma unroll
  for (int gi = 0; gi < 4; ++gi) {
    const uint32_t mode = (tagbyte >> (2 * gi)) & 3u;
    uint32_t e[2];
    if (mode == 0u) {
      e[0] = b3w[2 * gi] + cq[2 * gi];
      e[1] = b3w[2 * gi + 1] + cq[2 * gi + 1];
    } else if (mode == 1u) {
      uint32_t x4 = 0;
      if (o4 < esc_len) x4 = slot[L.off_esc + o4];
      else bad = true;
      o4 += 1;
      e[0] = b4w[2 * gi] + (cq[2 * gi] | (spread4(x4 & 15u) << 3));
      e[1] = b4w[2 * gi + 1] + (cq[2 * gi + 1] | (spread4(x4 >> 4) << 3));
    } else {
      const bool rawok = mode == 2u && oraw + 8 <= esc_len;
      if (!rawok) bad = true;
      e[0] = rawok ? load_u32_any(slot, L.off_esc + oraw) : 0u;
      e[1] = rawok ? load_u32_any(slot, L.off_esc + oraw + 4) : 0u;
      oraw += 8;
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {  // FP8 byte: sign (bit mw of sm) to bit 7, exponent, mantissa
      const uint32_t sm = sq[2 * gi + q];
      xw[2 * gi + q] = (((sm >> L.mw) & 0x01010101u) << 7) | ((e[q] & emask_w) << L.mw) | (sm & mmask_w);
    }
  }
  if (bad) report(a.status, GAAC_EFORMAT);
  __syncthreads();  // every unit has read the staged image
  if (kind == 0) {  // token u/4, channels 32(u%4)..+31
    uint4* d = reinterpret_cast<uint4*>(logical + (u >> 2) * kFp8Stride + 32 * (u & 3));
    d[0] = make_uint4(xw[0], xw[1], xw[2], xw[3]);
    d[1] = make_uint4(xw[4], xw[5], xw[6], xw[7]);
  } else {
#pragma unroll
    for (int el = 0; el < 32; ++el) {
      const int s = 32 * u + el;
      logical[v_token_of(s) * kFp8Stride + v_channel_of(s)] = static_cast<uint8_t>(xw[el >> 2] >> (8 * (el & 3)));
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 2; ++k) {  // 64 rows of 128 bytes, a whole row per 8 threads
    const int idx = u + kFp8Threads * k, t = idx >> 3, c16 = 16 * (idx & 7);
    *reinterpret_cast<uint4*>(out + tile * kTile + t * kD + c16) =
        *reinterpret_cast<const uint4*>(logical + t * kFp8Stride + c16);
  }
}

}  // namespace gaac

using namespace gaac;

extern "C" int gaac_fp8_slot_bytes(int fmt) {
  Fp8Layout L;
  return fp8_layout(fmt, &L) ? L.slot : 0;
}

extern "C" int gaac_fp8_calibrate(const uint8_t* x, int64_t n_tok, int64_t tok_stride, int n_kv_heads, int fmt,
                                  uint8_t* base3, uint8_t* base4, int32_t* d_status, void* stream) {
  (void)d_status;
  Fp8Layout L;
  if (x == nullptr || base3 == nullptr || base4 == nullptr || !fp8_layout(fmt, &L)) return GAAC_EINVAL;
  if (n_tok < 1 || n_tok > 65535 || n_kv_heads <= 0 || n_kv_heads > 65535 || tok_stride < n_kv_heads * kD)
    return GAAC_EINVAL;
  fp8_calibrate_kernel<<<n_kv_heads, kD, 0, static_cast<cudaStream_t>(stream)>>>(x, n_tok, tok_stride, L.ew, L.mw,
                                                                                  base3, base4);
  return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}

static int fp8_args(const uint8_t* tiles, int64_t n_tiles, int fmt, const uint8_t* tile_kind, const int32_t* tile_row,
                    int n_rows, const uint8_t* base3, const uint8_t* base4, uint8_t* slots, uint16_t* esc_len,
                    gaac_stats* stats, int32_t* d_status, Fp8Args* a) {
  if (tiles == nullptr || tile_kind == nullptr || tile_row == nullptr || base3 == nullptr || base4 == nullptr ||
      slots == nullptr || esc_len == nullptr || n_tiles < 0 || n_tiles > 0x7FFFFFFFLL || n_rows <= 0)
    return GAAC_EINVAL;
  if ((reinterpret_cast<uintptr_t>(tiles) & 15u) || (reinterpret_cast<uintptr_t>(slots) & 15u) ||
      (reinterpret_cast<uintptr_t>(base3) & 3u) || (reinterpret_cast<uintptr_t>(base4) & 3u))
    return GAAC_EINVAL;
  if (!fp8_layout(fmt, &a->L)) return GAAC_EINVAL;
  a->tiles = tiles;
  a->n_tiles = n_tiles;
  a->tile_kind = tile_kind;
  a->tile_row = tile_row;
  a->n_rows = n_rows;
  a->base3 = base3;
  a->base4 = base4;
  a->slots = slots;
  a->esc_len = esc_len;
  a->stats = stats;
  a->status = d_status;
  return GAAC_OK;
}

extern "C" int gaac_fp8_encode_tiles(const uint8_t* tiles, int64_t n_tiles, int fmt, const uint8_t* tile_kind,
                                     const int32_t* tile_row, int n_rows, const uint8_t* base3, const uint8_t* base4,
                                     uint8_t* slots, uint16_t* esc_len, gaac_stats* stats, int32_t* d_status,
                                     void* stream) {
  Fp8Args a;
  const int st = fp8_args(tiles, n_tiles, fmt, tile_kind, tile_row, n_rows, base3, base4, slots, esc_len, stats,
                          d_status, &a);
  if (st != GAAC_OK) return st;
  if (n_tiles == 0) return GAAC_OK;
  fp8_encode_kernel<<<static_cast<unsigned>(n_tiles), kFp8Threads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}

extern "C" int gaac_fp8_decompress_tiles(const uint8_t* slots, const uint16_t* esc_len, int64_t n_tiles, int fmt,
                                         const uint8_t* tile_kind, const int32_t* tile_row, int n_rows,
                                         const uint8_t* base3, const uint8_t* base4, uint8_t* tiles,
                                         int32_t* d_status, void* stream) {
  Fp8Args a;
  const int st = fp8_args(tiles, n_tiles, fmt, tile_kind, tile_row, n_rows, base3, base4,
                          const_cast<uint8_t*>(slots), const_cast<uint16_t*>(esc_len), nullptr, d_status, &a);
  if (st != GAAC_OK) return st;
  if (n_tiles == 0) return GAAC_OK;
  fp8_decompress_kernel<<<static_cast<unsigned>(n_tiles), kFp8Threads, 0, static_cast<cudaStream_t>(stream)>>>(
      a, tiles);
  return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}
