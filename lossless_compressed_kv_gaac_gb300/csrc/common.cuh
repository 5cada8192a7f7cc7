// Device-side building blocks of the GAAC library: tile format v3 constants,
// the packed exponent decoder, status reporting, mbarrier and bulk-copy PTX.
//
// Method: "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference
// on Personal Devices", section 3.1 (base-plus-offset exponent codes, 3-bit /
// 4-bit / raw groups of eight, sign and mantissa verbatim) and Appendix D
// (3-bit code plane, 2-bit tags, escape bytes).  The bit layout is format v3 as
// declared in gaac.h.
#pragma once

#include <cstdint>

#include "gaac.h"

namespace gaac {

constexpr int kD = 128;
constexpr int kBlock = 64;
constexpr int kTile = 8192;
constexpr int kOffCode = 8192;
constexpr int kOffTag = 11264;
constexpr int kOffDir = 11520;  // escape directory: 8 x u16, entry w = n4 | nraw << 9 over eighths 0..w
constexpr int kOffEsc = 11536;  // escape area: 4-bit escape bytes, then 8 exponent bytes per raw group
constexpr int kEscCap = 496;
constexpr int kDirUnits = 32;   // units per directory entry: an eighth = 128 groups = 1024 elements
constexpr int kSlot = 12032;
constexpr int kRawBytes = 16384;

__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------ storage order ----

// V tiles (format v3): element (t, c) of the tile sits at storage position
//   s = 1024 (2 (t/16) + c/64) + 32 (4 (c%8) + (t%8)/2) + 8 ((c/16)%4) + r,
//   r = (c%16)/8 + 2 (t%2) + 4 ((t%16)/8),
// so that unit 32 (2w + h) + 4g + q holds, for the 16-channel blocks
// 4h..4h+3, channels 16m+g and 16m+g+8 at tokens 16w + 2q + {0, 1, 8, 9}: one
// lane's share of a 16 x 16 (channels x tokens) tensor-core operand tile.  K
// tiles are token-major (s = t*128 + c).
__device__ __forceinline__ int v_storage_index(int t, int c) {
  return 1024 * (2 * (t >> 4) + (c >> 6)) + 32 * (4 * (c & 7) + ((t & 7) >> 1)) + 8 * ((c >> 4) & 3) +
         ((c >> 3) & 1) + 2 * (t & 1) + 4 * ((t >> 3) & 1);
}
__device__ __forceinline__ int v_token_of(int s) {
  const int u = s >> 5, r = s & 7;
  return 16 * (u >> 6) + 8 * (r >> 2) + 2 * (u & 3) + ((r >> 1) & 1);
}
__device__ __forceinline__ int v_channel_of(int s) {
  const int u = s >> 5, r = s & 7;
  return 16 * (4 * ((u >> 5) & 1) + ((s >> 3) & 3)) + 8 * (r & 1) + ((u >> 2) & 7);
}

// ---------------------------------------------------------------- codec ----

// Codes of one 16-element half-unit as four words, one code per byte lane
// (lane L of word q = element 4q+L of the half).  wh = W0 or W1 of the unit
// (half h), w2 = W2 of the unit.
__device__ __forceinline__ void extract_codes(uint32_t wh, uint32_t w2, int h, uint32_t c[4]) {
  c[0] = wh & 0x07070707u;
  c[1] = (wh >> 3) & 0x07070707u;
  c[2] = (w2 >> (3 * h)) & 0x07070707u;
  c[3] = ((wh >> 6) & 0x03030303u) | ((w2 >> (4 + h)) & 0x04040404u);
}

// Bit i of a 4-bit value moved to bit 0 of byte lane i.
__device__ __forceinline__ uint32_t spread4(uint32_t n) { return (n * 0x00204081u) & 0x01010101u; }

// Group counts of 16 two-bit tags: 4-bit groups (tag 1), raw groups (tag 2),
// reserved tags (3).
__device__ __forceinline__ int n4_of(uint32_t tags) {
  return __popc(tags & 0x55555555u & ~((tags >> 1) & 0x55555555u));
}
__device__ __forceinline__ int nraw_of(uint32_t tags) {
  return __popc((tags >> 1) & 0x55555555u & ~tags);
}
__device__ __forceinline__ bool reserved_in(uint32_t tags) { return (tags & (tags >> 1) & 0x55555555u) != 0u; }

// Table entry x: the escape byte x of a 4-bit group spread over two exponent
// words, bit j of x becoming bit 3 of byte lane j%4 of word j/4.
__device__ __forceinline__ uint2 spread_entry(uint32_t x) {
  return make_uint2(spread4(x & 15u) << 3, spread4(x >> 4) << 3);
}

// Four bytes of a slot image at any byte offset `off` (4-byte aligned image);
// reads no word past the one holding byte off + 3.
__device__ __forceinline__ uint32_t load_u32_any(const uint8_t* img, int off) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(img + (off & ~3));
  return (off & 3) ? __funnelshift_r(w[0], w[1], 8 * (off & 3)) : w[0];
}

// Exponent words of one half-unit (two groups of eight), format v3.  tagnib:
// the two groups' tags (bits 0-1 first group); b3/b4: base bytes laid out like
// the codes; img: the slot image; *o4: the 4-bit escape byte of the half's
// first 4-bit group (advanced past the half's 4-bit groups); *oraw: escape
// offset of the half's first raw group's exponents (advanced by 8 per raw
// group).  Sets *bad on a reserved tag or a read past esc_len (reads as 0).
__device__ __forceinline__ void half_exponents_v3(uint32_t wh, uint32_t w2, int h, uint32_t tagnib,
                                                  const uint32_t b3[4], const uint32_t b4[4], const uint8_t* img,
                                                  int* o4, int* oraw, int esc_len, uint32_t e[4], bool* bad) {
  uint32_t c[4];
  extract_codes(wh, w2, h, c);
#pragma unroll
  for (int gi = 0; gi < 2; ++gi) {
    const uint32_t m = (tagnib >> (2 * gi)) & 3u;
    const int q0 = 2 * gi;
    if (m == 0u) {
      e[q0] = b3[q0] + c[q0];
      e[q0 + 1] = b3[q0 + 1] + c[q0 + 1];
    } else if (m == 1u) {
      const bool in = *o4 < esc_len;
      if (!in) *bad = true;
      const uint32_t x = in ? img[kOffEsc + *o4] : 0u;
      e[q0] = b4[q0] + (c[q0] | (spread4(x & 15u) << 3));
      e[q0 + 1] = b4[q0 + 1] + (c[q0 + 1] | (spread4(x >> 4) << 3));
      *o4 += 1;
    } else {
      const bool in = m == 2u && *oraw + 8 <= esc_len;
      if (!in) *bad = true;
      e[q0] = in ? load_u32_any(img, kOffEsc + *oraw) : 0u;
      e[q0 + 1] = in ? load_u32_any(img, kOffEsc + *oraw + 4) : 0u;
      *oraw += 8;
    }
  }
}

// Four BF16 values from their sign|mantissa bytes and exponent bytes (byte
// lane L = element L), returned as two bf16x2 words: p01 = elements {0,1},
// p23 = elements {2,3} (lower element in the low half).
__device__ __forceinline__ void join_bf16x4(uint32_t sm, uint32_t e, uint32_t& p01, uint32_t& p23) {
  const uint32_t hi = (sm & 0x80808080u) | ((e >> 1) & 0x7F7F7F7Fu);
  const uint32_t lo = ((e << 7) & 0x80808080u) | (sm & 0x7F7F7F7Fu);
  p01 = __byte_perm(lo, hi, 0x5140);
  p23 = __byte_perm(lo, hi, 0x7362);
}

// Stages tokens [0, nv) of a tile (token t's 128 channels at src + t *
// tok_stride, 16-byte aligned) into `tile` in storage order; tokens past nv
// are zero.  Thread tid of 256 moves a quarter of token tid / 4.
__device__ __forceinline__ void stage_tile(uint16_t* tile, const uint16_t* src, int64_t tok_stride, int nv, int kind,
                                           int tid) {
  const int t = tid >> 2, part = tid & 3;
  uint4 w[4];
  if (t < nv) {
    const uint4* p = reinterpret_cast<const uint4*>(src + t * tok_stride + 32 * part);
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = p[i];
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = make_uint4(0, 0, 0, 0);
  }
  if (kind == 0) {
    uint4* d = reinterpret_cast<uint4*>(tile + t * kD + 32 * part);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = w[i];
  } else {
    const uint32_t* ws = reinterpret_cast<const uint32_t*>(w);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = 32 * part + 2 * i;
      tile[v_storage_index(t, c)] = static_cast<uint16_t>(ws[i] & 0xFFFFu);
      tile[v_storage_index(t, c + 1)] = static_cast<uint16_t>(ws[i] >> 16);
    }
  }
}

// Row stride (elements) of a token-major tile staged in shared memory: 8
// elements of padding put consecutive tokens 4 banks apart, so the scattered
// stores of V units (channels 16m+g, 16m+g+8 of four tokens per lane) spread
// over the banks.
constexpr int kLogicalStride = kD + 8;
constexpr int kLogicalElems = kBlock * kLogicalStride;

// Unit u's rebuilt values (pairs[m] = bf16x2 of storage elements 32u + 2m, +1)
// into a token-major [64][kLogicalStride] tile in shared memory.
__device__ __forceinline__ void unit_to_logical(uint16_t* logical, int kind, int u, const uint32_t pairs[16]) {
  if (kind == 0) {  // token u/4, channels 32(u%4)..+31
    uint4* d = reinterpret_cast<uint4*>(logical + (u >> 2) * kLogicalStride + 32 * (u & 3));
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = make_uint4(pairs[4 * i], pairs[4 * i + 1], pairs[4 * i + 2], pairs[4 * i + 3]);
  } else {
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const int s0 = 32 * u + 2 * m;
      logical[v_token_of(s0) * kLogicalStride + v_channel_of(s0)] = static_cast<uint16_t>(pairs[m] & 0xFFFFu);
      logical[v_token_of(s0 + 1) * kLogicalStride + v_channel_of(s0 + 1)] = static_cast<uint16_t>(pairs[m] >> 16);
    }
  }
}

// Copies the staged tile's 64 rows to dst (row t at dst + t * dst_stride elements, 16-byte aligned), rows
// t < nv only; 256 threads, each store instruction of a warp covering two whole 256-byte rows.
__device__ __forceinline__ void logical_to_global(const uint16_t* logical, uint16_t* dst, int64_t dst_stride, int nv,
                                                  int tid) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int idx = tid + 256 * k, t = idx >> 4, c8 = 8 * (idx & 15);
    if (t < nv)
      *reinterpret_cast<uint4*>(dst + t * dst_stride + c8) =
          *reinterpret_cast<const uint4*>(logical + t * kLogicalStride + c8);
  }
}

// Base bytes of unit u's 32 elements, four per word (word k = elements
// 4k..4k+3 of the unit), from a row of 128 per-channel bases.
__device__ __forceinline__ void unit_base_words(int kind, int u, const uint8_t* bg, uint32_t out[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (kind == 0) {  // K: element 4k+L of unit u is channel 32(u%4) + 4k + L
      out[k] = *reinterpret_cast<const uint32_t*>(bg + 32 * (u & 3) + 4 * k);
    } else {
      uint32_t w = 0u;
#pragma unroll
      for (int L = 0; L < 4; ++L) w |= static_cast<uint32_t>(bg[v_channel_of(32 * u + 4 * k + L)]) << (8 * L);
      out[k] = w;
    }
  }
}

// Exclusive prefixes of the 4-bit and raw group counts (packed n4 | nraw << 16)
// over the 64 tag words of a slot image, into word_prefix[0..63], and the tile
// totals into word_prefix[64].  Threads 0..31 of the CTA call it (one warp).
__device__ __forceinline__ void slot_word_prefix(const uint8_t* slot, int lane, int* word_prefix) {
  const uint32_t* tagw = reinterpret_cast<const uint32_t*>(slot + kOffTag);
  const int c0 = n4_of(tagw[lane]) | (nraw_of(tagw[lane]) << 16);
  const int c1 = n4_of(tagw[lane + 32]) | (nraw_of(tagw[lane + 32]) << 16);
  int i0 = c0, i1 = c1;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v0 = __shfl_up_sync(0xFFFFFFFFu, i0, d), v1 = __shfl_up_sync(0xFFFFFFFFu, i1, d);
    if (lane >= d) {
      i0 += v0;
      i1 += v1;
    }
  }
  const int tot0 = __shfl_sync(0xFFFFFFFFu, i0, 31);
  word_prefix[lane] = i0 - c0;
  word_prefix[lane + 32] = tot0 + i1 - c1;
  if (lane == 31) word_prefix[64] = tot0 + i1;
}

// Rebuilds code unit u (storage elements 32u..32u+31) of a slot image into
// pairs[m] = bf16x2 of storage elements 32u + 2m, 32u + 2m + 1.  word_prefix:
// slot_word_prefix's output for this image; b3w/b4w: the unit's base words
// (word k = elements 4k..4k+3, unit_base_words' layout).  Returns true when the
// unit fails a check of the format (a reserved tag, an escape read past
// esc_len, a directory entry or the totals differing from the tags).
__device__ __forceinline__ bool decode_slot_unit_w(const uint8_t* slot, int u, const uint32_t b3w[8],
                                                   const uint32_t b4w[8], int esc_len, const int* word_prefix,
                                                   uint32_t pairs[16]) {
  const uint32_t* tagw = reinterpret_cast<const uint32_t*>(slot + kOffTag);
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
  if (u == 255 && (dir[7] != ((tot4 & 0x1FF) | ((totraw & 0x7F) << 9)) || tot4 + 8 * totraw != esc_len))
    bad = true;
  const uint4* smp = reinterpret_cast<const uint4*>(slot + 32 * u);
  const uint4 s0 = smp[0], s1 = smp[1];
  uint32_t smw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) {  // signs back to their own bytes (stored one byte up, cyclically)
    const uint32_t sg = smw[j] & 0x80808080u;
    smw[j] = (smw[j] & 0x7F7F7F7Fu) | ((sg >> 8) | (sg << 24));
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const uint32_t b3[4] = {b3w[4 * hh], b3w[4 * hh + 1], b3w[4 * hh + 2], b3w[4 * hh + 3]};
    const uint32_t b4[4] = {b4w[4 * hh], b4w[4 * hh + 1], b4w[4 * hh + 2], b4w[4 * hh + 3]};
    uint32_t e[4];
    half_exponents_v3(hh == 0 ? W0 : W1, W2, hh, (tagbyte >> (4 * hh)) & 15u, b3, b4, slot, &o4, &oraw, esc_len, e,
                      &bad);
#pragma unroll
    for (int q = 0; q < 4; ++q) join_bf16x4(smw[4 * hh + q], e[q], pairs[8 * hh + 2 * q], pairs[8 * hh + 2 * q + 1]);
  }
  return bad;
}

// As decode_slot_unit_w, with the unit's base words read from the tile's 128
// bases b3g/b4g (K: word loads; V: byte gathers).
__device__ __forceinline__ bool decode_slot_unit(const uint8_t* slot, int kind, int u, const uint8_t* b3g,
                                                 const uint8_t* b4g, int esc_len, const int* word_prefix,
                                                 uint32_t pairs[16]) {
  uint32_t b3w[8], b4w[8];
  unit_base_words(kind, u, b3g, b3w);
  unit_base_words(kind, u, b4g, b4w);
  return decode_slot_unit_w(slot, u, b3w, b4w, esc_len, word_prefix, pairs);
}

// A V unit u's element 4k+L has channel v_channel_of(32u + 4k + L), which
// depends on u only through h = (u >> 5) & 1 and g = (u >> 2) & 7: 16 classes.
__device__ __forceinline__ int v_unit_class(int u) { return 8 * ((u >> 5) & 1) + ((u >> 2) & 7); }

// Base words of the 16 V unit classes, table[0 base3 | 1 base4][class][k]; one
// word per thread of 256.
__device__ __forceinline__ void fill_v_base_table(uint32_t (*table)[16][8], const uint8_t* b3g, const uint8_t* b4g,
                                                  int tid) {
  const int which = tid >> 7, cls = (tid >> 3) & 15, k = tid & 7;
  const int urep = 32 * (cls >> 3) + 4 * (cls & 7);  // a unit of the class
  const uint8_t* bg = which ? b4g : b3g;
  uint32_t w = 0u;
#pragma unroll
  for (int L = 0; L < 4; ++L) w |= static_cast<uint32_t>(bg[v_channel_of(32 * urep + 4 * k + L)]) << (8 * L);
  table[which][cls][k] = w;
}

// ------------------------------------------------------- mbarrier / bulk ----

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// One poll; the thread may sleep up to ~20 us inside it (woken early when the
// phase completes), so a waiting warp takes few issue slots from working warps.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(20000)
      : "memory");
  return ok != 0u;
}

// Bounded wait: gives up after `limit` polls and reports GAAC_ETIMEOUT.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* status,
                                          uint32_t limit = (1u << 17)) {
#pragma unroll 1
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  report(status, GAAC_ETIMEOUT);
  return false;
}

// 1-D bulk copy global -> this CTA's shared memory, completion counted on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// D += A * B, m16n8k16, BF16 inputs, FP32 accumulate.
__device__ __forceinline__ void mma_bf16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace gaac
