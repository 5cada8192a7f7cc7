// Device-side building blocks of the GAAC library: tile format v2 constants,
// the packed exponent decoder, status reporting, mbarrier and bulk-copy PTX.
//
// Method: "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference
// on Personal Devices", section 3.1 (base-plus-offset exponent codes, 3-bit /
// 4-bit / raw groups of eight, sign and mantissa verbatim) and Appendix D
// (3-bit code plane, 2-bit tags, escape bytes).  The bit layout is format v2 as
// declared in gaac.h.
#pragma once

#include <cstdint>

#include "gaac.h"

namespace gaac {

constexpr int kD = 128;
constexpr int kBlock = 64;
constexpr int kTile = 8192;
constexpr int kOffCode = 8192;
constexpr int kPlaneBytes = 1024;  // one code plane: 256 words
constexpr int kOffTag = 11264;
constexpr int kOffDir = 11520;  // escape directory: 8 x u16, entry w = escape bytes of eighths 0..w
constexpr int kOffEsc = 11536;  // escape bytes
constexpr int kEscCap = 496;
constexpr int kDirUnits = 32;   // units per directory entry: an eighth = 128 groups = 1024 elements
constexpr int kSlot = 12032;
constexpr int kRawBytes = 16384;

// Largest escape stream a tile can carry if every group is raw (5 bytes x 1024).
constexpr int kEscMaxAnyTile = 5120;

__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
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

// Escape bytes of 16 two-bit group tags (tag 1 -> 1 byte, tag 2 -> 5 bytes, 0 and 3 -> 0).
__device__ __forceinline__ int esc_count(uint32_t tags) {
  const uint32_t lo = tags & 0x55555555u, hi = (tags >> 1) & 0x55555555u;
  return __popc(lo & ~hi) + 5 * __popc(hi & ~lo);
}

// Exponent bytes of one half-unit (two groups).  tagnib: the two groups' tags
// (bits 0-1 first group).  b3/b4: base bytes of the 16 elements, laid out like
// the codes.  esc: escape area of the slot; esc_off: escape offset of the first
// group; esc_len: escape bytes present.  Sets *bad on a reserved tag or an
// escape read past esc_len.
__device__ __forceinline__ void half_exponents(uint32_t wh, uint32_t w2, int h, uint32_t tagnib,
                                               const uint32_t b3[4], const uint32_t b4[4],
                                               const uint8_t* esc, int esc_off, int esc_len,
                                               uint32_t e[4], bool* bad) {
  uint32_t c[4];
  extract_codes(wh, w2, h, c);
  if (tagnib == 0u) {
#pragma unroll
    for (int q = 0; q < 4; ++q) e[q] = b3[q] + c[q];
    return;
  }
  int off = esc_off;
#pragma unroll
  for (int gi = 0; gi < 2; ++gi) {
    const uint32_t m = (tagnib >> (2 * gi)) & 3u;
    const int q0 = 2 * gi;
    if (m == 0u) {
      e[q0] = b3[q0] + c[q0];
      e[q0 + 1] = b3[q0 + 1] + c[q0 + 1];
    } else if (m == 1u) {
      const bool in = off + 1 <= esc_len;  // never read past the escape bytes present
      if (!in) *bad = true;
      const uint32_t x = in ? esc[off] : 0u;
      e[q0] = b4[q0] + (c[q0] | (spread4(x & 15u) << 3));
      e[q0 + 1] = b4[q0 + 1] + (c[q0 + 1] | (spread4(x >> 4) << 3));
      off += 1;
    } else {
      const bool in = off + 5 <= esc_len;
      if (m == 3u || !in) *bad = true;
      uint32_t hi0 = 0, hi1 = 0;
#pragma unroll
      for (int k = 0; k < 5; ++k) {
        const uint32_t x = in ? esc[off + k] : 0u;
        hi0 |= spread4(x & 15u) << (3 + k);
        hi1 |= spread4(x >> 4) << (3 + k);
      }
      e[q0] = c[q0] | hi0;
      e[q0 + 1] = c[q0 + 1] | hi1;
      off += 5;
    }
  }
}

// Table entry x: the escape byte x of a 4-bit group spread over two exponent
// words, bit j of x becoming bit 3 of byte lane j%4 of word j/4.
__device__ __forceinline__ uint2 spread_entry(uint32_t x) {
  return make_uint2(spread4(x & 15u) << 3, spread4(x >> 4) << 3);
}

// Escape bytes of a group with tag m (0: 0, 1: 1, 2: 5; tag 3 counts 6 and is
// rejected by the caller).
__device__ __forceinline__ int esc_of_tag(uint32_t m) { return static_cast<int>((m & 1u) + 5u * (m >> 1)); }

// Exponent bytes of one half-unit (two groups of eight), without per-lane
// branches for the 3-bit and 4-bit modes.  tagnib: the two groups' tags (bits
// 0-1 first group); b3/b4: base bytes laid out like the codes; esc: escape area
// of the slot image (esc_len bytes valid); off: escape offset of the first
// group; lut: 256 spread_entry values.  Raw-mode groups take a rare branch.
// Sets *bad on a reserved tag or an escape read past esc_len (such bytes read as 0).
__device__ __forceinline__ void half_exponents_fast(uint32_t wh, uint32_t w2, int h, uint32_t tagnib,
                                                    const uint32_t b3[4], const uint32_t b4[4],
                                                    const uint8_t* esc, int off, int esc_len, const uint2* lut,
                                                    uint32_t e[4], bool* bad) {
  uint32_t c[4];
  extract_codes(wh, w2, h, c);
  const uint32_t m0 = tagnib & 3u, m1 = (tagnib >> 2) & 3u;
  const int off1 = off + esc_of_tag(m0);
  const uint32_t x0 = (m0 == 1u && off < esc_len) ? esc[off] : 0u;
  const uint32_t x1 = (m1 == 1u && off1 < esc_len) ? esc[off1] : 0u;
  const uint2 s0 = lut[x0], s1 = lut[x1];
  e[0] = (m0 != 0u ? b4[0] : b3[0]) + c[0] + s0.x;
  e[1] = (m0 != 0u ? b4[1] : b3[1]) + c[1] + s0.y;
  e[2] = (m1 != 0u ? b4[2] : b3[2]) + c[2] + s1.x;
  e[3] = (m1 != 0u ? b4[3] : b3[3]) + c[3] + s1.y;
  if ((m0 == 1u && off >= esc_len) || (m1 == 1u && off1 >= esc_len)) *bad = true;
  if (tagnib & 0xAu) {  // a raw-mode (or reserved) group: five escape bit planes
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
      const uint32_t m = gi == 0 ? m0 : m1;
      if (m >= 2u) {
        const int o = gi == 0 ? off : off1;
        const bool in = m == 2u && o + 5 <= esc_len;
        if (!in) *bad = true;
        uint32_t hi0 = 0, hi1 = 0;
#pragma unroll
        for (int k = 0; k < 5; ++k) {
          const uint32_t x = in ? esc[o + k] : 0u;
          hi0 |= spread4(x & 15u) << (3 + k);
          hi1 |= spread4(x >> 4) << (3 + k);
        }
        e[2 * gi] = c[2 * gi] | hi0;
        e[2 * gi + 1] = c[2 * gi + 1] | hi1;
      }
    }
  }
}

// Exponent bytes of one half-unit when the 4-bit-mode escape bytes of its unit
// have been gathered in advance: xw holds, in byte j, the escape byte of group j
// of the unit (0 unless that group is in 4-bit mode).  tb: the unit's tag byte;
// hh: which half.  Raw-mode groups are left for the caller (their words come out
// as base4 + code).  The tile must have been validated (no reserved tags).
__device__ __forceinline__ void half_exponents_gathered(uint32_t wh, uint32_t w2, int hh, uint32_t tb, uint32_t xw,
                                                        const uint32_t b3[4], const uint32_t b4[4],
                                                        const uint2* lut, uint32_t e[4]) {
  uint32_t c[4];
  extract_codes(wh, w2, hh, c);
  const uint32_t tagnib = (tb >> (4 * hh)) & 15u;
  const uint32_t xs = xw >> (16 * hh);
  const uint2 s0 = lut[xs & 0xFFu], s1 = lut[(xs >> 8) & 0xFFu];
  const bool w0 = (tagnib & 3u) != 0u, w1 = (tagnib & 12u) != 0u;
  e[0] = (w0 ? b4[0] : b3[0]) + c[0] + s0.x;
  e[1] = (w0 ? b4[1] : b3[1]) + c[1] + s0.y;
  e[2] = (w1 ? b4[2] : b3[2]) + c[2] + s1.x;
  e[3] = (w1 ? b4[3] : b3[3]) + c[3] + s1.y;
}

// Raw-mode group gi (0/1) of a half-unit: exponent words from the group's five
// escape bit planes at `esc` (already offset to the group).
__device__ __forceinline__ void raw_group_exponents(uint32_t wh, uint32_t w2, int hh, int gi, const uint8_t* esc,
                                                    uint32_t e[4]) {
  uint32_t c[4];
  extract_codes(wh, w2, hh, c);
  uint32_t hi0 = 0, hi1 = 0;
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    const uint32_t x = esc[k];
    hi0 |= spread4(x & 15u) << (3 + k);
    hi1 |= spread4(x >> 4) << (3 + k);
  }
  e[2 * gi] = c[2 * gi] | hi0;
  e[2 * gi + 1] = c[2 * gi + 1] | hi1;
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

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
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

// One non-blocking poll.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
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

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
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
