// Fused split-K GQA decode attention over the GAAC compressed cache.
//
// "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference on
// Personal Devices", section 3.2: attention reads the compressed tiles and
// rebuilds the values it needs on the fly (no decompressed copy of the cache
// in global memory); compressed blocks and the raw tail go through one
// softmax.  Section 3.3: the block table says per block whether it is a slot
// or a raw tile.
//
// GB300 design: one CTA of 352 threads per SM, grid (split, kv-head, sequence).
//  * Warp 10 (producer): one lane streams each 64-token block's K and V tile
//    images (only the bytes a slot uses) into a 3-stage shared-memory ring
//    with 1-D bulk copies tracked by mbarriers.
//  * Warps 0-7 (decoders): warp w rebuilds quarter w%4 (code units
//    [64q, 64q+64)) of the K (w < 4) or V tile into BF16 in a swizzled
//    shared-memory tile.  A lane owns two 32-element units.  The escape
//    directory gives the quarter's first escape byte, a packed warp scan each
//    unit's, and one byte permute gathers a unit's 4-bit escape bytes.
//    Exponents are rebuilt four at a time in 32-bit words (the bytes cannot
//    carry) and joined with the sign|mantissa word by two bit selects and a
//    byte rotation per four values.  Raw-mode groups are rare and patched
//    afterwards by the lane that owns them.
//  * Warps 8-9 (tensor-core warps) take alternate blocks: QK^T and PV^T with
//    ldmatrix + mma.sync m16n8k16 (bf16 in, fp32 accumulate), an online
//    softmax in the log2 domain that rescales only when a running maximum
//    rises, and P stored transposed (stmatrix) as a bf16 hi + lo pair so its
//    rounding stays near 2^-17.  Each warp keeps (m, l, acc) for its own
//    blocks; the two are merged when the split ends.
//  * The decoded tiles hold each group of four values in the order {0,2,1,3}
//    (the join's output order).  The QK^T contraction runs over channels in
//    that order (q's fragment follows it); the PV^T contraction runs over
//    tokens in that order (QK^T rows are permuted the same way, so P^T comes
//    out in it).
//  * q is pre-scaled by 2^-4 (exact for normal values) to keep q.k inside the
//    fp32 range for extreme keys; the factor is folded into the softmax scale.
//  * Partials (m, l, acc) per split go to the workspace; the last CTA of each
//    (sequence, kv-head) to finish, found with a device counter, merges them
//    with a log-sum-exp (the final split reduction) and resets the counter.
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"

namespace gaac {

constexpr int kDWarps = 16;                      // decoders: 0-7 K eighths, 8-15 V eighths
constexpr int kMGroupWarps = 4;                  // a tensor-core group: one 16-token / 32-channel share per warp
constexpr int kMGroups = 1;                      // groups take alternate blocks
constexpr int kMWarps = kMGroupWarps * kMGroups;
constexpr int kMWarp0 = kDWarps;
constexpr int kProducerWarp = kDWarps + kMWarps;
constexpr int kAttThreads = (kProducerWarp + 1) * 32;
constexpr int kStages = 3;                       // staging ring of K+V tile images
constexpr int kDecBufs = 3;                      // decoded BF16 K+V tiles
constexpr int kCtasPerSm = 1;
constexpr int kRPad = 8;                         // query heads per kv-head in the MMA N dimension
constexpr int kPtStride = 72;                    // bf16 per head row of P^T (64 tokens + pad): 144 B
constexpr int kQStride = 136;                    // bf16 per head row of q (128 channels + pad): 272 B
constexpr int kPartFloats = 2 * kRPad + kRPad * kD;
constexpr int kBarM = 1;                         // named barriers 1, 2: one per tensor-core group
constexpr int kBarMAll = kBarM + kMGroups;       // all tensor-core warps (end of the split)
constexpr uint32_t kJoinMask = 0x807F807Fu;      // sign and mantissa bits of a bf16x2 word
constexpr uint32_t kFull = 0xFFFFFFFFu;

struct StageMeta {
  int mode[2], esc[2];  // [K, V]
};

struct AttSmem {
  alignas(128) uint8_t stage[kStages][2][kRawBytes];  // K, V tile images
  alignas(128) uint8_t decK[kDecBufs][kTile * 2];      // BF16 K, rows = tokens (256 B), swizzled
  alignas(128) uint8_t decV[kDecBufs][kTile * 2];      // BF16 V, rows = channels (128 B), swizzled
  alignas(16) uint16_t pt[kMGroups][2][kRPad][kPtStride];  // per group: P^T hi, lo of its current block
  alignas(16) uint16_t qs[kRPad][kQStride];                 // q * 2^-4, channels in decoded order
  alignas(16) float wmax[kMGroups][kRPad][kMGroupWarps];    // per head: max of each warp's 16 scores
  alignas(16) float wl[kMGroups][kRPad][kMGroupWarps];      // per head: row sums of each warp (at the end)
  alignas(16) float xacc[kRPad][kD];                        // group 1's accumulators (at the end)
  float xm[kRPad];                                          // group 1's running maxima (at the end)
  uint2 lut[256];       // escape byte -> bit 3 spread into the byte lanes of two exponent words
  uint32_t tagl[256];   // tag byte -> gather selector (bits 0-15), escape bytes (16-23), needs a patch (24)
  StageMeta smeta[kStages];
  int dec_nv[kDecBufs];                   // tokens of the block in decoded buffer d
  alignas(8) uint8_t dec_bad[kDecBufs][8];  // K eighth failed its checks
  uint64_t stFull[kStages], stEmpty[kStages];
  uint64_t dkFull[kDecBufs], dvFull[kDecBufs], dkEmpty[kDecBufs], dvEmpty[kDecBufs];
  int last;
};

struct AttnArgs {
  const uint16_t* q;
  const int32_t* seq_lens;
  const gaac_entry* table;
  const uint8_t* slot_pool;
  int64_t n_slots;
  const uint16_t* raw_pool;
  int64_t n_raw;
  const uint8_t* base3;
  const uint8_t* base4;
  float scale_log2;  // scale * 16 * log2(e)
  int Hq, Hkv, r, max_blocks, n_splits;
  float* part;
  unsigned int* counters;  // [batch][Hkv] splits finished; zero between launches
  float* out;
  int32_t* status;
};

// ------------------------------------------------------------------ helpers

// bf16x2 times 2^-4; exact whenever the result is a normal number.
__device__ __forceinline__ uint32_t bf16x2_div16(uint32_t w) {
  const float lo = __uint_as_float(w << 16) * 0.0625f;
  const float hi = __uint_as_float(w & 0xFFFF0000u) * 0.0625f;
  return (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int warp_incl_scan(int x, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(kFull, x, d);
    if (lane >= d) x += v;
  }
  return x;
}

__device__ __forceinline__ unsigned int atomic_add_acq_rel(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void stsm_x4_trans(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(r0), "r"(r1),
               "r"(r2), "r"(r3)
               : "memory");
}

// Position p of a decoded row holds element quad_perm(p): each aligned group
// of four is stored {0,2,1,3}.  The map is its own inverse.
__device__ __forceinline__ int quad_perm(int p) { return (p & ~3) | ((p & 1) << 1) | ((p >> 1) & 1); }

// Byte offset of 16-byte chunk c (0..15) of token row t in a decoded K tile.
// The chunk's low three bits are XORed with the row (and bit 1 flipped in the
// upper half-row) so that ldmatrix over 8 rows and the decoders' 16-byte
// stores both touch 8 different bank groups.
__device__ __forceinline__ uint32_t kswz(int t, int c) {
  return static_cast<uint32_t>(t * 256 + 16 * ((c & 8) | ((c ^ t ^ ((c >> 3) << 1)) & 7)));
}
// Byte offset of 16-byte chunk c (0..7) of channel row ch in a decoded V tile.
__device__ __forceinline__ uint32_t vswz(int ch, int c) { return static_cast<uint32_t>(ch * 128 + 16 * ((c ^ ch) & 7)); }

// Four BF16 values from one sign|mantissa word of format v2 (byte L: mantissa
// of element L, sign of element (L+3)%4) and their exponent word (byte L =
// exponent of element L): p02 = elements {0, 2}, p13 = elements {1, 3}.
// Rotating the exponents left by 7 puts elements 0 and 2 in their bf16 fields
// and elements 1 and 3 in the fields of the same word rotated by one byte.
__device__ __forceinline__ void join_v2(uint32_t w, uint32_t e, uint32_t& p02, uint32_t& p13) {
  uint32_t r, t;
  asm("shf.l.wrap.b32 %0, %1, %1, 7;" : "=r"(r) : "r"(e));
  // lop3 0xE4: c ? a : b per bit, with c = kJoinMask (the sign and mantissa bits of a bf16x2 word)
  asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(p02) : "r"(w), "r"(r), "n"(kJoinMask));  // sign|mantissa from w
  asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(t) : "r"(r), "r"(w), "n"(kJoinMask));    // rotated frame
  p13 = __byte_perm(t, t, 0x0321);
}

// Everything the decoders need from a unit's tag byte (4 groups x 2 bits):
//  bits 0-15: byte permute selector that gathers the escape bytes of the
//    unit's 4-bit groups from the four escape bytes at the unit's offset (byte
//    j = group j's escape byte if group j is 4-bit and no raw group precedes it
//    in the unit, else a zero byte; the others are patched separately);
//  bits 16-23: the unit's escape bytes (1 per 4-bit group, 5 per raw group),
//    255 if a group has the reserved tag 3 (the quarter's total check fails);
//  bit 24: the unit has a raw group (patch_unit must run).
__device__ __forceinline__ uint32_t tag_entry(uint32_t tb) {
  uint32_t s = 0, rank = 0, bytes = 0;
  bool raw = false, reserved = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t t = (tb >> (2 * j)) & 3u;
    if (t == 3u) reserved = true;
    if (t >= 2u) raw = true;
    const uint32_t nib = (t == 1u && !raw) ? rank : 4u;  // 4: a zero byte of the second operand
    if (t == 1u) ++rank;
    bytes += t == 1u ? 1u : (t == 2u ? 5u : 0u);
    s |= nib << (4 * j);
  }
  return s | ((reserved ? 255u : bytes) << 16) | (raw ? (1u << 24) : 0u);
}

// The four escape bytes starting at escape offset `off` of a slot image.
__device__ __forceinline__ uint32_t escape_window(const uint8_t* img, int off) {
  const uint32_t* ew = reinterpret_cast<const uint32_t*>(img + kOffEsc);
  const uint32_t w0 = ew[off >> 2], w1 = ew[(off >> 2) + 1];
  return __funnelshift_r(w0, w1, 8 * (off & 3));
}

// Rebuilds 32-element unit u of a slot image into 16 bf16x2 words, in decoded
// order: word 2q+i of half h holds elements 16h+4q + {0,2} (i=0) / {1,3} (i=1).
// x: the unit's gathered 4-bit escape bytes (byte j = group j); b3/d43: the
// unit's base3 words and base4 - base3 (32-bit, modular: e stays exact), word
// i covering elements 4i..4i+3.  Raw groups and 4-bit groups after them come
// out wrong and are patched by patch_unit.
__device__ __forceinline__ void decode_unit(const uint8_t* img, int u, uint32_t tb, uint32_t x, const uint32_t b3[8],
                                            const uint32_t d43[8], const uint2* lut, uint32_t o[16]) {
  const uint32_t* cw = reinterpret_cast<const uint32_t*>(img + kOffCode);
  const uint32_t W0 = cw[u], W1 = cw[256 + u], W2 = cw[512 + u];
  const uint4 s0 = *reinterpret_cast<const uint4*>(img + 32 * u);
  const uint4 s1 = *reinterpret_cast<const uint4*>(img + 32 * u + 16);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    uint32_t c[4];
    extract_codes(hh ? W1 : W0, W2, hh, c);
    const uint2 sa = lut[(x >> (16 * hh)) & 0xFFu], sb = lut[(x >> (16 * hh + 8)) & 0xFFu];
    const uint32_t fa = (tb >> (4 * hh)) & 1u, fb = (tb >> (4 * hh + 2)) & 1u;  // 4-bit flags of the two groups
    uint32_t e[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t f = q < 2 ? fa : fb;
      const uint32_t s = q == 0 ? sa.x : (q == 1 ? sa.y : (q == 2 ? sb.x : sb.y));
      e[q] = (f ? b3[4 * hh + q] + d43[4 * hh + q] : b3[4 * hh + q]) + c[q] + s;  // base4 = base3 + d43
    }
    const uint4 sm = hh ? s1 : s0;
    join_v2(sm.x, e[0], o[8 * hh + 0], o[8 * hh + 1]);
    join_v2(sm.y, e[1], o[8 * hh + 2], o[8 * hh + 3]);
    join_v2(sm.z, e[2], o[8 * hh + 4], o[8 * hh + 5]);
    join_v2(sm.w, e[3], o[8 * hh + 6], o[8 * hh + 7]);
  }
}

// Decoded chunk j (0..3) of unit u of a K (kind 0) or V tile: byte offset.
__device__ __forceinline__ uint32_t unit_chunk(int kind, int u, int j) {
  return kind == 0 ? kswz(u >> 2, 4 * (u & 3) + j) : vswz(u >> 1, 4 * (u & 1) + j);
}

__device__ __forceinline__ void store_unit(uint8_t* dec, uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                           const uint32_t o[16]) {
  *reinterpret_cast<uint4*>(dec + c0) = make_uint4(o[0], o[1], o[2], o[3]);
  *reinterpret_cast<uint4*>(dec + c1) = make_uint4(o[4], o[5], o[6], o[7]);
  *reinterpret_cast<uint4*>(dec + c2) = make_uint4(o[8], o[9], o[10], o[11]);
  *reinterpret_cast<uint4*>(dec + c3) = make_uint4(o[12], o[13], o[14], o[15]);
}

// V tail (the open block): zero the decoded values of tokens >= nv in V unit
// u, whose tokens are 32(u%2)..+31, so that no stale value meets a zero
// probability.  Runs for one block per split at most.
__device__ __noinline__ void clear_tail(uint8_t* dec, int u, int nv) {
#pragma unroll 1
  for (int j = 0; j < 4; ++j) {
    const int t0 = 32 * (u & 1) + 8 * j;  // chunk j: tokens t0..t0+7 stored {0,2,1,3,4,6,5,7}
    if (t0 + 8 <= nv) continue;
    uint4* p = reinterpret_cast<uint4*>(dec + vswz(u >> 1, 4 * (u & 1) + j));
    uint4 w = *p;
    w.x &= (t0 < nv ? 0x0000FFFFu : 0u) | (t0 + 2 < nv ? 0xFFFF0000u : 0u);
    w.y &= (t0 + 1 < nv ? 0x0000FFFFu : 0u) | (t0 + 3 < nv ? 0xFFFF0000u : 0u);
    w.z &= (t0 + 4 < nv ? 0x0000FFFFu : 0u) | (t0 + 6 < nv ? 0xFFFF0000u : 0u);
    w.w &= (t0 + 5 < nv ? 0x0000FFFFu : 0u) | (t0 + 7 < nv ? 0xFFFF0000u : 0u);
    *p = w;
  }
}

// Re-decodes the groups of unit u that decode_unit cannot: raw groups (their
// exponent bits 3..7 are five escape bit planes) and 4-bit groups placed after
// a raw group.  off: the unit's first escape byte.  Rewrites those groups'
// 16-byte chunks in the decoded tile.
__device__ __forceinline__ void patch_unit(const uint8_t* img, int kind, int u, uint32_t tb, int off,
                                           const uint8_t* b4g, const uint2* lut, uint8_t* dec) {
  uint32_t fix = 0;
  bool raw = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t t = (tb >> (2 * j)) & 3u;
    if (t == 2u || (t == 1u && raw)) fix |= 1u << j;
    if (t == 2u) raw = true;
  }
  const uint32_t* cw = reinterpret_cast<const uint32_t*>(img + kOffCode);
  const uint8_t* esc = img + kOffEsc;
#pragma unroll 1
  while (fix) {
    const int j = __ffs(fix) - 1;
    fix &= fix - 1;
    const uint32_t t = (tb >> (2 * j)) & 3u;
    const int o = off + esc_count(tb & ((1u << (2 * j)) - 1u));
    const int hh = j >> 1;
    uint32_t c[4];
    extract_codes(hh ? cw[256 + u] : cw[u], cw[512 + u], hh, c);
    const uint32_t ca = (j & 1) ? c[2] : c[0], cb = (j & 1) ? c[3] : c[1];
    const uint2 smw = *reinterpret_cast<const uint2*>(img + 32 * u + 8 * j);
    uint32_t ea, eb;
    if (t == 1u) {
      uint32_t ba, bb;
      if (kind == 0) {
        const int ch = 32 * (u & 3) + 8 * j;
        ba = *reinterpret_cast<const uint32_t*>(b4g + ch);
        bb = *reinterpret_cast<const uint32_t*>(b4g + ch + 4);
      } else {
        ba = bb = 0x01010101u * b4g[u >> 1];
      }
      const uint2 s = lut[esc[o]];
      ea = ba + ca + s.x;
      eb = bb + cb + s.y;
    } else {
      uint32_t h0 = 0, h1 = 0;
#pragma unroll
      for (int k = 0; k < 5; ++k) {
        const uint2 s = lut[esc[o + k]];  // bit plane 3+k: spread to bit 3, shifted up by k
        h0 |= s.x << k;
        h1 |= s.y << k;
      }
      ea = ca | h0;
      eb = cb | h1;
    }
    uint32_t w[4];
    join_v2(smw.x, ea, w[0], w[1]);
    join_v2(smw.y, eb, w[2], w[3]);
    *reinterpret_cast<uint4*>(dec + unit_chunk(kind, u, j)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Raw tile (BF16 in storage order) unit u into decoded order.
__device__ __forceinline__ void raw_unit(const uint8_t* img, int u, uint32_t o[16]) {
  const uint4* src = reinterpret_cast<const uint4*>(img + 64 * u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 w = src[i];
    o[4 * i + 0] = __byte_perm(w.x, w.y, 0x5410);  // elements {0, 2} of the quad
    o[4 * i + 1] = __byte_perm(w.x, w.y, 0x7632);  // elements {1, 3}
    o[4 * i + 2] = __byte_perm(w.z, w.w, 0x5410);
    o[4 * i + 3] = __byte_perm(w.z, w.w, 0x7632);
  }
}

// ------------------------------------------------------------------ decoders

// One decoder warp: eighth e8 (code units [32 e8, 32 e8 + 32)) of every
// block's K (kind 0) or V (kind 1) tile; lane l owns unit 32 e8 + l.  A K unit
// is one token's channel block l%4, a V unit one half of channel 16 e8 + l/2,
// so a lane's window bases never change.  Both kinds run this one code path.
__device__ __forceinline__ void decoder_warp(const AttnArgs& a, AttSmem& sm, int h, int blk0, int n_my, int len,
                                             int kind, int e8, int lane) {
  const uint8_t* b3g = a.base3 + (kind * a.Hkv + h) * kD;
  const uint8_t* b4g = a.base4 + (kind * a.Hkv + h) * kD;
  const int u = kDirUnits * e8 + lane;
  uint32_t b3[8], d43[8];
  if (kind == 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      b3[i] = *reinterpret_cast<const uint32_t*>(b3g + 32 * (u & 3) + 4 * i);
      d43[i] = *reinterpret_cast<const uint32_t*>(b4g + 32 * (u & 3) + 4 * i) - b3[i];
    }
  } else {
    const uint32_t x3 = 0x01010101u * b3g[u >> 1], x4 = 0x01010101u * b4g[u >> 1];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      b3[i] = x3;
      d43[i] = x4 - x3;
    }
  }
  const uint32_t c0 = unit_chunk(kind, u, 0), c1 = unit_chunk(kind, u, 1), c2 = unit_chunk(kind, u, 2),
                 c3 = unit_chunk(kind, u, 3);
  uint64_t* dec_full = kind ? sm.dvFull : sm.dkFull;
  uint64_t* dec_empty = kind ? sm.dvEmpty : sm.dkEmpty;
  int st = 0, db = 0;
  uint32_t sph = 0u, dph = 0u;  // parity of the current lap of the staging ring / decoded buffers
#pragma unroll 1
  for (int j = 0; j < n_my; ++j) {
    mbar_wait(&sm.stFull[st], sph, a.status);
    // the decoded buffer is needed only at the stores: poll it now, wait there if it was not free
    const bool dfree = j < kDecBufs || mbar_test_wait(&dec_empty[db], dph ^ 1u);
    const int mode = sm.smeta[st].mode[kind], esc_len = sm.smeta[st].esc[kind];
    const int nv = min(kBlock, len - (blk0 + j) * kBlock);
    const uint8_t* img = sm.stage[st][kind];
    uint8_t* dec = kind ? sm.decV[db] : sm.decK[db];
    const bool slot = mode == GAAC_MODE_SLOT;
    // Slot bookkeeping, read without waiting for the mode (the bytes are harmless for other modes):
    // the escape directory gives the eighth's first escape byte, a warp scan of the units' counts each
    // unit's (escape bytes are in unit order); the eighth's total must match the directory.
    const uint16_t* dir = reinterpret_cast<const uint16_t*>(img + kOffDir);
    const int start = e8 ? dir[e8 - 1] : 0, end = dir[e8];
    const uint32_t tb = img[kOffTag + u];
    const uint32_t te = sm.tagl[tb];
    const int cnt = (te >> 16) & 0xFF;
    const int incl = warp_incl_scan(cnt, lane);
    const int off = min(max(start + incl - cnt, 0), kEscCap);  // clamped: reads stay in the image
    const int total = __shfl_sync(kFull, incl, 31);
    uint32_t o[16];
    if (slot) {
      decode_unit(img, u, tb, __byte_perm(escape_window(img, off), 0u, te & 0xFFFFu), b3, d43, sm.lut, o);
    } else {
      raw_unit(img, u, o);
    }
    bool bad = !slot && mode != GAAC_MODE_RAW;
    if (slot) {
      bad = start > end || end > esc_len || start + total != end;
      if (bad && lane == 0) report(a.status, GAAC_EFORMAT);
    }
    if (bad) {  // no valid data: zeros (K blocks are also masked by the tensor-core warps)
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i] = 0u;
    }
    if (!dfree) mbar_wait(&dec_empty[db], dph ^ 1u, a.status);
    store_unit(dec, c0, c1, c2, c3, o);
    // Every escape offset used below lies inside [start, end) and end <= 496.
    if (slot && !bad && (te >> 24)) patch_unit(img, kind, u, tb, off, b4g, sm.lut, dec);  // raw groups: rare
    if (kind == 1 && nv < kBlock) clear_tail(dec, u, nv);
    if (kind == 0 && lane == 0) {
      sm.dec_bad[db][e8] = bad ? 1 : 0;
      if (e8 == 0) sm.dec_nv[db] = nv;
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&sm.stEmpty[st]);
      mbar_arrive(&dec_full[db]);
    }
    if (++st == kStages) {
      st = 0;
      sph ^= 1u;
    }
    if (++db == kDecBufs) {
      db = 0;
      dph ^= 1u;
    }
  }
}

// ------------------------------------------------------------------ producer

__device__ __forceinline__ void producer_lane(const AttnArgs& a, AttSmem& sm, int b, int h, int blk0, int n_my) {
  const gaac_entry* tab = a.table + ((static_cast<size_t>(b) * a.max_blocks + blk0) * a.Hkv + h) * 2;
  const size_t stride = static_cast<size_t>(a.Hkv) * 2;
  uint2 curK = make_uint2(0u, 0u), curV = make_uint2(0u, 0u);
  if (n_my > 0) {
    curK = *reinterpret_cast<const uint2*>(tab);
    curV = *reinterpret_cast<const uint2*>(tab + 1);
  }
#pragma unroll 1
  for (int j = 0; j < n_my; ++j) {
    uint2 nxtK = curK, nxtV = curV;
    if (j + 1 < n_my) {
      nxtK = *reinterpret_cast<const uint2*>(tab + (j + 1) * stride);
      nxtV = *reinterpret_cast<const uint2*>(tab + (j + 1) * stride + 1);
    }
    const int st = j % kStages;
    if (j >= kStages) mbar_wait(&sm.stEmpty[st], ((j / kStages) & 1) ^ 1, a.status);
    StageMeta m;
    uint32_t bytes[2];
    const void* src[2];
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      const uint2 cur = kv ? curV : curK;
      const uint32_t index = cur.x, esc_len = cur.y & 0xFFFFu, emode = (cur.y >> 16) & 0xFFu;
      bytes[kv] = 0;
      src[kv] = nullptr;
      m.mode[kv] = GAAC_MODE_NONE;
      m.esc[kv] = 0;
      if (emode == GAAC_MODE_SLOT && static_cast<int64_t>(index) < a.n_slots && esc_len <= kEscCap) {
        m.mode[kv] = GAAC_MODE_SLOT;
        m.esc[kv] = static_cast<int>(esc_len);
        bytes[kv] = (kOffEsc + esc_len + 15u) & ~15u;
        src[kv] = a.slot_pool + static_cast<size_t>(index) * kSlot;
      } else if (emode == GAAC_MODE_RAW && static_cast<int64_t>(index) < a.n_raw) {
        m.mode[kv] = GAAC_MODE_RAW;
        bytes[kv] = kRawBytes;
        src[kv] = a.raw_pool + static_cast<size_t>(index) * kTile;
      } else {
        report(a.status, GAAC_EFORMAT);
      }
    }
    sm.smeta[st] = m;
    mbar_arrive_expect_tx(&sm.stFull[st], bytes[0] + bytes[1]);
    if (bytes[0]) bulk_g2s(sm.stage[st][0], src[0], bytes[0], &sm.stFull[st]);
    if (bytes[1]) bulk_g2s(sm.stage[st][1], src[1], bytes[1], &sm.stFull[st]);
    curK = nxtK;
    curV = nxtV;
  }
  // Every issued copy was consumed by the decoders; after a timed-out wait,
  // wait once more (bounded) so that no copy is still landing at exit.
#pragma unroll 1
  for (int i = max(0, n_my - kStages); i < n_my; ++i)
    mbar_wait(&sm.stFull[i % kStages], (i / kStages) & 1, a.status, 1u << 10);
}

// ------------------------------------------------------------- tensor cores

// A tensor-core group of four warps shares each of its blocks (group gr takes
// blocks gr, gr+2, ...): warp w scores tokens [16w, 16w+16) (QK^T) and
// accumulates channels [32w, 32w+32) (PV^T).  The block maximum per head goes
// through shared memory, so the group's warps keep the same running maximum;
// the two groups' partials are merged when the split ends.
__device__ __forceinline__ void tensor_warp(const AttnArgs& a, AttSmem& sm, int n_my, float* part, int gr, int w,
                                            int lane) {
  const int g = lane >> 2, tq = lane & 3;
  // ldmatrix row of this lane inside a 16-row tile: matrix m = lane/8 covers rows 8(m%2).., columns 8(m/2)..
  const int lrow = ((lane >> 3) & 1) * 8 + (lane & 7);
  const int lcol = lane >> 4;
  const int tg = quad_perm(g);
  float acc[2][4];  // channel tiles 2w, 2w+1
#pragma unroll
  for (int ct = 0; ct < 2; ++ct) acc[ct][0] = acc[ct][1] = acc[ct][2] = acc[ct][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2tq, 2tq+1 (log2 domain)
  // q as the B operand of QK^T: two k-steps per ldmatrix (chunk lane/8 of the head row lane%8)
  uint32_t qf[16];
  {
    const uint32_t qsa = smem_addr(&sm.qs[lane & 7][0]) + 16u * (lane >> 3);
#pragma unroll
    for (int k2 = 0; k2 < 4; ++k2) ldsm_x4(qsa + 64u * k2, qf[4 * k2], qf[4 * k2 + 1], qf[4 * k2 + 2], qf[4 * k2 + 3]);
  }
  const uint32_t pth = smem_addr(&sm.pt[gr][0][0][0]);
  // P^T store: matrices (hi rows 0-7, hi rows 8-15, lo rows 0-7, lo rows 8-15) of this warp's 16 positions
  const uint32_t pst = pth + static_cast<uint32_t>((lane >> 4) * kRPad * kPtStride * 2 + (lane & 7) * kPtStride * 2 +
                                                   (2 * w + ((lane >> 3) & 1)) * 16);
  // P^T as B of one k-step: matrices (hi k0-7, hi k8-15, lo k0-7, lo k8-15)
  const uint32_t pba = pth + static_cast<uint32_t>((lane >> 4) * kRPad * kPtStride * 2 + (lane & 7) * kPtStride * 2 +
                                                   16 * ((lane >> 3) & 1));
  uint32_t koff[8], voff[8];  // swizzled ldmatrix offsets: K row 16w + quad_perm(lrow) per k-step; V rows per (k-step, tile)
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) koff[ks] = kswz(16 * w + quad_perm(lrow), 2 * ks + lcol);  // rows follow V's token order
#pragma unroll
  for (int kt = 0; kt < 4; ++kt)
#pragma unroll
    for (int ct = 0; ct < 2; ++ct) voff[2 * kt + ct] = vswz(32 * w + 16 * ct + lrow, 2 * kt + lcol);

#pragma unroll 1
  for (int j = gr; j < n_my; j += kMGroups) {
    const int db = j % kDecBufs;
    const uint32_t par = (j / kDecBufs) & 1;
    mbar_wait(&sm.dkFull[db], par, a.status);
    const int nv = sm.dec_nv[db];
    const uint2 badw = *reinterpret_cast<const uint2*>(sm.dec_bad[db]);  // one byte per K eighth
    const bool kbad = (badw.x | badw.y) != 0u;
    // ---- S = K q^T for tokens 16w..16w+15: 8 k-steps in two accumulation chains
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t kb = smem_addr(sm.decK[db]);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(kb + koff[ks], a0, a1, a2, a3);
      mma_bf16(ks & 1 ? sb : sa, a0, a1, a2, a3, qf[2 * ks], qf[2 * ks + 1]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.dkEmpty[db]);
    const bool ok0 = !kbad && 16 * w + tg < nv, ok1 = !kbad && 16 * w + 8 + tg < nv;
    float s0 = ok0 ? (sa[0] + sb[0]) * a.scale_log2 : -INFINITY;
    float s1 = ok0 ? (sa[1] + sb[1]) * a.scale_log2 : -INFINITY;
    float s2 = ok1 ? (sa[2] + sb[2]) * a.scale_log2 : -INFINITY;
    float s3 = ok1 ? (sa[3] + sb[3]) * a.scale_log2 : -INFINITY;
    float x0 = fmaxf(s0, s2), x1 = fmaxf(s1, s3);
#pragma unroll
    for (int d = 4; d < 32; d <<= 1) {
      x0 = fmaxf(x0, __shfl_xor_sync(kFull, x0, d));
      x1 = fmaxf(x1, __shfl_xor_sync(kFull, x1, d));
    }
    if (g == 0) {
      sm.wmax[gr][2 * tq][w] = x0;
      sm.wmax[gr][2 * tq + 1][w] = x1;
    }
    named_bar_sync(kBarM + gr, kMGroupWarps * 32);  // block maxima of the group's warps written
    const float4 ma = *reinterpret_cast<const float4*>(&sm.wmax[gr][2 * tq][0]);
    const float4 mb = *reinterpret_cast<const float4*>(&sm.wmax[gr][2 * tq + 1][0]);
    const float n0 = fmaxf(m0, fmaxf(fmaxf(ma.x, ma.y), fmaxf(ma.z, ma.w)));
    const float n1 = fmaxf(m1, fmaxf(fmaxf(mb.x, mb.y), fmaxf(mb.z, mb.w)));
    if (n0 != m0 || n1 != m1) {  // a running maximum rises: rescale (rare after the first blocks)
      const float al0 = n0 == -INFINITY ? 1.f : fast_exp2(m0 - n0);
      const float al1 = n1 == -INFINITY ? 1.f : fast_exp2(m1 - n1);
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int ct = 0; ct < 2; ++ct) {
        acc[ct][0] *= al0;
        acc[ct][1] *= al1;
        acc[ct][2] *= al0;
        acc[ct][3] *= al1;
      }
      m0 = n0;
      m1 = n1;
    }
    const float p0 = m0 == -INFINITY ? 0.f : fast_exp2(s0 - m0);
    const float p1 = m1 == -INFINITY ? 0.f : fast_exp2(s1 - m1);
    const float p2 = m0 == -INFINITY ? 0.f : fast_exp2(s2 - m0);
    const float p3 = m1 == -INFINITY ? 0.f : fast_exp2(s3 - m1);
    l0 += p0 + p2;
    l1 += p1 + p3;
    const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
    const uint32_t r01 = pack_bf16x2(p0 - __uint_as_float(h01 << 16), p1 - __uint_as_float(h01 & 0xFFFF0000u));
    const uint32_t r23 = pack_bf16x2(p2 - __uint_as_float(h23 << 16), p3 - __uint_as_float(h23 & 0xFFFF0000u));
    stsm_x4_trans(pst, h01, h23, r01, r23);  // P^T[head][16w + row]
    named_bar_sync(kBarM + gr, kMGroupWarps * 32);  // P^T of the block complete
    // ---- acc += V^T P for channels 32w..32w+31: 4 k-steps of 16 tokens
    mbar_wait(&sm.dvFull[db], par, a.status);
    const uint32_t vb = smem_addr(sm.decV[db]);
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      uint32_t bh0, bh1, bl0, bl1;
      ldsm_x4(pba + 32u * kt, bh0, bh1, bl0, bl1);
#pragma unroll
      for (int ct = 0; ct < 2; ++ct) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(vb + voff[2 * kt + ct], a0, a1, a2, a3);
        mma_bf16(acc[ct], a0, a1, a2, a3, bh0, bh1);
        mma_bf16(acc[ct], a0, a1, a2, a3, bl0, bl1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.dvEmpty[db]);
  }
  // ---- the split's partial: l summed over lanes and warps; group 1 hands (m, l, acc) to group 0, which
  // merges the two with a log-sum-exp and writes the partial
#pragma unroll
  for (int d = 4; d < 32; d <<= 1) {
    l0 += __shfl_xor_sync(kFull, l0, d);
    l1 += __shfl_xor_sync(kFull, l1, d);
  }
  if (g == 0) {
    sm.wl[gr][2 * tq][w] = l0;
    sm.wl[gr][2 * tq + 1][w] = l1;
  }
  if (gr == kMGroups - 1 && gr > 0) {
    if (w == 0 && g == 0) {
      sm.xm[2 * tq] = m0;
      sm.xm[2 * tq + 1] = m1;
    }
#pragma unroll
    for (int ct = 0; ct < 2; ++ct) {
      const int cA = 32 * w + 16 * ct + g, cB = cA + 8;
      sm.xacc[2 * tq][cA] = acc[ct][0];
      sm.xacc[2 * tq + 1][cA] = acc[ct][1];
      sm.xacc[2 * tq][cB] = acc[ct][2];
      sm.xacc[2 * tq + 1][cB] = acc[ct][3];
    }
  }
  named_bar_sync(kBarMAll, kMWarps * 32);
  if (gr != 0) return;
  float wt[2][2];  // [head 2tq + i][own group, group 1]
  float mm[2], ll[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float4 la = *reinterpret_cast<const float4*>(&sm.wl[0][2 * tq + i][0]);
    const float lown = (la.x + la.y) + (la.z + la.w);
    const float mo = i ? m1 : m0;
    if (kMGroups > 1) {
      const float mx = sm.xm[2 * tq + i];
      const float M = fmaxf(mo, mx);
      mm[i] = M;
      wt[i][0] = mo == -INFINITY ? 0.f : fast_exp2(mo - M);
      wt[i][1] = mx == -INFINITY ? 0.f : fast_exp2(mx - M);
      const float4 lb = *reinterpret_cast<const float4*>(&sm.wl[kMGroups - 1][2 * tq + i][0]);
      ll[i] = wt[i][0] * lown + wt[i][1] * ((lb.x + lb.y) + (lb.z + lb.w));
    } else {
      mm[i] = mo;
      wt[i][0] = 1.f;
      wt[i][1] = 0.f;
      ll[i] = lown;
    }
  }
  if (w == 0 && g == 0) {
    part[4 * tq + 0] = mm[0];
    part[4 * tq + 1] = ll[0];
    part[4 * tq + 2] = mm[1];
    part[4 * tq + 3] = ll[1];
  }
  float* pa = part + 2 * kRPad;
#pragma unroll
  for (int ct = 0; ct < 2; ++ct) {
    const int cA = 32 * w + 16 * ct + g, cB = cA + 8;
    if (kMGroups > 1) {
      pa[(2 * tq) * kD + cA] = wt[0][0] * acc[ct][0] + wt[0][1] * sm.xacc[2 * tq][cA];
      pa[(2 * tq + 1) * kD + cA] = wt[1][0] * acc[ct][1] + wt[1][1] * sm.xacc[2 * tq + 1][cA];
      pa[(2 * tq) * kD + cB] = wt[0][0] * acc[ct][2] + wt[0][1] * sm.xacc[2 * tq][cB];
      pa[(2 * tq + 1) * kD + cB] = wt[1][0] * acc[ct][3] + wt[1][1] * sm.xacc[2 * tq + 1][cB];
    } else {
      pa[(2 * tq) * kD + cA] = acc[ct][0];
      pa[(2 * tq + 1) * kD + cA] = acc[ct][1];
      pa[(2 * tq) * kD + cB] = acc[ct][2];
      pa[(2 * tq + 1) * kD + cB] = acc[ct][3];
    }
  }
}

// Log-sum-exp merge of the n_splits partials (m, l, acc) of one (sequence,
// kv-head) into out[b, h*r + n, :] = sum_s w_s acc_s / sum_s w_s l_s with
// w_s = 2^(m_s - max_s m_s) per head n (the final split reduction).  Runs on
// the CTA that finished last, so it is a tail on the critical path: each
// thread owns one float4 column of the output and a subset of the splits,
// issues that subset's loads ten at a time and folds them in with its own
// running maximum; the subsets are then combined the same way in shared
// memory.  The staging ring is free by then and holds that exchange.
// base: the first partial of the pair; out: its first output row.
__device__ __noinline__ void merge_splits(const float* base, int ns, int r, float* out, AttSmem& sm, int tid) {
  constexpr int kBatch = 10;
  const int o4n = r * (kD / 4);  // float4 columns of the r x 128 output
  const int groups = kAttThreads / o4n;
  const int o4 = tid % o4n, grp = tid / o4n;
  const int n = o4 / (kD / 4), c4 = o4 % (kD / 4);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f, mt = -INFINITY;
  if (grp < groups) {
    const float* pcol = base + 2 * kRPad + n * kD + 4 * c4;
    for (int sp0 = grp; sp0 < ns; sp0 += kBatch * groups) {
      float2 ml[kBatch];
      float4 v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int sp = sp0 + u * groups;
        if (sp < ns) {
          ml[u] = __ldcg(reinterpret_cast<const float2*>(base + static_cast<size_t>(sp) * kPartFloats + 2 * n));
          v[u] = __ldcg(reinterpret_cast<const float4*>(pcol + static_cast<size_t>(sp) * kPartFloats));
        } else {
          ml[u] = make_float2(-INFINITY, 0.f);
          v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float mb = mt;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) mb = fmaxf(mb, ml[u].x);
      if (mb != -INFINITY) {
        const float al = mt == -INFINITY ? 0.f : fast_exp2(mt - mb);
        acc.x *= al;
        acc.y *= al;
        acc.z *= al;
        acc.w *= al;
        den *= al;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const float w = ml[u].x == -INFINITY ? 0.f : fast_exp2(ml[u].x - mb);
          acc.x += w * v[u].x;
          acc.y += w * v[u].y;
          acc.z += w * v[u].z;
          acc.w += w * v[u].w;
          den += w * ml[u].y;
        }
        mt = mb;
      }
    }
  }
  float4* xa = reinterpret_cast<float4*>(sm.stage[0][0]);  // [groups][o4n] accumulators
  float2* xm = reinterpret_cast<float2*>(sm.stage[1][0]);  // [groups][o4n] (running max, denominator)
  if (grp < groups && groups > 1) {
    xa[grp * o4n + o4] = acc;
    xm[grp * o4n + o4] = make_float2(mt, den);
  }
  __syncthreads();
  if (tid < o4n) {
    float mx = mt;
    for (int gi = 1; gi < groups; ++gi) mx = fmaxf(mx, xm[gi * o4n + o4].x);
    if (mx != -INFINITY) {
      const float al = mt == -INFINITY ? 0.f : fast_exp2(mt - mx);
      acc.x *= al;
      acc.y *= al;
      acc.z *= al;
      acc.w *= al;
      den *= al;
      for (int gi = 1; gi < groups; ++gi) {
        const float2 md = xm[gi * o4n + o4];
        if (md.x == -INFINITY) continue;
        const float w = fast_exp2(md.x - mx);
        const float4 x = xa[gi * o4n + o4];
        acc.x += w * x.x;
        acc.y += w * x.y;
        acc.z += w * x.z;
        acc.w += w * x.w;
        den += w * md.y;
      }
    }
    float* o = out + n * kD + 4 * c4;
    const float inv = den > 0.f ? 1.f / den : 0.f;
    o[0] = acc.x * inv;
    o[1] = acc.y * inv;
    o[2] = acc.z * inv;
    o[3] = acc.w * inv;
  }
}


__global__ void __launch_bounds__(kAttThreads, kCtasPerSm) attn_split_kernel(AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  AttSmem& sm = *reinterpret_cast<AttSmem*>(smem_raw);
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int len = a.seq_lens[b];
  if (len < 0 || len > a.max_blocks * kBlock) {
    if (tid == 0) report(a.status, GAAC_EINVAL);
    len = 0;
  }
  // This split's blocks of the sequence: an even share of its blocks.
  const int nblk = (len + kBlock - 1) / kBlock;
  const int per = (nblk + a.n_splits - 1) / a.n_splits;
  const int blk0 = split * per;
  const int n_my = max(0, min(nblk, blk0 + per) - blk0);

  for (int x = tid; x < 256; x += kAttThreads) {
    sm.lut[x] = spread_entry(static_cast<uint32_t>(x));
    sm.tagl[x] = tag_entry(static_cast<uint32_t>(x));
  }
  // q of the kv-head's query heads, times 2^-4, channels in decoded order (the B operand of QK^T)
  for (int x = tid; x < kRPad * kD / 2; x += kAttThreads) {
    const int n = x / (kD / 2), p = 2 * (x % (kD / 2));  // positions p, p+1 hold channels quad_perm(p), quad_perm(p+1)
    uint32_t w = 0u;
    if (n < a.r) {
      const uint16_t* qrow = a.q + (static_cast<size_t>(b) * a.Hq + h * a.r + n) * kD;
      w = bf16x2_div16(static_cast<uint32_t>(qrow[quad_perm(p)]) | (static_cast<uint32_t>(qrow[quad_perm(p + 1)]) << 16));
    }
    *reinterpret_cast<uint32_t*>(&sm.qs[n][p]) = w;
  }
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.stFull[s], 1);
      mbar_init(&sm.stEmpty[s], kDWarps);
    }
#pragma unroll
    for (int d = 0; d < kDecBufs; ++d) {
      mbar_init(&sm.dkFull[d], kDWarps / 2);
      mbar_init(&sm.dvFull[d], kDWarps / 2);
      mbar_init(&sm.dkEmpty[d], kMGroupWarps);
      mbar_init(&sm.dvEmpty[d], kMGroupWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int r = a.r;
  float* part = a.part + ((static_cast<size_t>(b) * a.Hkv + h) * a.n_splits + split) * kPartFloats;
  if (warp < kDWarps) {
    decoder_warp(a, sm, h, blk0, n_my, len, warp / (kDWarps / 2), warp % (kDWarps / 2), lane);
  } else if (warp < kProducerWarp) {
    tensor_warp(a, sm, n_my, part, (warp - kMWarp0) / kMGroupWarps, (warp - kMWarp0) % kMGroupWarps, lane);
  } else if (lane == 0) {
    producer_lane(a, sm, b, h, blk0, n_my);
  }

  // ---------------------------------------------------------------- split merge (final reduction)
  // The last CTA of a (sequence, kv-head) to finish merges the partials of all
  // its splits with a log-sum-exp; the counter goes back to zero for the next
  // launch.  No CTA ever waits for another.
  // Release/acquire through the counter: the barrier orders every thread's
  // partial stores before thread 0's acq_rel add, and the add orders the other
  // splits' stores before this CTA's loads (the barrier passes that on).
  __syncthreads();
  unsigned int* counter = a.counters + static_cast<size_t>(b) * a.Hkv + h;
  if (tid == 0) sm.last = atomic_add_acq_rel(counter, 1u) == static_cast<unsigned int>(a.n_splits - 1);
  __syncthreads();
  if (!sm.last) return;
  merge_splits(a.part + (static_cast<size_t>(b) * a.Hkv + h) * a.n_splits * kPartFloats, a.n_splits, r,
               a.out + (static_cast<size_t>(b) * a.Hq + h * r) * kD, sm, tid);
  if (tid == 0) *counter = 0u;
}

static int device_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

static bool prepare_kernel() {
  static bool done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (!done[dev]) {
    if (cudaFuncSetAttribute(attn_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(AttSmem))) != cudaSuccess)
      return false;
    done[dev] = true;
  }
  return true;
}

}  // namespace gaac

using namespace gaac;

extern "C" int gaac_attention_auto_splits(int batch, int n_kv_heads, int max_blocks) {
  if (batch <= 0 || n_kv_heads <= 0 || max_blocks <= 0) return 1;
  const long long target = static_cast<long long>(kCtasPerSm) * device_sms();  // one wave of resident CTAs
  const long long pairs = static_cast<long long>(batch) * n_kv_heads;
  long long s = (target + pairs - 1) / pairs;
  if (s > max_blocks) s = max_blocks;
  return static_cast<int>(s < 1 ? 1 : s);
}

static size_t partials_bytes(int batch, int n_kv_heads, int n_splits) {
  return static_cast<size_t>(batch) * n_kv_heads * n_splits * kPartFloats * sizeof(float);
}

extern "C" size_t gaac_attention_workspace(int batch, int n_kv_heads, int max_blocks, int n_splits) {
  if (n_splits <= 0) n_splits = gaac_attention_auto_splits(batch, n_kv_heads, max_blocks);
  if (batch <= 0 || n_kv_heads <= 0) return 0;
  const size_t counters = (static_cast<size_t>(batch) * n_kv_heads * sizeof(unsigned int) + 15) & ~static_cast<size_t>(15);
  return partials_bytes(batch, n_kv_heads, n_splits) + counters;
}

extern "C" int gaac_decode_attention(const uint16_t* q, int batch, int n_q_heads, int n_kv_heads, int max_blocks,
                                     const int32_t* seq_lens, const gaac_entry* table, const gaac_pools* pools,
                                     const uint8_t* base3, const uint8_t* base4, float scale, int n_splits,
                                     float* out, void* workspace, size_t workspace_bytes, int32_t* d_status,
                                     void* stream) {
  if (q == nullptr || seq_lens == nullptr || table == nullptr || pools == nullptr || pools->slot_pool == nullptr ||
      pools->raw_pool == nullptr || pools->n_slots < 0 || pools->n_raw < 0 || base3 == nullptr ||
      base4 == nullptr || out == nullptr || workspace == nullptr)
    return GAAC_EINVAL;
  if (batch <= 0 || batch > 65535 || n_kv_heads <= 0 || n_kv_heads > 65535 || n_q_heads <= 0 ||
      n_q_heads % n_kv_heads != 0 || n_q_heads / n_kv_heads > GAAC_MAX_GQA || max_blocks <= 0 ||
      max_blocks > (1 << 24) || !std::isfinite(scale))
    return GAAC_EINVAL;
  if ((reinterpret_cast<uintptr_t>(q) & 15u) || (reinterpret_cast<uintptr_t>(pools->slot_pool) & 15u) ||
      (reinterpret_cast<uintptr_t>(pools->raw_pool) & 15u) || (reinterpret_cast<uintptr_t>(base3) & 15u) ||
      (reinterpret_cast<uintptr_t>(base4) & 15u) || (reinterpret_cast<uintptr_t>(workspace) & 15u) ||
      (reinterpret_cast<uintptr_t>(out) & 3u))
    return GAAC_EINVAL;
  if (n_splits <= 0) n_splits = gaac_attention_auto_splits(batch, n_kv_heads, max_blocks);
  if (n_splits > max_blocks) n_splits = max_blocks;
  if (workspace_bytes < gaac_attention_workspace(batch, n_kv_heads, max_blocks, n_splits)) return GAAC_EINVAL;
  if (!prepare_kernel()) return GAAC_ECUDA;
  AttnArgs a;
  a.q = q;
  a.seq_lens = seq_lens;
  a.table = table;
  a.slot_pool = pools->slot_pool;
  a.n_slots = pools->n_slots;
  a.raw_pool = pools->raw_pool;
  a.n_raw = pools->n_raw;
  a.base3 = base3;
  a.base4 = base4;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 16.0 * 1.4426950408889634);
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.r = n_q_heads / n_kv_heads;
  a.max_blocks = max_blocks;
  a.n_splits = n_splits;
  a.part = static_cast<float*>(workspace);
  a.counters = reinterpret_cast<unsigned int*>(static_cast<char*>(workspace) + partials_bytes(batch, n_kv_heads, n_splits));
  a.out = out;
  a.status = d_status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  attn_split_kernel<<<dim3(n_splits, n_kv_heads, batch), kAttThreads, sizeof(AttSmem), st>>>(a);
  return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}

// ------------------------------------------------------------------------
// Allocation-free variant.  Some callers cannot hand the library a workspace
// allocated at call time: a serving loop that has frozen its device memory
// plan, a plugin whose host owns every allocation, or code that must not call
// into an allocator on the decode path.  This entry point runs the same kernel with
// its split partials in a fixed scratch array that lives in the
// library itself.
constexpr size_t kStaticScratchBytes = GAAC_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_attn_scratch[kStaticScratchBytes];

// Device address of g_attn_scratch on the current device, looked up once per
// device (the host-side name is only a stand-in and must not reach a kernel).
static void* static_scratch_address() {
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || p == nullptr) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

extern "C" int gaac_decode_attention_noalloc(const uint16_t* q, int batch, int n_q_heads, int n_kv_heads,
                                             int max_blocks, const int32_t* seq_lens, const gaac_entry* table,
                                             const gaac_pools* pools, const uint8_t* base3, const uint8_t* base4,
                                             float scale, int n_splits, float* out, int32_t* d_status,
                                             void* stream) {
  if (batch <= 0 || n_kv_heads <= 0 || max_blocks <= 0) return GAAC_EINVAL;
  int ns = n_splits <= 0 ? gaac_attention_auto_splits(batch, n_kv_heads, max_blocks) : n_splits;
  if (ns > max_blocks) ns = max_blocks;
  if (gaac_attention_workspace(batch, n_kv_heads, max_blocks, ns) > kStaticScratchBytes) return GAAC_EINVAL;
  void* scratch = static_scratch_address();
  if (scratch == nullptr) return GAAC_ECUDA;
  // The merge counters must start at zero; clear them on every call so that a
  // call never depends on how an earlier one ended.
  const size_t cbytes = static_cast<size_t>(batch) * n_kv_heads * sizeof(unsigned int);
  if (cudaMemsetAsync(static_cast<char*>(scratch) + partials_bytes(batch, n_kv_heads, ns), 0, cbytes,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GAAC_ECUDA;
  return gaac_decode_attention(q, batch, n_q_heads, n_kv_heads, max_blocks, seq_lens, table, pools, base3, base4,
                               scale, ns, out, scratch, kStaticScratchBytes, d_status, stream);
}
