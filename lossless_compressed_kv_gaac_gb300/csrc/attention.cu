// Fused split-K GQA decode attention over the GAAC compressed cache.
//
// "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference on
// Personal Devices", section 3.2: attention reads the compressed tiles and
// rebuilds the values it needs on the fly (no decompressed copy of the cache
// in global memory); compressed blocks and the raw tail go through one
// softmax.  Section 3.3: the block table says per block whether it is a slot
// or a raw tile.
//
// GB300 design: one CTA of 384 threads per SM, grid (split, kv-head, sequence).
//  * The CTA streams its split's 64-token blocks through a ring of shared-
//    memory stages: each block's K and V tile images (only the bytes a slot
//    uses) arrive by 1-D bulk copies tracked by an mbarrier per stage.  There
//    is no copy warp: the last warp to finish reading a stage issues its
//    refill with the next block for it.
//  * Twelve warps form three groups of four; group gr takes blocks gr, gr+3, ...
//    of the split, and warp w of a group takes tokens [16w, 16w+16) of each.
//    Each warp keeps its own online-softmax state (m, l, acc) over its tokens;
//    the twelve states are merged with a log-sum-exp when the split ends.
//  * 256-channel heads (two 128-channel half-heads): the two CTAs of a head
//    form a cluster; each decodes its own half-head's K and V tiles, and the
//    warps exchange partial scores with st.async stores into the peer's shared
//    memory (completed on the peer's mbarrier) before the softmax.
//  * Per block a lane rebuilds two K units and two V units (32 elements each)
//    straight into tensor-core operand registers, with no shared-memory copy
//    of the decoded tile:
//      - K units 64w + lane and 64w + 32 + lane are tokens 16w + g and
//        16w + 8 + g (g = lane/4), channel block lane%4: exactly the B operand
//        of S^T = q K^T over eight tokens (mma.sync m16n8k16, q as A with the
//        8 query heads in rows 0-7 and channels in the order the decoder
//        emits them);
//      - the S^T accumulators of the two token octets are, lane for lane, the
//        B operand (P^T) of O^T += V^T P^T, so softmax needs no data movement;
//      - V tiles are stored in operand order (format v3), so V units 64w +
//        lane and 64w + 32 + lane are the A operands of four 16-channel tiles
//        each for this warp's 16 tokens.
//  * Decode of a unit: the escape directory gives the eighth's first 4-bit
//    escape byte and raw group; one warp scan of four packed counts gives each
//    unit's; one byte permute gathers a unit's 4-bit escape bytes.  Exponents
//    are rebuilt four at a time in 32-bit words and joined with the
//    sign|mantissa word by two bit selects and a byte rotation per four
//    values.  Raw groups (their eight exponents in the escape area) are
//    re-joined by the lanes that own them.
//  * Softmax in the log2 domain; rescales only when a running maximum rises;
//    P goes to the tensor cores as a bf16 hi + lo pair (rounding near 2^-17).
//  * q is pre-scaled by +-2^-4 (exact for normal values; the sign is that of
//    the softmax scale) so that q.k stays inside the fp32 range for extreme
//    keys.  Running maxima are kept on these raw scores and only a score's
//    difference from its maximum is multiplied by |scale| * 16 * log2(e), so
//    no unshifted scaled logit is ever formed: a score whose logit is within
//    the fp32 range never overflows, and a difference that does is a weight
//    of exactly zero.
//  * Partials (m, l, acc) per split go to the workspace; the last CTA of each
//    (sequence, kv-head) to finish, found with a device counter, merges them
//    with a log-sum-exp (the final split reduction) and resets the counter.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "common.cuh"

namespace gaac {

constexpr int kGroupWarps = 4;                    // token quarters of a block
constexpr int kGroups = 3;                        // warp groups, alternate blocks
constexpr int kCWarps = kGroupWarps * kGroups;    // compute warps
constexpr int kAttThreads = kCWarps * 32;
// Staging ring depth: 6 stages of K+V images for 128-channel heads, 4 of K0+K1+V for 256-channel heads
// (two half-heads).  Block j of a split uses stage j % depth.
template <int KH>
constexpr int stages_of() { return KH == 1 ? 6 : 4; }

constexpr int kCtasPerSm = 1;
constexpr int kRPad = 8;                          // query heads per kv-head in the MMA rows
constexpr int kPartFloats = 2 * kRPad + kRPad * kD;
constexpr uint32_t kJoinMask = 0x807F807Fu;       // sign and mantissa bits of a bf16x2 word
constexpr uint32_t kFull = 0xFFFFFFFFu;

struct StageMeta {
  int mode[3], esc[3];  // [K half 0, (K half 1,) V]
};

// NH: 128-channel half-heads per attention head (1, or 2 for 256-channel heads).
// KH: K half-head images a CTA decodes per block: NH, or 1 when the two CTAs
// of a 256-channel head form a cluster and exchange their partial scores.
template <int NH, int KH>
struct AttSmem {
  static constexpr int kStages = stages_of<KH>();
  // Block j uses stage j % kStages and is read by group j % kGroups.  The depth must be a multiple of the
  // group count, so that one group reads every block of a stage, in order: a group then never waits on a
  // stage whose previous phase has not completed (a parity wait would take that phase for done).
  static_assert(kStages % kGroups == 0, "each stage must belong to one warp group");
  static constexpr int kPairs = NH > KH ? kCWarps : 1;  // score mailboxes (cluster pairs only)
  alignas(128) uint8_t stage[kStages][KH + 1][kRawBytes];  // K half-head images, then the V image
  uint2 lut[256];                 // escape byte -> bit 3 spread into the byte lanes of two exponent words
  uint32_t tagl[256];             // tag byte -> gather selector, counts, raw groups (tag_entry)
  alignas(16) uint8_t kbases[KH][2][kD];  // K: [image][base3|base4][channel]
  StageMeta smeta[kStages];
  alignas(16) uint2 qf[KH][8][32];       // q^T B-operand pairs [image][k-step][lane] of S = K q^T
  alignas(16) uint4 vbw[2][2][32];        // V base words [unit][base3 | base4][lane], groups 0-3
  unsigned int stDone[kStages];           // warps of the group done reading the stage's current block
  float wm[kCWarps][kRPad];       // per warp and head: running maximum (end of split)
  float wl[kCWarps][kRPad];       // per warp and head: denominator (end of split)
  float ww[kCWarps][kRPad];       // per warp and head: merge weight (end of split)
  uint64_t stFull[kStages];
  alignas(16) float4 mail[kPairs][2][32];  // [warp][buffer][lane]: the peer CTA's partial scores of a block
  uint64_t mFull[kPairs][2];               // the peer's 512 bytes landed in mail[warp][buffer]
  uint64_t mEmpty[kPairs][2];              // the peer's warp has read this warp's partials from its mailbox
  alignas(16) float4 ack[kPairs][2];       // landing slots of the peer's acknowledgements (16 bytes each)
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
  float qmul;       // q multiplier: 2^-4 times the sign of the softmax scale (0 for a zero scale)
  float c_log2;     // |scale| * 16 * log2(e): raw-score differences to log2 weights (1 for a zero scale)
  int Hq, Hkv, r, max_blocks, n_splits;  // Hkv: attention kv-heads (of NH half-heads each)
  float* part;
  unsigned int* counters;  // [batch][NH * Hkv] splits finished; zero between launches
  float* out;
  int32_t* status;
};

// ------------------------------------------------------------- timeline
// Opt-in per-CTA timeline (built only with -DGAAC_TIMELINE; the default
// library has none of it): %globaltimer stamps of each CTA's start (after the
// dependent-launch wait), of every block's copy issue, landing (the first warp
// of its group through the stage wait, after it began waiting at arrive) and
// release (the group's last warp done
// with the stage), of the end of the split's blocks and of the CTA's exit
// (after the merge, for the CTA that merges).  Read with gaac_timeline_fetch.
#ifdef GAAC_TIMELINE
constexpr int kTlCtas = 1024, kTlBlocks = 256;
struct TlCta {
  unsigned long long start, split_end, exit, merged;
  unsigned long long issue[kTlBlocks], arrive[kTlBlocks], land[kTlBlocks], release[kTlBlocks];
};
__device__ TlCta g_timeline[kTlCtas];
__device__ __forceinline__ unsigned long long tl_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ TlCta* tl_cta() {
  const unsigned id = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  return id < kTlCtas ? &g_timeline[id] : nullptr;
}
#define GAAC_TL(...) \
  do {               \
    __VA_ARGS__;     \
  } while (0)
#else
#define GAAC_TL(...) \
  do {               \
  } while (0)
#endif

// ------------------------------------------------------------------ helpers

// bf16x2 times f (+-2^-4 or 0); exact whenever the result is a normal number or zero.
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t w, float f) {
  const float lo = __uint_as_float(w << 16) * f;
  const float hi = __uint_as_float(w & 0xFFFF0000u) * f;
  return (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Transpose of an 8 x 8 matrix of 16-bit values held one row pair per lane (lane (g, tq): row g, columns
// 2tq, 2tq+1): the result holds row g, columns 2tq, 2tq+1 of the transpose.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t x, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t v = __shfl_up_sync(kFull, x, d);
    if (lane >= d) x += v;
  }
  return x;
}

__device__ __forceinline__ unsigned int atomic_add_acq_rel(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Four BF16 values from one sign|mantissa word of format v3 (byte L: mantissa
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
//  bits 0-15: byte permute selector that gathers the unit's 4-bit escape
//    bytes from the four escape bytes at the unit's offset (byte j = group j's
//    escape byte if group j is 4-bit, else a zero byte);
//  byte 2: the 4-bit groups, plus 32 per reserved tag, so that a reserved tag
//    breaks its eighth's check against the escape directory;
//  byte 3: the raw groups.
// Bytes 2 and 3 of two units' entries are the packed counts of the warp scan.
__device__ __forceinline__ uint32_t tag_entry(uint32_t tb) {
  uint32_t sel = 0, n4 = 0, nr = 0, rsv = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t t = (tb >> (2 * j)) & 3u;
    sel |= (t == 1u ? n4 : 4u) << (4 * j);  // 4: a zero byte of the second operand
    if (t == 1u) ++n4;
    if (t == 2u) ++nr;
    if (t == 3u) ++rsv;
  }
  return sel | ((n4 + 32u * rsv) << 16) | (nr << 24);
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds8(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

// The four escape bytes starting at escape offset `off` (clamped into the escape area).
__device__ __forceinline__ uint32_t escape_window(const uint8_t* img, int off) {
  off = min(off, kEscCap);
  const uint32_t a = smem_addr(img) + kOffEsc + 4 * (off >> 2);
  const uint32_t w0 = lds32(a), w1 = lds32(a + 4);
  return __funnelshift_r(w0, w1, 8 * (off & 3));
}

// Rebuilds 32-element unit u of a slot image into 16 bf16x2 words: word 2m+i
// holds elements 4m + {0,2} (i=0) / {1,3} (i=1).  x: the unit's gathered 4-bit
// escape bytes (byte j = group j); b3/b4: the unit's base3 and base4 words
// base3 (32-bit, modular: e stays exact), word 2i and 2i+1 covering group i.
// A raw group comes out right when its base3 words hold its exponents (raw_bases).
__device__ __forceinline__ void decode_unit(const uint8_t* img, int u, uint32_t tb, uint32_t x, const uint32_t b3[8],
                                            const uint32_t b4[8], const uint2* lut, uint32_t o[16]) {
  const uint32_t ib = smem_addr(img);
  const uint32_t W0 = lds32(ib + kOffCode + 4 * u), W1 = lds32(ib + kOffCode + 1024 + 4 * u);
  const uint32_t W2 = lds32(ib + kOffCode + 2048 + 4 * u);
  const uint4 s0 = lds128(ib + 32 * u), s1 = lds128(ib + 32 * u + 16);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    uint32_t c[4];
    extract_codes(hh ? W1 : W0, W2, hh, c);
    const uint32_t lb = smem_addr(lut);
    const uint2 sa = lds64(lb + 8 * ((x >> (16 * hh)) & 0xFFu)), sb = lds64(lb + 8 * ((x >> (16 * hh + 8)) & 0xFFu));
    const uint32_t fa = (tb >> (4 * hh)) & 1u, fb = (tb >> (4 * hh + 2)) & 1u;  // 4-bit flags of the two groups
    uint32_t e[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t f = q < 2 ? fa : fb;
      const uint32_t sp = q == 0 ? sa.x : (q == 1 ? sa.y : (q == 2 ? sb.x : sb.y));
      e[q] = (f ? b4[4 * hh + q] : b3[4 * hh + q]) + c[q] + sp;
    }
    const uint4 sm = hh ? s1 : s0;
    join_v2(sm.x, e[0], o[8 * hh + 0], o[8 * hh + 1]);
    join_v2(sm.y, e[1], o[8 * hh + 2], o[8 * hh + 3]);
    join_v2(sm.z, e[2], o[8 * hh + 4], o[8 * hh + 5]);
    join_v2(sm.w, e[3], o[8 * hh + 6], o[8 * hh + 7]);
  }
}

// Raw groups of a unit take their exponents as base words: a raw group's codes are zero and its escape
// selector byte is zero, so decode_unit's exponent sum is the base word itself.  The eight exponent bytes of
// each raw group start at escape offset `oraw` (clamped into the area); b3: the unit's base3 words, those of
// its raw groups replaced.
__device__ __forceinline__ void raw_bases(const uint8_t* img, uint32_t tb, int oraw, uint32_t b3[8]) {
  // one pass per raw group of this lane (bit 2gi of m set for raw group gi), not per group position
  uint32_t m = (tb >> 1) & ~tb & 0x55u;
#pragma unroll 1
  while (m != 0u) {
    const int bit = __ffs(m) - 1;
    m &= m - 1u;
    const int at = kOffEsc + min(oraw, kEscCap - 8);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(img + (at & ~3));
    const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], sh = 8u * static_cast<uint32_t>(at & 3);
    const uint32_t x0 = __funnelshift_r(w0, w1, sh), x1 = __funnelshift_r(w1, w2, sh);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      if (bit == 2 * g) {
        b3[2 * g] = x0;
        b3[2 * g + 1] = x1;
      }
    }
    oraw += 8;
  }
}

// Raw tile (BF16 in storage order) unit u into the decoder's word order.
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

// The lane's two units of one tile image (units 64w + lane and 64w + 32 +
// lane, in eighths 2w and 2w+1), rebuilt into oA / oB; badA / badB: the
// eighth failed its checks (its words are then meaningless).  Slot bookkeeping: the
// directory gives each eighth's first 4-bit escape byte and raw group, one
// warp scan of the four packed counts (at most 4 per unit, 128 per eighth)
// each unit's.
template <class Smem>
__device__ __forceinline__ void tile_units(const AttnArgs& a, const Smem& sm, const uint8_t* img, int mode,
                                           int esc_len, int w, int lane, const uint32_t b3A[8],
                                           const uint32_t b4A[8], const uint32_t b3B[8], const uint32_t b4B[8],
                                           uint32_t oA[16], uint32_t oB[16], bool& badA, bool& badB) {
  const int uA = 64 * w + lane, uB = uA + 32;
  if (mode == GAAC_MODE_SLOT) {
    const uint16_t* dir = reinterpret_cast<const uint16_t*>(img + kOffDir);
    const uint32_t d0 = w ? dir[2 * w - 1] : 0u, dA = dir[2 * w], dB = dir[2 * w + 1], d7 = dir[7];
    const uint32_t ib = smem_addr(img), tl = smem_addr(sm.tagl);
    const uint32_t tbA = lds8(ib + kOffTag + uA), tbB = lds8(ib + kOffTag + uB);
    const uint32_t teA = lds32(tl + 4 * tbA), teB = lds32(tl + 4 * tbB);
    const uint32_t cnt = __byte_perm(teA, teB, 0x7362);  // 4-bit A, 4-bit B, raw A, raw B
    const uint32_t incl = warp_incl_scan(cnt, lane);
    const uint32_t tot = __shfl_sync(kFull, incl, 31), ex = incl - cnt;
    const int rawbase = static_cast<int>(d7 & 0x1FFu);
    const int o4A = static_cast<int>((d0 & 0x1FFu) + (ex & 0xFFu));
    const int o4B = static_cast<int>((dA & 0x1FFu) + ((ex >> 8) & 0xFFu));
    const int orA = rawbase + 8 * static_cast<int>((d0 >> 9) + ((ex >> 16) & 0xFFu));
    const int orB = rawbase + 8 * static_cast<int>((dA >> 9) + (ex >> 24));
    uint32_t eA[8], eB[8];  // base3 words, raw groups' exponents in their place (raw groups: rare)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      eA[i] = b3A[i];
      eB[i] = b3B[i];
    }
    if (teA >> 24) raw_bases(img, tbA, orA, eA);
    if (teB >> 24) raw_bases(img, tbB, orB, eB);
    decode_unit(img, uA, tbA, __byte_perm(escape_window(img, o4A), 0u, teA & 0xFFFFu), eA, b4A, sm.lut, oA);
    decode_unit(img, uB, tbB, __byte_perm(escape_window(img, o4B), 0u, teB & 0xFFFFu), eB, b4B, sm.lut, oB);
    // Checks of the format, on warp-uniform values (no vote): the directory entry after each eighth must be
    // the one before it plus the eighth's counts from the tags (exact arithmetic: the counts of a valid image
    // never fill their fields), and the totals must give esc_len.  A reserved tag counts 32 four-bit groups.
    const bool totals = rawbase + 8 * static_cast<int>(d7 >> 9) != esc_len;
    badA = totals || ((d0 + (tot & 0xFFu) + (((tot >> 16) & 0xFFu) << 9)) & 0xFFFFu) != dA;
    badB = totals || ((dA + ((tot >> 8) & 0xFFu) + ((tot >> 24) << 9)) & 0xFFFFu) != dB;
  } else {
    badA = badB = mode != GAAC_MODE_RAW;
    if (!badA) {
      raw_unit(img, uA, oA);
      raw_unit(img, uB, oB);
    }
  }
  // The words of a unit that failed its checks are left as they are (no branch here, between the decode
  // and the MMAs): a bad K eighth's scores are masked in the softmax and a bad V eighth's operands are
  // cleared just before the PV MMAs.
}

// ------------------------------------------------------------------ producer

// Source and byte count of one table entry's tile image (only the bytes a
// slot uses); nullptr with mode NONE for an entry that fails its checks.
__device__ __forceinline__ const void* tile_source(const AttnArgs& a, uint2 e, uint32_t& bytes, int& mode, int& esc) {
  const uint32_t index = e.x, esc_len = e.y & 0xFFFFu, emode = (e.y >> 16) & 0xFFu;
  if (emode == GAAC_MODE_SLOT && static_cast<int64_t>(index) < a.n_slots && esc_len <= kEscCap) {
    mode = GAAC_MODE_SLOT;
    esc = static_cast<int>(esc_len);
    bytes = (kOffEsc + esc_len + 15u) & ~15u;
    return a.slot_pool + static_cast<size_t>(index) * kSlot;
  }
  esc = 0;
  if (emode == GAAC_MODE_RAW && static_cast<int64_t>(index) < a.n_raw) {
    mode = GAAC_MODE_RAW;
    bytes = kRawBytes;
    return a.raw_pool + static_cast<size_t>(index) * kTile;
  }
  mode = GAAC_MODE_NONE;
  bytes = 0;
  return nullptr;
}

// Table entries of block blk for attention head H and output half hf: the K
// entries of the head's NH half-heads, then the V entry of half-head NH*H + hf.
template <int NH, int KH>
__device__ __forceinline__ void block_entries(const AttnArgs& a, int b, int H, int hf, int blk, uint2 e[KH + 1]) {
  const gaac_entry* t = a.table + (static_cast<size_t>(b) * a.max_blocks + blk) * (NH * a.Hkv) * 2;
#pragma unroll
  for (int j = 0; j < KH; ++j) e[j] = *reinterpret_cast<const uint2*>(t + (NH * H + (KH == NH ? j : hf)) * 2);
  e[KH] = *reinterpret_cast<const uint2*>(t + (NH * H + hf) * 2 + 1);
}

// One thread starts the bulk copies of a block's images into stage st (a free
// stage); stFull[st] completes when all have landed.
template <int NH, int KH>
__device__ __forceinline__ void issue_block(const AttnArgs& a, AttSmem<NH, KH>& sm, int st, const uint2 e[KH + 1],
                                            [[maybe_unused]] int j) {
  GAAC_TL(if (TlCta* c = tl_cta()) if (j < kTlBlocks) c->issue[j] = tl_now());
  StageMeta m;
  uint32_t bytes[KH + 1], total = 0;
  const void* src[KH + 1];
  bool ok = true;
#pragma unroll
  for (int i = 0; i <= KH; ++i) {
    src[i] = tile_source(a, e[i], bytes[i], m.mode[i], m.esc[i]);
    ok = ok && src[i] != nullptr;
    total += bytes[i];
  }
  if (!ok) report(a.status, GAAC_EFORMAT);
  sm.smeta[st] = m;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier generic reads of the stage, then async writes
  mbar_arrive_expect_tx(&sm.stFull[st], total);
#pragma unroll
  for (int i = 0; i <= KH; ++i)
    if (bytes[i]) bulk_g2s(sm.stage[st][i], src[i], bytes[i], &sm.stFull[st]);
}

__device__ __forceinline__ unsigned int atomic_add_acq_rel_cta(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.add.acq_rel.cta.shared::cta.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_addr(p)), "r"(v) : "memory");
  return old;
}

// ------------------------------------------------------ cluster pair (DSMEM)

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of this CTA's shared variable p in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

// Asynchronous 16-byte store into another CTA's shared memory that completes its bytes on that CTA's
// mbarrier `bar` (which expects them with arrive.expect_tx).
__device__ __forceinline__ void st_async_f4(uint32_t addr, float x, float y, float z, float w, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
               "f"(x), "f"(y), "f"(z), "f"(w), "r"(bar)
               : "memory");
}

// All threads of both CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------ compute warps

// Warp w of group gr: tokens [16w, 16w+16) of blocks gr, gr + kGroups, ...
// Lane (g, tq) = (lane/4, lane%4).  Returns the warp's (m, l) per head through
// shared memory and its accumulators in acc (O^T fragments: acc[m][0..3] =
// channels 16m+g, 16m+g+8 x heads 2tq, 2tq+1).
// K unit base words of half-head `half`: channels 32tq..32tq+31, word i = channels 32tq + 4i..+3.
template <int NH, int KH>
__device__ __forceinline__ void k_bases(const AttSmem<NH, KH>& sm, int half, int tq, uint32_t kb3[8], uint32_t kb4[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    kb3[i] = *reinterpret_cast<const uint32_t*>(&sm.kbases[half][0][32 * tq + 4 * i]);
    kb4[i] = *reinterpret_cast<const uint32_t*>(&sm.kbases[half][1][32 * tq + 4 * i]);
  }
}

// The group's last warp to finish reading stage st refills it with block jn (entries ne, read by lane 0).
template <int NH, int KH>
__device__ __forceinline__ void release_stage(const AttnArgs& a, AttSmem<NH, KH>& sm, int st, int jn, int n_my,
                                              int lane, const uint2 ne[KH + 1]) {
  __syncwarp();
  if (lane == 0 && atomic_add_acq_rel_cta(&sm.stDone[st], 1u) == kGroupWarps - 1) {
    sm.stDone[st] = 0u;
    GAAC_TL(if (TlCta* c = tl_cta()) if (jn - AttSmem<NH, KH>::kStages < kTlBlocks) c->release[jn - AttSmem<NH, KH>::kStages] = tl_now());
    if (jn < n_my) issue_block<NH, KH>(a, sm, st, ne, jn);
  }
}

// RAW: the uncompressed BF16 path (every tile a raw tile): the warp loads its K and V units straight
// into operand registers, releases the stage before any MMA, and has no decode.
template <int NH, int KH, bool RAW>
__device__ __forceinline__ void compute_warp(const AttnArgs& a, AttSmem<NH, KH>& sm, int b, int H, int hf, int blk0,
                                             int n_my, int len, int gr, int w, int cw, int lane, float acc[8][4]) {
  constexpr int kStages = AttSmem<NH, KH>::kStages;
  const int g = lane >> 2, tq = lane & 3;
  uint32_t kb3[8], kb4[8];  // one half-head: loaded once (NH = 1) or per half and block (NH = 2)
  // K base words are reloaded from shared memory per block (registers are scarce at 12 warps per SM)
  [[maybe_unused]] uint32_t peer_mail = 0u, peer_full = 0u, peer_empty = 0u, peer_ack = 0u;  // the peer's mailbox
  if constexpr (NH > KH) {
    const uint32_t peer = cluster_rank() ^ 1u;
    peer_mail = peer_addr(&sm.mail[cw][0][lane], peer);
    peer_full = peer_addr(&sm.mFull[cw][0], peer);
    peer_empty = peer_addr(&sm.mEmpty[cw][0], peer);
    peer_ack = peer_addr(&sm.ack[cw][0], peer);
  }
  int it = 0;  // this warp's block count
#pragma unroll
  for (int m = 0; m < 8; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
  // Scores S = K q^T of the warp's 16 tokens: rows g and g+8 (tokens tA, tB of the two octets), columns
  // 2tq, 2tq+1.  A column is a query head; with r <= 4 query heads per kv-head, columns 4-7 repeat
  // heads 0-3 (`packed`): their lanes run the same softmax and feed the low parts of P to the same PV MMA
  // in which columns 0-3 take the high parts.  Running maxima m0, m1 and sums l0, l1 per column.
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int tA = 16 * w + g, tB = tA + 8;        // tokens of S rows g, g+8
  const int vA = 16 * w + 2 * tq, vB = vA + 8;   // tokens of the V operand's columns 2tq, 2tq+1
  const bool packed = a.r <= 4;
  bool fmt_bad = false;  // a tile this warp read failed the format checks (reported once, at the end)
  // BF16 path: q's B-operand registers stay in registers across blocks
  [[maybe_unused]] uint32_t qb0[8], qb1[8];
  if constexpr (RAW) {
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const uint2 qv = sm.qf[0][m][lane];
      qb0[m] = qv.x;
      qb1[m] = qv.y;
    }
  }
  // Table entries of the block each stage takes next, read one iteration of the group ahead so that a
  // refill never waits for them: ne serves this iteration's refill (block j + kStages), nn the next one's.
  uint2 ne[KH + 1], nn[KH + 1];
#pragma unroll
  for (int i = 0; i <= KH; ++i) ne[i] = nn[i] = make_uint2(0u, 0u);
  if (lane == 0 && gr + kStages < n_my) block_entries<NH, KH>(a, b, H, hf, blk0 + gr + kStages, ne);
#pragma unroll 1
  for (int j = gr; j < n_my; j += kGroups, ++it) {
    const int st = j % kStages, jn = j + kStages;  // jn: the block this stage takes next
    if (lane == 0 && jn + kGroups < n_my) block_entries<NH, KH>(a, b, H, hf, blk0 + jn + kGroups, nn);
    GAAC_TL(if (w == 0 && lane == 0) if (TlCta* c = tl_cta()) if (j < kTlBlocks) c->arrive[j] = tl_now());
    mbar_wait(&sm.stFull[st], static_cast<uint32_t>(j / kStages) & 1u, a.status);
    GAAC_TL(if (w == 0 && lane == 0) if (TlCta* c = tl_cta()) if (j < kTlBlocks) c->land[j] = tl_now());
    const StageMeta meta = sm.smeta[st];
    const int nv = min(kBlock, len - (blk0 + j) * kBlock);
    // ---- S = K q^T for tokens tA (row g) and tB (row g+8), summed over this CTA's K images: the K units
    // of the two tokens are the A operand (k-step m: a0, a2 = token tA, a1, a3 = token tB), q^T the B
    // operand; even and odd k-steps go to two accumulators (a chain of four MMAs each)
    float sc[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
    bool kbadA = false, kbadB = false, vbadA = false, vbadB = false;
    uint32_t oA[16], oB[16];  // the V operands of this warp's 16 tokens
    if constexpr (RAW) {
      static_assert(NH == 1 && KH == 1, "the BF16 path serves 128-channel heads");
      const int uA = 64 * w + lane, uB = uA + 32;
      uint32_t kA[16], kB[16];
      raw_unit(sm.stage[st][0], uA, kA);
      raw_unit(sm.stage[st][0], uB, kB);
      raw_unit(sm.stage[st][1], uA, oA);
      raw_unit(sm.stage[st][1], uB, oB);
      release_stage<NH, KH>(a, sm, st, jn, n_my, lane, ne);
      kbadA = kbadB = meta.mode[0] != GAAC_MODE_RAW;
      vbadA = vbadB = meta.mode[1] != GAAC_MODE_RAW;
#pragma unroll
      for (int m = 0; m < 8; m += 2) {
        mma_bf16(sc, kA[2 * m], kB[2 * m], kA[2 * m + 1], kB[2 * m + 1], qb0[m], qb1[m]);
        mma_bf16(s1, kA[2 * m + 2], kB[2 * m + 2], kA[2 * m + 3], kB[2 * m + 3], qb0[m + 1], qb1[m + 1]);
      }
    } else {
#pragma unroll 1
      for (int half = 0; half < KH; ++half) {
        k_bases(sm, half, tq, kb3, kb4);
        uint32_t oA[16], oB[16];
        bool bA, bB;
        tile_units(a, sm, sm.stage[st][half], meta.mode[half], meta.esc[half], w, lane, kb3, kb4, kb3, kb4, oA, oB,
                   bA, bB);
        kbadA = kbadA || bA;
        kbadB = kbadB || bB;
        // q^T (scaled by 2^-4) as the B operand: for k-step m the lane's K registers hold channels
        // 32tq + 4m + {0,2} (first) and {1,3} (second) of its two tokens, and its q pair the same channels
        // of column g
#pragma unroll
        for (int m = 0; m < 8; m += 2) {
          const uint2 q0 = sm.qf[half][m][lane], q1 = sm.qf[half][m + 1][lane];
          mma_bf16(sc, oA[2 * m], oB[2 * m], oA[2 * m + 1], oB[2 * m + 1], q0.x, q0.y);
          mma_bf16(s1, oA[2 * m + 2], oB[2 * m + 2], oA[2 * m + 3], oB[2 * m + 3], q1.x, q1.y);
        }
      }
      if constexpr (NH > KH) {
        // 256-channel heads as a cluster pair: the scores are this CTA's half-head partial plus the peer's.
        // Each lane posts its partials (NaN for a unit that failed its checks) into the peer's mailbox now,
        // as asynchronous stores that complete on the peer's barrier, and takes the peer's after the V
        // decode; both CTAs add S0 + S1 (exact-commutative), so their softmax weights are identical.
        const int bb = it & 1;
        if (it >= 2) {  // the peer has read this buffer's previous use: its 16-byte acknowledgement landed
          if (lane == 0) mbar_arrive_expect_tx(&sm.mEmpty[cw][bb], sizeof(float4));
          mbar_wait(&sm.mEmpty[cw][bb], static_cast<uint32_t>((it >> 1) + 1) & 1u, a.status);
        }
        st_async_f4(peer_mail + bb * 32 * sizeof(float4), kbadA ? NAN : sc[0] + s1[0],
                    kbadA ? NAN : sc[1] + s1[1], kbadB ? NAN : sc[2] + s1[2], kbadB ? NAN : sc[3] + s1[3],
                    peer_full + bb * sizeof(uint64_t));
      }
      // ---- V units of the same tokens (independent of the scores: decoded while the MMAs above run)
      uint32_t vb3[2][8], vb4[2][8];  // word 2i and 2i+1 serve group i
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
        const uint4 x3 = sm.vbw[hv][0][lane];
        const uint4 x4 = sm.vbw[hv][1][lane];
        vb3[hv][0] = vb3[hv][1] = x3.x;
        vb3[hv][2] = vb3[hv][3] = x3.y;
        vb3[hv][4] = vb3[hv][5] = x3.z;
        vb3[hv][6] = vb3[hv][7] = x3.w;
        vb4[hv][0] = vb4[hv][1] = x4.x;
        vb4[hv][2] = vb4[hv][3] = x4.y;
        vb4[hv][4] = vb4[hv][5] = x4.z;
        vb4[hv][6] = vb4[hv][7] = x4.w;
      }
      tile_units(a, sm, sm.stage[st][KH], meta.mode[KH], meta.esc[KH], w, lane, vb3[0], vb4[0], vb3[1], vb4[1], oA,
                 oB, vbadA, vbadB);
      // The stage is read: the group's last warp to get here refills it with block jn.
      release_stage<NH, KH>(a, sm, st, jn, n_my, lane, ne);
    }  // compressed path
    if constexpr (NH > KH) {  // take the peer's partial scores of this block (posted above)
      const int bb = it & 1;
      if (lane == 0) mbar_arrive_expect_tx(&sm.mFull[cw][bb], 32 * sizeof(float4));
      mbar_wait(&sm.mFull[cw][bb], static_cast<uint32_t>(it >> 1) & 1u, a.status);
      const float4 X = sm.mail[cw][bb][lane];
      // Acknowledge with an asynchronous store into the peer's ack slot that completes on its mEmpty; its
      // payload is an OR over the warp of the loaded scores' bits, so it cannot issue before every lane's
      // load has returned.
      {
        const uint32_t dep = __reduce_or_sync(kFull, __float_as_uint(X.x) | __float_as_uint(X.y) |
                                                         __float_as_uint(X.z) | __float_as_uint(X.w));
        if (lane == 0)
          st_async_f4(peer_ack + bb * sizeof(float4), __uint_as_float(dep), 0.f, 0.f, 0.f,
                      peer_empty + bb * sizeof(uint64_t));
      }
      sc[0] = (kbadA ? NAN : sc[0] + s1[0]) + X.x;
      sc[1] = (kbadA ? NAN : sc[1] + s1[1]) + X.y;
      sc[2] = (kbadB ? NAN : sc[2] + s1[2]) + X.z;
      sc[3] = (kbadB ? NAN : sc[3] + s1[3]) + X.w;
      s1[0] = s1[1] = s1[2] = s1[3] = 0.f;
      kbadA = __any_sync(kFull, isnan(sc[0]) || isnan(sc[1]));
      kbadB = __any_sync(kFull, isnan(sc[2]) || isnan(sc[3]));
    }
    // ---- online softmax of columns 2tq, 2tq+1 over the warp's 16 tokens, on raw scores (q/16).k: only the
    // differences from the running maxima are scaled to the log2 domain
    fmt_bad = fmt_bad || kbadA || kbadB || vbadA || vbadB;
    const float x0 = (!kbadA && tA < nv) ? sc[0] + s1[0] : -INFINITY;  // token tA, column 2tq
    const float x1 = (!kbadA && tA < nv) ? sc[1] + s1[1] : -INFINITY;  // token tA, column 2tq+1
    const float x2 = (!kbadB && tB < nv) ? sc[2] + s1[2] : -INFINITY;  // token tB
    const float x3 = (!kbadB && tB < nv) ? sc[3] + s1[3] : -INFINITY;
    float b0 = fmaxf(x0, x2), b1 = fmaxf(x1, x3);
#pragma unroll
    for (int d = 4; d < 32; d <<= 1) {  // over the eight lanes g of each column pair
      b0 = fmaxf(b0, __shfl_xor_sync(kFull, b0, d));
      b1 = fmaxf(b1, __shfl_xor_sync(kFull, b1, d));
    }
    const float n0 = fmaxf(m0, b0), n1 = fmaxf(m1, b1);
    const float cl = a.c_log2;
    if (__any_sync(kFull, n0 != m0 || n1 != m1)) {  // a running maximum rises: rescale (rare after the first blocks)
      const float al0 = m0 == -INFINITY ? 0.f : fast_exp2((m0 - n0) * cl);
      const float al1 = m1 == -INFINITY ? 0.f : fast_exp2((m1 - n1) * cl);
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        acc[m][0] *= al0;
        acc[m][2] *= al0;
        acc[m][1] *= al1;
        acc[m][3] *= al1;
      }
      m0 = n0;
      m1 = n1;
    }
    const float p0 = m0 != -INFINITY ? fast_exp2((x0 - m0) * cl) : 0.f;
    const float p2 = m0 != -INFINITY ? fast_exp2((x2 - m0) * cl) : 0.f;
    const float p1 = m1 != -INFINITY ? fast_exp2((x1 - m1) * cl) : 0.f;
    const float p3 = m1 != -INFINITY ? fast_exp2((x3 - m1) * cl) : 0.f;
    l0 += p0 + p2;
    l1 += p1 + p3;
    // P as bf16 high and low parts (rows = tokens, columns 2tq, 2tq+1), then transposed per octet into the
    // B operand P^T of O^T += V^T P^T (lane (g, tq): tokens 2tq, 2tq+1 of the octet, column g)
    const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
    const uint32_t l01 = pack_bf16x2(p0 - __uint_as_float(h01 << 16), p1 - __uint_as_float(h01 & 0xFFFF0000u));
    const uint32_t l23 = pack_bf16x2(p2 - __uint_as_float(h23 << 16), p3 - __uint_as_float(h23 & 0xFFFF0000u));
    // ---- O^T += V^T P^T over the 16 tokens, eight 16-channel tiles
    if (nv < kBlock || vbadA || vbadB) {
      // the open block: values of tokens past the sequence must not meet a zero weight; a V eighth that
      // failed its checks contributes nothing
      const uint32_t mlo = (vA < nv ? 0x0000FFFFu : 0u) | (vA + 1 < nv ? 0xFFFF0000u : 0u);
      const uint32_t mhi = (vB < nv ? 0x0000FFFFu : 0u) | (vB + 1 < nv ? 0xFFFF0000u : 0u);
      const uint32_t kA = vbadA ? 0u : 0xFFFFFFFFu, kB = vbadB ? 0u : 0xFFFFFFFFu;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        oA[4 * i] &= mlo & kA;
        oA[4 * i + 1] &= mlo & kA;
        oA[4 * i + 2] &= mhi & kA;
        oA[4 * i + 3] &= mhi & kA;
        oB[4 * i] &= mlo & kB;
        oB[4 * i + 1] &= mlo & kB;
        oB[4 * i + 2] &= mhi & kB;
        oB[4 * i + 3] &= mhi & kB;
      }
    }
    if (packed) {  // columns 0-3: high parts, columns 4-7: low parts of the same heads
      const uint32_t pA = movmatrix_trans(tq < 2 ? h01 : l01), pB = movmatrix_trans(tq < 2 ? h23 : l23);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        mma_bf16(acc[i], oA[4 * i], oA[4 * i + 1], oA[4 * i + 2], oA[4 * i + 3], pA, pB);
        mma_bf16(acc[4 + i], oB[4 * i], oB[4 * i + 1], oB[4 * i + 2], oB[4 * i + 3], pA, pB);
      }
    } else {
      const uint32_t hA = movmatrix_trans(h01), hB = movmatrix_trans(h23);
      const uint32_t lA = movmatrix_trans(l01), lB = movmatrix_trans(l23);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        mma_bf16(acc[i], oA[4 * i], oA[4 * i + 1], oA[4 * i + 2], oA[4 * i + 3], hA, hB);
        mma_bf16(acc[4 + i], oB[4 * i], oB[4 * i + 1], oB[4 * i + 2], oB[4 * i + 3], hA, hB);
        mma_bf16(acc[i], oA[4 * i], oA[4 * i + 1], oA[4 * i + 2], oA[4 * i + 3], lA, lB);
        mma_bf16(acc[4 + i], oB[4 * i], oB[4 * i + 1], oB[4 * i + 2], oB[4 * i + 3], lA, lB);
      }
    }
#pragma unroll
    for (int i = 0; i <= KH; ++i) ne[i] = nn[i];
  }
  if constexpr (NH > KH) {
    // The acknowledgements of this warp's last posts (one per buffer used) are still owed: take them, so that
    // no asynchronous store is on its way to this CTA when it exits.
#pragma unroll 1
    for (int u = max(0, it - 2); u < it; ++u) {
      const int bb = u & 1;
      if (lane == 0) mbar_arrive_expect_tx(&sm.mEmpty[cw][bb], sizeof(float4));
      mbar_wait(&sm.mEmpty[cw][bb], static_cast<uint32_t>(u >> 1) & 1u, a.status);
    }
  }
  if (fmt_bad && lane == 0) report(a.status, GAAC_EFORMAT);
#pragma unroll
  for (int d = 4; d < 32; d <<= 1) {
    l0 += __shfl_xor_sync(kFull, l0, d);
    l1 += __shfl_xor_sync(kFull, l1, d);
  }
  if (packed) {  // fold the low-part columns 4-7 into the high-part columns 0-3 of the same heads
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[m][k] += __shfl_xor_sync(kFull, acc[m][k], 2);
  }
  if (g == 0) {  // columns 4-7 of a packed warp hold no head of their own
    const bool own = !packed || tq < 2;
    sm.wm[cw][2 * tq] = own ? m0 : -INFINITY;
    sm.wm[cw][2 * tq + 1] = own ? m1 : -INFINITY;
    sm.wl[cw][2 * tq] = own ? l0 : 0.f;
    sm.wl[cw][2 * tq + 1] = own ? l1 : 0.f;
  }
}

// Log-sum-exp merge of the n_splits partials (m, l, acc) of one (sequence,
// kv-head) into out[b, h*r + n, :] = sum_s w_s acc_s / sum_s w_s l_s with
// w_s = 2^((m_s - max_s m_s) cl) per head n (the final split reduction; m_s are
// raw-score maxima, cl converts their differences to the log2 domain).  Runs on
// the CTA that finished last, so it is a tail on the critical path: each
// thread owns one float4 column of the output and a subset of the splits,
// issues that subset's loads ten at a time and folds them in with its own
// running maximum; the subsets are then combined the same way in shared
// memory.  The staging ring is free by then and holds that exchange.
// base: the first partial of the pair; out: its first output row.
template <int NH, class Smem>
__device__ __noinline__ void merge_splits(const float* base, int ns, int r, float cl, float* out, Smem& sm, int tid) {
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
        const float al = mt == -INFINITY ? 0.f : fast_exp2((mt - mb) * cl);
        acc.x *= al;
        acc.y *= al;
        acc.z *= al;
        acc.w *= al;
        den *= al;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const float w = ml[u].x == -INFINITY ? 0.f : fast_exp2((ml[u].x - mb) * cl);
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
      const float al = mt == -INFINITY ? 0.f : fast_exp2((mt - mx) * cl);
      acc.x *= al;
      acc.y *= al;
      acc.z *= al;
      acc.w *= al;
      den *= al;
      for (int gi = 1; gi < groups; ++gi) {
        const float2 md = xm[gi * o4n + o4];
        if (md.x == -INFINITY) continue;
        const float w = fast_exp2((md.x - mx) * cl);
        const float4 x = xa[gi * o4n + o4];
        acc.x += w * x.x;
        acc.y += w * x.y;
        acc.z += w * x.z;
        acc.w += w * x.w;
        den += w * md.y;
      }
    }
    float* o = out + n * (NH * kD) + 4 * c4;  // rows of NH * 128 channels
    const float inv = den > 0.f ? 1.f / den : 0.f;
    o[0] = acc.x * inv;
    o[1] = acc.y * inv;
    o[2] = acc.z * inv;
    o[3] = acc.w * inv;
  }
}


// Grid (split, NH * Hkv, batch): CTA y serves attention head H = y / NH and
// output channels [128 hf, 128 hf + 128) of it (hf = y % NH), reading the V
// tile of half-head NH*H + hf.  KH = NH: the CTA also reads the K tiles of all
// NH half-heads.  KH = 1 < NH: the NH CTAs of a head form a cluster; each
// reads the K tile of its own half-head and the pair exchanges partial scores
// through distributed shared memory, so every K tile is decoded once.
template <int NH, int KH, bool RAW>
__global__ void __launch_bounds__(kAttThreads, kCtasPerSm) attn_split_kernel(AttnArgs a) {
  constexpr int kStages = AttSmem<NH, KH>::kStages;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  AttSmem<NH, KH>& sm = *reinterpret_cast<AttSmem<NH, KH>*>(smem_raw);
  const int split = blockIdx.x, y = blockIdx.y, b = blockIdx.z;
  const int H = y / NH, hf = y % NH, nkv = NH * a.Hkv;  // nkv: half-heads in the table and the bases
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Launched as a programmatic dependent of the previous kernel on the stream, the CTA may already be
  // resident while that kernel finishes.  Meanwhile its first blocks' images are prefetched into L2 from a
  // guess of the length and table (the previous kernel may still write them: a stale or torn guess only
  // wastes a prefetch, and every address is checked against the pools), then the CTA waits for that
  // kernel (and its memory) before any read it relies on.  A no-op wait for an ordinary launch.
  if (tid < kStages) {
    const int glen = *reinterpret_cast<const volatile int32_t*>(a.seq_lens + b);
    if (glen > 0 && glen <= a.max_blocks * kBlock) {
      const int gper = (a.max_blocks + a.n_splits - 1) / a.n_splits;
      const int gblk = split * gper + tid;
      if (tid < gper && gblk * kBlock < glen) {
        uint2 e[KH + 1];
        block_entries<NH, KH>(a, b, H, hf, gblk, e);
#pragma unroll
        for (int i = 0; i <= KH; ++i) {
          uint32_t bytes;
          int mode, esc;
          const void* src = tile_source(a, e[i], bytes, mode, esc);
          if (src != nullptr)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
        }
      }
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  GAAC_TL(if (tid == 0) if (TlCta* c = tl_cta()) { c->start = tl_now(); c->merged = 0ull; });
  int len = a.seq_lens[b];
  if (len < 0 || len > a.max_blocks * kBlock) {
    if (tid == 0) report(a.status, GAAC_EINVAL);
    len = 0;
  }
  // This split's blocks of the sequence: chunks of `per` blocks, the same for every sequence of the
  // launch, so a shorter sequence uses fewer splits (at least one) and the others leave at once.
  const int nblk = (len + kBlock - 1) / kBlock;
  const int per = (a.max_blocks + a.n_splits - 1) / a.n_splits;
  const int n_used = max(1, (nblk + per - 1) / per);  // splits of this sequence, and partials its merge takes
  if (split >= n_used) return;
  const int blk0 = split * per;
  const int n_my = max(0, min(nblk, blk0 + per) - blk0);

  // The first blocks' copies start before anything else: lane st initialises
  // stage st's barrier and issues block st into it (later blocks are issued as
  // stages free up), so the tables below are built while the copies land.
  if (tid < kStages) {
    mbar_init(&sm.stFull[tid], 1);
    sm.stDone[tid] = 0u;
  }
  if (NH > KH && tid < 2 * AttSmem<NH, KH>::kPairs) {
    mbar_init(&sm.mFull[tid / 2][tid % 2], 1);   // lane 0's expect_tx; the peer's bytes complete it
    mbar_init(&sm.mEmpty[tid / 2][tid % 2], 1);  // lane 0 of the peer's warp, after reading
  }
  fence_mbar_init();
  if (tid < min(n_my, kStages)) {
    uint2 e[KH + 1];
    block_entries<NH, KH>(a, b, H, hf, blk0 + tid, e);
    issue_block<NH, KH>(a, sm, tid, e, tid);
  }

  for (int x = tid; x < (RAW ? 0 : 256); x += kAttThreads) {  // decode tables (compressed path only)
    sm.lut[x] = spread_entry(static_cast<uint32_t>(x));
    sm.tagl[x] = tag_entry(static_cast<uint32_t>(x));
  }
  for (int x = tid; x < (RAW ? 0 : KH * 2 * kD); x += kAttThreads) {  // K: [image][base3|base4][channel]
    const int half = x / (2 * kD), which = (x / kD) & 1, c = x % kD;
    sm.kbases[half][which][c] = (which ? a.base4 : a.base3)[(NH * H + (KH == NH ? half : hf)) * kD + c];
  }
  // V unit base words: group i of the lane's unit hv holds channels 16m+g and 16m+g+8 (m = 4hv + i, g =
  // lane/4) in byte lanes 0, 2 and 1, 3 of both of its exponent words
  for (int x = tid; x < (RAW ? 0 : 32 * 2 * 4); x += kAttThreads) {
    const int ln = x / 8, hv = (x / 4) % 2, i = x % 4;
    const int cA = 16 * (4 * hv + i) + ln / 4;
    const uint8_t* v3 = a.base3 + (nkv + NH * H + hf) * kD;
    const uint8_t* v4 = a.base4 + (nkv + NH * H + hf) * kD;
    const uint32_t x3 = v3[cA] | (static_cast<uint32_t>(v3[cA + 8]) << 8);
    const uint32_t x4 = v4[cA] | (static_cast<uint32_t>(v4[cA + 8]) << 8);
    reinterpret_cast<uint32_t*>(&sm.vbw[hv][0][ln])[i] = x3 | (x3 << 16);
    reinterpret_cast<uint32_t*>(&sm.vbw[hv][1][ln])[i] = x4 | (x4 << 16);
  }
  // q of the kv-head's query heads, times 2^-4 (and the sign of the scale), as B-operand pairs of
  // S = K q^T: for half `half`, lane (g, tq) and k-step m, (channels 128 half + 32tq + 4m + {0, 2},
  // ... + {1, 3}) of column g's head: head g, or g % 4 when the kv-head has at most 4 query heads
  // (columns 4-7 repeat heads 0-3); columns without a head are zero
  for (int x = tid; x < KH * 32 * 8 * 2; x += kAttThreads) {
    const int half = x / 512, ln = (x / 16) % 32, tq = ln % 4, m = (x / 2) % 8, odd = x % 2;
    const int n = a.r <= 4 ? (ln / 4) & 3 : ln / 4;
    uint32_t v = 0u;
    if (n < a.r) {
      const uint16_t* qrow = a.q + (static_cast<size_t>(b) * a.Hq + H * a.r + n) * (NH * kD) +
                             kD * (KH == NH ? half : hf) + 32 * tq + 4 * m + odd;
      v = bf16x2_mul(static_cast<uint32_t>(qrow[0]) | (static_cast<uint32_t>(qrow[2]) << 16), a.qmul);
    }
    reinterpret_cast<uint32_t*>(&sm.qf[half][m][ln])[odd] = v;
  }
  __syncthreads();  // barriers initialised, tables built
  if constexpr (NH > KH) cluster_sync();  // the peer's mailbox barriers exist before any remote arrival

  const int r = a.r;
  float* part = a.part + ((static_cast<size_t>(b) * nkv + y) * a.n_splits + split) * kPartFloats;
  float acc[8][4];
  compute_warp<NH, KH, RAW>(a, sm, b, H, hf, blk0, n_my, len, warp / kGroupWarps, warp % kGroupWarps, warp, lane,
                            acc);
  // The next kernel on the stream may be scheduled now (it waits for this one before its first read).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    // Every issued copy was waited for by its group; after a timed-out wait,
    // wait once more (bounded) so that no copy is still landing at exit.
#pragma unroll 1
    for (int i = max(0, n_my - kStages); i < n_my; ++i)
      mbar_wait(&sm.stFull[i % kStages], (i / kStages) & 1, a.status, 1u << 10);
  }
  __syncthreads();  // every stage consumed: the ring becomes merge scratch
  GAAC_TL(if (tid == 0) if (TlCta* c = tl_cta()) c->split_end = tl_now());
  // ---- merge of the compute warps' states: weights 2^(m_w - max_w m_w) per head
  if (tid < kCWarps * kRPad) {
    const int cw = tid / kRPad, n = tid % kRPad;
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kCWarps; ++i) mx = fmaxf(mx, sm.wm[i][n]);
    const float mw = sm.wm[cw][n];
    sm.ww[cw][n] = mw == -INFINITY ? 0.f : fast_exp2((mw - mx) * a.c_log2);
    if (cw == 0) {
      float lt = 0.f;
#pragma unroll
      for (int i = 0; i < kCWarps; ++i) {
        const float mi = sm.wm[i][n];
        lt += (mi == -INFINITY ? 0.f : fast_exp2((mi - mx) * a.c_log2)) * sm.wl[i][n];
      }
      part[2 * n] = mx;
      part[2 * n + 1] = lt;
    }
  }
  float* xacc = reinterpret_cast<float*>(sm.stage[0][0]);  // [warp][head][channel]
  {
    const int g = lane >> 2, tq = lane & 3;
    float* xw = xacc + warp * kRPad * kD;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int c0 = 16 * m + g;
      xw[(2 * tq) * kD + c0] = acc[m][0];
      xw[(2 * tq + 1) * kD + c0] = acc[m][1];
      xw[(2 * tq) * kD + c0 + 8] = acc[m][2];
      xw[(2 * tq + 1) * kD + c0 + 8] = acc[m][3];
    }
  }
  __syncthreads();
  float* pa = part + 2 * kRPad;
  for (int x = tid; x < kRPad * kD; x += kAttThreads) {
    const int n = x / kD;
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kCWarps; ++i) s += sm.ww[i][n] * xacc[i * kRPad * kD + x];
    pa[x] = s;
  }

  // ---------------------------------------------------------------- split merge (final reduction)
  // The last CTA of a (sequence, kv-head) to finish merges the partials of all
  // its splits with a log-sum-exp; the counter goes back to zero for the next
  // launch.  No CTA ever waits for another.
  // Release/acquire through the counter: the barrier orders every thread's
  // partial stores before thread 0's acq_rel add, and the add orders the other
  // splits' stores before this CTA's loads (the barrier passes that on).
  __syncthreads();
  if constexpr (NH > KH) cluster_sync();  // no remote arrival is still on its way to this CTA
  unsigned int* counter = a.counters + static_cast<size_t>(b) * nkv + y;
  if (tid == 0) sm.last = atomic_add_acq_rel(counter, 1u) == static_cast<unsigned int>(n_used - 1);
  __syncthreads();
  GAAC_TL(if (tid == 0) if (TlCta* c = tl_cta()) c->exit = tl_now());
  if (!sm.last) return;
  merge_splits<NH>(a.part + (static_cast<size_t>(b) * nkv + y) * a.n_splits * kPartFloats, n_used, r, a.c_log2,
                   a.out + (static_cast<size_t>(b) * a.Hq + H * r) * (NH * kD) + kD * hf, sm, tid);
  if (tid == 0) *counter = 0u;
  GAAC_TL(if (tid == 0) if (TlCta* c = tl_cta()) c->merged = tl_now());
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

template <int NH, int KH, bool RAW>
static bool prepare_kernel() {
  static bool done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (!done[dev]) {
    if (cudaFuncSetAttribute(attn_split_kernel<NH, KH, RAW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(AttSmem<NH, KH>))) != cudaSuccess)
      return false;
    done[dev] = true;
  }
  return true;
}

// Launch configuration of the cluster-pair kernel for 256-channel heads: clusters of the NH CTAs of a head.
template <int NH, int KH>
static cudaLaunchConfig_t pair_config(dim3 grid, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kAttThreads, 1, 1);
  cfg.dynamicSmemBytes = sizeof(AttSmem<NH, KH>);
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = NH;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Clusters of the pair kernel that can be resident at once (0 if unknown), cached per device.
template <int NH, int KH>
static int pair_max_clusters() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pair_config<NH, KH>(dim3(1, NH, 1), nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attn_split_kernel<NH, KH, false>, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = -1;
    }
    cached[dev] = n;
  }
  return cached[dev] > 0 ? cached[dev] : 0;
}

}  // namespace gaac

using namespace gaac;

// Split count for sequences of up to max_blocks blocks: each (sequence, kv-head) is cut into chunks of
// ceil(max_blocks / s) blocks, one CTA per chunk, one resident CTA per SM.  The count minimises the
// launch's length for full sequences, waves x (chunk + a CTA's fixed cost), the fixed cost (ramp-up of
// its first copies, partial and merge) being worth about kCtaCostBlocks blocks; ties go to fewer splits.
constexpr int kCtaCostBlocks = 4;
extern "C" int gaac_attention_auto_splits(int batch, int n_kv_heads, int max_blocks) {
  if (batch <= 0 || n_kv_heads <= 0 || max_blocks <= 0) return 1;
  const long long slots = static_cast<long long>(kCtasPerSm) * device_sms();
  const long long pairs = static_cast<long long>(batch) * n_kv_heads;
  long long best = 1, best_cost = -1;
  const long long smax = std::min<long long>(max_blocks, std::max<long long>(1, 64 * slots / pairs));
  for (long long s = 1; s <= smax; ++s) {
    const long long chunk = (max_blocks + s - 1) / s;
    if (s > 1 && (max_blocks + chunk - 1) / chunk < s) continue;  // the same chunks as a smaller count
    const long long waves = (pairs * s + slots - 1) / slots;
    const long long cost = waves * (chunk + kCtaCostBlocks);
    if (best_cost < 0 || cost < best_cost) {
      best = s;
      best_cost = cost;
    }
  }
  return static_cast<int>(best);
}

static size_t partials_bytes(int batch, int n_kv_heads, int n_splits) {
  return static_cast<size_t>(batch) * n_kv_heads * n_splits * kPartFloats * sizeof(float);
}

// The merge counters open the workspace (one u32 per (sequence, kv-head), rounded up to 16 bytes), so
// their place does not depend on the split count and a workspace reused with another count still
// finds them at zero; the split partials follow.
static size_t counters_bytes(int batch, int n_kv_heads) {
  return (static_cast<size_t>(batch) * n_kv_heads * sizeof(unsigned int) + 15) & ~static_cast<size_t>(15);
}

extern "C" size_t gaac_attention_workspace(int batch, int n_kv_heads, int max_blocks, int n_splits) {
  if (n_splits <= 0) n_splits = gaac_attention_auto_splits(batch, n_kv_heads, max_blocks);
  if (batch <= 0 || n_kv_heads <= 0) return 0;
  return counters_bytes(batch, n_kv_heads) + partials_bytes(batch, n_kv_heads, n_splits);
}

// Checks and launch shared by the 128- and 256-channel entry points; n_kv_heads
// counts attention kv-heads, each of NH half-heads in the table and the bases.
// clear_counters: zero the workspace's merge counters on the stream once every
// check has passed (a call that fails a check enqueues nothing).  RAW: the
// uncompressed BF16 kernel (128-channel heads only).
template <int NH, bool RAW = false>
static int launch_attention(const uint16_t* q, int batch, int n_q_heads, int n_kv_heads, int max_blocks,
                            const int32_t* seq_lens, const gaac_entry* table, const gaac_pools* pools,
                            const uint8_t* base3, const uint8_t* base4, float scale, int n_splits, float* out,
                            void* workspace, size_t workspace_bytes, int32_t* d_status, void* stream,
                            bool clear_counters = false) {
  if (q == nullptr || seq_lens == nullptr || table == nullptr || pools == nullptr || (!RAW && pools->slot_pool == nullptr) ||
      pools->raw_pool == nullptr || pools->n_slots < 0 || pools->n_raw < 0 || base3 == nullptr ||
      base4 == nullptr || out == nullptr || workspace == nullptr)
    return GAAC_EINVAL;
  if (batch <= 0 || batch > 65535 || n_kv_heads <= 0 || NH * n_kv_heads > 65535 || n_q_heads <= 0 ||
      n_q_heads % n_kv_heads != 0 || n_q_heads / n_kv_heads > GAAC_MAX_GQA || max_blocks <= 0 ||
      max_blocks > (1 << 24) || !std::isfinite(scale))
    return GAAC_EINVAL;
  if ((reinterpret_cast<uintptr_t>(q) & 15u) || (reinterpret_cast<uintptr_t>(pools->slot_pool) & 15u) ||  // null passes
      (reinterpret_cast<uintptr_t>(pools->raw_pool) & 15u) || (reinterpret_cast<uintptr_t>(base3) & 15u) ||
      (reinterpret_cast<uintptr_t>(base4) & 15u) || (reinterpret_cast<uintptr_t>(workspace) & 15u) ||
      (reinterpret_cast<uintptr_t>(out) & 3u))
    return GAAC_EINVAL;
  constexpr int KH = 1;  // 256-channel heads: the two CTAs of a head form a cluster and share the scores
  const int nkv = NH * n_kv_heads;  // CTAs per (sequence, split) and half-heads in the table
  static_assert(!RAW || NH == 1, "the BF16 kernel serves 128-channel heads");
  if (!prepare_kernel<NH, KH, RAW>()) return GAAC_ECUDA;
  if (n_splits <= 0) {
    n_splits = gaac_attention_auto_splits(batch, nkv, max_blocks);
    if (NH > KH) {  // one wave of resident clusters
      const long long per_split = static_cast<long long>(batch) * n_kv_heads;
      const int mc = pair_max_clusters<NH, KH>();
      if (mc > 0 && per_split * n_splits > mc) n_splits = static_cast<int>(max(1ll, mc / per_split));
    }
  }
  if (n_splits > max_blocks) n_splits = max_blocks;
  if (workspace_bytes < gaac_attention_workspace(batch, nkv, max_blocks, n_splits)) return GAAC_EINVAL;
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
  // Scores are (q * qmul) . k; weights 2^((s - m) * c_log2) = e^(scale (q.k - max q.k)).  The sign of
  // the scale goes into q (exactly), so the running maxima are maxima of the logits for either sign.
  a.qmul = scale > 0.f ? 0.0625f : (scale < 0.f ? -0.0625f : 0.f);
  a.c_log2 = scale != 0.f ? static_cast<float>(std::fabs(static_cast<double>(scale)) * 16.0 * 1.4426950408889634) : 1.f;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.r = n_q_heads / n_kv_heads;
  a.max_blocks = max_blocks;
  a.n_splits = n_splits;
  a.counters = static_cast<unsigned int*>(workspace);
  a.part = reinterpret_cast<float*>(static_cast<char*>(workspace) + counters_bytes(batch, nkv));
  a.out = out;
  a.status = d_status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (clear_counters &&
      cudaMemsetAsync(a.counters, 0, static_cast<size_t>(batch) * nkv * sizeof(unsigned int), st) != cudaSuccess)
    return GAAC_ECUDA;
  if (NH > KH) {
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pair_config<NH, KH>(dim3(n_splits, nkv, batch), st, attr);
    if (cudaLaunchKernelEx(&cfg, attn_split_kernel<NH, KH, false>, a) != cudaSuccess) return GAAC_ECUDA;
  } else {
    // Programmatic dependent launch: the grid is set up while the previous kernel on the stream drains.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_splits, nkv, batch);
    cfg.blockDim = dim3(kAttThreads, 1, 1);
    cfg.dynamicSmemBytes = sizeof(AttSmem<NH, KH>);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, attn_split_kernel<NH, KH, RAW>, a) != cudaSuccess) return GAAC_ECUDA;
  }
  return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}

extern "C" int gaac_decode_attention(const uint16_t* q, int batch, int n_q_heads, int n_kv_heads, int max_blocks,
                                     const int32_t* seq_lens, const gaac_entry* table, const gaac_pools* pools,
                                     const uint8_t* base3, const uint8_t* base4, float scale, int n_splits,
                                     float* out, void* workspace, size_t workspace_bytes, int32_t* d_status,
                                     void* stream) {
  return launch_attention<1>(q, batch, n_q_heads, n_kv_heads, max_blocks, seq_lens, table, pools, base3, base4, scale,
                             n_splits, out, workspace, workspace_bytes, d_status, stream);
}

extern "C" int gaac_decode_attention_bf16(const uint16_t* q, int batch, int n_q_heads, int n_kv_heads,
                                          int max_blocks, const int32_t* seq_lens, const gaac_entry* table,
                                          const gaac_pools* pools, float scale, int n_splits, float* out,
                                          void* workspace, size_t workspace_bytes, int32_t* d_status, void* stream) {
  // The BF16 kernel reads no bases; any aligned non-null pointer satisfies the shared checks.
  const uint8_t* unused = reinterpret_cast<const uint8_t*>(pools ? pools->raw_pool : nullptr);
  return launch_attention<1, true>(q, batch, n_q_heads, n_kv_heads, max_blocks, seq_lens, table, pools, unused,
                                   unused, scale, n_splits, out, workspace, workspace_bytes, d_status, stream);
}

extern "C" int gaac_decode_attention_hd256(const uint16_t* q, int batch, int n_q_heads, int n_kv_heads,
                                           int max_blocks, const int32_t* seq_lens, const gaac_entry* table,
                                           const gaac_pools* pools, const uint8_t* base3, const uint8_t* base4,
                                           float scale, int n_splits, float* out, void* workspace,
                                           size_t workspace_bytes, int32_t* d_status, void* stream) {
  return launch_attention<2>(q, batch, n_q_heads, n_kv_heads, max_blocks, seq_lens, table, pools, base3, base4, scale,
                             n_splits, out, workspace, workspace_bytes, d_status, stream);
}

#ifdef GAAC_TIMELINE
// Copies the per-CTA timeline of the last attention launch (CTA id = x + X (y + Y z)) to host memory.
extern "C" GAAC_API int gaac_timeline_fetch(void* host_dst, size_t bytes, size_t* cta_bytes, int* n_ctas,
                                            int* n_blocks) {
  if (cta_bytes) *cta_bytes = sizeof(TlCta);
  if (n_ctas) *n_ctas = kTlCtas;
  if (n_blocks) *n_blocks = kTlBlocks;
  if (host_dst == nullptr) return GAAC_OK;
  if (bytes > sizeof(g_timeline)) bytes = sizeof(g_timeline);
  return cudaMemcpyFromSymbol(host_dst, g_timeline, bytes) == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}
#endif

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
  // The merge counters must start at zero: every call clears the ones it uses (after its argument
  // checks, so a rejected call leaves the array untouched) and never depends on how an earlier call ended.
  return launch_attention<1>(q, batch, n_q_heads, n_kv_heads, max_blocks, seq_lens, table, pools, base3, base4,
                             scale, ns, out, scratch, kStaticScratchBytes, d_status, stream, true);
}
