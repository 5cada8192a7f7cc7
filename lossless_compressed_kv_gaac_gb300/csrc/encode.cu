// Block encoder (prefill), O(1) appender and seal of the GAAC cache.
//
// "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference on
// Personal Devices":
//  - section 3.1: per-channel base-plus-offset exponent codes; a group of eight
//    takes the 3-bit mode if every offset from base3 fits [0,7], else the 4-bit
//    mode if every offset from base4 fits [0,15], else the raw mode; sign and
//    mantissa are stored unchanged;
//  - section 3.3 / Figure 3: complete blocks are encoded once into
//    fixed-capacity slots, oversized blocks stay BF16, the incomplete tail is a
//    BF16 block that is encoded when it fills ("fill-then-finalize").  With
//    GAAC_OPEN_COMPRESSED the open block is kept in its slot instead, and an
//    append re-encodes only the groups that gain the new token.
//
// One CTA of 256 threads encodes one tile; thread u owns the 32-element code
// unit u (storage elements 32u..32u+31), i.e. exactly one tag byte and one
// word of each code plane.  Tile layout: format v3 (gaac.h).
#include <cuda_runtime.h>

#include "common.cuh"

namespace gaac {

constexpr int kEncThreads = 256;

// Shared state of one tile's encode (every encoder kernel).
struct EncCommon {
  uint32_t vtab[2][16][8];  // base3 / base4 words of the unit classes (V: 16, K: 4)
  int warp_sums[kEncThreads / 32];
  int mode_counts[4];
  uint32_t raw_idx;
  int ok;
};

// One tile staged in storage order (the appender and the tile-batch encoder).
struct EncShared : EncCommon {
  alignas(16) uint16_t tile[kTile];
};

// The block encoder: the tile token-major with padded rows (filled by
// asynchronous copies); a V tile is then rearranged into storage order in place.
struct EncBlockShared : EncCommon {
  alignas(16) uint16_t raw[kLogicalElems];
};

// Token of storage element s (format v3).
__device__ __forceinline__ int token_of(int kind, int s) { return kind == 0 ? (s >> 7) : v_token_of(s); }

// V staging: thread tid takes token t, channels 32p .. 32p+31.  Storage
// elements 2m and 2m+1 are channels c and c+8 of one token, so the thread
// stores each such pair as one word; this assignment puts a warp's 32 stores
// of an instruction in 16 distinct banks.
__device__ __forceinline__ void v_pair_slice(int tid, int& t, int& p) {
  const int l = tid & 31, w = tid >> 5;
  t = (l & 1) | (((l >> 3) & 1) << 1) | (((l >> 4) & 1) << 2) | (((l >> 1) & 1) << 3) | ((w & 3) << 4);
  p = ((l >> 2) & 1) | (((w >> 2) & 1) << 1);
}

// 16-byte chunk positions of the block encoder's staged tile.  A unit's four
// chunks are read by one thread, a warp's 8 threads of one shared-memory
// phase taking 8 consecutive units; XOR-ing each unit's chunk index with a
// function of the unit puts those 8 reads in 8 distinct bank groups.
//  V (storage order, 64-byte units): chunk j of unit u lies at j ^ ((u >> 1) & 3).
//  K (token-major rows of kLogicalStride): chunk c of a row (channels 8c ..
//    8c+7) lies at c ^ ((c >> 2) & 2), i.e. unit u's chunk j at j ^ (u & 2).
//    (A V tile's token-major rows, read once by the rearrangement, stay plain.)
__device__ __forceinline__ int v_chunk_swz(int u) { return (u >> 1) & 3; }
__device__ __forceinline__ int k_chunk_swz(int u) { return u & 2; }
__device__ __forceinline__ int k_row_chunk(int c) { return c ^ ((c >> 2) & 2); }

// Stores channels 32p .. 32p+31 of token t (x[i] = channels 32p + 8i .. + 7) into a V tile in storage order
// (kSwz: with the block encoder's chunk swizzle).
template <bool kSwz = false>
__device__ __forceinline__ void store_v_pairs(uint16_t* tile, int t, int p, const uint4 x[4]) {
  // word index of storage element v_storage_index(t, 32p + 16m + j) / 2 = base + 64j + 4m (j < 8)
  const int base = 1024 * (t >> 4) + 512 * (p >> 1) + 16 * ((t >> 1) & 3) + 8 * (p & 1) + (t & 1) + 2 * ((t >> 3) & 1);
  // Bit 2 of base is clear and base + 4m stays below the next multiple of 32, so base + 4m = base ^ 4m; the
  // offsets 128i leave bits 0-6 alone.  The swizzle reads unit bits 5-6, the same for every m and i, so it
  // is one XOR on base (words 64j, j even) and one on base + 64 (j odd).
  const int e0 = kSwz ? base ^ (v_chunk_swz(base >> 4) << 2) : base;
  const int e1 = kSwz ? (base + 64) ^ (v_chunk_swz((base + 64) >> 4) << 2) : base + 64;
  uint32_t* tw = reinterpret_cast<uint32_t*>(tile);
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const uint32_t aw[4] = {x[2 * m].x, x[2 * m].y, x[2 * m].z, x[2 * m].w};                  // channels c
    const uint32_t bw[4] = {x[2 * m + 1].x, x[2 * m + 1].y, x[2 * m + 1].z, x[2 * m + 1].w};  // c + 8
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      tw[(e0 ^ (4 * m)) + 128 * i] = __byte_perm(aw[i], bw[i], 0x5410);
      tw[(e1 ^ (4 * m)) + 128 * i] = __byte_perm(aw[i], bw[i], 0x7632);
    }
  }
}

// Stages tokens [0, nv) of a tile (token t's 128 channels at src + t * tok_stride,
// 16-byte aligned) into `tile` in storage order; tokens past nv are zero.
//  K (token-major storage): 16-byte chunk q = tid + 256i is token q / 16,
//    channels 8(q % 16) .. +7, so a warp's loads and stores are contiguous.
//  V: v_pair_slice / store_v_pairs.
__device__ __forceinline__ void stage_tile_enc(uint16_t* tile, const uint16_t* src, int64_t tok_stride, int nv,
                                               int kind, int tid) {
  if (kind == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int q = tid + kEncThreads * i, t = q >> 4, col = 8 * (q & 15);
      uint4 x = make_uint4(0, 0, 0, 0);
      if (t < nv) x = *reinterpret_cast<const uint4*>(src + t * tok_stride + col);
      *reinterpret_cast<uint4*>(tile + t * kD + col) = x;
    }
    return;
  }
  int t, p;
  v_pair_slice(tid, t, p);
  uint4 x[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) x[i] = make_uint4(0, 0, 0, 0);
  if (t < nv) {
    const uint4* g = reinterpret_cast<const uint4*>(src + t * tok_stride + 32 * p);
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = g[i];
  }
  store_v_pairs(tile, t, p, x);
}

// Exponent bytes of four BF16 values (w0 = elements 0, 1; w1 = elements 2, 3):
// byte L = exponent of element L.  Shifting a word of two BF16 values right by
// 7 puts their exponents in bytes 0 and 2.
__device__ __forceinline__ uint32_t exponent_word(uint32_t w0, uint32_t w1) {
  return __byte_perm(w0 >> 7, w1 >> 7, 0x6420);
}

// The escape byte of a 4-bit group from its two words of 4-bit offsets: bit L
// (bit 4 + L) = bit 3 of byte L of d4a (d4b).  Multiplying the four masked bits
// 3 + 8L by 2^25 + 2^18 + 2^11 + 2^4 lands bit L at 28 + L; every other product
// term stays below bit 24 or leaves the word, so nothing carries into 24..31.
__device__ __forceinline__ uint32_t escape_byte(uint32_t d4a, uint32_t d4b) {
  return (((d4a & 0x08080808u) * 0x02040810u) >> 28) | (((d4b & 0x08080808u) * 0x02040810u) >> 24);
}

// The group loop element by element (open tiles, whose absent elements take no
// part; bases outside the calibrated ranges).  Rare, so kept out of line: the
// word-wide loop then gets the registers.
struct UnitCodes {
  uint32_t W[3], esc4, tagbyte, counts;
  int n4, nraw;
};

template <bool kOpen>
__device__ __noinline__ void encode_groups_elementwise(const uint16_t* unit, int kind, int u, const EncCommon* sh,
                                                       int cls, int n_present, int sw, UnitCodes* out) {
  const uint4* src = reinterpret_cast<const uint4*>(unit);
  uint32_t W[3] = {0, 0, 0};
  uint32_t esc4 = 0, tagbyte = 0, counts = 0;
  int n4 = 0, nraw = 0;
#pragma unroll
  for (int gi = 0; gi < 4; ++gi) {
    int e[8], b3[8], b4[8];
    bool pres[8];
    bool fits3 = true, fits4 = true;
    const uint4 gq = src[gi ^ sw];  // the group's 8 values
    const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
    const uint32_t b3q[2] = {sh->vtab[0][cls][2 * gi], sh->vtab[0][cls][2 * gi + 1]};  // four bases per word
    const uint32_t b4q[2] = {sh->vtab[1][cls][2 * gi], sh->vtab[1][cls][2 * gi + 1]};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int el = 8 * gi + j;
      pres[j] = !kOpen || token_of(kind, 32 * u + el) < n_present;
      const uint32_t x = (gw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
      e[j] = (x >> 7) & 0xFF;
      b3[j] = (b3q[j >> 2] >> (8 * (j & 3))) & 0xFFu;
      b4[j] = (b4q[j >> 2] >> (8 * (j & 3))) & 0xFFu;
      const int o3 = e[j] - b3[j], o4 = e[j] - b4[j];
      fits3 = fits3 && (!pres[j] || ((o3 >= 0) && (o3 <= 7)));
      fits4 = fits4 && (!pres[j] || ((o4 >= 0) && (o4 <= 15)));
    }
    const uint32_t mode = fits3 ? 0u : (fits4 ? 1u : 2u);
    tagbyte |= mode << (2 * gi);
    counts += mode == 0u ? 1u : (mode == 1u ? 0x10000u : 0u);
    uint32_t eb = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t cd = 0;  // raw groups keep code 0: their exponents are escape bytes
      if (!pres[j]) {
        // absent element: code and escape bit zero
      } else if (mode == 0u) {
        cd = static_cast<uint32_t>(e[j] - b3[j]) & 7u;
      } else if (mode == 1u) {
        const uint32_t off = static_cast<uint32_t>(e[j] - b4[j]) & 0xFFu;
        cd = off & 7u;
        eb |= ((off >> 3) & 1u) << j;
      }
      // format v3 placement: element 16h + 4q + L of the unit goes to byte lane L of W[h] (q = 0: bits
      // 0-2, q = 1: bits 3-5, q = 3: bits 6-7 with its third bit in W[2] bit 6+h) or of W[2] (q = 2: bits 3h..)
      const int h = gi >> 1, q = (8 * (gi & 1) + j) >> 2, L = j & 3;
      if (q == 0) W[h] |= cd << (8 * L);
      if (q == 1) W[h] |= cd << (8 * L + 3);
      if (q == 2) W[2] |= cd << (8 * L + 3 * h);
      if (q == 3) {
        W[h] |= (cd & 3u) << (8 * L + 6);
        W[2] |= ((cd >> 2) & 1u) << (8 * L + 6 + h);
      }
    }
    if (mode == 1u) {
      esc4 |= eb << (8 * n4);
      n4 += 1;
    }
    if (mode == 2u) nraw += 1;
  }
  out->W[0] = W[0];
  out->W[1] = W[1];
  out->W[2] = W[2];
  out->esc4 = esc4;
  out->tagbyte = tagbyte;
  out->counts = counts;
  out->n4 = n4;
  out->nraw = nraw;
}

// The per-CTA tables of encode_tile_cta: the base words of the unit classes
// (V: the 16 classes of v_unit_class; K: class u % 4, element 4k+L of unit u
// being channel 32(u%4) + 4k + L) and the statistics counter.  Returns whether
// one of this thread's bases lies outside the calibrated ranges (base3 <= 248,
// base4 <= 240), for which a word subtraction decides a group's fit exactly
// (the tile then takes the element-by-element path).  A barrier must follow
// before the tables are read.
__device__ __forceinline__ bool base_tables(EncCommon* sh, int kind, const uint8_t* __restrict__ b3g,
                                            const uint8_t* __restrict__ b4g, int u) {
  if (u == 0) sh->mode_counts[0] = 0;
  if (kind == 1) {
    fill_v_base_table(sh->vtab, b3g, b4g, u);
  } else if (u < 64) {
    const int which = u >> 5, c = (u >> 3) & 3, k = u & 7;
    sh->vtab[which][c][k] = *reinterpret_cast<const uint32_t*>((which ? b4g : b3g) + 32 * c + 4 * k);
  }
  bool odd_base = false;
  if (u < kD / 4) {
    const uint32_t w3 = reinterpret_cast<const uint32_t*>(b3g)[u], w4 = reinterpret_cast<const uint32_t*>(b4g)[u];
#pragma unroll
    for (int L = 0; L < 4; ++L) odd_base = odd_base || ((w3 >> (8 * L)) & 0xFFu) > 248u || ((w4 >> (8 * L)) & 0xFFu) > 240u;
  }
  return odd_base;
}

// Encodes a staged tile into `slot` (global, 16-byte aligned) unless its
// escape stream exceeds the capacity.  `unit`: this thread's 32 values (code
// unit u = threadIdx.x, storage elements 32u .. 32u+31; 16-byte aligned).  Returns the escape length, or -1 when
// the tile must stay raw (then nothing is written).  CTA-uniform result; all
// 256 threads must call it.
//
// n_present < 64 encodes an open tile (the incomplete last block of a
// prefill): elements of tokens >= n_present are absent (the staged tile must
// hold zero there); they take no part in their group's mode, and their codes and
// escape bits are zero.  kOpen = false compiles the sealed-tile encoder
// (n_present is then ignored: every token present).
//
// odd < 0: the routine builds the base tables itself (base_tables); odd = 0 or
// 1: the caller built them (and put a barrier after) and passes whether any
// base lies outside the calibrated ranges.
template <bool kOpen>
__device__ __noinline__ int encode_tile_cta(EncCommon* sh, const uint16_t* unit, int kind,
                                           const uint8_t* __restrict__ b3g, const uint8_t* __restrict__ b4g,
                                           uint8_t* __restrict__ slot, gaac_stats* stats, int n_present = kBlock,
                                           int odd = -1, int sw = 0) {
  const int u = threadIdx.x;
  const int lane = u & 31, warp = u >> 5;
  const uint4* src = reinterpret_cast<const uint4*>(unit);  // the unit's 32 values, 4 quads of 8
  const bool any_odd = odd >= 0 ? odd != 0 : __syncthreads_or(base_tables(sh, kind, b3g, b4g, u)) != 0;
  const bool word_fit = !kOpen && !any_odd;
  const int cls = kind == 0 ? (u & 3) : v_unit_class(u);

  uint32_t W[3] = {0, 0, 0};  // the unit's code-plane words, filled code by code
  uint32_t esc4 = 0;  // the unit's 4-bit escape bytes, little-endian, in group order
  int n4 = 0, nraw = 0;
  uint32_t tagbyte = 0;
  uint32_t counts = 0;  // 3-bit groups | 4-bit groups << 16 (raw: the rest of the tile's 1024)

  if (word_fit) {
    // Four elements per word: E = exponent bytes, D = E - base.  With every
    // base3 <= 248, a group fits the 3-bit mode iff no byte of E - base3 (either
    // word) has a bit above bit 2: when all bytes are in [0, 7] nothing
    // borrows, and the lowest byte that is out of range is exact modulo 256 and
    // lies in [8, 255] (a negative offset is at least -248).  Likewise 4 bits
    // with base4 <= 240.  In a group that fits, D holds the offsets themselves.
#pragma unroll
    for (int gi = 0; gi < 4; ++gi) {
      const uint4 gq = src[gi ^ sw];  // the group's 8 values
      const uint32_t b3q[2] = {sh->vtab[0][cls][2 * gi], sh->vtab[0][cls][2 * gi + 1]};
      const uint32_t b4q[2] = {sh->vtab[1][cls][2 * gi], sh->vtab[1][cls][2 * gi + 1]};
      const uint32_t E0 = exponent_word(gq.x, gq.y), E1 = exponent_word(gq.z, gq.w);
      const uint32_t d3a = E0 - b3q[0], d3b = E1 - b3q[1], d4a = E0 - b4q[0], d4b = E1 - b4q[1];
      const bool fits3 = ((d3a | d3b) & 0xF8F8F8F8u) == 0u, fits4 = ((d4a | d4b) & 0xF0F0F0F0u) == 0u;
      const uint32_t mode = fits3 ? 0u : (fits4 ? 1u : 2u);
      tagbyte |= mode << (2 * gi);
      counts += mode == 0u ? 1u : (mode == 1u ? 0x10000u : 0u);
      // codes: the offsets (3-bit), their low three bits (4-bit), zero (raw)
      const uint32_t c0 = fits3 ? d3a : (fits4 ? (d4a & 0x07070707u) : 0u);
      const uint32_t c1 = fits3 ? d3b : (fits4 ? (d4b & 0x07070707u) : 0u);
      // format v3 placement (word k = 2gi, 2gi+1 is q = k % 4 of half h = gi / 2): q = 0 in bits 0-2 and
      // q = 1 in bits 3-5 of W[h]; q = 2 in bits 3h.. of W[2]; q = 3 in bits 6-7 of W[h], third bit in W[2]
      // bit 6+h (every byte lane L the element 4q+L of the half)
      const int h = gi >> 1;
      if ((gi & 1) == 0) {
        W[h] |= c0 | (c1 << 3);
      } else {
        W[2] |= (c0 << (3 * h)) | ((c1 & 0x04040404u) << (4 + h));
        W[h] |= (c1 & 0x03030303u) << 6;
      }
      if (mode == 1u) {
        esc4 |= escape_byte(d4a, d4b) << (8 * n4);
        n4 += 1;
      }
      if (mode == 2u) nraw += 1;
    }
  } else {
    UnitCodes uc;
    encode_groups_elementwise<kOpen>(unit, kind, u, sh, cls, n_present, sw, &uc);
    W[0] = uc.W[0];
    W[1] = uc.W[1];
    W[2] = uc.W[2];
    esc4 = uc.esc4;
    tagbyte = uc.tagbyte;
    counts = uc.counts;
    n4 = uc.n4;
    nraw = uc.nraw;
  }

  // Exclusive scans over the CTA (unit order = group order) of the 4-bit and
  // raw group counts, packed in one word (each total is at most 1024).
  const int packed = n4 | (nraw << 16);
  int incl = packed;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) sh->warp_sums[warp] = incl;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kEncThreads / 32; ++w) {
    const int s = sh->warp_sums[w];
    if (w < warp) before += s;
    total += s;
  }
  const int excl = before + incl - packed;
  const int off4 = excl & 0xFFFF, offraw = excl >> 16;
  const int tot4 = total & 0xFFFF, totraw = total >> 16;
  const int esc = tot4 + 8 * totraw;
  if (esc > kEscCap || slot == nullptr) return -1;

  // Sign|mantissa plane: each byte keeps its mantissa and takes the sign of the
  // previous element of its aligned group of four (cyclically).
  uint32_t smb[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {  // word j: elements 4j..4j+3 from two staged words
    const uint4 gq = src[(j >> 1) ^ sw];
    const uint32_t w0 = (j & 1) ? gq.z : gq.x, w1 = (j & 1) ? gq.w : gq.y;
    // byte L: the mantissa (low byte, bits 0-6) of element L and the sign (high byte, bit 7) of element (L+3)%4
    // mantissas from the low bytes of the four values (bytes 0, 2 of each word); the sign bytes (high bytes
    // 1, 3) of elements 3, 0, 1, 2 into bytes 0-3
    smb[j] = (__byte_perm(w0, w1, 0x6420) & 0x7F7F7F7Fu) | (__byte_perm(w0, w1, 0x5317) & 0x80808080u);
  }
  uint4* smdst = reinterpret_cast<uint4*>(slot + 32 * u);
  smdst[0] = make_uint4(smb[0], smb[1], smb[2], smb[3]);
  smdst[1] = make_uint4(smb[4], smb[5], smb[6], smb[7]);
  uint32_t* cw = reinterpret_cast<uint32_t*>(slot + kOffCode);
  cw[u] = W[0];
  cw[256 + u] = W[1];
  cw[512 + u] = W[2];
  slot[kOffTag + u] = static_cast<uint8_t>(tagbyte);
  uint8_t* escp = slot + kOffEsc;
  for (int k = 0; k < n4; ++k) escp[off4 + k] = static_cast<uint8_t>(esc4 >> (8 * k));
  if (nraw) {  // raw groups: their eight exponents, after all 4-bit escape bytes of the tile
    int r = tot4 + 8 * offraw;
#pragma unroll
    for (int gi = 0; gi < 4; ++gi) {
      if (((tagbyte >> (2 * gi)) & 3u) != 2u) continue;
#pragma unroll
      for (int j = 0; j < 8; ++j)  // the exponent of element 8gi + j (zero where absent)
        escp[r + j] = static_cast<uint8_t>(unit[8 * (gi ^ sw) + j] >> 7);
      r += 8;
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int at = 2 * u + i;  // 0..511
    if (at >= esc && at < kEscCap) escp[at] = 0;
  }
  if ((u & (kDirUnits - 1)) == kDirUnits - 1) {  // directory entry of eighth u / 32
    const int w = u / kDirUnits;
    const uint32_t entry = ((off4 + n4) & 0x1FF) | (((offraw + nraw) & 0x7F) << 9);
    slot[kOffDir + 2 * w] = static_cast<uint8_t>(entry & 0xFFu);
    slot[kOffDir + 2 * w + 1] = static_cast<uint8_t>(entry >> 8);
  }
  if (stats != nullptr) {  // a sealed tile: all 1024 groups counted
    const uint32_t warp_counts = __reduce_add_sync(0xFFFFFFFFu, counts);
    if (lane == 0) atomicAdd(reinterpret_cast<unsigned int*>(&sh->mode_counts[0]), warp_counts);
    __syncthreads();
    if (u == 0) {
      const uint32_t c = static_cast<uint32_t>(sh->mode_counts[0]);
      const unsigned long long n3 = c & 0xFFFFu, n4g = c >> 16;
      atomicAdd(&stats->groups[0], n3);
      atomicAdd(&stats->groups[1], n4g);
      atomicAdd(&stats->groups[2], 1024ull - n3 - n4g);
      atomicAdd(&stats->escape_bytes, static_cast<unsigned long long>(esc));
      atomicAdd(&stats->slot_tiles, 1ull);
    }
  }
  return esc;
}

__device__ __forceinline__ gaac_entry make_entry(uint32_t index, int esc, int mode, int n_tok) {
  gaac_entry e;
  e.index = index;
  e.esc_len = static_cast<uint16_t>(esc);
  e.mode = static_cast<uint8_t>(mode);
  e.n_tok = static_cast<uint8_t>(n_tok);
  return e;
}

// Pops one raw tile index from the free list; thread 0 only.  Returns false on exhaustion.
__device__ __forceinline__ bool pop_raw(const gaac_pools& pools, uint32_t* idx, int32_t* status) {
  const unsigned long long pos = atomicAdd(reinterpret_cast<unsigned int*>(pools.raw_cursor), 1u);
  if (static_cast<long long>(pos) >= pools.n_raw_free) {
    report(status, GAAC_EPOOL);
    return false;
  }
  const uint32_t v = pools.raw_free != nullptr ? pools.raw_free[pos] : static_cast<uint32_t>(pos);
  if (static_cast<long long>(v) >= pools.n_raw) {
    report(status, GAAC_EPOOL);
    return false;
  }
  *idx = v;
  return true;
}

struct EncodeArgs {
  const uint16_t* k;
  const uint16_t* v;
  int64_t seq_stride, tok_stride, n_tok;
  const int32_t* seq_lens;
  int n_kv_heads, max_blocks;
  const uint8_t* base3;
  const uint8_t* base4;
  gaac_entry* table;
  const uint32_t* slot_ids;
  gaac_pools pools;
  gaac_stats* stats;
  unsigned flags;
  int32_t* status;
};

// 16-byte asynchronous global -> shared copy; src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Work item (x, blk, b) of the block encoder, the CTA's grid coordinates: x =
// h*2 + kind, block blk of sequence b.  nv = tokens of the block present (0:
// the block is past the sequence; -1: the sequence length is invalid).
struct BlockItem {
  int b, blk, h, kind, nv;
};

__device__ __forceinline__ BlockItem block_item(const EncodeArgs& a, uint32_t x, uint32_t blk, uint32_t b) {
  BlockItem it;
  it.h = static_cast<int>(x >> 1);
  it.kind = static_cast<int>(x & 1u);
  it.blk = static_cast<int>(blk);
  it.b = static_cast<int>(b);
  const int len = a.seq_lens[it.b];
  if (len < 0 || len > a.max_blocks * kBlock || len > a.n_tok)
    it.nv = -1;
  else
    it.nv = max(0, min(kBlock, len - it.blk * kBlock));
  return it;
}

// Starts the copies of an item's tile into a token-major buffer with padded rows
// (tokens past the sequence are filled with zeros) as one commit group.
__device__ __forceinline__ void prefetch_block(const EncodeArgs& a, const BlockItem& it, uint16_t* buf, int tid) {
  if (it.nv > 0) {
    const uint16_t* src = (it.kind == 0 ? a.k : a.v) + static_cast<int64_t>(it.b) * a.seq_stride +
                          static_cast<int64_t>(it.blk) * kBlock * a.tok_stride + it.h * kD;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int q = tid + kEncThreads * j, t = q >> 4, col = 8 * (q & 15);
      const bool in = t < it.nv;
      const int at = it.kind == 0 ? k_row_chunk(q & 15) : (q & 15);  // K rows swizzled, V rows plain
      cp_async16(buf + t * kLogicalStride + 8 * at, in ? src + t * a.tok_stride + col : src, in ? 16u : 0u);
    }
  }
  cp_async_commit();
}

// Table entry of an item.
__device__ __forceinline__ size_t item_entry(const EncodeArgs& a, const BlockItem& it) {
  return ((static_cast<size_t>(it.b) * a.max_blocks + it.blk) * a.n_kv_heads + it.h) * 2 + it.kind;
}

// Whether an item is encoded into its slot (a full block, or the open last block kept in its slot).
__device__ __forceinline__ bool item_to_slot(const EncodeArgs& a, const BlockItem& it) {
  return it.nv > 0 && (it.nv == kBlock || (a.flags & GAAC_OPEN_COMPRESSED)) && a.slot_ids != nullptr;
}

// Encodes an item, staged in `buf`; all threads call it.  The base tables are
// built (any_odd: a base outside the calibrated ranges) and, for an item going
// to a slot, slot_id is its slot.
__device__ __forceinline__ void encode_block_item(const EncodeArgs& a, const BlockItem& it, EncBlockShared& sh,
                                                  const uint16_t* buf, int tid, size_t eidx, uint32_t slot_id,
                                                  bool any_odd) {
  if (it.nv <= 0) {
    if (tid == 0) {
      a.table[eidx] = make_entry(0, 0, GAAC_MODE_NONE, 0);
      if (it.nv < 0) report(a.status, GAAC_EINVAL);
    }
    return;
  }
  const int kind = it.kind, h = it.h, nv = it.nv;
  const uint16_t* unit;
  int sw;  // the unit's chunk swizzle
  if (kind == 1) {  // V: rearrange the token-major tile into storage order
    int t, p;
    v_pair_slice(tid, t, p);
    uint4 x[4];
    const uint4* row = reinterpret_cast<const uint4*>(buf + t * kLogicalStride + 32 * p);
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = row[j];
    __syncthreads();  // every thread holds its slice: the buffer takes storage order in place
    store_v_pairs<true>(sh.raw, t, p, x);
    __syncthreads();
    unit = sh.raw + 32 * tid;
    sw = v_chunk_swz(tid);
  } else {  // K: storage order is token-major; unit u = token u/4, channels 32(u%4) .. +31
    unit = buf + (tid >> 2) * kLogicalStride + 32 * (tid & 3);
    sw = k_chunk_swz(tid);
  }
  const uint8_t* b3 = a.base3 + (kind * a.n_kv_heads + h) * kD;
  const uint8_t* b4 = a.base4 + (kind * a.n_kv_heads + h) * kD;
  if (item_to_slot(a, it)) {
    uint8_t* slot = nullptr;
    if (static_cast<int64_t>(slot_id) < a.pools.n_slots) {
      slot = a.pools.slot_pool + static_cast<size_t>(slot_id) * kSlot;
    } else if (tid == 0) {
      report(a.status, GAAC_EPOOL);
    }
    const int esc = nv == kBlock ? encode_tile_cta<false>(&sh, unit, kind, b3, b4, slot, a.stats, kBlock, any_odd, sw)
                                 : encode_tile_cta<true>(&sh, unit, kind, b3, b4, slot, nullptr, nv, any_odd, sw);
    if (esc >= 0) {
      if (tid == 0) a.table[eidx] = make_entry(slot_id, esc, GAAC_MODE_SLOT, nv);
      return;
    }
  }
  // Raw tile (storage order): overflow fallback of a full block, or the open tail.
  if (tid == 0) {
    uint32_t idx = 0;
    sh.ok = pop_raw(a.pools, &idx, a.status) ? 1 : 0;
    sh.raw_idx = idx;
  }
  __syncthreads();
  if (!sh.ok) {
    if (tid == 0) a.table[eidx] = make_entry(0, 0, GAAC_MODE_NONE, 0);
    return;
  }
  uint4* dst = reinterpret_cast<uint4*>(a.pools.raw_pool + static_cast<size_t>(sh.raw_idx) * kTile);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int q = tid + kEncThreads * j;  // 16-byte chunk q: storage elements 8q .. 8q+7
    const uint16_t* from = kind == 1 ? buf + 8 * (q ^ v_chunk_swz(q >> 2))
                                     : buf + (q >> 4) * kLogicalStride + 8 * k_row_chunk(q & 15);
    dst[q] = *reinterpret_cast<const uint4*>(from);
  }
  if (tid == 0) {
    a.table[eidx] = make_entry(sh.raw_idx, 0, GAAC_MODE_RAW, nv);
    if (a.stats != nullptr && a.slot_ids != nullptr)
      atomicAdd(nv == kBlock ? &a.stats->raw_tiles : &a.stats->tail_tiles, 1ull);
  }
}

// One CTA per item.  (A persistent variant that copied the next item's tile
// while encoding the current one was slower: the scheduler already overlaps
// the copies of some CTAs with the encoding of others.)
__global__ void __launch_bounds__(kEncThreads, 7) encode_blocks_kernel(EncodeArgs a) {
  extern __shared__ __align__(16) uint8_t enc_smem[];
  EncBlockShared& sh = *reinterpret_cast<EncBlockShared*>(enc_smem);
  const int tid = threadIdx.x;
  const BlockItem it = block_item(a, blockIdx.x, blockIdx.y, blockIdx.z);
  prefetch_block(a, it, sh.raw, tid);
  // while the copies land: the item's slot and the base tables of its (kind, head)
  const size_t eidx = item_entry(a, it);
  const uint32_t slot_id = item_to_slot(a, it) ? a.slot_ids[eidx] : 0u;
  const int row = (it.kind * a.n_kv_heads + it.h) * kD;
  const bool odd = base_tables(&sh, it.kind, a.base3 + row, a.base4 + row, tid);
  cp_async_wait<0>();
  const bool any_odd = __syncthreads_or(odd) != 0;
  encode_block_item(a, it, sh, sh.raw, tid, eidx, slot_id, any_odd);
}

// ------------------------------------------------ open block, one token --
//
// Adding token `pos` to an open slot changes only the groups that hold it:
// the 16 groups of that token (K: an eighth of the tile holds 8 tokens), or
// 64 groups of the V operand order, all inside the two eighths of the token's
// 16-token quarter.  One thread per group of the affected eighths rebuilds its
// group's present elements from the slot, adds the token's elements, and
// re-encodes the group; groups that do not hold the token keep their mode and
// move their escape bytes.  Earlier eighths keep their 4-bit escape bytes in
// place and their raw bytes shift with the new number of 4-bit bytes; later
// eighths hold no token yet (no escapes).  The result is the open image of
// the first pos + 1 tokens, byte for byte.

struct OpenShared {
  uint8_t esc_old[kEscCap + 16];
  uint8_t esc_new[kEscCap + 16];
  uint16_t tok[kD];  // the new token's 128 values
  int warp_old[kEncThreads / 32];
  int warp_new[kEncThreads / 32];
  int bad;
};

// Tokens of the 8 elements of group G (storage 8G..8G+7).
__device__ __forceinline__ int group_token(int kind, int G, int j) { return token_of(kind, 8 * G + j); }

// Base bytes of group G's 8 elements as two byte-lane words.
__device__ __forceinline__ void group_bases(int kind, int G, const uint8_t* bg, uint32_t& w0, uint32_t& w1) {
  if (kind == 0) {  // K: channels 8 (G % 16) .. + 7
    const uint2 v = *reinterpret_cast<const uint2*>(bg + 8 * (G & 15));
    w0 = v.x;
    w1 = v.y;
  } else {
    w0 = w1 = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      w0 |= static_cast<uint32_t>(bg[v_channel_of(8 * G + j)]) << (8 * j);
      w1 |= static_cast<uint32_t>(bg[v_channel_of(8 * G + 4 + j)]) << (8 * j);
    }
  }
}

__device__ __forceinline__ int block_excl_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int x = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += x;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < kEncThreads / 32; ++w) {
    const int x = warp_sums[w];
    if (w < warp) before += x;
    total += x;
  }
  return before + incl - v;
}

// Returns the new escape length (the slot updated), -1 if the escape stream
// would outgrow the slot (nothing written), or -2 if the open image fails its
// checks (nothing written).  All kEncThreads threads call it; os->tok holds
// the token.  esc_old: the entry's escape length.
__device__ int open_append_groups(OpenShared* os, uint8_t* slot, int kind, int pos, int esc_old,
                                  const uint8_t* __restrict__ b3g, const uint8_t* __restrict__ b4g, gaac_stats* stats) {
  const int tid = threadIdx.x;
  const int nA = kind == 0 ? 128 : 256;                 // groups of the affected eighths
  const int A0 = kind == 0 ? (pos >> 3) : 2 * (pos >> 4);  // first affected eighth
  const int A1 = A0 + (kind == 0 ? 0 : 1);
  const uint16_t* dir = reinterpret_cast<const uint16_t*>(slot + kOffDir);
  const uint32_t d7 = dir[7], dprev = A0 ? dir[A0 - 1] : 0u;
  const int n4_old = d7 & 0x1FF, nraw_old = d7 >> 9;
  const int p4 = dprev & 0x1FF, praw = dprev >> 9;  // counts of the eighths before A0
  if (tid == 0) os->bad = 0;
  __syncthreads();
  if (tid == 0 && n4_old + 8 * nraw_old != esc_old) os->bad = 1;
  for (int b = tid; b < kEscCap + 16; b += kEncThreads) {
    os->esc_old[b] = b < esc_old ? slot[kOffEsc + b] : 0;
    os->esc_new[b] = 0;
  }
  const bool act = tid < nA;
  const int G = 128 * A0 + tid, u = G >> 2, gi = G & 3;
  uint32_t m_old = 0u;
  if (act) m_old = (slot[kOffTag + u] >> (2 * gi)) & 3u;
  if (act && m_old == 3u) os->bad = 1;
  __syncthreads();
  // old escape offsets of the affected groups
  int tot_old;
  const int ex_old = block_excl_scan(act ? ((m_old == 1u) | ((m_old == 2u) << 16)) : 0, os->warp_old, tot_old);
  const int o4_old = p4 + (ex_old & 0xFFFF);
  const int oraw_old = n4_old + 8 * (praw + (ex_old >> 16));
  // the group's tokens: does it hold token pos?
  bool touched = false;
#pragma unroll
  for (int j = 0; j < 8; ++j) touched = touched || (act && group_token(kind, G, j) == pos);
  uint32_t m_new = m_old;
  uint32_t smw[2] = {0u, 0u}, C[2] = {0u, 0u}, ew[2] = {0u, 0u}, esc4 = 0u;
  if (act && m_old == 1u) esc4 = o4_old < kEscCap ? os->esc_old[o4_old] : 0u;
  if (act && m_old == 2u) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      ew[j >> 2] |= static_cast<uint32_t>(oraw_old + j < kEscCap ? os->esc_old[oraw_old + j] : 0u) << (8 * (j & 3));
  }
  if (touched) {
    uint32_t b3w[2], b4w[2];
    group_bases(kind, G, b3g, b3w[0], b3w[1]);
    group_bases(kind, G, b4g, b4w[0], b4w[1]);
    // old codes: words 2(gi & 1) and 2(gi & 1) + 1 of the half's extraction
    const uint32_t* cw = reinterpret_cast<const uint32_t*>(slot + kOffCode);
    const int h = gi >> 1;
    uint32_t c[4];
    extract_codes(h ? cw[256 + u] : cw[u], cw[512 + u], h, c);
    const uint32_t c0 = c[2 * (gi & 1)], c1 = c[2 * (gi & 1) + 1];
    // old exponents (valid where an element was present)
    uint32_t eo[2];
    if (m_old == 0u) {
      eo[0] = b3w[0] + c0;
      eo[1] = b3w[1] + c1;
    } else if (m_old == 1u) {
      eo[0] = b4w[0] + (c0 | (spread4(esc4 & 15u) << 3));
      eo[1] = b4w[1] + (c1 | (spread4(esc4 >> 4) << 3));
    } else {
      eo[0] = ew[0];
      eo[1] = ew[1];
    }
    // old sign|mantissa bytes, signs back in their own bytes
    const uint2 sraw = *reinterpret_cast<const uint2*>(slot + 8 * G);
    uint32_t so[2] = {sraw.x, sraw.y};
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t sg = so[q] & 0x80808080u;
      so[q] = (so[q] & 0x7F7F7F7Fu) | ((sg >> 8) | (sg << 24));
    }
    // present elements after the append: old ones and the token's
    uint32_t e[2] = {0u, 0u}, sm[2] = {0u, 0u};
    bool f3 = true, f4 = true;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = group_token(kind, G, j), q = j >> 2, sh8 = 8 * (j & 3);
      uint32_t ej = 0u, sj = 0u;
      if (t < pos) {
        ej = (eo[q] >> sh8) & 0xFFu;
        sj = (so[q] >> sh8) & 0xFFu;
      } else if (t == pos) {
        const int ch = kind == 0 ? ((8 * G + j) & (kD - 1)) : v_channel_of(8 * G + j);
        const uint32_t x = os->tok[ch];
        ej = (x >> 7) & 0xFFu;
        sj = ((x >> 8) & 0x80u) | (x & 0x7Fu);
      }
      e[q] |= ej << sh8;
      sm[q] |= sj << sh8;
      if (t <= pos) {
        const int o3 = static_cast<int>(ej) - static_cast<int>((b3w[q] >> sh8) & 0xFFu);
        const int o4 = static_cast<int>(ej) - static_cast<int>((b4w[q] >> sh8) & 0xFFu);
        f3 = f3 && o3 >= 0 && o3 <= 7;
        f4 = f4 && o4 >= 0 && o4 <= 15;
      }
    }
    m_new = f3 ? 0u : (f4 ? 1u : 2u);
    // codes (byte lanes: C[0] elements 0-3, C[1] elements 4-7), escape byte, raw exponents
    esc4 = 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = group_token(kind, G, j), q = j >> 2, sh8 = 8 * (j & 3);
      if (t > pos) continue;  // absent: code and escape bit zero
      const uint32_t ej = (e[q] >> sh8) & 0xFFu;
      uint32_t cd = 0u;
      if (m_new == 0u) {
        cd = (ej - ((b3w[q] >> sh8) & 0xFFu)) & 7u;
      } else if (m_new == 1u) {
        const uint32_t off = (ej - ((b4w[q] >> sh8) & 0xFFu)) & 0xFFu;
        cd = off & 7u;
        esc4 |= ((off >> 3) & 1u) << j;
      }
      C[q] |= cd << sh8;
    }
    ew[0] = m_new == 2u ? e[0] : 0u;
    ew[1] = m_new == 2u ? e[1] : 0u;
#pragma unroll
    for (int q = 0; q < 2; ++q) {  // signs rotated one byte within each aligned group of four
      const uint32_t sg = sm[q] & 0x80808080u;
      smw[q] = (sm[q] & 0x7F7F7F7Fu) | ((sg << 8) | (sg >> 24));
    }
  }
  // new escape offsets
  int tot_new;
  const int ex_new = block_excl_scan(act ? ((m_new == 1u) | ((m_new == 2u) << 16)) : 0, os->warp_new, tot_new);
  const int n4_new = p4 + (tot_new & 0xFFFF);  // no 4-bit groups after the affected eighths
  const int nraw_new = praw + (tot_new >> 16);
  const int esc_new = n4_new + 8 * nraw_new;
  if (os->bad) return -2;
  if (esc_new > kEscCap) return -1;
  // the new escape area in shared memory: earlier 4-bit bytes in place, earlier raw bytes shifted, then
  // the affected groups' bytes at their new offsets
  for (int b = tid; b < kEscCap; b += kEncThreads) {
    if (b < p4)
      os->esc_new[b] = os->esc_old[b];
    else if (b >= n4_new && b < n4_new + 8 * praw)
      os->esc_new[b] = os->esc_old[b - n4_new + n4_old];
  }
  if (act && m_new == 1u) os->esc_new[p4 + (ex_new & 0xFFFF)] = static_cast<uint8_t>(esc4);
  if (act && m_new == 2u) {
    const int at = n4_new + 8 * (praw + (ex_new >> 16));
#pragma unroll
    for (int j = 0; j < 8; ++j) os->esc_new[at + j] = static_cast<uint8_t>(ew[j >> 2] >> (8 * (j & 3)));
  }
  // touched groups: sign|mantissa bytes; touched units (all four groups touched): code words, tag byte
  if (touched) *reinterpret_cast<uint2*>(slot + 8 * G) = make_uint2(smw[0], smw[1]);
  const int h = gi >> 1;
  uint32_t wH = 0u, w2 = 0u;
  if (touched) {
    if ((gi & 1) == 0) {
      wH = C[0] | (C[1] << 3);
    } else {
      wH = (C[1] & 0x03030303u) << 6;
      w2 = (C[0] << (3 * h)) | (((C[1] >> 2) & 0x01010101u) << (6 + h));
    }
  }
  uint32_t tagbits = touched ? (m_new << (2 * gi)) : 0u;
  wH |= __shfl_xor_sync(0xFFFFFFFFu, wH, 1);  // groups 0+1 -> W0, groups 2+3 -> W1
  w2 |= __shfl_xor_sync(0xFFFFFFFFu, w2, 1);
  w2 |= __shfl_xor_sync(0xFFFFFFFFu, w2, 2);
  tagbits |= __shfl_xor_sync(0xFFFFFFFFu, tagbits, 1);
  tagbits |= __shfl_xor_sync(0xFFFFFFFFu, tagbits, 2);
  if (touched) {
    uint32_t* cw = reinterpret_cast<uint32_t*>(slot + kOffCode);
    if (gi == 0) {
      cw[u] = wH;
      cw[512 + u] = w2;
      slot[kOffTag + u] = static_cast<uint8_t>(tagbits);
    } else if (gi == 2) {
      cw[256 + u] = wH;
    }
  }
  // directory: the affected eighths' entries from the scan, later entries the totals
  if (act && (tid & 127) == 127) {
    const int w = A0 + (tid >> 7);
    const int incl = ex_new + ((m_new == 1u) | ((m_new == 2u) << 16));
    const uint32_t entry = static_cast<uint32_t>((p4 + (incl & 0xFFFF)) & 0x1FF) |
                           (static_cast<uint32_t>((praw + (incl >> 16)) & 0x7F) << 9);
    *reinterpret_cast<uint16_t*>(slot + kOffDir + 2 * w) = static_cast<uint16_t>(entry);
  }
  if (tid > A1 && tid < 8) {
    const uint32_t entry = static_cast<uint32_t>(n4_new & 0x1FF) | (static_cast<uint32_t>(nraw_new & 0x7F) << 9);
    *reinterpret_cast<uint16_t*>(slot + kOffDir + 2 * tid) = static_cast<uint16_t>(entry);
  }
  __syncthreads();
  for (int b = tid; b < kEscCap / 4; b += kEncThreads)
    reinterpret_cast<uint32_t*>(slot + kOffEsc)[b] = reinterpret_cast<const uint32_t*>(os->esc_new)[b];
  if (stats != nullptr) {  // the block seals: count its groups' modes
    __syncthreads();
    const uint32_t tb = slot[kOffTag + tid];
    const int c4 = n4_of(tb), cr = nraw_of(tb);
    int t4;
    block_excl_scan(c4 | (cr << 16), os->warp_old, t4);
    if (tid == 0) {
      const int n4 = t4 & 0xFFFF, nr = t4 >> 16;
      atomicAdd(&stats->groups[0], static_cast<unsigned long long>(1024 - n4 - nr));
      atomicAdd(&stats->groups[1], static_cast<unsigned long long>(n4));
      atomicAdd(&stats->groups[2], static_cast<unsigned long long>(nr));
      atomicAdd(&stats->escape_bytes, static_cast<unsigned long long>(esc_new));
      atomicAdd(&stats->slot_tiles, 1ull);
    }
  }
  return esc_new;
}

struct AppendArgs {
  const uint16_t* k_new;
  const uint16_t* v_new;
  int32_t* seq_lens;
  int n_kv_heads, max_blocks;
  const uint8_t* base3;
  const uint8_t* base4;
  gaac_entry* table;
  const uint32_t* slot_ids;
  gaac_pools pools;
  gaac_stats* stats;
  unsigned flags;
  int32_t* status;
  int bump;  // 1: the CTAs of a sequence form one cluster and its first CTA advances the length
};

// How one append reaches its block.
enum AppendPath { kFail = 0, kRawTail = 1, kRawFresh = 2, kOpenNew = 3, kOpenSlot = 4 };

// grid (2*n_kv_heads, batch): x = h*2 + kind.
__global__ void __launch_bounds__(kEncThreads) append_kernel(AppendArgs a) {
  __shared__ EncShared sh;
  __shared__ OpenShared os;
  __shared__ int word_prefix[65];
  __shared__ int esc_old;
  const int h = blockIdx.x >> 1, kind = blockIdx.x & 1, b = blockIdx.y;
  const int tid = threadIdx.x;
  // Launched as a programmatic dependent: wait for the previous kernel on the stream (and its memory)
  // before the first read, then let the length bump that follows be scheduled.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int len = a.seq_lens[b];
  if (a.bump) {
    // Every CTA of the sequence (one cluster) has read the length before the first one advances it.
    asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (blockIdx.x == 0 && tid == 0) a.seq_lens[b] = len + 1;
  }
  if (len < 0 || len >= a.max_blocks * kBlock) {
    if (tid == 0) report(a.status, GAAC_EINVAL);
    return;
  }
  const int blk = len / kBlock, pos = len % kBlock;
  const size_t eidx = ((static_cast<size_t>(b) * a.max_blocks + blk) * a.n_kv_heads + h) * 2 + kind;
  gaac_entry* ep = a.table + eidx;
  const bool open_c = (a.flags & GAAC_OPEN_COMPRESSED) != 0u;
  if (tid == 0) {
    const gaac_entry e = *ep;
    int path = kFail;
    uint32_t idx = 0;
    if (e.mode == GAAC_MODE_RAW) {  // a raw tail (from prefill, a hand-over or an overflow)
      if (e.n_tok == pos && static_cast<int64_t>(e.index) < a.pools.n_raw) {
        path = kRawTail;
        idx = e.index;
      } else {
        report(a.status, GAAC_EFORMAT);
      }
    } else if (pos == 0) {  // the block opens
      if (open_c) {
        idx = a.slot_ids[eidx];
        if (static_cast<int64_t>(idx) < a.pools.n_slots)
          path = kOpenNew;
        else
          report(a.status, GAAC_EPOOL);
      } else if (pop_raw(a.pools, &idx, a.status)) {
        path = kRawFresh;
      }
    } else if (open_c && e.mode == GAAC_MODE_SLOT && e.n_tok == pos &&
               static_cast<int64_t>(e.index) < a.pools.n_slots && e.esc_len <= kEscCap) {
      path = kOpenSlot;
      idx = e.index;
      esc_old = e.esc_len;
    } else {
      report(a.status, GAAC_EFORMAT);
    }
    sh.raw_idx = idx;
    sh.ok = path;
  }
  __syncthreads();
  const int path = sh.ok;
  if (path == kFail) return;
  const uint8_t* b3 = a.base3 + (kind * a.n_kv_heads + h) * kD;
  const uint8_t* b4 = a.base4 + (kind * a.n_kv_heads + h) * kD;
  const uint16_t x_new =
      tid < kD ? (kind == 0 ? a.k_new : a.v_new)[(static_cast<size_t>(b) * a.n_kv_heads + h) * kD + tid] : 0;
  const int s_new = kind == 0 ? pos * kD + tid : v_storage_index(pos, tid & (kD - 1));

  if (path >= kOpenNew) {
    // The open block lives in its slot: only the groups holding the new token
    // are rebuilt and re-encoded (open_append_groups).
    const uint32_t slot_id = sh.raw_idx;
    uint8_t* slot = a.pools.slot_pool + static_cast<size_t>(slot_id) * kSlot;
    if (tid < kD) os.tok[tid] = x_new;
    if (path == kOpenNew) {  // a fresh slot: every byte of the empty image is zero
      uint4* z = reinterpret_cast<uint4*>(slot);
      for (int i = tid; i < kSlot / 16; i += kEncThreads) z[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    const bool sealing = pos + 1 == kBlock;
    const int esc = open_append_groups(&os, slot, kind, pos, path == kOpenSlot ? esc_old : 0, b3, b4,
                                       sealing ? a.stats : nullptr);
    if (esc == -2) {
      if (tid == 0) report(a.status, GAAC_EFORMAT);
      return;
    }
    if (esc >= 0) {
      if (tid == 0) *ep = make_entry(slot_id, esc, GAAC_MODE_SLOT, pos + 1);
      return;
    }
    // The escape stream would outgrow the slot (it only grows as tokens
    // arrive, so the full block would not fit either; the slot is untouched):
    // the block continues as a raw tile holding its tokens so far.
    bool bad = false;
    uint4* mine = reinterpret_cast<uint4*>(sh.tile + 32 * tid);
    if (path == kOpenSlot) {
      if (tid < 32) slot_word_prefix(slot, tid, word_prefix);
      __syncthreads();
      uint32_t pairs[16];
      bad = decode_slot_unit(slot, kind, tid, b3, b4, esc_old, word_prefix, pairs);
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const int s0 = 32 * tid + 2 * m;
        const uint32_t lo = token_of(kind, s0) < pos ? (pairs[m] & 0xFFFFu) : 0u;
        const uint32_t hi = token_of(kind, s0 + 1) < pos ? (pairs[m] & 0xFFFF0000u) : 0u;
        pairs[m] = lo | hi;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) mine[i] = make_uint4(pairs[4 * i], pairs[4 * i + 1], pairs[4 * i + 2], pairs[4 * i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) mine[i] = make_uint4(0, 0, 0, 0);
    }
    if (__syncthreads_or(bad)) {
      if (tid == 0) report(a.status, GAAC_EFORMAT);
      return;
    }
    if (tid < kD) sh.tile[s_new] = x_new;
    if (tid == 0) {
      uint32_t idx = 0;
      sh.ok = pop_raw(a.pools, &idx, a.status) ? 1 : 0;
      sh.raw_idx = idx;
    }
    __syncthreads();
    if (!sh.ok) return;
    uint4* dst = reinterpret_cast<uint4*>(a.pools.raw_pool + static_cast<size_t>(sh.raw_idx) * kTile);
    const uint4* src = reinterpret_cast<const uint4*>(sh.tile);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[tid + kEncThreads * i] = src[tid + kEncThreads * i];
    if (tid == 0) {
      *ep = make_entry(sh.raw_idx, 0, GAAC_MODE_RAW, pos + 1);
      if (a.stats != nullptr) atomicAdd(sealing ? &a.stats->raw_tiles : &a.stats->tail_tiles, 1ull);
    }
    return;
  }

  // Raw tail: write the token in place; encode the block once when it fills.
  uint16_t* raw = a.pools.raw_pool + static_cast<size_t>(sh.raw_idx) * kTile;
  if (path == kRawFresh) {
    uint4* d = reinterpret_cast<uint4*>(raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[tid + kEncThreads * i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
  }
  if (tid < kD) raw[s_new] = x_new;
  if (pos + 1 < kBlock) {
    if (tid == 0) *ep = make_entry(sh.raw_idx, 0, GAAC_MODE_RAW, pos + 1);
    return;
  }
  // The block is full: seal it (encode once; it is never re-encoded).
  __syncthreads();
  {
    const uint4* src = reinterpret_cast<const uint4*>(raw);
    uint4* d = reinterpret_cast<uint4*>(sh.tile);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[tid + kEncThreads * i] = src[tid + kEncThreads * i];
  }
  __syncthreads();
  if (a.slot_ids == nullptr) {  // an all-raw cache: the full tail stays a raw tile
    if (tid == 0) {
      *ep = make_entry(sh.raw_idx, 0, GAAC_MODE_RAW, kBlock);
      if (a.stats != nullptr) atomicAdd(&a.stats->raw_tiles, 1ull);
    }
    return;
  }
  const uint32_t slot_id = a.slot_ids[eidx];
  uint8_t* slot = nullptr;
  if (static_cast<int64_t>(slot_id) < a.pools.n_slots) {
    slot = a.pools.slot_pool + static_cast<size_t>(slot_id) * kSlot;
  } else if (tid == 0) {
    report(a.status, GAAC_EPOOL);
  }
  const int esc = encode_tile_cta<false>(&sh, sh.tile + 32 * tid, kind, b3, b4, slot, a.stats);
  if (esc >= 0 && blk + 1 < a.max_blocks) {
    // The raw tile becomes the next block's empty tail: clear it so that a tail
    // always holds zeros past its last token.
    uint4* d = reinterpret_cast<uint4*>(raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[tid + kEncThreads * i] = make_uint4(0, 0, 0, 0);
  }
  if (tid == 0) {
    if (esc >= 0) {
      *ep = make_entry(slot_id, esc, GAAC_MODE_SLOT, kBlock);
      if (blk + 1 < a.max_blocks) ep[static_cast<size_t>(a.n_kv_heads) * 2] = make_entry(sh.raw_idx, 0, GAAC_MODE_RAW, 0);
    } else {
      *ep = make_entry(sh.raw_idx, 0, GAAC_MODE_RAW, kBlock);
      if (a.stats != nullptr) atomicAdd(&a.stats->raw_tiles, 1ull);
    }
  }
}

struct EncodeTilesArgs {
  const uint16_t* tiles;  // [n][64][128] BF16, token-major
  const uint8_t* kind;
  const int32_t* row;
  int n_rows;
  const uint8_t* base3;
  const uint8_t* base4;
  uint8_t* slots;
  uint16_t* esc_len;
  gaac_stats* stats;
  int32_t* status;
};

// grid (n_tiles): one CTA encodes one tile of the batch.
__global__ void __launch_bounds__(kEncThreads, 6) encode_tiles_kernel(EncodeTilesArgs a) {
  __shared__ EncShared sh;
  const int64_t i = blockIdx.x;
  const int tid = threadIdx.x;
  const int kind = a.kind[i], r = a.row[i];
  if (kind > 1 || r < 0 || r >= a.n_rows) {
    if (tid == 0) {
      a.esc_len[i] = 0xFFFFu;
      report(a.status, GAAC_EINVAL);
    }
    return;
  }
  stage_tile_enc(sh.tile, a.tiles + i * kTile, kD, kBlock, kind, tid);
  __syncthreads();
  const int esc = encode_tile_cta<false>(&sh, sh.tile + 32 * tid, kind, a.base3 + r * kD, a.base4 + r * kD,
                                         a.slots + i * kSlot, a.stats);
  if (tid == 0) a.esc_len[i] = esc >= 0 ? static_cast<uint16_t>(esc) : 0xFFFFu;
}

__global__ void bump_lens_kernel(int32_t* lens, int batch) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the append kernel has read every length
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < batch) lens[i] += 1;
}

// Whether clusters of n append CTAs (one sequence's tiles) can be launched on this device, cached per
// device and size; sizes above 8 need the non-portable cluster attribute.  The first question is not
// answered while `st` is being captured into a graph (the two-kernel form serves that call).
static bool append_cluster_ok(int n, cudaStream_t st) {
  if (n < 1 || n > 16) return false;
  static signed char cached[64][17] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (cached[dev][n] == 0) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
      cudaGetLastError();
      return false;
    }
    bool ok = n <= 8 || cudaFuncSetAttribute(append_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                            cudaSuccess;
    if (ok) {
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = n;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(n, 1);
      cfg.blockDim = dim3(kEncThreads);
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      ok = cudaOccupancyMaxActiveClusters(&clusters, append_kernel, &cfg) == cudaSuccess && clusters > 0;
    }
    cudaGetLastError();
    cached[dev][n] = ok ? 1 : -1;
  }
  return cached[dev][n] > 0;
}

}  // namespace gaac

using namespace gaac;

// Sets the block encoder's dynamic shared-memory size on the current device (once).
static bool prepare_encode_blocks() {
  static bool done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (!done[dev]) {
    if (cudaFuncSetAttribute(encode_blocks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(EncBlockShared))) != cudaSuccess)
      return false;
    done[dev] = true;
  }
  return true;
}

static bool pools_ok(const gaac_pools* p) {
  return p != nullptr && p->slot_pool != nullptr && p->raw_pool != nullptr && p->raw_cursor != nullptr &&
         p->n_slots >= 0 && p->n_raw >= 0 && p->n_raw_free >= 0 &&
         (reinterpret_cast<uintptr_t>(p->slot_pool) & 15u) == 0 && (reinterpret_cast<uintptr_t>(p->raw_pool) & 15u) == 0;
}

extern "C" int gaac_encode_blocks_ex(const uint16_t* k, const uint16_t* v, int64_t seq_stride, int64_t tok_stride,
                                     int64_t n_tok, const int32_t* seq_lens, int batch, int n_kv_heads,
                                     int max_blocks, const uint8_t* base3, const uint8_t* base4, gaac_entry* table,
                                     const uint32_t* slot_ids, const gaac_pools* pools, gaac_stats* stats,
                                     unsigned flags, int32_t* d_status, void* stream) {
  if (k == nullptr || v == nullptr || seq_lens == nullptr || base3 == nullptr || base4 == nullptr ||
      table == nullptr || !pools_ok(pools) || (flags & ~static_cast<unsigned>(GAAC_OPEN_COMPRESSED)))
    return GAAC_EINVAL;
  if (batch <= 0 || n_kv_heads <= 0 || max_blocks <= 0 || max_blocks > 65535 || batch > 65535 ||
      n_kv_heads > 1024)
    return GAAC_EINVAL;
  if (tok_stride < static_cast<int64_t>(n_kv_heads) * kD || (tok_stride & 7) || (seq_stride & 7) ||
      (reinterpret_cast<uintptr_t>(k) & 15u) || (reinterpret_cast<uintptr_t>(v) & 15u) ||
      (reinterpret_cast<uintptr_t>(base3) & 15u) || (reinterpret_cast<uintptr_t>(base4) & 15u))
    return GAAC_EINVAL;
  if (n_tok < 0) return GAAC_EINVAL;
  EncodeArgs a{k, v, seq_stride, tok_stride, n_tok, seq_lens, n_kv_heads, max_blocks, base3, base4, table, slot_ids,
               *pools, stats, flags, d_status};
  if (!prepare_encode_blocks()) return GAAC_ECUDA;
  // one CTA per (h*2 + kind, block, sequence): the argument checks above keep every dimension in range
  const dim3 grid(static_cast<unsigned>(2 * n_kv_heads), static_cast<unsigned>(max_blocks), static_cast<unsigned>(batch));
  encode_blocks_kernel<<<grid, kEncThreads, sizeof(EncBlockShared), static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}

extern "C" int gaac_encode_blocks(const uint16_t* k, const uint16_t* v, int64_t seq_stride, int64_t tok_stride,
                                  int64_t n_tok, const int32_t* seq_lens, int batch, int n_kv_heads, int max_blocks,
                                  const uint8_t* base3, const uint8_t* base4, gaac_entry* table,
                                  const uint32_t* slot_ids, const gaac_pools* pools, gaac_stats* stats,
                                  int32_t* d_status, void* stream) {
  return gaac_encode_blocks_ex(k, v, seq_stride, tok_stride, n_tok, seq_lens, batch, n_kv_heads, max_blocks, base3,
                               base4, table, slot_ids, pools, stats, 0u, d_status, stream);
}

extern "C" int gaac_append_ex(const uint16_t* k_new, const uint16_t* v_new, int32_t* seq_lens, int batch,
                              int n_kv_heads, int max_blocks, const uint8_t* base3, const uint8_t* base4,
                              gaac_entry* table, const uint32_t* slot_ids, const gaac_pools* pools,
                              gaac_stats* stats, unsigned flags, int32_t* d_status, void* stream) {
  if (k_new == nullptr || v_new == nullptr || seq_lens == nullptr || base3 == nullptr || base4 == nullptr ||
      table == nullptr || !pools_ok(pools) || (flags & ~static_cast<unsigned>(GAAC_OPEN_COMPRESSED)) ||
      (slot_ids == nullptr && (flags & GAAC_OPEN_COMPRESSED)))
    return GAAC_EINVAL;
  if (batch <= 0 || batch > 65535 || n_kv_heads <= 0 || n_kv_heads > 1024 || max_blocks <= 0) return GAAC_EINVAL;
  if ((reinterpret_cast<uintptr_t>(base3) & 15u) || (reinterpret_cast<uintptr_t>(base4) & 15u)) return GAAC_EINVAL;
  AppendArgs a{k_new, v_new, seq_lens, n_kv_heads, max_blocks, base3, base4, table, slot_ids, *pools,
               stats, flags, d_status, 0};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Programmatic dependents of their predecessor on the stream (each waits for it before any read): a
  // launch is set up while the previous kernel runs.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * n_kv_heads, batch);
  cfg.blockDim = dim3(kEncThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // One launch: the 2 * n_kv_heads CTAs of a sequence as one thread-block cluster, whose first CTA
  // advances the length once all have read it.  Otherwise (more than 16 CTAs per sequence, or clusters of
  // that size not schedulable) a second small kernel advances the lengths.
  if (append_cluster_ok(2 * n_kv_heads, st)) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2 * n_kv_heads;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
    a.bump = 1;
    if (cudaLaunchKernelEx(&cfg, append_kernel, a) != cudaSuccess) return GAAC_ECUDA;
    return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
  }
  if (cudaLaunchKernelEx(&cfg, append_kernel, a) != cudaSuccess) return GAAC_ECUDA;
  cfg.gridDim = dim3((batch + 255) / 256);
  cfg.blockDim = dim3(256);
  if (cudaLaunchKernelEx(&cfg, bump_lens_kernel, seq_lens, batch) != cudaSuccess) return GAAC_ECUDA;
  return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}

extern "C" int gaac_append(const uint16_t* k_new, const uint16_t* v_new, int32_t* seq_lens, int batch,
                           int n_kv_heads, int max_blocks, const uint8_t* base3, const uint8_t* base4,
                           gaac_entry* table, const uint32_t* slot_ids, const gaac_pools* pools,
                           gaac_stats* stats, int32_t* d_status, void* stream) {
  return gaac_append_ex(k_new, v_new, seq_lens, batch, n_kv_heads, max_blocks, base3, base4, table, slot_ids, pools,
                        stats, 0u, d_status, stream);
}

extern "C" int gaac_encode_tiles(const uint16_t* tiles, int64_t n_tiles, const uint8_t* tile_kind,
                                 const int32_t* tile_row, int n_rows, const uint8_t* base3, const uint8_t* base4,
                                 uint8_t* slots, uint16_t* esc_len, gaac_stats* stats, int32_t* d_status,
                                 void* stream) {
  if (tiles == nullptr || tile_kind == nullptr || tile_row == nullptr || base3 == nullptr || base4 == nullptr ||
      slots == nullptr || esc_len == nullptr || n_rows <= 0)
    return GAAC_EINVAL;
  if (n_tiles < 0 || n_tiles > 0x7FFFFFFF || (reinterpret_cast<uintptr_t>(tiles) & 15u) ||
      (reinterpret_cast<uintptr_t>(slots) & 15u) || (reinterpret_cast<uintptr_t>(base3) & 3u) ||
      (reinterpret_cast<uintptr_t>(base4) & 3u))
    return GAAC_EINVAL;
  if (n_tiles == 0) return GAAC_OK;
  EncodeTilesArgs a{tiles, tile_kind, tile_row, n_rows, base3, base4, slots, esc_len, stats, d_status};
  encode_tiles_kernel<<<static_cast<unsigned>(n_tiles), kEncThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}
