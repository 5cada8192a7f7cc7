// The nested 2-bit-mode ablation format: calibrate, encode and decode tile
// batches.  Not used by the cache; it exists to measure the trade the GAAC
// page's section 4.7.2 (Table 4) reports: a 2-bit mode nested inside the 3-bit
// one raises the compression ratio a little and makes decoding slower, because
// a code width that varies per group needs a running bit offset.
//
// Format (declared in gaac.h): format v3's sign|mantissa plane, tags (3 =
// 2-bit group) and escape area, with the three code planes replaced by one
// code stream (16 bits per 2-bit group, 24 per 3-bit or 4-bit group, none per
// raw group, groups in order) and a directory of u32 entries that also holds
// the code-stream bit count at each eighth of the tile.
//
// One CTA of 256 threads per tile; thread u owns the 32-element code unit u,
// and warp w the eighth w (units 32w..32w+31): the bit offset of a unit is
// its eighth's directory entry plus a warp scan of the units' widths.
#include <cuda_runtime.h>

#include "common.cuh"

namespace gaac {

constexpr int kNOffCode = 8192;
constexpr int kNOffTag = 11264;
constexpr int kNOffDir = 11520;
constexpr int kNOffEsc = 11552;
constexpr int kNSlot = 12048;
constexpr int kNCodeWords = 768;  // code stream capacity: 1024 groups x 24 bits
constexpr int kNThreads = 256;
constexpr uint32_t kM2 = 3u;      // tag of a 2-bit group

static_assert(kNSlot == GAAC_NESTED_SLOT_BYTES, "nested slot size");

// Bits a group's codes take in the stream.
__device__ __forceinline__ int group_bits(uint32_t mode) { return mode == kM2 ? 16 : (mode == 2u ? 0 : 24); }

// ------------------------------------------------------------- calibrate ----

// One CTA per kv-head, one thread per channel: 256-bin histogram column,
// best 4-exponent window, ties to the smallest base.
__global__ void __launch_bounds__(kD) nested_calibrate_kernel(const uint16_t* __restrict__ x, int64_t n_tok,
                                                              int64_t tok_stride, uint8_t* __restrict__ base2) {
  extern __shared__ uint16_t hist[];  // [256][128]
  const int h = blockIdx.x, c = threadIdx.x;
  for (int bin = 0; bin < 256; ++bin) hist[bin * kD + c] = 0;
  const uint16_t* p = x + static_cast<int64_t>(h) * kD + c;
  for (int64_t t = 0; t < n_tok; ++t) hist[((p[t * tok_stride] >> 7) & 0xFFu) * kD + c] += 1;
  int sum = 0;
  for (int i = 0; i < 4; ++i) sum += hist[i * kD + c];
  int best = sum, arg = 0;
  for (int b = 1; b + 4 <= 256; ++b) {
    sum += hist[(b + 3) * kD + c] - hist[(b - 1) * kD + c];
    if (sum > best) {
      best = sum;
      arg = b;
    }
  }
  base2[h * kD + c] = static_cast<uint8_t>(arg);
}

// ---------------------------------------------------------------- encode ----

struct NestedArgs {
  const uint16_t* tiles;  // encode: input; decode: output ([n][64][128] BF16, token-major)
  uint16_t* tiles_out;
  const uint8_t* kind;
  const int32_t* row;
  int n_rows;
  const uint8_t* base2;
  const uint8_t* base3;
  const uint8_t* base4;
  uint8_t* slots;
  const uint8_t* slots_in;
  uint16_t* esc_len;
  const uint16_t* esc_in;
  int32_t* status;
};

struct NestedEncShared {
  alignas(16) uint16_t tile[kTile];
  alignas(16) uint32_t code[kNCodeWords];
  int warp_cnt[kNThreads / 32];
  int warp_bits[kNThreads / 32];
};

// value (at most 24 bits) placed at bit p (a multiple of 8, p + 24 <= 96) of the 96-bit (lo, hi) accumulator.
__device__ __forceinline__ void put_field(uint64_t& lo, uint32_t& hi, uint32_t value, int p) {
  if (p < 64) {
    lo |= static_cast<uint64_t>(value) << p;
    if (p > 40) hi |= value >> (64 - p);
  } else {
    hi |= value << (p - 64);
  }
}

__global__ void __launch_bounds__(kNThreads, 4) nested_encode_kernel(NestedArgs a) {
  __shared__ NestedEncShared sh;
  const int64_t i = blockIdx.x;
  const int u = threadIdx.x, lane = u & 31, warp = u >> 5;
  const int kind = a.kind[i], r = a.row[i];
  if (kind > 1 || r < 0 || r >= a.n_rows) {
    if (u == 0) {
      a.esc_len[i] = 0xFFFFu;
      report(a.status, GAAC_EINVAL);
    }
    return;
  }
  stage_tile(sh.tile, a.tiles + i * kTile, kD, kBlock, kind, u);
#pragma unroll
  for (int k = 0; k < 3; ++k) sh.code[u + kNThreads * k] = 0u;
  __syncthreads();

  uint32_t xw[16];
  {
    const uint4* src = reinterpret_cast<const uint4*>(sh.tile + 32 * u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 w = src[k];
      xw[4 * k] = w.x;
      xw[4 * k + 1] = w.y;
      xw[4 * k + 2] = w.z;
      xw[4 * k + 3] = w.w;
    }
  }
  uint32_t b2w[8], b3w[8], b4w[8];
  unit_base_words(kind, u, a.base2 + r * kD, b2w);
  unit_base_words(kind, u, a.base3 + r * kD, b3w);
  unit_base_words(kind, u, a.base4 + r * kD, b4w);

  uint32_t smb[8], ew[8];
  uint64_t acc_lo = 0;
  uint32_t acc_hi = 0;
  int p = 0, n4 = 0, nraw = 0;
  uint32_t esc4 = 0, tagbyte = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) smb[k] = ew[k] = 0u;
#pragma unroll
  for (int gi = 0; gi < 4; ++gi) {
    int e[8], o2[8], o3[8], o4[8];
    bool f2 = true, f3 = true, f4 = true;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int el = 8 * gi + j;
      const uint32_t x = (xw[el >> 1] >> (16 * (el & 1))) & 0xFFFFu;
      e[j] = (x >> 7) & 0xFF;
      ew[el >> 2] |= static_cast<uint32_t>(e[j]) << (8 * (el & 3));
      smb[el >> 2] |= (((x >> 8) & 0x80u) | (x & 0x7Fu)) << (8 * (el & 3));
      const int sh8 = 8 * (el & 3);
      o2[j] = e[j] - static_cast<int>((b2w[el >> 2] >> sh8) & 0xFFu);
      o3[j] = e[j] - static_cast<int>((b3w[el >> 2] >> sh8) & 0xFFu);
      o4[j] = e[j] - static_cast<int>((b4w[el >> 2] >> sh8) & 0xFFu);
      f2 = f2 && o2[j] >= 0 && o2[j] <= 3;
      f3 = f3 && o3[j] >= 0 && o3[j] <= 7;
      f4 = f4 && o4[j] >= 0 && o4[j] <= 15;
    }
    const uint32_t mode = f2 ? kM2 : (f3 ? 0u : (f4 ? 1u : 2u));
    tagbyte |= mode << (2 * gi);
    uint32_t field = 0, eb = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (mode == kM2) field |= static_cast<uint32_t>(o2[j]) << (2 * j);
      if (mode == 0u) field |= static_cast<uint32_t>(o3[j]) << (3 * j);
      if (mode == 1u) {
        field |= (static_cast<uint32_t>(o4[j]) & 7u) << (3 * j);
        eb |= ((static_cast<uint32_t>(o4[j]) >> 3) & 1u) << j;
      }
    }
    put_field(acc_lo, acc_hi, field, p);
    p += group_bits(mode);
    if (mode == 1u) {
      esc4 |= eb << (8 * n4);
      n4 += 1;
    }
    if (mode == 2u) nraw += 1;
  }

  // CTA scans (unit order = group order): counts packed n4 | nraw << 16, and code bits.
  const int packed = n4 | (nraw << 16);
  int inc_c = packed, inc_b = p;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int vc = __shfl_up_sync(0xFFFFFFFFu, inc_c, d), vb = __shfl_up_sync(0xFFFFFFFFu, inc_b, d);
    if (lane >= d) {
      inc_c += vc;
      inc_b += vb;
    }
  }
  if (lane == 31) {
    sh.warp_cnt[warp] = inc_c;
    sh.warp_bits[warp] = inc_b;
  }
  __syncthreads();
  int before_c = 0, total_c = 0, before_b = 0;
#pragma unroll
  for (int w = 0; w < kNThreads / 32; ++w) {
    const int c = sh.warp_cnt[w];
    if (w < warp) {
      before_c += c;
      before_b += sh.warp_bits[w];
    }
    total_c += c;
  }
  const int ex_c = before_c + inc_c - packed, off_bits = before_b + inc_b - p;
  const int off4 = ex_c & 0xFFFF, offraw = ex_c >> 16, tot4 = total_c & 0xFFFF, totraw = total_c >> 16;
  const int esc = tot4 + 8 * totraw;
  if (esc > kEscCap) {
    if (u == 0) a.esc_len[i] = 0xFFFFu;
    return;
  }
  // Code bits into the shared stream (neighbouring units share boundary words).
  {
    const int wi = off_bits >> 5, s = off_bits & 31;
    const uint32_t v0 = static_cast<uint32_t>(acc_lo), v1 = static_cast<uint32_t>(acc_lo >> 32), v2 = acc_hi;
    uint32_t w[4];
    w[0] = v0 << s;
    w[1] = s ? (v0 >> (32 - s)) | (v1 << s) : v1;
    w[2] = s ? (v1 >> (32 - s)) | (v2 << s) : v2;
    w[3] = s ? v2 >> (32 - s) : 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (w[k] != 0u && wi + k < kNCodeWords) atomicOr(&sh.code[wi + k], w[k]);
  }
  uint8_t* slot = a.slots + i * kNSlot;
#pragma unroll
  for (int k = 0; k < 8; ++k) {  // signs rotated one byte within each aligned group of four, as format v3
    const uint32_t sg = smb[k] & 0x80808080u;
    smb[k] = (smb[k] & 0x7F7F7F7Fu) | ((sg << 8) | (sg >> 24));
  }
  uint4* smdst = reinterpret_cast<uint4*>(slot + 32 * u);
  smdst[0] = make_uint4(smb[0], smb[1], smb[2], smb[3]);
  smdst[1] = make_uint4(smb[4], smb[5], smb[6], smb[7]);
  slot[kNOffTag + u] = static_cast<uint8_t>(tagbyte);
  uint8_t* escp = slot + kNOffEsc;
  for (int k = 0; k < n4; ++k) escp[off4 + k] = static_cast<uint8_t>(esc4 >> (8 * k));
  if (nraw) {
    int at = tot4 + 8 * offraw;
#pragma unroll
    for (int gi = 0; gi < 4; ++gi) {
      if (((tagbyte >> (2 * gi)) & 3u) != 2u) continue;
#pragma unroll
      for (int j = 0; j < 8; ++j) escp[at + j] = static_cast<uint8_t>(ew[2 * gi + (j >> 2)] >> (8 * (j & 3)));
      at += 8;
    }
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int at = 2 * u + k;
    if (at >= esc && at < kEscCap) escp[at] = 0;
  }
  if (lane == 31) {  // directory entry of eighth `warp`: counts and bits over groups [0, 128 (warp + 1))
    const uint32_t entry = static_cast<uint32_t>((off4 + n4) & 0x1FF) | (static_cast<uint32_t>((offraw + nraw) & 0x7F) << 9) |
                           (static_cast<uint32_t>(off_bits + p) << 16);
    *reinterpret_cast<uint32_t*>(slot + kNOffDir + 4 * warp) = entry;
  }
  __syncthreads();
  uint32_t* cdst = reinterpret_cast<uint32_t*>(slot + kNOffCode);
#pragma unroll
  for (int k = 0; k < 3; ++k) cdst[u + kNThreads * k] = sh.code[u + kNThreads * k];
  if (u == 0) a.esc_len[i] = static_cast<uint16_t>(esc);
}

// ---------------------------------------------------------------- decode ----

// Four byte lanes from four consecutive w-bit fields of g (w = 2 or 3).
__device__ __forceinline__ uint32_t fields_to_bytes(uint32_t g, int w) {
  const uint32_t m = (1u << w) - 1u;
  return (g & m) | (((g >> w) & m) << 8) | (((g >> (2 * w)) & m) << 16) | (((g >> (3 * w)) & m) << 24);
}

__global__ void __launch_bounds__(kNThreads, 6) nested_decode_kernel(NestedArgs a) {
  __shared__ alignas(16) uint16_t logical[kLogicalElems];
  __shared__ uint32_t vbt[2][16][8];  // V: base3 / base4 words of the unit classes
  __shared__ uint32_t vbt2[16][8];    // V: base2 words
  const int64_t i = blockIdx.x;
  const int u = threadIdx.x, lane = u & 31, warp = u >> 5;
  const int esc = a.esc_in[i];
  if (esc == 0xFFFF) return;
  const int kind = a.kind[i], r = a.row[i];
  if (kind > 1 || r < 0 || r >= a.n_rows || esc > kEscCap) {
    if (u == 0) report(a.status, GAAC_EINVAL);
    return;
  }
  const uint8_t* slot = a.slots_in + i * kNSlot;
  if (kind == 1) {  // V base words of the 16 unit classes (base3, base4, then base2)
    fill_v_base_table(vbt, a.base3 + r * kD, a.base4 + r * kD, u);
    if (u < 128) {
      const int cls = (u >> 3) & 15, k = u & 7, urep = 32 * (cls >> 3) + 4 * (cls & 7);
      uint32_t w = 0u;
#pragma unroll
      for (int L = 0; L < 4; ++L) w |= static_cast<uint32_t>(a.base2[r * kD + v_channel_of(32 * urep + 4 * k + L)]) << (8 * L);
      vbt2[cls][k] = w;
    }
  }
  const uint32_t* dir = reinterpret_cast<const uint32_t*>(slot + kNOffDir);
  const uint32_t tagbyte = slot[kNOffTag + u];
  int bits_u = 0, n4 = 0, nraw = 0;
#pragma unroll
  for (int gi = 0; gi < 4; ++gi) {
    const uint32_t m = (tagbyte >> (2 * gi)) & 3u;
    bits_u += group_bits(m);
    n4 += m == 1u;
    nraw += m == 2u;
  }
  // Warp scan over the eighth's units: n4 | nraw << 8 | bits << 16 (each sum fits its field).
  const uint32_t packed = static_cast<uint32_t>(n4) | (static_cast<uint32_t>(nraw) << 8) |
                          (static_cast<uint32_t>(bits_u) << 16);
  uint32_t incl = packed;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += v;
  }
  const uint32_t ex = incl - packed, tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
  const uint32_t prev = warp ? dir[warp - 1] : 0u, cur = dir[warp], last = dir[7];
  const int p4 = prev & 0x1FF, praw = (prev >> 9) & 0x7F, pbits = prev >> 16;
  bool bad = ((p4 + (tot & 0xFF)) & 0x1FF) != (cur & 0x1FF) || ((praw + ((tot >> 8) & 0xFF)) & 0x7F) != ((cur >> 9) & 0x7F) ||
             pbits + static_cast<int>(tot >> 16) != static_cast<int>(cur >> 16);
  const int rawbase = last & 0x1FF;
  if (rawbase + 8 * static_cast<int>((last >> 9) & 0x7F) != esc) bad = true;
  int o4 = p4 + static_cast<int>(ex & 0xFF);
  int oraw = rawbase + 8 * (praw + static_cast<int>((ex >> 8) & 0xFF));
  const int off_bits = pbits + static_cast<int>(ex >> 16);
  // The unit's (at most 96) code bits, starting at bit 0 of (x0, x1, x2).
  uint32_t x0, x1, x2;
  {
    const uint32_t* cw = reinterpret_cast<const uint32_t*>(slot + kNOffCode);
    const int wi = off_bits >> 5, s = off_bits & 31;
    uint32_t c[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) c[k] = wi + k < kNCodeWords ? cw[wi + k] : 0u;
    x0 = __funnelshift_r(c[0], c[1], s);
    x1 = __funnelshift_r(c[1], c[2], s);
    x2 = __funnelshift_r(c[2], c[3], s);
  }
  const uint64_t lo = static_cast<uint64_t>(x0) | (static_cast<uint64_t>(x1) << 32);
  uint32_t b2w[8], b3w[8], b4w[8];
  if (kind == 0) {
    unit_base_words(0, u, a.base2 + r * kD, b2w);
    unit_base_words(0, u, a.base3 + r * kD, b3w);
    unit_base_words(0, u, a.base4 + r * kD, b4w);
  } else {  // V: from the table of the 16 unit classes, as the format-v3 decoder
    __syncthreads();
    const int cls = v_unit_class(u);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      b2w[k] = vbt2[cls][k];
      b3w[k] = vbt[0][cls][k];
      b4w[k] = vbt[1][cls][k];
    }
  }
  const uint4* smp = reinterpret_cast<const uint4*>(slot + 32 * u);
  const uint4 s0 = smp[0], s1 = smp[1];
  uint32_t smw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  uint32_t pairs[16];
  int pbit = 0;
#pragma unroll
  for (int gi = 0; gi < 4; ++gi) {
    const uint32_t m = (tagbyte >> (2 * gi)) & 3u;
    uint32_t f;  // the group's field, bits pbit.. of the unit's window
    if (pbit < 64)
      f = static_cast<uint32_t>(lo >> pbit) | (pbit > 32 ? x2 << (64 - pbit) : 0u);
    else
      f = x2 >> (pbit - 64);
    uint32_t e[2];
    if (m == kM2) {
      e[0] = b2w[2 * gi] + fields_to_bytes(f, 2);
      e[1] = b2w[2 * gi + 1] + fields_to_bytes(f >> 8, 2);
    } else if (m == 0u) {
      e[0] = b3w[2 * gi] + fields_to_bytes(f, 3);
      e[1] = b3w[2 * gi + 1] + fields_to_bytes(f >> 12, 3);
    } else if (m == 1u) {
      const bool in = o4 < esc;
      if (!in) bad = true;
      const uint32_t xb = in ? slot[kNOffEsc + o4] : 0u;
      e[0] = b4w[2 * gi] + (fields_to_bytes(f, 3) | (spread4(xb & 15u) << 3));
      e[1] = b4w[2 * gi + 1] + (fields_to_bytes(f >> 12, 3) | (spread4(xb >> 4) << 3));
      o4 += 1;
    } else {
      const bool in = oraw + 8 <= esc;
      if (!in) bad = true;
      e[0] = in ? load_u32_any(slot, kNOffEsc + oraw) : 0u;
      e[1] = in ? load_u32_any(slot, kNOffEsc + oraw + 4) : 0u;
      oraw += 8;
    }
    pbit += group_bits(m);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint32_t sm = smw[2 * gi + q];
      const uint32_t sg = sm & 0x80808080u;  // signs back to their own bytes
      sm = (sm & 0x7F7F7F7Fu) | ((sg >> 8) | (sg << 24));
      join_bf16x4(sm, e[q], pairs[4 * gi + 2 * q], pairs[4 * gi + 2 * q + 1]);
    }
  }
  if (bad) report(a.status, GAAC_EFORMAT);
  unit_to_logical(logical, kind, u, pairs);
  __syncthreads();
  logical_to_global(logical, a.tiles_out + i * kTile, kD, kBlock, u);
}

}  // namespace gaac

using namespace gaac;

extern "C" int gaac_nested_calibrate(const uint16_t* x, int64_t n_tok, int64_t tok_stride, int n_kv_heads,
                                     uint8_t* base2, int32_t* d_status, void* stream) {
  (void)d_status;
  if (x == nullptr || base2 == nullptr) return GAAC_EINVAL;
  if (n_tok < 1 || n_tok > 65535 || n_kv_heads <= 0 || n_kv_heads > 65535 ||
      tok_stride < static_cast<int64_t>(n_kv_heads) * kD)
    return GAAC_EINVAL;
  const size_t smem = 256 * kD * sizeof(uint16_t);
  static bool attr_done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GAAC_ECUDA;
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(nested_calibrate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return GAAC_ECUDA;
    attr_done[dev] = true;
  }
  nested_calibrate_kernel<<<n_kv_heads, kD, smem, static_cast<cudaStream_t>(stream)>>>(x, n_tok, tok_stride, base2);
  return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}

static bool nested_common_ok(int64_t n_tiles, const uint8_t* kind, const int32_t* row, int n_rows, const uint8_t* b2,
                             const uint8_t* b3, const uint8_t* b4) {
  return kind != nullptr && row != nullptr && b2 != nullptr && b3 != nullptr && b4 != nullptr && n_rows > 0 &&
         n_tiles >= 0 && n_tiles <= 0x7FFFFFFF && (reinterpret_cast<uintptr_t>(b2) & 3u) == 0 &&
         (reinterpret_cast<uintptr_t>(b3) & 3u) == 0 && (reinterpret_cast<uintptr_t>(b4) & 3u) == 0;
}

extern "C" int gaac_nested_encode_tiles(const uint16_t* tiles, int64_t n_tiles, const uint8_t* tile_kind,
                                        const int32_t* tile_row, int n_rows, const uint8_t* base2,
                                        const uint8_t* base3, const uint8_t* base4, uint8_t* slots,
                                        uint16_t* esc_len, int32_t* d_status, void* stream) {
  if (tiles == nullptr || slots == nullptr || esc_len == nullptr ||
      !nested_common_ok(n_tiles, tile_kind, tile_row, n_rows, base2, base3, base4) ||
      (reinterpret_cast<uintptr_t>(tiles) & 15u) || (reinterpret_cast<uintptr_t>(slots) & 15u))
    return GAAC_EINVAL;
  if (n_tiles == 0) return GAAC_OK;
  NestedArgs a{tiles, nullptr, tile_kind, tile_row, n_rows, base2, base3, base4, slots, nullptr, esc_len, nullptr,
               d_status};
  nested_encode_kernel<<<static_cast<unsigned>(n_tiles), kNThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}

extern "C" int gaac_nested_decode_tiles(const uint8_t* slots, const uint16_t* esc_len, int64_t n_tiles,
                                        const uint8_t* tile_kind, const int32_t* tile_row, int n_rows,
                                        const uint8_t* base2, const uint8_t* base3, const uint8_t* base4,
                                        uint16_t* tiles, int32_t* d_status, void* stream) {
  if (tiles == nullptr || slots == nullptr || esc_len == nullptr ||
      !nested_common_ok(n_tiles, tile_kind, tile_row, n_rows, base2, base3, base4) ||
      (reinterpret_cast<uintptr_t>(tiles) & 15u) || (reinterpret_cast<uintptr_t>(slots) & 15u))
    return GAAC_EINVAL;
  if (n_tiles == 0) return GAAC_OK;
  NestedArgs a{nullptr, tiles, tile_kind, tile_row, n_rows, base2, base3, base4, nullptr, slots, nullptr, esc_len,
               d_status};
  nested_decode_kernel<<<static_cast<unsigned>(n_tiles), kNThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}
