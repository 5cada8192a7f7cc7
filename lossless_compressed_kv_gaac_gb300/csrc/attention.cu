// Fused split-K GQA decode attention over the GAAC compressed cache.
//
// "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference on
// Personal Devices", section 3.2: attention reads the compressed tiles and
// rebuilds the values it needs on the fly (no decompressed copy of the cache);
// compressed blocks and the raw tail go through one softmax.  Section 3.3: the
// block table says per block whether it is a slot or a raw tile.
//
// GB300 design
//  * grid (split, kv-head, sequence); 160 threads: warp 4 is a producer that
//    streams each 64-token block's K and V tile bytes (only the bytes the slot
//    uses) into a 3-stage shared-memory ring with 1-D bulk copies tracked by
//    mbarriers; warps 0-3 consume.
//  * The exponent decoder works on four elements per 32-bit operation and
//    writes BF16 pairs straight into mma.sync m16n8k16 fragments: QK^T with
//    16 tokens x 8 query heads per warp (K token-major, channels permuted so
//    each thread's 32 channels are contiguous), PV^T with 32 channels x 8 heads
//    per warp (V channel-major, each thread's 16 tokens contiguous).  No
//    decompressed tile is ever written back to shared memory.
//  * The producer warp also checks each slot image's tag plane and gathers the
//    escape bytes of 4-bit-mode groups per 32-element unit (into the unused
//    tail of the stage region), so consumers decode without per-lane branches.
//  * Online softmax in the log2 domain, shared by the CTA through a small score
//    buffer and one named barrier per block; P enters the PV product as a
//    bf16 hi + lo pair so its rounding stays near 2^-17.
//  * q is pre-scaled by 2^-4 (exact for normal values) to keep q.k inside the
//    fp32 range for extreme keys; the factor is folded into the softmax scale.
//  * Partials (m, l, acc) per split go to the workspace; the last CTA of each
//    (sequence, kv-head) to finish, found with a device counter, merges them with
//    a log-sum-exp (the final split reduction) and resets the counter.
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"

namespace gaac {

// Warp roles: warps 0-3 take K (decode, QK^T, softmax), warps 4-7 take V
// (decode, PV), warp 8 streams tiles.  K warps run up to two blocks ahead of V
// warps; P crosses over through a double-buffered shared-memory buffer.
constexpr int kKWarps = 4, kVWarps = 4;
constexpr int kProducerWarp = kKWarps + kVWarps;
constexpr int kAttThreads = (kProducerWarp + 1) * 32;
#ifndef GAAC_ATT_STAGES
#define GAAC_ATT_STAGES 3
#endif
#ifndef GAAC_ATT_CTAS_PER_SM
#define GAAC_ATT_CTAS_PER_SM 2
#endif
constexpr int kStages = GAAC_ATT_STAGES;
constexpr int kCtasPerSm = GAAC_ATT_CTAS_PER_SM;
constexpr int kRPad = 8;     // query heads per kv-head in the MMA N dimension
constexpr int kPStride = 72;  // bf16 per head row of the probability buffer (64 + pad)
constexpr int kPartFloats = 2 * kRPad + kRPad * kD;
// named barriers (0 is __syncthreads)
constexpr int kBarK = 1;           // the 4 K warps
constexpr int kBarPFull = 2;       // + parity: P of a block written (K arrive, V sync)
constexpr int kBarPEmpty = 4;      // + parity: P of a block read (V arrive, K sync)

struct TileMeta {
  int mode, esc;
};

struct AttSmem {
  alignas(128) uint8_t ringK[kStages][kRawBytes];
  alignas(128) uint8_t ringV[kStages][kRawBytes];
  alignas(16) uint16_t P[2][2][kRPad][kPStride];  // [block parity][hi, lo][head][token] bf16 probabilities
  alignas(16) float wmax[2][kRPad][kKWarps];       // [parity][head][K warp] max over the warp's 16 scores
  alignas(16) float wsum[2][kRPad][kKWarps];       // [parity][head][K warp] sum of the warp's 16 probabilities
  alignas(16) float alpha[2][kRPad];               // [parity][head] rescale factor of the running sums
  uint2 lut[256];                                  // escape byte -> spread bits of a 4-bit group
  TileMeta metaK[kStages], metaV[kStages];
  uint64_t fullK[kStages], emptyK[kStages], fullV[kStages], emptyV[kStages];
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

// bf16x2 times 2^-4; exact whenever the result is a normal number.
__device__ __forceinline__ uint32_t bf16x2_div16(uint32_t w) {
  const float lo = __uint_as_float(w << 16) * 0.0625f;
  const float hi = __uint_as_float(w & 0xFFFF0000u) * 0.0625f;
  return (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
}

__device__ __forceinline__ uint16_t to_bf16(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int warp_sum(int x) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, d);
  return x;
}

__device__ __forceinline__ int warp_incl_scan(int x, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, x, d);
    if (lane >= d) x += v;
  }
  return x;
}

// Per consumer warp and slot image.  Warp w decodes exactly the 32-element
// units [64w, 64w+64) of the tile (K: its 16 tokens, V: its 32 channels), whose
// tags are tag words [16w, 16w+16).  Returns the escape bytes before that range
// and checks the whole tag plane (no reserved tag; escape bytes add up to
// esc_len), a decision every warp takes identically.
__device__ __forceinline__ bool range_escape_base(const uint8_t* tile, int esc_len, int warp, int lane,
                                                  int& before) {
  const uint32_t* tw = reinterpret_cast<const uint32_t*>(tile + kOffTag);
  const uint32_t wa = tw[lane], wb = tw[lane + 32];
  const int ca = esc_count(wa), cb = esc_count(wb);
  const bool reserved = ((wa & (wa >> 1)) | (wb & (wb >> 1))) & 0x55555555u;
  const int bnd = 16 * warp;
  const int red = warp_sum(((lane < bnd ? ca : 0) + (lane + 32 < bnd ? cb : 0)) | ((ca + cb) << 16));
  before = red & 0xFFFF;
  return !__any_sync(0xFFFFFFFFu, reserved) && (red >> 16) == esc_len;
}

// Escape bytes of the 4-bit-mode groups among the groups of tag byte/nibble
// `tags` (ngroups groups, escape offset of the first at `off`), gathered as
// byte j for group j (0 for the other groups).
template <int NG>
__device__ __forceinline__ uint32_t gather_groups(const uint8_t* esc, uint32_t tags, int off) {
  uint32_t x = 0;
#pragma unroll
  for (int j = 0; j < NG; ++j) {
    const uint32_t m = (tags >> (2 * j)) & 3u;
    if (m == 1u) x |= static_cast<uint32_t>(esc[off]) << (8 * j);
    off += esc_of_tag(m);
  }
  return x;
}

// Exponents of one half-unit (16 elements) into 8 bf16x2 words.  xw16: the two
// groups' gathered 4-bit escape bytes; off: escape offset of its first group
// (used only for raw-mode groups).
__device__ __forceinline__ void decode_half(const uint8_t* tile, uint32_t Wh, uint32_t W2, int hh, uint32_t tagnib,
                                            uint32_t xw16, int off, const uint4 sm, const uint32_t b3[4],
                                            const uint32_t b4[4], const uint2* lut, uint32_t out[8]) {
  uint32_t c[4];
  extract_codes(Wh, W2, hh, c);
  const uint2 s0 = lut[xw16 & 0xFFu], s1 = lut[(xw16 >> 8) & 0xFFu];
  const bool g0 = (tagnib & 3u) != 0u, g1 = (tagnib & 12u) != 0u;
  uint32_t e[4];
  e[0] = (g0 ? b4[0] : b3[0]) + c[0] + s0.x;
  e[1] = (g0 ? b4[1] : b3[1]) + c[1] + s0.y;
  e[2] = (g1 ? b4[2] : b3[2]) + c[2] + s1.x;
  e[3] = (g1 ? b4[3] : b3[3]) + c[3] + s1.y;
  if (tagnib & 0xAu) {  // a raw-mode group in this half (rare): five escape bit planes
    const uint8_t* esc = tile + kOffEsc;
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
      const uint32_t m = (tagnib >> (2 * gi)) & 3u;
      if (m == 2u) {
        const int o = off + (gi == 0 ? 0 : esc_of_tag(tagnib & 3u));
        uint32_t hi0 = 0, hi1 = 0;
#pragma unroll
        for (int k = 0; k < 5; ++k) {
          const uint32_t x = esc[o + k];
          hi0 |= spread4(x & 15u) << (3 + k);
          hi1 |= spread4(x >> 4) << (3 + k);
        }
        e[2 * gi] = c[2 * gi] | hi0;
        e[2 * gi + 1] = c[2 * gi + 1] | hi1;
      }
    }
  }
  join_bf16x4(sm.x, e[0], out[0], out[1]);
  join_bf16x4(sm.y, e[1], out[2], out[3]);
  join_bf16x4(sm.z, e[2], out[4], out[5]);
  join_bf16x4(sm.w, e[3], out[6], out[7]);
}

__device__ __forceinline__ void load8(const uint8_t* p, uint32_t out[8]) {
  const uint4 a = reinterpret_cast<const uint4*>(p)[0], b = reinterpret_cast<const uint4*>(p)[1];
  out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
  out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
}

__device__ __forceinline__ unsigned int atomic_add_acq_rel(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void named_bar_arrive(int id, int threads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Producer lane for one tile kind (kv 0 = K, 1 = V): streams the tile of every
// block of the split into its ring, prefetching the next table entry while it
// waits for a free slot.
__device__ __forceinline__ void stream_tiles(const AttnArgs& a, AttSmem& sm, int kv, int b, int h, int blk0, int n_my) {
  const gaac_entry* tab = a.table + ((static_cast<size_t>(b) * a.max_blocks + blk0) * a.Hkv + h) * 2 + kv;
  const size_t stride = static_cast<size_t>(a.Hkv) * 2;
  uint8_t(*ring)[kRawBytes] = kv ? sm.ringV : sm.ringK;
  TileMeta* meta = kv ? sm.metaV : sm.metaK;
  uint64_t* full = kv ? sm.fullV : sm.fullK;
  uint64_t* empty = kv ? sm.emptyV : sm.emptyK;
  uint2 cur = make_uint2(0u, 0u);
  if (n_my > 0) cur = *reinterpret_cast<const uint2*>(tab);
  for (int j = 0; j < n_my; ++j) {
    uint2 nxt = cur;
    if (j + 1 < n_my) nxt = *reinterpret_cast<const uint2*>(tab + (j + 1) * stride);
    const int st = j % kStages;
    if (j >= kStages) mbar_wait(&empty[st], ((j / kStages) & 1) ^ 1, a.status);
    const uint32_t index = cur.x, esc_len = cur.y & 0xFFFFu, emode = (cur.y >> 16) & 0xFFu;
    uint32_t bytes = 0;
    const void* src = nullptr;
    TileMeta tm{GAAC_MODE_NONE, 0};
    if (emode == GAAC_MODE_SLOT && static_cast<int64_t>(index) < a.n_slots && esc_len <= kEscCap) {
      tm = TileMeta{GAAC_MODE_SLOT, static_cast<int>(esc_len)};
      bytes = kOffEsc + ((esc_len + 15u) & ~15u);
      src = a.slot_pool + static_cast<size_t>(index) * kSlot;
    } else if (emode == GAAC_MODE_RAW && static_cast<int64_t>(index) < a.n_raw) {
      tm = TileMeta{GAAC_MODE_RAW, 0};
      bytes = kRawBytes;
      src = a.raw_pool + static_cast<size_t>(index) * kTile;
    } else {
      report(a.status, GAAC_EFORMAT);
    }
    meta[st] = tm;
    mbar_arrive_expect_tx(&full[st], bytes);
    if (bytes) bulk_g2s(ring[st], src, bytes, &full[st]);
    cur = nxt;
  }
}

// Log-sum-exp merge of the n_splits partials (m, l, acc) of one (sequence,
// kv-head) into out[b, h*r + n, :] = sum_s w_s acc_s / sum_s w_s l_s with
// w_s = 2^(m_s - max_s m_s) per head n (the final split reduction).  Runs on
// the CTA that finished last, so it is a tail on the critical path: each
// thread owns one float4 column of the output and a subset of the splits,
// issues that subset's loads ten at a time and folds them in with its own
// running maximum; the subsets are then combined the same way in shared
// memory.  The ring buffers are free by then and hold that exchange.
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
  float4* xa = reinterpret_cast<float4*>(sm.ringK);  // [groups][o4n] accumulators
  float2* xm = reinterpret_cast<float2*>(sm.ringV);  // [groups][o4n] (running max, denominator)
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
  const int nblk = (len + kBlock - 1) / kBlock;
  const int per = (a.max_blocks + a.n_splits - 1) / a.n_splits;
  const int blk0 = split * per;
  const int n_my = max(0, min(nblk, blk0 + per) - blk0);

  for (int x = tid; x < 256; x += kAttThreads) sm.lut[x] = spread_entry(static_cast<uint32_t>(x));
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.fullK[s], 1);
      mbar_init(&sm.fullV[s], 1);
      mbar_init(&sm.emptyK[s], kKWarps);
      mbar_init(&sm.emptyV[s], kVWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int g = lane >> 2, tq = lane & 3;
  const int r = a.r;
  float* part = a.part + ((static_cast<size_t>(b) * a.Hkv + h) * a.n_splits + split) * kPartFloats;

  if (warp == kProducerWarp) {  // ------------------------------------------------ producer
    if (lane < 2) stream_tiles(a, sm, lane, b, h, blk0, n_my);
  } else if (warp < kKWarps) {  // ------------------------------------------------ K warps
    const int kw = warp;
    uint32_t qf[16];
    if (g < r) {
      const uint4* qp =
          reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(b) * a.Hq + h * r + g) * kD + 32 * tq);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 w = qp[i];
        qf[4 * i] = bf16x2_div16(w.x);
        qf[4 * i + 1] = bf16x2_div16(w.y);
        qf[4 * i + 2] = bf16x2_div16(w.z);
        qf[4 * i + 3] = bf16x2_div16(w.w);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) qf[i] = 0u;
    }
    uint32_t k3[8], k4[8];
    {
      const uint4* p3 = reinterpret_cast<const uint4*>(a.base3 + h * kD + 32 * tq);
      const uint4* p4 = reinterpret_cast<const uint4*>(a.base4 + h * kD + 32 * tq);
      const uint4 x0 = p3[0], x1 = p3[1], y0 = p4[0], y1 = p4[1];
      k3[0] = x0.x; k3[1] = x0.y; k3[2] = x0.z; k3[3] = x0.w;
      k3[4] = x1.x; k3[5] = x1.y; k3[6] = x1.z; k3[7] = x1.w;
      k4[0] = y0.x; k4[1] = y0.y; k4[2] = y0.z; k4[3] = y0.w;
      k4[4] = y1.x; k4[5] = y1.y; k4[6] = y1.z; k4[7] = y1.w;
    }
    float m0 = -INFINITY, m1 = -INFINITY;  // running max of heads 2tq, 2tq+1 (log2 domain)
    const int t0 = 16 * kw + g, t1 = t0 + 8;
    for (int i = 0; i < n_my; ++i) {
      const int st = i % kStages, par = i & 1;
      mbar_wait(&sm.fullK[st], (i / kStages) & 1, a.status);
      const TileMeta md = sm.metaK[st];
      const int nv = min(kBlock, len - (blk0 + i) * kBlock);
      const uint8_t* tK = sm.ringK[st];
      int modeK = md.mode;
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
      if (modeK == GAAC_MODE_SLOT) {
        int before;
        if (!range_escape_base(tK, md.esc, kw, lane, before)) {
          modeK = GAAC_MODE_NONE;
          if (kw == 0 && lane == 0) report(a.status, GAAC_EFORMAT);
        } else {
          // this lane's units: uA = 4*t0 + tq = 64kw + lane, uB = uA + 32 (range positions lane, lane + 32)
          const uint32_t tbA = tK[kOffTag + 64 * kw + lane], tbB = tK[kOffTag + 64 * kw + 32 + lane];
          const int cA = esc_count(tbA), cB = esc_count(tbB);
          const int sc = warp_incl_scan(cA | (cB << 16), lane);
          const int totA = __shfl_sync(0xFFFFFFFFu, sc, 31) & 0xFFFF;
          const int offA = before + (sc & 0xFFFF) - cA;
          const int offB = before + totA + (sc >> 16) - cB;
          const uint32_t xA = gather_groups<4>(tK + kOffEsc, tbA, offA);
          const uint32_t xB = gather_groups<4>(tK + kOffEsc, tbB, offB);
          const uint32_t* cw = reinterpret_cast<const uint32_t*>(tK + kOffCode);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t ka[8], kb[8];
            const int uA = 4 * t0 + tq, uB = 4 * t1 + tq;
            const uint32_t nibA = (tbA >> (4 * hh)) & 15u, nibB = (tbB >> (4 * hh)) & 15u;
            const int hoA = offA + (hh ? esc_count(tbA & 15u) : 0), hoB = offB + (hh ? esc_count(tbB & 15u) : 0);
            decode_half(tK, cw[256 * hh + uA], cw[512 + uA], hh, nibA, xA >> (16 * hh), hoA,
                        *reinterpret_cast<const uint4*>(tK + 128 * t0 + 32 * tq + 16 * hh), k3 + 4 * hh,
                        k4 + 4 * hh, sm.lut, ka);
            decode_half(tK, cw[256 * hh + uB], cw[512 + uB], hh, nibB, xB >> (16 * hh), hoB,
                        *reinterpret_cast<const uint4*>(tK + 128 * t1 + 32 * tq + 16 * hh), k3 + 4 * hh,
                        k4 + 4 * hh, sm.lut, kb);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int ks = 4 * hh + j;
              mma_bf16(j & 1 ? sb : sa, ka[2 * j], kb[2 * j], ka[2 * j + 1], kb[2 * j + 1], qf[2 * ks],
                       qf[2 * ks + 1]);
            }
          }
        }
      } else if (modeK == GAAC_MODE_RAW) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t ka[8], kb[8];
          load8(tK + 256 * t0 + 64 * tq + 32 * hh, ka);
          load8(tK + 256 * t1 + 64 * tq + 32 * hh, kb);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int ks = 4 * hh + j;
            mma_bf16(j & 1 ? sb : sa, ka[2 * j], kb[2 * j], ka[2 * j + 1], kb[2 * j + 1], qf[2 * ks], qf[2 * ks + 1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.emptyK[st]);  // the K tile is no longer read
      const bool ok0 = t0 < nv && modeK != GAAC_MODE_NONE, ok1 = t1 < nv && modeK != GAAC_MODE_NONE;
      // scores: (t0, head 2tq), (t0, 2tq+1), (t1, 2tq), (t1, 2tq+1)
      const float s0 = ok0 ? (sa[0] + sb[0]) * a.scale_log2 : -INFINITY;
      const float s1 = ok0 ? (sa[1] + sb[1]) * a.scale_log2 : -INFINITY;
      const float s2 = ok1 ? (sa[2] + sb[2]) * a.scale_log2 : -INFINITY;
      const float s3 = ok1 ? (sa[3] + sb[3]) * a.scale_log2 : -INFINITY;
      float x0 = fmaxf(s0, s2), x1 = fmaxf(s1, s3);
#pragma unroll
      for (int d = 4; d < 32; d <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xFFFFFFFFu, x0, d));
        x1 = fmaxf(x1, __shfl_xor_sync(0xFFFFFFFFu, x1, d));
      }
      if (g == 0) {
        sm.wmax[par][2 * tq][kw] = x0;
        sm.wmax[par][2 * tq + 1][kw] = x1;
      }
      named_bar_sync(kBarK, kKWarps * 32);
      const float4 wa = *reinterpret_cast<const float4*>(&sm.wmax[par][2 * tq][0]);
      const float4 wb = *reinterpret_cast<const float4*>(&sm.wmax[par][2 * tq + 1][0]);
      const float n0 = fmaxf(m0, fmaxf(fmaxf(wa.x, wa.y), fmaxf(wa.z, wa.w)));
      const float n1 = fmaxf(m1, fmaxf(fmaxf(wb.x, wb.y), fmaxf(wb.z, wb.w)));
      const float al0 = n0 == -INFINITY ? 1.f : fast_exp2(m0 - n0);
      const float al1 = n1 == -INFINITY ? 1.f : fast_exp2(m1 - n1);
      const float p0 = n0 == -INFINITY ? 0.f : fast_exp2(s0 - n0);
      const float p2 = n0 == -INFINITY ? 0.f : fast_exp2(s2 - n0);
      const float p1 = n1 == -INFINITY ? 0.f : fast_exp2(s1 - n1);
      const float p3 = n1 == -INFINITY ? 0.f : fast_exp2(s3 - n1);
      m0 = n0;
      m1 = n1;
      float y0 = p0 + p2, y1 = p1 + p3;
#pragma unroll
      for (int d = 4; d < 32; d <<= 1) {
        y0 += __shfl_xor_sync(0xFFFFFFFFu, y0, d);
        y1 += __shfl_xor_sync(0xFFFFFFFFu, y1, d);
      }
      if (i >= 2) named_bar_sync(kBarPEmpty + par, (kKWarps + kVWarps) * 32);  // V warps are done with P[par]
      if (g == 0) {
        sm.wsum[par][2 * tq][kw] = y0;
        sm.wsum[par][2 * tq + 1][kw] = y1;
        if (kw == 0) {
          sm.alpha[par][2 * tq] = al0;
          sm.alpha[par][2 * tq + 1] = al1;
        }
      }
      {
        uint16_t* Ph = &sm.P[par][0][0][0];
        uint16_t* Pl = &sm.P[par][1][0][0];
        const float pv[4] = {p0, p1, p2, p3};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int head = 2 * tq + (j & 1), tok = j < 2 ? t0 : t1;
          const uint16_t hb = to_bf16(pv[j]);
          Ph[head * kPStride + tok] = hb;
          Pl[head * kPStride + tok] = to_bf16(pv[j] - __uint_as_float(static_cast<uint32_t>(hb) << 16));
        }
      }
      named_bar_arrive(kBarPFull + par, (kKWarps + kVWarps) * 32);
    }
    if (kw == 0 && g == 0) {
      part[4 * tq] = m0;      // head 2tq
      part[4 * tq + 2] = m1;  // head 2tq + 1
    }
  } else {  // ---------------------------------------------------------------------- V warps
  const int vw = warp - kKWarps;
  uint32_t v3[4], v4[4];  // [mi*2 + hb]: channel 32vw + 16mi + g + 8hb, byte replicated
#pragma unroll
  for (int mi = 0; mi < 2; ++mi) {
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const int c = 32 * vw + 16 * mi + g + 8 * hb;
      v3[2 * mi + hb] = 0x01010101u * a.base3[(a.Hkv + h) * kD + c];
      v4[2 * mi + hb] = 0x01010101u * a.base4[(a.Hkv + h) * kD + c];
    }
  }
  float accH[2][4], accL[2][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int j = 0; j < 4; ++j) accH[mi][j] = accL[mi][j] = 0.f;
  float lg = 0.f;  // running sum of head g
  for (int i = 0; i < n_my; ++i) {
    const int st = i % kStages, par = i & 1;
    mbar_wait(&sm.fullV[st], (i / kStages) & 1, a.status);
    const TileMeta md = sm.metaV[st];
    const int nv = min(kBlock, len - (blk0 + i) * kBlock);
    const uint8_t* tV = sm.ringV[st];
    int modeV = md.mode;
    uint32_t va[2][8], vb[2][8];
    if (modeV == GAAC_MODE_SLOT) {
      int before;
      if (!range_escape_base(tV, md.esc, vw, lane, before)) {
        modeV = GAAC_MODE_NONE;
        if (vw == 0 && lane == 0) report(a.status, GAAC_EFORMAT);
      } else {
        // half-unit k = 2*mi + hb: channel c, unit u = 2c + tq/2, half tq%2; its range position
        // (in half-units) is 64*mi + 32*hb + lane, so each k is a lane-ordered segment of 32.
        const uint32_t* cw = reinterpret_cast<const uint32_t*>(tV + kOffCode);
        const int hh = tq & 1;
        uint32_t nib[4];
        int cnt[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int u = 64 * vw + 32 * (k >> 1) + 16 * (k & 1) + 2 * g + (tq >> 1);
          nib[k] = (static_cast<uint32_t>(tV[kOffTag + u]) >> (4 * hh)) & 15u;
          cnt[k] = esc_count(nib[k]);
        }
        const int s01 = warp_incl_scan(cnt[0] | (cnt[1] << 16), lane);
        const int s23 = warp_incl_scan(cnt[2] | (cnt[3] << 16), lane);
        const int t01 = __shfl_sync(0xFFFFFFFFu, s01, 31), t23 = __shfl_sync(0xFFFFFFFFu, s23, 31);
        int ho[4];
        ho[0] = before + (s01 & 0xFFFF) - cnt[0];
        ho[1] = before + (t01 & 0xFFFF) + (s01 >> 16) - cnt[1];
        ho[2] = before + (t01 & 0xFFFF) + (t01 >> 16) + (s23 & 0xFFFF) - cnt[2];
        ho[3] = before + (t01 & 0xFFFF) + (t01 >> 16) + (t23 & 0xFFFF) + (s23 >> 16) - cnt[3];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = 32 * vw + 16 * (k >> 1) + g + 8 * (k & 1);
          const int u = 2 * c + (tq >> 1);
          const uint32_t xw = gather_groups<2>(tV + kOffEsc, nib[k], ho[k]);
          const uint32_t b3[4] = {v3[k], v3[k], v3[k], v3[k]}, b4[4] = {v4[k], v4[k], v4[k], v4[k]};
          decode_half(tV, cw[256 * hh + u], cw[512 + u], hh, nib[k], xw, ho[k],
                      *reinterpret_cast<const uint4*>(tV + 64 * c + 16 * tq), b3, b4, sm.lut,
                      (k & 1) ? vb[k >> 1] : va[k >> 1]);
        }
      }
    }
    if (modeV == GAAC_MODE_RAW) {
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int cA = 32 * vw + 16 * mi + g;
        load8(tV + 128 * cA + 32 * tq, va[mi]);
        load8(tV + 128 * (cA + 8) + 32 * tq, vb[mi]);
      }
    } else if (modeV == GAAC_MODE_NONE) {
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int j = 0; j < 8; ++j) va[mi][j] = vb[mi][j] = 0u;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.emptyV[st]);  // the V tile is no longer read
    if (nv < kBlock) {  // the open tail: tokens past the sequence must not reach the product
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int tt = 16 * tq + 2 * m;
        const uint32_t keep = (tt < nv ? 0x0000FFFFu : 0u) | (tt + 1 < nv ? 0xFFFF0000u : 0u);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          va[mi][m] &= keep;
          vb[mi][m] &= keep;
        }
      }
    }
    named_bar_sync(kBarPFull + par, (kKWarps + kVWarps) * 32);  // P of block i is written
    uint32_t ph[8], pl[8];
    load8(reinterpret_cast<const uint8_t*>(&sm.P[par][0][g][16 * tq]), ph);
    load8(reinterpret_cast<const uint8_t*>(&sm.P[par][1][g][16 * tq]), pl);
    const float4 ws = *reinterpret_cast<const float4*>(&sm.wsum[par][g][0]);
    const float alg = sm.alpha[par][g], al0 = sm.alpha[par][2 * tq], al1 = sm.alpha[par][2 * tq + 1];
    if (i + 2 < n_my) named_bar_arrive(kBarPEmpty + par, (kKWarps + kVWarps) * 32);
    lg = lg * alg + ((ws.x + ws.y) + (ws.z + ws.w));
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
      accH[mi][0] *= al0; accH[mi][1] *= al1; accH[mi][2] *= al0; accH[mi][3] *= al1;
      accL[mi][0] *= al0; accL[mi][1] *= al1; accL[mi][2] *= al0; accL[mi][3] *= al1;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(accH[mi], va[mi][2 * ks], vb[mi][2 * ks], va[mi][2 * ks + 1], vb[mi][2 * ks + 1], ph[2 * ks],
                 ph[2 * ks + 1]);
        mma_bf16(accL[mi], va[mi][2 * ks], vb[mi][2 * ks], va[mi][2 * ks + 1], vb[mi][2 * ks + 1], pl[2 * ks],
                 pl[2 * ks + 1]);
      }
    }
  }
  // Every issued copy was awaited (K warps and V warps consumed every stage);
  // after a timed-out wait, wait once more (bounded) so that no copy is still
  // landing when the CTA exits.
  if (vw == 0 && lane == 0) {
    for (int i = max(0, n_my - kStages); i < n_my; ++i) {
      mbar_wait(&sm.fullK[i % kStages], (i / kStages) & 1, a.status, 1u << 10);
      mbar_wait(&sm.fullV[i % kStages], (i / kStages) & 1, a.status, 1u << 10);
    }
  }
  if (vw == 0 && tq == 0) part[2 * g + 1] = lg;
#pragma unroll
  for (int mi = 0; mi < 2; ++mi) {
    const int cA = 32 * vw + 16 * mi + g, cB = cA + 8;
    float* pa = part + 2 * kRPad;
    pa[(2 * tq) * kD + cA] = accH[mi][0] + accL[mi][0];
    pa[(2 * tq + 1) * kD + cA] = accH[mi][1] + accL[mi][1];
    pa[(2 * tq) * kD + cB] = accH[mi][2] + accL[mi][2];
    pa[(2 * tq + 1) * kD + cB] = accH[mi][3] + accL[mi][3];
  }
  }

  // ---------------------------------------------------------------- split merge (final reduction)
  // The last CTA of a (sequence, kv-head) to finish merges the partials of all
  // its splits with a log-sum-exp; the counter goes back to zero for the next
  // launch.  No CTA ever waits for another.  The merge is a short tail on the
  // critical path, so it keeps many independent L2 loads in flight: one round
  // for the per-head maxima, then every thread streams its share of the splits'
  // accumulators (eight at a time) and the CTA adds the shares up in shared memory.
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
// into an allocator on the decode path.  This entry point runs the same two
// kernels with their split partials in a fixed scratch array that lives in the
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
