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
//  * Online softmax in the log2 domain, shared by the CTA through a small score
//    buffer and one named barrier per block; P enters the PV product as a
//    bf16 hi + lo pair so its rounding stays near 2^-17.
//  * q is pre-scaled by 2^-4 (exact for normal values) to keep q.k inside the
//    fp32 range for extreme keys; the factor is folded into the softmax scale.
//  * Partials (m, l, acc) per split go to the workspace; a combine kernel merges
//    them with a log-sum-exp.
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"

namespace gaac {

constexpr int kAttWarps = 4;
constexpr int kAttThreads = (kAttWarps + 1) * 32;
constexpr int kStages = 3;
constexpr int kStageBytes = 2 * kRawBytes;  // K region + V region
constexpr int kSStride = 68;                // floats per head row of the score buffer
constexpr int kRPad = 8;                    // query heads per kv-head in the MMA N dimension
constexpr int kPartFloats = 2 * kRPad + kRPad * kD;

struct StageMeta {
  int modeK, modeV, escK, escV;
};

struct AttSmem {
  alignas(128) uint8_t stage[kStages][kStageBytes];
  alignas(16) float S[2][kRPad][kSStride];
  StageMeta meta[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
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
  int32_t* status;
};

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

// Exclusive prefix of escape bytes over the 64 tag words of a slot image:
// lane l returns the prefixes of words l and l+32.
__device__ __forceinline__ void tag_word_prefix(const uint8_t* tile, int lane, int& pre_lo, int& pre_hi) {
  const uint32_t* tw = reinterpret_cast<const uint32_t*>(tile + kOffTag);
  const int c0 = esc_count(tw[lane]), c1 = esc_count(tw[lane + 32]);
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
  pre_lo = i0 - c0;
  pre_hi = tot0 + i1 - c1;
}

// K token t, channels 32tq..32tq+31 -> 16 bf16x2 words (channel pairs 32tq+2m, +1).
__device__ __forceinline__ void k_raw(const uint8_t* tile, int t, int tq, uint32_t out[16]) {
  const uint4* p = reinterpret_cast<const uint4*>(tile + 256 * t + 64 * tq);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 w = p[i];
    out[4 * i] = w.x;
    out[4 * i + 1] = w.y;
    out[4 * i + 2] = w.z;
    out[4 * i + 3] = w.w;
  }
}

__device__ __forceinline__ void k_slot(const uint8_t* tile, int t, int tq, const uint32_t k3[8],
                                       const uint32_t k4[8], int word_pre, int esc_len, uint32_t out[16],
                                       bool* bad) {
  const int u = 4 * t + tq;
  const uint32_t* cw = reinterpret_cast<const uint32_t*>(tile + kOffCode);
  const uint32_t W0 = cw[u], W1 = cw[256 + u], W2 = cw[512 + u];
  const uint32_t tagbyte = tile[kOffTag + u];
  const uint4* sp = reinterpret_cast<const uint4*>(tile + 128 * t + 32 * tq);
  const uint4 s0 = sp[0], s1 = sp[1];
  const uint32_t smw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  int esc0 = 0, esc1 = 0;
  if (tagbyte != 0u) {
    const uint32_t tword = *reinterpret_cast<const uint32_t*>(tile + kOffTag + 4 * t);
    esc0 = word_pre + esc_count(tword & ((1u << (8 * tq)) - 1u));
    esc1 = esc0 + esc_count(tagbyte & 15u);
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    uint32_t e[4];
    half_exponents(hh == 0 ? W0 : W1, W2, hh, (tagbyte >> (4 * hh)) & 15u, k3 + 4 * hh, k4 + 4 * hh,
                   tile + kOffEsc, hh == 0 ? esc0 : esc1, esc_len, e, bad);
#pragma unroll
    for (int q = 0; q < 4; ++q) join_bf16x4(smw[4 * hh + q], e[q], out[8 * hh + 2 * q], out[8 * hh + 2 * q + 1]);
  }
}

// V channel c, tokens 16tq..16tq+15 -> 8 bf16x2 words (token pairs 16tq+2m, +1).
__device__ __forceinline__ void v_raw(const uint8_t* tile, int c, int tq, uint32_t out[8]) {
  const uint4* p = reinterpret_cast<const uint4*>(tile + 128 * c + 32 * tq);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 w = p[i];
    out[4 * i] = w.x;
    out[4 * i + 1] = w.y;
    out[4 * i + 2] = w.z;
    out[4 * i + 3] = w.w;
  }
}

__device__ __forceinline__ void v_slot(const uint8_t* tile, int c, int tq, uint32_t b3w, uint32_t b4w, int word_pre,
                                       int esc_len, uint32_t out[8], bool* bad) {
  const int u = 2 * c + (tq >> 1), hh = tq & 1;
  const uint32_t* cw = reinterpret_cast<const uint32_t*>(tile + kOffCode);
  const uint32_t Wh = cw[256 * hh + u], W2 = cw[512 + u];
  const uint32_t tagnib = (static_cast<uint32_t>(tile[kOffTag + u]) >> (4 * hh)) & 15u;
  const uint4 s = *reinterpret_cast<const uint4*>(tile + 64 * c + 16 * tq);
  int esc0 = 0;
  if (tagnib != 0u) {
    const uint32_t tword = *reinterpret_cast<const uint32_t*>(tile + kOffTag + 4 * (c >> 1));
    esc0 = word_pre + esc_count(tword & ((1u << (16 * (c & 1) + 4 * tq)) - 1u));
  }
  const uint32_t b3[4] = {b3w, b3w, b3w, b3w}, b4[4] = {b4w, b4w, b4w, b4w};
  uint32_t e[4];
  half_exponents(Wh, W2, hh, tagnib, b3, b4, tile + kOffEsc, esc0, esc_len, e, bad);
  join_bf16x4(s.x, e[0], out[0], out[1]);
  join_bf16x4(s.y, e[1], out[2], out[3]);
  join_bf16x4(s.z, e[2], out[4], out[5]);
  join_bf16x4(s.w, e[3], out[6], out[7]);
}

__global__ void __launch_bounds__(kAttThreads, 2) attn_split_kernel(AttnArgs a) {
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

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kAttWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kAttWarps) {  // ------------------------------------ producer
    if (lane == 0) {
      for (int i = 0; i < n_my; ++i) {
        const int st = i % kStages;
        if (i >= kStages) mbar_wait(&sm.empty[st], ((i / kStages) & 1) ^ 1, a.status);
        const gaac_entry* ep =
            a.table + ((static_cast<size_t>(b) * a.max_blocks + blk0 + i) * a.Hkv + h) * 2;
        uint32_t bytes[2];
        const void* src[2];
        int mode[2], esc[2];
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          const gaac_entry e = ep[kv];
          bytes[kv] = 0;
          src[kv] = nullptr;
          esc[kv] = 0;
          if (e.mode == GAAC_MODE_SLOT && static_cast<int64_t>(e.index) < a.n_slots && e.esc_len <= kEscCap) {
            mode[kv] = GAAC_MODE_SLOT;
            esc[kv] = e.esc_len;
            bytes[kv] = kOffEsc + ((e.esc_len + 15) & ~15);
            src[kv] = a.slot_pool + static_cast<size_t>(e.index) * kSlot;
          } else if (e.mode == GAAC_MODE_RAW && static_cast<int64_t>(e.index) < a.n_raw) {
            mode[kv] = GAAC_MODE_RAW;
            bytes[kv] = kRawBytes;
            src[kv] = a.raw_pool + static_cast<size_t>(e.index) * kTile;
          } else {
            mode[kv] = GAAC_MODE_NONE;
            report(a.status, GAAC_EFORMAT);
          }
        }
        sm.meta[st] = StageMeta{mode[0], mode[1], esc[0], esc[1]};
        mbar_arrive_expect_tx(&sm.full[st], bytes[0] + bytes[1]);
        if (bytes[0]) bulk_g2s(sm.stage[st], src[0], bytes[0], &sm.full[st]);
        if (bytes[1]) bulk_g2s(sm.stage[st] + kRawBytes, src[1], bytes[1], &sm.full[st]);
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int g = lane >> 2, tq = lane & 3;
  const int r = a.r;
  uint32_t qf[16];
  if (g < r) {
    const uint4* qp = reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(b) * a.Hq + h * r + g) * kD + 32 * tq);
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
  uint32_t v3[4], v4[4];  // [mi*2 + (0: channel g, 1: channel g+8)]
#pragma unroll
  for (int mi = 0; mi < 2; ++mi) {
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const int c = 32 * warp + 16 * mi + g + 8 * hb;
      v3[2 * mi + hb] = 0x01010101u * a.base3[(a.Hkv + h) * kD + c];
      v4[2 * mi + hb] = 0x01010101u * a.base4[(a.Hkv + h) * kD + c];
    }
  }
  float acc[2][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[mi][j] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;
  bool bad = false;
  const int t0 = 16 * warp + g, t1 = t0 + 8;

  for (int i = 0; i < n_my; ++i) {
    const int st = i % kStages;
    mbar_wait(&sm.full[st], (i / kStages) & 1, a.status);
    const StageMeta md = sm.meta[st];
    const int nv = min(kBlock, len - (blk0 + i) * kBlock);
    const uint8_t* tK = sm.stage[st];
    const uint8_t* tV = tK + kRawBytes;

    // ---- S = (q/16) K^T for tokens t0, t1 of this warp's 16-token slice
    uint32_t ka[16], kb[16];
    if (md.modeK == GAAC_MODE_SLOT) {
      int pre_lo = 0, pre_hi = 0;
      if (md.escK > 0) tag_word_prefix(tK, lane, pre_lo, pre_hi);
      const int src = warp < 2 ? pre_lo : pre_hi;
      const int wp0 = __shfl_sync(0xFFFFFFFFu, src, t0 & 31);
      const int wp1 = __shfl_sync(0xFFFFFFFFu, src, t1 & 31);
      k_slot(tK, t0, tq, k3, k4, wp0, md.escK, ka, &bad);
      k_slot(tK, t1, tq, k3, k4, wp1, md.escK, kb, &bad);
    } else if (md.modeK == GAAC_MODE_RAW) {
      k_raw(tK, t0, tq, ka);
      k_raw(tK, t1, tq, kb);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) ka[j] = kb[j] = 0u;
    }
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) mma_bf16(s, ka[2 * ks], kb[2 * ks], ka[2 * ks + 1], kb[2 * ks + 1], qf[2 * ks], qf[2 * ks + 1]);
    const bool ok0 = t0 < nv && md.modeK != GAAC_MODE_NONE, ok1 = t1 < nv && md.modeK != GAAC_MODE_NONE;
    float* Sb = &sm.S[i & 1][0][0];
    Sb[(2 * tq) * kSStride + t0] = ok0 ? s[0] * a.scale_log2 : -INFINITY;
    Sb[(2 * tq + 1) * kSStride + t0] = ok0 ? s[1] * a.scale_log2 : -INFINITY;
    Sb[(2 * tq) * kSStride + t1] = ok1 ? s[2] * a.scale_log2 : -INFINITY;
    Sb[(2 * tq + 1) * kSStride + t1] = ok1 ? s[3] * a.scale_log2 : -INFINITY;
    named_bar_sync(1, kAttWarps * 32);

    // ---- online softmax for head g over this thread's tokens 16tq..16tq+15
    float p[16];
    {
      const float4* sr = reinterpret_cast<const float4*>(Sb + g * kSStride + 16 * tq);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 v = sr[j];
        p[4 * j] = v.x;
        p[4 * j + 1] = v.y;
        p[4 * j + 2] = v.z;
        p[4 * j + 3] = v.w;
      }
    }
    float mx = p[0];
#pragma unroll
    for (int j = 1; j < 16; ++j) mx = fmaxf(mx, p[j]);
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
    const float m_new = fmaxf(m_run, mx);
    float alpha;
    if (m_new == -INFINITY) {
      alpha = 1.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) p[j] = 0.f;
    } else {
      alpha = exp2f(m_run - m_new);
#pragma unroll
      for (int j = 0; j < 16; ++j) p[j] = exp2f(p[j] - m_new);
    }
    float ls = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) ls += p[j];
    ls += __shfl_xor_sync(0xFFFFFFFFu, ls, 1);
    ls += __shfl_xor_sync(0xFFFFFFFFu, ls, 2);
    l_run = l_run * alpha + ls;
    m_run = m_new;
    uint32_t ph[8], pl[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      ph[j] = pack_bf16x2(p[2 * j], p[2 * j + 1]);
      const float h0 = __uint_as_float(ph[j] << 16), h1 = __uint_as_float(ph[j] & 0xFFFF0000u);
      pl[j] = pack_bf16x2(p[2 * j] - h0, p[2 * j + 1] - h1);
    }
    const float al0 = __shfl_sync(0xFFFFFFFFu, alpha, 8 * tq);
    const float al1 = __shfl_sync(0xFFFFFFFFu, alpha, 8 * tq + 4);
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
      acc[mi][0] *= al0;
      acc[mi][1] *= al1;
      acc[mi][2] *= al0;
      acc[mi][3] *= al1;
    }

    // ---- O^T += V^T P^T for channels 32warp + 16mi + {g, g+8}
    int vpre_lo = 0, vpre_hi = 0;
    if (md.modeV == GAAC_MODE_SLOT && md.escV > 0) tag_word_prefix(tV, lane, vpre_lo, vpre_hi);
    const int vsrc = warp < 2 ? vpre_lo : vpre_hi;
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
      const int cA = 32 * warp + 16 * mi + g, cB = cA + 8;
      uint32_t va[8], vb[8];
      const int wpA = __shfl_sync(0xFFFFFFFFu, vsrc, (cA >> 1) & 31);
      const int wpB = __shfl_sync(0xFFFFFFFFu, vsrc, (cB >> 1) & 31);
      if (md.modeV == GAAC_MODE_SLOT) {
        v_slot(tV, cA, tq, v3[2 * mi], v4[2 * mi], wpA, md.escV, va, &bad);
        v_slot(tV, cB, tq, v3[2 * mi + 1], v4[2 * mi + 1], wpB, md.escV, vb, &bad);
      } else if (md.modeV == GAAC_MODE_RAW) {
        v_raw(tV, cA, tq, va);
        v_raw(tV, cB, tq, vb);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) va[j] = vb[j] = 0u;
      }
      if (nv < kBlock) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int tt = 16 * tq + 2 * m;
          const uint32_t keep = (tt < nv ? 0x0000FFFFu : 0u) | (tt + 1 < nv ? 0xFFFF0000u : 0u);
          va[m] &= keep;
          vb[m] &= keep;
        }
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(acc[mi], va[2 * ks], vb[2 * ks], va[2 * ks + 1], vb[2 * ks + 1], ph[2 * ks], ph[2 * ks + 1]);
        mma_bf16(acc[mi], va[2 * ks], vb[2 * ks], va[2 * ks + 1], vb[2 * ks + 1], pl[2 * ks], pl[2 * ks + 1]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[st]);
  }
  if (bad) report(a.status, GAAC_EFORMAT);
  // Every issued copy was awaited above; after a timed-out wait, wait once
  // more (bounded) so that no copy is still landing when the CTA exits.
  if (warp == 0 && lane == 0) {
    for (int i = max(0, n_my - kStages); i < n_my; ++i)
      mbar_wait(&sm.full[i % kStages], (i / kStages) & 1, a.status, 1u << 20);
  }

  float* part = a.part + ((static_cast<size_t>(b) * a.Hkv + h) * a.n_splits + split) * kPartFloats;
  if (warp == 0 && tq == 0) {
    part[2 * g] = m_run;
    part[2 * g + 1] = l_run;
  }
#pragma unroll
  for (int mi = 0; mi < 2; ++mi) {
    const int cA = 32 * warp + 16 * mi + g, cB = cA + 8;
    float* pa = part + 2 * kRPad;
    pa[(2 * tq) * kD + cA] = acc[mi][0];
    pa[(2 * tq + 1) * kD + cA] = acc[mi][1];
    pa[(2 * tq) * kD + cB] = acc[mi][2];
    pa[(2 * tq + 1) * kD + cB] = acc[mi][3];
  }
}

// grid (Hq, batch), 128 threads: log-sum-exp merge of the split partials.
__global__ void __launch_bounds__(kD) attn_combine_kernel(const float* __restrict__ part, int Hq, int Hkv, int r,
                                                          int n_splits, float* __restrict__ out) {
  const int hq = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
  const int h = hq / r, n = hq % r;
  const float* base = part + (static_cast<size_t>(b) * Hkv + h) * n_splits * kPartFloats;
  float m = -INFINITY;
  for (int s = 0; s < n_splits; ++s) m = fmaxf(m, base[static_cast<size_t>(s) * kPartFloats + 2 * n]);
  float num = 0.f, den = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < n_splits; ++s) {
      const float* ps = base + static_cast<size_t>(s) * kPartFloats;
      const float ms = ps[2 * n];
      if (ms == -INFINITY) continue;
      const float w = exp2f(ms - m);
      den += ps[2 * n + 1] * w;
      num += ps[2 * kRPad + n * kD + c] * w;
    }
  }
  out[(static_cast<size_t>(b) * Hq + hq) * kD + c] = den > 0.f ? num / den : 0.f;
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
  const long long target = 2LL * device_sms();  // two CTAs per SM
  const long long pairs = static_cast<long long>(batch) * n_kv_heads;
  long long s = (target + pairs - 1) / pairs;
  if (s > max_blocks) s = max_blocks;
  return static_cast<int>(s < 1 ? 1 : s);
}

extern "C" size_t gaac_attention_workspace(int batch, int n_kv_heads, int max_blocks, int n_splits) {
  if (n_splits <= 0) n_splits = gaac_attention_auto_splits(batch, n_kv_heads, max_blocks);
  if (batch <= 0 || n_kv_heads <= 0) return 0;
  return static_cast<size_t>(batch) * n_kv_heads * n_splits * kPartFloats * sizeof(float);
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
  a.status = d_status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  attn_split_kernel<<<dim3(n_splits, n_kv_heads, batch), kAttThreads, sizeof(AttSmem), st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return GAAC_ECUDA;
  attn_combine_kernel<<<dim3(n_q_heads, batch), kD, 0, st>>>(a.part, n_q_heads, n_kv_heads, a.r, n_splits, out);
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
  return gaac_decode_attention(q, batch, n_q_heads, n_kv_heads, max_blocks, seq_lens, table, pools, base3, base4,
                               scale, ns, out, scratch, kStaticScratchBytes, d_status, stream);
}
