// Calibration of the per-head-channel exponent windows.
//
// "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference on
// Personal Devices", section 3.1: each head-channel gets one window of 8 and one
// of 16 consecutive exponents, fixed from calibration data (section 4.7.1
// studies which data).  Here the window is the one holding the most calibration
// exponents; ties go to the smallest base.
//
// One CTA per kv-head, one thread per channel: the thread owns its channel's
// 256-bin histogram column in shared memory (no atomics), loads are coalesced
// across the 128 channels of a token.
#include <cuda_runtime.h>

#include "common.cuh"

namespace gaac {

__global__ void __launch_bounds__(kD) calibrate_kernel(const uint16_t* __restrict__ x, int64_t n_tok,
                                                       int64_t tok_stride, uint8_t* __restrict__ base3,
                                                       uint8_t* __restrict__ base4) {
  extern __shared__ uint16_t hist[];  // [256][128]
  const int h = blockIdx.x, c = threadIdx.x;
  for (int bin = 0; bin < 256; ++bin) hist[bin * kD + c] = 0;
  const uint16_t* p = x + static_cast<int64_t>(h) * kD + c;
  for (int64_t t = 0; t < n_tok; ++t) {
    const uint32_t e = (p[t * tok_stride] >> 7) & 0xFFu;
    hist[e * kD + c] += 1;
  }
  // Sliding windows over the bins; strict '>' keeps the smallest base on ties.
  int best3 = 0, arg3 = 0, best4 = 0, arg4 = 0, sum8 = 0, sum16 = 0;
  for (int i = 0; i < 16; ++i) {
    const int v = hist[i * kD + c];
    sum16 += v;
    if (i < 8) sum8 += v;
  }
  best3 = sum8;
  best4 = sum16;
  for (int b = 1; b + 8 <= 256; ++b) {
    sum8 += hist[(b + 7) * kD + c] - hist[(b - 1) * kD + c];
    if (sum8 > best3) {
      best3 = sum8;
      arg3 = b;
    }
  }
  for (int b = 1; b + 16 <= 256; ++b) {
    sum16 += hist[(b + 15) * kD + c] - hist[(b - 1) * kD + c];
    if (sum16 > best4) {
      best4 = sum16;
      arg4 = b;
    }
  }
  base3[h * kD + c] = static_cast<uint8_t>(arg3);
  base4[h * kD + c] = static_cast<uint8_t>(arg4);
}

}  // namespace gaac

using namespace gaac;

extern "C" int gaac_calibrate(const uint16_t* x, int64_t n_tok, int64_t tok_stride, int n_kv_heads, uint8_t* base3,
                              uint8_t* base4, int32_t* d_status, void* stream) {
  (void)d_status;
  if (x == nullptr || base3 == nullptr || base4 == nullptr) return GAAC_EINVAL;
  if (n_tok < 1 || n_tok > 65535 || n_kv_heads <= 0 || n_kv_heads > 65535 ||
      tok_stride < static_cast<int64_t>(n_kv_heads) * kD)
    return GAAC_EINVAL;
  const size_t smem = 256 * kD * sizeof(uint16_t);
  static bool attr_done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GAAC_ECUDA;
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(calibrate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return GAAC_ECUDA;
    attr_done[dev] = true;
  }
  calibrate_kernel<<<n_kv_heads, kD, smem, static_cast<cudaStream_t>(stream)>>>(x, n_tok, tok_stride, base3, base4);
  return cudaGetLastError() == cudaSuccess ? GAAC_OK : GAAC_ECUDA;
}
