// quant.cu - MXFP8 quantiser (E4M3 elements, 32-element blocks, E8M0
// scales).
//
// "Accelerating dropless MoE in JAX with NVIDIA Transformer Engine", 03:
// group-aware MXFP8 quantisation (blocks never straddle two experts' token
// groups); "Prime Intellect releases Prime Mega MoE" (MarkTechPost): MXFP8 on
// Blackwell.  Element and scale formats: OCP MX v1.0.
//
// Rule per 32-element block: s = floor(log2(amax)) - 8 clamped to
// [-127, 127]; codes = E4M3(x * 2^-s), nearest-even, saturating to +-448;
// scale byte = s + 127.  For a finite fp32 amax with biased exponent field f,
// floor(log2(amax)) - 8 = f - 135 for normal numbers, and zero / subnormal
// amax (f = 0) gives s <= -127, so the clamped exponent is max(f - 135, -127)
// and the scale byte is max(f - 8, 0).  Multiplying by 2^-s is exact, so the
// only rounding is the hardware E4M3 conversion (round-to-nearest-even with
// saturation to the largest finite value).
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

__device__ __forceinline__ int mx_scale_byte(float amax) {
  const int f = (__float_as_uint(amax) >> 23) & 0xFF;
  return f > 8 ? f - 8 : 0;
}

// 2^-s as fp32 for a scale byte b (s = b - 127, so 2^-s = 2^(127 - b)).
__device__ __forceinline__ float mx_inv_scale(int b) {
  return __uint_as_float((uint32_t)(254 - b) << 23);
}

// Byte index of the scale of (MN index mn, 32-element K block kb) in the
// tensor-core scale-factor layout: 512-byte atoms cover 128 MN indices x 4 K
// blocks, atom (mn/128, kb/4) at (mn/128) * kgroups + kb/4, and inside an atom
// byte (mn % 32) * 16 + ((mn / 32) % 4) * 4 + kb % 4.  Copied to tensor memory
// with tcgen05.cp (32x128b, replicated to the four lane quarters), row mn
// reads lane mn, column mn / 32, byte kb % 4.
__device__ __forceinline__ size_t mma_scale_index(int64_t mn, int kb, int64_t kgroups) {
  return ((size_t)(mn >> 7) * kgroups + (kb >> 2)) * 512 + (size_t)(mn & 31) * 16 +
         (size_t)((mn >> 5) & 3) * 4 + (kb & 3);
}

__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// axis 1: one thread per 32-element block of a row (64 contiguous bytes in,
// 32 bytes of codes + 1 scale byte out).
// LAYOUT 0: scales [R, C/32]; LAYOUT 1: tensor-core atoms with K along the
// columns (rows padded to 128 with scale byte 0, their codes untouched).
template <int LAYOUT>
__global__ void __launch_bounds__(256) quant_rowwise_kernel(const __nv_bfloat16* __restrict__ src,
                                                            int R, int C, int ld,
                                                            uint8_t* __restrict__ q,
                                                            uint8_t* __restrict__ scales) {
  const int nbc = C / 32;
  const int Rp = LAYOUT == 1 ? (R + 127) / 128 * 128 : R;
  const int64_t nblk = (int64_t)Rp * nbc;
  for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nblk;
       b += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(b / nbc), cb = (int)(b - (int64_t)r * nbc);
    if (LAYOUT == 1 && r >= R) {
      scales[mma_scale_index(r, cb, C / 128)] = 0;
      continue;
    }
    const uint4* s = reinterpret_cast<const uint4*>(src + (size_t)r * ld + cb * 32);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(s + i);
      w[4 * i + 0] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
    const int sb = mx_scale_byte(amax);
    const float inv = mx_inv_scale(sb);
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t p0 = e4m3x2(bf16_lo(w[2 * i]) * inv, bf16_hi(w[2 * i]) * inv);
      const uint32_t p1 = e4m3x2(bf16_lo(w[2 * i + 1]) * inv, bf16_hi(w[2 * i + 1]) * inv);
      o[i] = p0 | (p1 << 16);
    }
    uint4* d = reinterpret_cast<uint4*>(q + (size_t)r * C + cb * 32);
    d[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d[1] = make_uint4(o[4], o[5], o[6], o[7]);
    if (LAYOUT == 1)
      scales[mma_scale_index(r, cb, C / 128)] = (uint8_t)sb;
    else
      scales[(size_t)r * nbc + cb] = (uint8_t)sb;
  }
}

// axis 0: one thread per (32-row block, column pair).  Lanes take adjacent
// column pairs, so every row access of a warp is one contiguous segment.
// LAYOUT 0: scales [R/32, C]; LAYOUT 1: tensor-core atoms with K along the
// rows (MN index = column, kgroups = ceil(R / 128)).
template <int LAYOUT>
__global__ void __launch_bounds__(256) quant_colwise_kernel(const __nv_bfloat16* __restrict__ src,
                                                            int R, int C, int ld,
                                                            const int32_t* __restrict__ go, int G,
                                                            uint8_t* __restrict__ q,
                                                            uint8_t* __restrict__ scales,
                                                            int32_t* status) {
  int rows = R;
  if (go) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      for (int g = 0; g <= G; ++g)
        if ((go[g] & 31) || go[g] < 0 || go[g] > R || (g > 0 && go[g] < go[g - 1])) {
          report(status, MOE_ERR_INVALID_ARG);
          break;
        }
    }
    rows = go[G];
    if (rows > R || rows < 0) return;
  }
  const int npair = C / 2;
  const int nrb = rows / 32;
  const int64_t n = (int64_t)nrb * npair;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int rb = (int)(i / npair), cp = (int)(i - (int64_t)rb * npair);
    const uint32_t* s = reinterpret_cast<const uint32_t*>(src + (size_t)rb * 32 * ld + 2 * cp);
    uint32_t w[32];
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      w[r] = __ldg(s + (size_t)r * (ld / 2));
      a0 = fmaxf(a0, fabsf(bf16_lo(w[r])));
      a1 = fmaxf(a1, fabsf(bf16_hi(w[r])));
    }
    const int sb0 = mx_scale_byte(a0), sb1 = mx_scale_byte(a1);
    const float inv0 = mx_inv_scale(sb0), inv1 = mx_inv_scale(sb1);
    uint16_t* d = reinterpret_cast<uint16_t*>(q + (size_t)rb * 32 * C + 2 * cp);
#pragma unroll
    for (int r = 0; r < 32; ++r) d[(size_t)r * (C / 2)] = e4m3x2(bf16_lo(w[r]) * inv0, bf16_hi(w[r]) * inv1);
    if (LAYOUT == 1) {
      const int64_t kg = (R + 127) / 128;
      scales[mma_scale_index(2 * cp, rb, kg)] = (uint8_t)sb0;
      scales[mma_scale_index(2 * cp + 1, rb, kg)] = (uint8_t)sb1;
    } else {
      scales[(size_t)rb * C + 2 * cp] = (uint8_t)sb0;
      scales[(size_t)rb * C + 2 * cp + 1] = (uint8_t)sb1;
    }
  }
}

int grid_cap() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return (sms > 0 ? sms : 1) * 8;
}

}  // namespace

cudaError_t launch_quantize(const void* src, int R, int C, int ld, int axis,
                            const int32_t* group_offsets, int G, uint8_t* q, uint8_t* scales,
                            int32_t* status, cudaStream_t s, int layout) {
  const int Rp = layout == 1 && axis == 1 ? (R + 127) / 128 * 128 : R;
  const int64_t work = axis == 1 ? (int64_t)Rp * (C / 32) : (int64_t)(R / 32) * (C / 2);
  if (work == 0 && !group_offsets) return cudaSuccess;
  int64_t blocks = (work + 255) / 256;
  const int cap = grid_cap();
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const __nv_bfloat16* x = (const __nv_bfloat16*)src;
  if (axis == 1 && layout == 1)
    quant_rowwise_kernel<1><<<(int)blocks, 256, 0, s>>>(x, R, C, ld, q, scales);
  else if (axis == 1)
    quant_rowwise_kernel<0><<<(int)blocks, 256, 0, s>>>(x, R, C, ld, q, scales);
  else if (layout == 1)
    quant_colwise_kernel<1><<<(int)blocks, 256, 0, s>>>(x, R, C, ld, group_offsets, G, q, scales,
                                                        status);
  else
    quant_colwise_kernel<0><<<(int)blocks, 256, 0, s>>>(x, R, C, ld, group_offsets, G, q, scales,
                                                        status);
  return cudaGetLastError();
}

}  // namespace moe
