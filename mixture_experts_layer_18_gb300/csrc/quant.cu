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

// Both quantisations of one bf16 tensor from a single read, tensor-core
// scale layout: row-wise (blocks of 32 along each row; MN = rows, K = the
// C columns) and column-wise (blocks of 32 rows down each column; MN =
// columns, K = rows, kgroups = ceil(R / 128)).  A block of 256 threads
// stages a 64-row x 128-column tile (two 32-row blocks) in shared memory,
// finds its 256 column-block maxima (one per thread) and its row-block
// maxima (pairs of threads, one shuffle), then every thread encodes 16
// consecutive elements of a row twice and writes each set of 16 codes with
// one 16-byte store (eight threads cover a row: coalesced); the next tile's
// loads are issued before this one is encoded.  Codes and scale bytes are those of the
// two kernels above.  Rows at or past `rows` (a device value, e.g. the
// padded row total) are neither read nor written; they start on a 32-row
// boundary.  qc == nullptr skips the column-wise output.
// SRC: 0 = row r of src; 1 = token row assign_of_row[r] / k of src (the
// dispatch gather; pad rows read as 0); 2 = the same gather, with the
// column-wise encoding taken of gate[a] * row rounded to bf16 (the
// gate-scaled gradient rows of the weight-gradient GEMM).
template <int SRC>
__global__ void __launch_bounds__(256, 4) quant_dual_kernel(
    const __nv_bfloat16* __restrict__ src, int R, int C, int ld, const int32_t* __restrict__ rows_dev,
    const int32_t* __restrict__ assign_of_row, int k, int n_assign, const float* __restrict__ gate,
    int32_t* status, uint8_t* __restrict__ qr, uint8_t* __restrict__ sr, uint8_t* __restrict__ qc,
    uint8_t* __restrict__ sc) {
  constexpr int TR = 64;                             // tile rows (two 32-row blocks)
  constexpr int PITCH = 68;                          // words per tile row (272 B)
  __shared__ __align__(16) uint32_t tile[TR][PITCH];                  // TR rows x 128 bf16
  __shared__ __align__(16) uint32_t tileg[SRC == 2 ? TR : 1][PITCH];  // bf16(gate * row)
  __shared__ float s_cinv[2][128];                   // column-wise 2^-s per (row block, column)
  const int rows = rows_dev ? min(*rows_dev, R) : R;
  const int nct = C / 128, nrt = (rows + TR - 1) / TR;
  const int64_t ntiles = (int64_t)nrt * nct;
  const int64_t kg_rows = (R + 127) / 128;
  // this thread's four 16-byte chunks of a tile (and, gathered, their gate)
  uint4 v[4];
  float gv[4];
  auto fetch = [&](int64_t t) {
    const int rt = (int)(t / nct), ct = (int)(t - (int64_t)rt * nct);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ch = threadIdx.x + 256 * i;
      const int r = rt * TR + (ch >> 4), c = ch & 15;
      v[i] = make_uint4(0, 0, 0, 0);
      gv[i] = 0.f;
      if (r < rows) {
        if constexpr (SRC == 0) {
          v[i] = __ldg(reinterpret_cast<const uint4*>(src + (size_t)r * ld + ct * 128) + c);
        } else {
          const int a = assign_of_row[r];
          const bool ok = a >= 0 && a < n_assign;
          if (a >= n_assign && c == 0) report(status, MOE_ERR_BAD_INDEX);
          if (ok) {
            v[i] = __ldg(reinterpret_cast<const uint4*>(src + (size_t)(a / k) * ld + ct * 128) + c);
            if constexpr (SRC == 2) gv[i] = gate[a];
          }
        }
      }
    }
  };
  int64_t t = blockIdx.x;
  if (t < ntiles) fetch(t);
  for (; t < ntiles; t += gridDim.x) {
    const int rt = (int)(t / nct), ct = (int)(t - (int64_t)rt * nct);
    const int r0 = rt * TR, c0 = ct * 128;
    const int nrb = min(TR, rows - r0) / 32;        // 32-row blocks of this tile (1 or 2)
    __syncthreads();   // previous tile fully consumed
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ch = threadIdx.x + 256 * i;
      const int r = ch >> 4, c = ch & 15;
      *reinterpret_cast<uint4*>(&tile[r][4 * c]) = v[i];
      if constexpr (SRC == 2) {
        const float g = gv[i];
        *reinterpret_cast<uint4*>(&tileg[r][4 * c]) =
            make_uint4(pack_bf16(g * bf16_lo(v[i].x), g * bf16_hi(v[i].x)),
                       pack_bf16(g * bf16_lo(v[i].y), g * bf16_hi(v[i].y)),
                       pack_bf16(g * bf16_lo(v[i].z), g * bf16_hi(v[i].z)),
                       pack_bf16(g * bf16_lo(v[i].w), g * bf16_hi(v[i].w)));
      }
    }
    __syncthreads();
    if (t + gridDim.x < ntiles) fetch(t + gridDim.x);   // next tile's loads overlap this one
    const uint32_t (*ctile)[PITCH] = SRC == 2 ? tileg : tile;   // column-wise source
    // column maxima: thread = (row block, column)
    if (qc) {
      const int rb = threadIdx.x >> 7, c = threadIdx.x & 127;
      if (rb < nrb) {
        float am = 0.f;
#pragma unroll 8
        for (int r = 0; r < 32; ++r) {
          const uint32_t w = ctile[32 * rb + r][c >> 1];
          am = fmaxf(am, fabsf((c & 1) ? bf16_hi(w) : bf16_lo(w)));
        }
        const int sb = mx_scale_byte(am);
        s_cinv[rb][c] = mx_inv_scale(sb);
        sc[mma_scale_index(c0 + c, (r0 >> 5) + rb, kg_rows)] = (uint8_t)sb;
      }
    }
    // row-wise: thread = (row, 16-column group); it and its neighbour
    // (group ^ 1) form one 32-column block
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int er = (threadIdx.x >> 3) + 32 * p, eg = threadIdx.x & 7;
      if (er >= 32 * nrb) break;
      uint32_t w[8];
      const uint4 v0 = *reinterpret_cast<const uint4*>(&tile[er][8 * eg]);
      const uint4 v1 = *reinterpret_cast<const uint4*>(&tile[er][8 * eg + 4]);
      w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
      w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
      float am = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) am = fmaxf(am, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
      const int sb = mx_scale_byte(am);
      const float inv = mx_inv_scale(sb);
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t p0 = e4m3x2(bf16_lo(w[2 * i]) * inv, bf16_hi(w[2 * i]) * inv);
        const uint32_t p1 = e4m3x2(bf16_lo(w[2 * i + 1]) * inv, bf16_hi(w[2 * i + 1]) * inv);
        o[i] = p0 | (p1 << 16);
      }
      *reinterpret_cast<uint4*>(qr + (size_t)(r0 + er) * C + c0 + 16 * eg) =
          make_uint4(o[0], o[1], o[2], o[3]);
      if ((eg & 1) == 0) sr[mma_scale_index(r0 + er, (c0 >> 5) + (eg >> 1), nct)] = (uint8_t)sb;
    }
    if (qc) {
      __syncthreads();   // column scales ready
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int er = (threadIdx.x >> 3) + 32 * p, eg = threadIdx.x & 7;
        if (er >= 32 * nrb) break;
        uint32_t w[8];
        const uint4 v0 = *reinterpret_cast<const uint4*>(&ctile[er][8 * eg]);
        const uint4 v1 = *reinterpret_cast<const uint4*>(&ctile[er][8 * eg + 4]);
        w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
        w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float* ci = &s_cinv[p][16 * eg + 4 * i];
          o[i] = (uint32_t)e4m3x2(bf16_lo(w[2 * i]) * ci[0], bf16_hi(w[2 * i]) * ci[1]) |
                 ((uint32_t)e4m3x2(bf16_lo(w[2 * i + 1]) * ci[2], bf16_hi(w[2 * i + 1]) * ci[3]) << 16);
        }
        *reinterpret_cast<uint4*>(qc + (size_t)(r0 + er) * C + c0 + 16 * eg) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
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

cudaError_t launch_quantize_dual(const void* src, int R, int C, int ld, const int32_t* rows_dev,
                                 uint8_t* qr, uint8_t* sr, uint8_t* qc, uint8_t* sc,
                                 cudaStream_t s, const DualGather* gather) {
  const int64_t tiles = (int64_t)((R + 63) / 64) * (C / 128);
  if (tiles == 0) return cudaSuccess;
  const int cap = grid_cap();
  const int blocks = (int)(tiles < cap ? tiles : cap);
  const __nv_bfloat16* x = (const __nv_bfloat16*)src;
  if (!gather)
    quant_dual_kernel<0><<<blocks, 256, 0, s>>>(x, R, C, ld, rows_dev, nullptr, 1, 0, nullptr,
                                                nullptr, qr, sr, qc, sc);
  else if (!gather->gate)
    quant_dual_kernel<1><<<blocks, 256, 0, s>>>(x, R, C, ld, rows_dev, gather->assign_of_row,
                                                gather->k, gather->n_assign, nullptr,
                                                gather->status, qr, sr, qc, sc);
  else
    quant_dual_kernel<2><<<blocks, 256, 0, s>>>(x, R, C, ld, rows_dev, gather->assign_of_row,
                                                gather->k, gather->n_assign, gather->gate,
                                                gather->status, qr, sr, qc, sc);
  return cudaGetLastError();
}

}  // namespace moe
