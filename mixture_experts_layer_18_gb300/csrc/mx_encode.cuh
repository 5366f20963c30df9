// mx_encode.cuh - MXFP8 encoding rules shared by the quantiser kernels and
// the GEMM epilogue that encodes the SwiGLU output directly.
//
// OCP Microscaling Formats (MX) v1.0, MXFP8: E4M3 elements in blocks of 32
// sharing one E8M0 scale; "Accelerating dropless MoE in JAX with NVIDIA
// Transformer Engine", 03 (MXFP8 quantisation, group-aware along tokens).
#pragma once

#include <cuda_fp8.h>
#include <cstdint>

namespace moe {

// Scale byte of a block with max |x| = amax: s = floor(log2(amax)) - 8
// (E4M3's largest exponent), clamped at -127, stored as s + 127.
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

// Scale slots (MN indices in the atom layout above) of B operands of the
// block-scaled GEMMs, whose tiles are kMxTileN = 192 B columns wide: each
// expert segment of `seg` indices is cut into 192-wide tiles and every tile
// gets two whole atoms (256 slots, the last 64 unused), so the scales of a
// tile start on an atom boundary and fill the tensor-memory scale columns of
// its MMAs in order.  Index m of segment e has slot
// e * mx_tile_slots(seg) + mx_tile_pos(m).
constexpr int kMxTileN = 192;
__host__ __device__ __forceinline__ int64_t mx_tile_slots(int64_t seg) {
  return (seg + kMxTileN - 1) / kMxTileN * 256;
}
// slot of index m inside its segment (32-bit, constant divisor)
__device__ __forceinline__ int mx_tile_pos(int m) {
  return (m / kMxTileN) * 256 + m % kMxTileN;
}

// Two E4M3 codes (round to nearest even, saturating), lo in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

}  // namespace moe
