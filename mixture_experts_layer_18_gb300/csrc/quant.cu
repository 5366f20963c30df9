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
#include "mx_encode.cuh"

namespace moe {

namespace {

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
// stages 128-row x 128-column tiles in shared memory with asynchronous
// copies, double-buffered (the next tile's copies are in flight while this
// one is encoded).  Threads 0-127 each take a column pair of a 32-row block
// (its 32 words in registers: maxima, codes, 2-byte stores down the
// column, 64 contiguous bytes per warp and row); threads 128-255 each take
// (row, 32-column block) tasks (16 words: maximum, codes, two 16-byte
// stores).  Codes and scale bytes are those of the two kernels above.
// Rows at or past `rows` (a device value, e.g. the padded row total) are
// neither read nor written; they start on a 32-row boundary.  qc == nullptr
// skips the column-wise output.  Gathered passes copy each tile's row
// assignments into shared memory two tiles ahead of its data copies, and
// its gates beside its data, all with asynchronous copies, so no thread ever
// waits on a global index load before issuing a tile's copies.
// SRC: 0 = row r of src; 1 = token row assign_of_row[r] / k of src (the
// dispatch gather; pad rows read as 0); 2 = the same gather, with the
// column-wise encoding taken of gate[a] * row rounded to bf16 (the
// gate-scaled gradient rows of the weight-gradient GEMM).
constexpr int kDualRows = 128;                     // tile rows (32-row blocks of K)
constexpr int kDualPitch = 68;                     // words per tile row (272 B)
constexpr int kDualTileWords = kDualRows * kDualPitch;

// 16-byte asynchronous copy global -> shared; src_bytes 0 writes zeros.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes)
               : "memory");
}
// 4-byte asynchronous copy global -> shared; src_bytes 0 writes zeros.
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(smem_dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev() {   // all but the newest group landed
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// Running max of |x| over bf16 pairs: for non-negative bf16 values the bit
// patterns order like the numbers, so clearing the sign bits and taking a
// per-halfword unsigned max gives both maxima at once (finite and infinite
// inputs; the same result as fmaxf of the absolute values).
__device__ __forceinline__ uint32_t absmax2(uint32_t acc, uint32_t w) {
  return __vmaxu2(acc, w & 0x7FFF7FFFu);
}
__device__ __forceinline__ float absmax_lo(uint32_t acc) { return __uint_as_float(acc << 16); }
__device__ __forceinline__ float absmax_hi(uint32_t acc) { return __uint_as_float(acc & 0xFFFF0000u); }

// two tile buffers, then gates [2][rows] and row assignments [3][rows]
template <int SRC>
size_t dual_smem_bytes() {
  return (size_t)2 * kDualTileWords * 4 + 5 * kDualRows * 4;
}

// Column index of the transposed column-wise output for column c: the
// block-scaled gate/up GEMM reads W13's encoding with 96 gate and 96 up
// columns per 192-wide tile (perm 1, C = 2I), the others in order.
__device__ __forceinline__ int dual_perm(int c, int C, int perm) {
  if (!perm) return c;
  const int half = C / 2, tn = kMxTileN / 2;
  return c < half ? (c / tn) * kMxTileN + c % tn : ((c - half) / tn) * kMxTileN + tn + (c - half) % tn;
}

template <int SRC>
__global__ void __launch_bounds__(256, 3) quant_dual_kernel(
    const __nv_bfloat16* __restrict__ src, int R, int C, int ld, const int32_t* __restrict__ rows_dev,
    const int32_t* __restrict__ assign_of_row, int k, int n_assign, const float* __restrict__ gate,
    int32_t* status, uint8_t* __restrict__ qr, uint8_t* __restrict__ sr, uint8_t* __restrict__ qc,
    uint8_t* __restrict__ sc, DualOut out) {
  constexpr int TR = kDualRows, PITCH = kDualPitch;
  extern __shared__ __align__(16) uint32_t dsm[];
  uint32_t (*tbuf)[TR][PITCH] = reinterpret_cast<uint32_t (*)[TR][PITCH]>(dsm);   // [2]
  float* s_g = reinterpret_cast<float*>(dsm + 2 * kDualTileWords);   // [2][TR] gates (SRC 2)
  int32_t* s_a = reinterpret_cast<int32_t*>(s_g + 2 * TR);            // [3][TR] assignments
  const int rows = rows_dev ? min(*rows_dev, R) : R;
  const int nct = C / 128, nrt = (rows + TR - 1) / TR;
  const int64_t ntiles = (int64_t)nrt * nct;
  const int64_t kg_rows = (R + 127) / 128;
  // Gathered tiles: the assignment of each row of tile t lands in slot
  // (t's iteration) % 3 two tiles before the tile's data copies are issued
  // (rows at or past `rows` read as 0 and are skipped by the row test).
  auto copy_rows = [&](int64_t t, int slot) {
    if (SRC != 0 && threadIdx.x < TR) {
      const int r = (int)(t / nct) * TR + threadIdx.x;
      const bool in = r < rows;
      cp_async4(&s_a[slot * TR + threadIdx.x], assign_of_row + (in ? r : 0), in ? 4 : 0);
    }
  };
  // issue this thread's 16-byte copies of tile t into buffer b (gathered:
  // token rows from the assignments in `slot`, and each row's gate)
  constexpr int NCH = TR / 16;                     // 16-byte chunks per thread per tile
  auto issue = [&](int64_t t, int b, int slot) {
    const int rt = (int)(t / nct), ct = (int)(t - (int64_t)rt * nct);
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int ch = threadIdx.x + 256 * i;
      const int rl = ch >> 4, c = ch & 15;
      const int r = rt * TR + rl;
      const __nv_bfloat16* p = src;
      int bytes = 0;
      if constexpr (SRC == 0) {
        if (r < rows) {
          p = src + (size_t)r * ld + ct * 128 + 8 * c;
          bytes = 16;
        }
      } else {
        const int a = r < rows ? s_a[slot * TR + rl] : -1;
        if (a >= n_assign && c == 0) report(status, MOE_ERR_BAD_INDEX);
        const bool ok = a >= 0 && a < n_assign;
        if (ok) {
          p = src + (size_t)(a / k) * ld + ct * 128 + 8 * c;
          bytes = 16;
        }
        if (SRC == 2 && c == 0) cp_async4(&s_g[b * TR + rl], ok ? gate + a : gate, ok ? 4 : 0);
      }
      cp_async16(&tbuf[b][rl][4 * c], p, bytes);
    }
  };
  int64_t t = blockIdx.x;
  const int64_t G = gridDim.x;
  if constexpr (SRC != 0) {
    if (t < ntiles) copy_rows(t, 0);
    if (t + G < ntiles) copy_rows(t + G, 1);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
  }
  if (t < ntiles) {
    issue(t, 0, 0);
    if (t + 2 * G < ntiles) copy_rows(t + 2 * G, 2);
  }
  cp_async_commit();
  if constexpr (SRC != 0) __syncthreads();   // slot 0 is read before it is refilled
  for (int b = 0, j = 0; t < ntiles; t += G, b ^= 1, ++j) {
    const int rt = (int)(t / nct), ct = (int)(t - (int64_t)rt * nct);
    const int r0 = rt * TR, c0 = ct * 128;
    const int nrb = min(TR, rows - r0) / 32;        // 32-row blocks of this tile
    if (t + G < ntiles) {
      issue(t + G, b ^ 1, (j + 1) % 3);            // next tile's copies in flight
      // slot j % 3 (this tile's assignments) was read before the last barrier
      if (t + 3 * G < ntiles) copy_rows(t + 3 * G, j % 3);
    }
    cp_async_commit();
    cp_async_wait_prev();
    __syncthreads();   // tile t in buffer b, from every thread's copies
    const uint32_t (*tile)[PITCH] = tbuf[b];
    // B-operand outputs: the tile's rows lie in one segment (segment lengths
    // are multiples of 128), so its segment index is computed once
    const int64_t rseg = out.row_seg > 0 ? r0 / out.row_seg : 0;
    const int64_t rslot0 = out.row_seg > 0 ? rseg * mx_tile_slots(out.row_seg) : 0;
    const int rbase = out.row_seg > 0 ? (int)(r0 - rseg * out.row_seg) : 0;
    const int64_t cseg = out.col_ld > 0 ? r0 / out.col_seg : 0;
    const int ckr0 = out.col_ld > 0 ? (int)(r0 - cseg * out.col_seg) : 0;
    if (threadIdx.x < 128 && qc && out.col_ld > 0) {
      // column-wise, stored transposed (K-major B): thread = one column of
      // the tile, whose codes for the tile's 32-row blocks are consecutive
      // bytes of its output row, written as whole 32-byte pieces in turn
      const int c = threadIdx.x, j = c >> 1, hi = c & 1;
      const int pc = dual_perm(c0 + c, C, out.col_perm);
      const int64_t orow = cseg * C + pc;
      const int64_t kg = (out.col_seg + 127) / 128;
      const int64_t slot = cseg * mx_tile_slots(C) + mx_tile_pos(pc);
      uint4* dst = reinterpret_cast<uint4*>(qc + (size_t)orow * out.col_ld + ckr0);
      for (int rb = 0; rb < nrb; ++rb) {
        float v[32];
        float am = 0.f;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
          const uint32_t wv = tile[32 * rb + r][j];
          float x = hi ? bf16_hi(wv) : bf16_lo(wv);
          if constexpr (SRC == 2)   // gate-scaled rows, rounded to bf16 once
            x = __bfloat162float(__float2bfloat16_rn(s_g[b * TR + 32 * rb + r] * x));
          v[r] = x;
          am = fmaxf(am, fabsf(x));
        }
        const int sbc = mx_scale_byte(am);
        const float inv = mx_inv_scale(sbc);
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          o[i] = (uint32_t)e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv) |
                 ((uint32_t)e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv) << 16);
        dst[2 * rb] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[2 * rb + 1] = make_uint4(o[4], o[5], o[6], o[7]);
        sc[mma_scale_index(slot, (ckr0 >> 5) + rb, kg)] = (uint8_t)sbc;
      }
    } else if (threadIdx.x < 128) {
      // column-wise: thread = (32-row block, column pair); the 32 words of
      // its two columns in registers, maxima and codes from them
      for (int rb = threadIdx.x >> 6; rb < nrb; rb += 2) {
        if (!qc) break;
        const int j = threadIdx.x & 63;
        uint32_t w[32];
        uint32_t acc = 0;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
          w[r] = tile[32 * rb + r][j];
          if constexpr (SRC == 2) {   // gate-scaled rows, rounded to bf16 once
            const float g = s_g[b * TR + 32 * rb + r];
            w[r] = pack_bf16(g * bf16_lo(w[r]), g * bf16_hi(w[r]));
          }
          acc = absmax2(acc, w[r]);
        }
        const int sb0 = mx_scale_byte(absmax_lo(acc)), sb1 = mx_scale_byte(absmax_hi(acc));
        const float inv0 = mx_inv_scale(sb0), inv1 = mx_inv_scale(sb1);
        uint16_t* d = reinterpret_cast<uint16_t*>(qc + (size_t)(r0 + 32 * rb) * C + c0 + 2 * j);
#pragma unroll
        for (int r = 0; r < 32; ++r)
          d[(size_t)r * (C / 2)] = e4m3x2(bf16_lo(w[r]) * inv0, bf16_hi(w[r]) * inv1);
        sc[mma_scale_index(c0 + 2 * j, (r0 >> 5) + rb, kg_rows)] = (uint8_t)sb0;
        sc[mma_scale_index(c0 + 2 * j + 1, (r0 >> 5) + rb, kg_rows)] = (uint8_t)sb1;
      }
    } else {
      // row-wise: thread = (row, 32-column block), tile rows x 4 tasks over
      // threads 128-255
      for (int task = threadIdx.x - 128; qr && task < 32 * nrb * 4; task += 128) {
        const int er = task >> 2, bb = task & 3;
        uint32_t w[16];
        uint32_t acc = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = *reinterpret_cast<const uint4*>(&tile[er][16 * bb + 4 * i]);
          w[4 * i + 0] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) acc = absmax2(acc, w[i]);
        const int sbv = mx_scale_byte(fmaxf(absmax_lo(acc), absmax_hi(acc)));
        const float inv = mx_inv_scale(sbv);
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t p0 = e4m3x2(bf16_lo(w[2 * i]) * inv, bf16_hi(w[2 * i]) * inv);
          const uint32_t p1 = e4m3x2(bf16_lo(w[2 * i + 1]) * inv, bf16_hi(w[2 * i + 1]) * inv);
          o[i] = p0 | (p1 << 16);
        }
        uint4* d = reinterpret_cast<uint4*>(qr + (size_t)(r0 + er) * C + c0 + 32 * bb);
        d[0] = make_uint4(o[0], o[1], o[2], o[3]);
        d[1] = make_uint4(o[4], o[5], o[6], o[7]);
        const int64_t mn = out.row_seg > 0 ? rslot0 + mx_tile_pos(rbase + er) : r0 + er;
        sr[mma_scale_index(mn, (c0 >> 5) + bb, nct)] = (uint8_t)sbv;
      }
    }
    __syncthreads();   // buffer b and its gates are free for the next tiles
  }
  cp_async_wait_all();
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
                                 cudaStream_t s, const DualGather* gather, const DualOut* outp) {
  const DualOut out = outp ? *outp : DualOut{};
  if (out.col_ld > 0 && (out.col_seg <= 0 || out.col_seg % 128 || out.col_ld % 16 ||
                         (out.col_perm && (C / 2) % (kMxTileN / 2))))
    return cudaErrorInvalidValue;
  const int64_t tiles = (int64_t)((R + kDualRows - 1) / kDualRows) * (C / 128);
  if (tiles == 0) return cudaSuccess;
  const __nv_bfloat16* x = (const __nv_bfloat16*)src;
  // per context (the attribute belongs to one): shared-memory opt-in and the
  // resident block count, so the grid is exactly one wave and every block
  // strides over the same number of tiles
  static CtxCache<int> resident[3];
  int blocks = 0;
  auto setup = [&](auto kern, size_t bytes, int which) {
    int n = 0;
    const cudaError_t e = resident[which].get(&n, [&](int* v) {
      cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
      if (r != cudaSuccess) return r;
      int per_sm = 0, dev = 0, sms = 0;
      r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, bytes);
      if (r == cudaSuccess && per_sm < 1) r = cudaErrorInvalidConfiguration;
      if (r == cudaSuccess) r = cudaGetDevice(&dev);
      if (r == cudaSuccess) r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      *v = per_sm * (sms > 0 ? sms : 1);
      return r;
    });
    if (e != cudaSuccess) return false;
    blocks = (int)(tiles < n ? tiles : n);
    return true;
  };
  if (!gather) {
    const size_t sm = dual_smem_bytes<0>();
    if (!setup(quant_dual_kernel<0>, sm, 0)) return cudaErrorInvalidValue;
    quant_dual_kernel<0><<<blocks, 256, sm, s>>>(x, R, C, ld, rows_dev, nullptr, 1, 0, nullptr,
                                                 nullptr, qr, sr, qc, sc, out);
  } else if (!gather->gate) {
    const size_t sm = dual_smem_bytes<1>();
    if (!setup(quant_dual_kernel<1>, sm, 1)) return cudaErrorInvalidValue;
    quant_dual_kernel<1><<<blocks, 256, sm, s>>>(x, R, C, ld, rows_dev, gather->assign_of_row,
                                                 gather->k, gather->n_assign, nullptr,
                                                 gather->status, qr, sr, qc, sc, out);
  } else {
    const size_t sm = dual_smem_bytes<2>();
    if (!setup(quant_dual_kernel<2>, sm, 2)) return cudaErrorInvalidValue;
    quant_dual_kernel<2><<<blocks, 256, sm, s>>>(x, R, C, ld, rows_dev, gather->assign_of_row,
                                                 gather->k, gather->n_assign, gather->gate,
                                                 gather->status, qr, sr, qc, sc, out);
  }
  return cudaGetLastError();
}

}  // namespace moe
