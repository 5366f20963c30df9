// gather.cu - HBM-bound data movement of the expert layer: the on-device
// dispatch (gather of token rows into expert-major order) and the combine
// (per-token sum of its k expert rows), plus the d(gate) reduction.
//
// "Accelerating dropless MoE in JAX with NVIDIA Transformer Engine",
// "Optimisation 2: dispatch and combine": dispatch reorders token copies by
// expert, combine returns them to token order and sums the expert outputs.
// On one GPU both are local: a gather by row map, and a deterministic
// gather-by-token sum in a fixed slot order (no atomics).
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ int grid_warps() { return (gridDim.x * blockDim.x) >> 5; }
__device__ __forceinline__ int global_warp() { return (blockIdx.x * blockDim.x + threadIdx.x) >> 5; }

// Dispatch in token order: dst[row_of_assign[t*k + j]] = src[t] for every
// slot j, then pad rows (assign_of_row < 0) = 0.  A warp takes one
// (token, 4 KB column chunk) unit: it reads the chunk once and writes it to
// the token's k rows, so each source row crosses HBM once however far apart
// the expert order puts its copies.
constexpr int kDispatchNV = 8;   // 16-byte vectors per lane per unit
__global__ void __launch_bounds__(kThreads) dispatch_rows_kernel(
    const uint4* __restrict__ src, uint4* __restrict__ dst, int vec_per_row, int T, int k,
    int n_assign, const int32_t* __restrict__ row_of_assign,
    const int32_t* __restrict__ assign_of_row, const int32_t* __restrict__ padded_offsets, int E,
    int32_t* status) {
  const int rows = padded_offsets[E];
  const int lane = threadIdx.x & 31;
  const int chunk = 32 * kDispatchNV;
  const int nch = (vec_per_row + chunk - 1) / chunk;
  const int64_t units = (int64_t)T * nch;
  for (int64_t u = global_warp(); u < units; u += grid_warps()) {
    const int t = (int)(u / nch);
    const int c0 = (int)(u - (int64_t)t * nch) * chunk;
    int my = -1;                       // lane j < k: destination row of slot j
    if (lane < k) {
      my = row_of_assign[(size_t)t * k + lane];
      if (my < 0 || my >= rows) {
        report(status, MOE_ERR_BAD_INDEX);
        my = -1;
      }
    }
    const uint4* sp = src + (size_t)t * vec_per_row;
    uint4 v[kDispatchNV];
#pragma unroll
    for (int i = 0; i < kDispatchNV; ++i) {
      const int c = c0 + i * 32 + lane;
      if (c < vec_per_row) v[i] = __ldg(sp + c);
    }
    for (int j = 0; j < k; ++j) {
      const int r = __shfl_sync(0xffffffffu, my, j);
      if (r < 0) continue;
      uint4* d = dst + (size_t)r * vec_per_row;
#pragma unroll
      for (int i = 0; i < kDispatchNV; ++i) {
        const int c = c0 + i * 32 + lane;
        if (c < vec_per_row) d[c] = v[i];
      }
    }
  }
  // pad rows, and rows whose assignment index is out of range, are zero:
  // each lane tests one row, the warp clears the flagged rows together
  for (int64_t rb = (int64_t)global_warp() * 32; rb < rows; rb += (int64_t)grid_warps() * 32) {
    const int64_t r = rb + lane;
    const int a = r < rows ? assign_of_row[r] : 0;
    if (r < rows && a >= n_assign) report(status, MOE_ERR_BAD_INDEX);
    unsigned m = __ballot_sync(0xffffffffu, r < rows && (a < 0 || a >= n_assign));
    while (m) {
      const int i = __ffs(m) - 1;
      m &= m - 1;
      uint4* d = dst + (size_t)(rb + i) * vec_per_row;
      for (int c = lane; c < vec_per_row; c += 32) d[c] = make_uint4(0, 0, 0, 0);
    }
  }
}

// dY_perm[r] = dY[t], dYg_perm[r] = gate[a] * dY[t] (t = a / k); pad rows 0
// (the fp32 mode's backward; bf16 needs dY_perm alone, from the dispatch).
template <typename Elt>
__global__ void __launch_bounds__(kThreads) gather_grad_kernel(
    const uint4* __restrict__ dY, uint4* __restrict__ dYp, uint4* __restrict__ dYgp,
    int vec_per_row, int k, int n_assign, const int32_t* __restrict__ assign_of_row,
    const float* __restrict__ gate, const int32_t* __restrict__ padded_offsets, int E,
    int32_t* status) {
  const int rows = padded_offsets[E];
  const int lane = threadIdx.x & 31;
  for (int r = global_warp(); r < rows; r += grid_warps()) {
    const int a = assign_of_row[r];
    uint4* d0 = dYp + (size_t)r * vec_per_row;
    uint4* d1 = dYgp + (size_t)r * vec_per_row;
    if (a < 0 || a >= n_assign) {
      if (a >= n_assign && lane == 0) report(status, MOE_ERR_BAD_INDEX);
      for (int c = lane; c < vec_per_row; c += 32) {
        d0[c] = make_uint4(0, 0, 0, 0);
        d1[c] = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    const float g = gate[a];
    const uint4* s = dY + (size_t)(a / k) * vec_per_row;
    for (int c = lane; c < vec_per_row; c += 32) {
      const uint4 v = __ldg(s + c);
      d0[c] = v;
      uint4 w;
      if constexpr (sizeof(Elt) == 2) {
        w.x = pack_bf16(g * bf16_lo(v.x), g * bf16_hi(v.x));
        w.y = pack_bf16(g * bf16_lo(v.y), g * bf16_hi(v.y));
        w.z = pack_bf16(g * bf16_lo(v.z), g * bf16_hi(v.z));
        w.w = pack_bf16(g * bf16_lo(v.w), g * bf16_hi(v.w));
      } else {
        w.x = __float_as_uint(g * __uint_as_float(v.x));
        w.y = __float_as_uint(g * __uint_as_float(v.y));
        w.z = __float_as_uint(g * __uint_as_float(v.z));
        w.w = __float_as_uint(g * __uint_as_float(v.w));
      }
      d1[c] = w;
    }
  }
}

// out[t] = sum_{j < k} src[row_of_assign[t*k + j]] in fp32, j ascending.
// One warp per token; each lane owns 16-byte column slices.
template <typename Elt>
__global__ void __launch_bounds__(kThreads) combine_kernel(
    const uint4* __restrict__ src, uint4* __restrict__ out, int T, int vec_per_row, int k,
    const int32_t* __restrict__ row_of_assign, int64_t max_rows, int32_t* status) {
  const int lane = threadIdx.x & 31;
  for (int t = global_warp(); t < T; t += grid_warps()) {
    int rows[kMaxTopK];
    bool bad = false;
    for (int j = 0; j < k; ++j) {
      rows[j] = row_of_assign[(size_t)t * k + j];
      if (rows[j] < 0 || rows[j] >= max_rows) bad = true;
    }
    if (bad && lane == 0) report(status, MOE_ERR_BAD_INDEX);
    for (int c = lane; c < vec_per_row; c += 32) {
      constexpr int EPV = 16 / sizeof(Elt);   // elements per 16-byte vector
      float acc[EPV];
#pragma unroll
      for (int i = 0; i < EPV; ++i) acc[i] = 0.f;
      for (int j = 0; j < k && !bad; ++j) {
        const uint4 v = __ldg(src + (size_t)rows[j] * vec_per_row + c);
        if constexpr (sizeof(Elt) == 2) {
          acc[0] += bf16_lo(v.x); acc[1] += bf16_hi(v.x);
          acc[2] += bf16_lo(v.y); acc[3] += bf16_hi(v.y);
          acc[4] += bf16_lo(v.z); acc[5] += bf16_hi(v.z);
          acc[6] += bf16_lo(v.w); acc[7] += bf16_hi(v.w);
        } else {
          acc[0] += __uint_as_float(v.x); acc[1] += __uint_as_float(v.y);
          acc[2] += __uint_as_float(v.z); acc[3] += __uint_as_float(v.w);
        }
      }
      uint4 w;
      if constexpr (sizeof(Elt) == 2) {
        w.x = pack_bf16(acc[0], acc[1]);
        w.y = pack_bf16(acc[2], acc[3]);
        w.z = pack_bf16(acc[4], acc[5]);
        w.w = pack_bf16(acc[6], acc[7]);
      } else {
        w.x = __float_as_uint(acc[0]); w.y = __float_as_uint(acc[1]);
        w.z = __float_as_uint(acc[2]); w.w = __float_as_uint(acc[3]);
      }
      out[(size_t)t * vec_per_row + c] = w;
    }
  }
}

// dgate[a] = sum_{n < nt} partial[row_of_assign[a] * nt + n], n ascending.
__global__ void dgate_reduce_kernel(const float* __restrict__ partial, int nt, int n_assign,
                                    const int32_t* __restrict__ row_of_assign, int64_t max_rows,
                                    float* __restrict__ dgate, int32_t* status) {
  for (int a = blockIdx.x * blockDim.x + threadIdx.x; a < n_assign; a += gridDim.x * blockDim.x) {
    const int r = row_of_assign[a];
    if (r < 0 || r >= max_rows) {
      report(status, MOE_ERR_BAD_INDEX);
      dgate[a] = 0.f;
      continue;
    }
    float s = 0.f;
    for (int n = 0; n < nt; ++n) s += partial[(size_t)r * nt + n];
    dgate[a] = s;
  }
}

// fp32 batched transpose through a padded 32x32 shared tile.
__global__ void __launch_bounds__(256) transpose_f32_kernel(const float* __restrict__ src,
                                                            float* __restrict__ dst, int64_t R,
                                                            int C, int64_t ld_dst) {
  __shared__ float tile[32][33];
  const int64_t b = blockIdx.z;
  const float* s = src + b * R * C;
  float* d = dst + b * (int64_t)C * ld_dst;
  const int c0 = blockIdx.x * 32;
  for (int64_t r0 = (int64_t)blockIdx.y * 32; r0 < R; r0 += (int64_t)gridDim.y * 32) {
    for (int i = threadIdx.y; i < 32; i += 8) {
      const int64_t r = r0 + i;
      const int c = c0 + threadIdx.x;
      if (r < R && c < C) tile[i][threadIdx.x] = s[r * C + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += 8) {
      const int c = c0 + i;
      const int64_t r = r0 + threadIdx.x;
      if (c < C && r < R) d[(int64_t)c * ld_dst + r] = tile[threadIdx.x][i];
    }
    __syncthreads();
  }
}

int num_sms() {
  static CtxCache<int> cache;
  int n = 0;
  cache.get(&n, [](int* v) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
    return e;
  });
  return n > 0 ? n : 1;
}

int grid_for_rows(int64_t rows) {
  // enough warps for one row each, capped at 8 resident blocks per SM
  const int64_t want = (rows + (kThreads / 32) - 1) / (kThreads / 32);
  const int64_t cap = (int64_t)num_sms() * 8;
  return (int)(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_gather_rows(const void* src, void* dst, int H, int elem_bytes, int k,
                               int n_assign, const int32_t* assign_of_row,
                               const int32_t* row_of_assign, const int32_t* padded_offsets,
                               int E, int64_t max_rows, int32_t* status, cudaStream_t s) {
  const int vec = H * elem_bytes / 16;
  const int T = n_assign / k;
  const int nch = (vec + 32 * kDispatchNV - 1) / (32 * kDispatchNV);
  const int64_t units = (int64_t)T * nch;
  dispatch_rows_kernel<<<grid_for_rows(units > max_rows / 32 ? units : max_rows / 32), kThreads, 0,
                         s>>>((const uint4*)src, (uint4*)dst, vec, T, k, n_assign, row_of_assign,
                              assign_of_row, padded_offsets, E, status);
  return cudaGetLastError();
}

cudaError_t launch_gather_grad(const void* dY, void* dY_perm, void* dYg_perm, int H,
                               int elem_bytes, int k, int n_assign, const int32_t* assign_of_row,
                               const float* gate, const int32_t* padded_offsets, int E,
                               int64_t max_rows, int32_t* status, cudaStream_t s) {
  const int vec = H * elem_bytes / 16;
  if (elem_bytes == 2)
    gather_grad_kernel<__nv_bfloat16><<<grid_for_rows(max_rows), kThreads, 0, s>>>(
        (const uint4*)dY, (uint4*)dY_perm, (uint4*)dYg_perm, vec, k, n_assign, assign_of_row,
        gate, padded_offsets, E, status);
  else
    gather_grad_kernel<float><<<grid_for_rows(max_rows), kThreads, 0, s>>>(
        (const uint4*)dY, (uint4*)dY_perm, (uint4*)dYg_perm, vec, k, n_assign, assign_of_row,
        gate, padded_offsets, E, status);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* src_perm, void* out, int T, int H, int elem_bytes, int k,
                           const int32_t* row_of_assign, int64_t max_rows, int32_t* status,
                           cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int vec = H * elem_bytes / 16;
  if (elem_bytes == 2)
    combine_kernel<__nv_bfloat16><<<grid_for_rows(T), kThreads, 0, s>>>(
        (const uint4*)src_perm, (uint4*)out, T, vec, k, row_of_assign, max_rows, status);
  else
    combine_kernel<float><<<grid_for_rows(T), kThreads, 0, s>>>(
        (const uint4*)src_perm, (uint4*)out, T, vec, k, row_of_assign, max_rows, status);
  return cudaGetLastError();
}

cudaError_t launch_transpose_f32(const float* src, float* dst, int nb, int64_t R, int C,
                                 int64_t ld_dst, cudaStream_t s) {
  if (nb == 0 || R == 0 || C == 0) return cudaSuccess;
  const int64_t ry = (R + 31) / 32;
  dim3 grid((C + 31) / 32, (unsigned)(ry < 65535 ? ry : 65535), nb);
  transpose_f32_kernel<<<grid, dim3(32, 8), 0, s>>>(src, dst, R, C, ld_dst);
  return cudaGetLastError();
}

cudaError_t launch_dgate_reduce(const float* partial, int nt, int n_assign,
                                const int32_t* row_of_assign, int64_t max_rows, float* dgate,
                                int32_t* status, cudaStream_t s) {
  if (n_assign == 0) return cudaSuccess;
  const int blocks = (n_assign + 255) / 256;
  dgate_reduce_kernel<<<blocks < 4096 ? blocks : 4096, 256, 0, s>>>(
      partial, nt, n_assign, row_of_assign, max_rows, dgate, status);
  return cudaGetLastError();
}

}  // namespace moe
