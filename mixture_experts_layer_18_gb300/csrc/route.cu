// route.cu - top-k router and permutation builder.
//
// Router: "Prime Intellect releases Prime Mega MoE" (MarkTechPost), "In
// brief": each token goes to its top-8 of 128 experts.  Gates are the
// softmax over all experts renormalised over the chosen ones, which equals
// exp(l_j - m) / sum_{i in top-k} exp(l_i - m) with m the largest logit.
// Permutation: "Accelerating dropless MoE in JAX with NVIDIA Transformer
// Engine", 02 (dropless: every assignment kept, ragged per-expert groups)
// and "Optimisation 2" (dispatch reorders token copies by expert locally).
// Storage groups are padded to 128 rows so that every 128-row GEMM tile
// belongs to one expert; the logical counts stay unpadded.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kBwdThreads = 256;

// Block shape of the router: 32 warps (4 tokens each, side by side) while a
// token's logits fit in 4 registers per lane; larger E keeps 8 warps and
// fewer tokens in flight per warp so the logits stay in registers.
template <int VPL> struct RouteShape {
  static constexpr int THREADS = VPL <= 8 ? 1024 : 256;
  static constexpr int NT = kRouteTokPerBlock / (THREADS / 32);   // tokens per warp
  static constexpr int ILP = VPL <= 4 ? 4 : (VPL <= 8 ? 2 : 1);  // processed side by side
};

// One warp per token; ILP tokens of a warp are processed side by side
// (independent shuffle chains, so their latencies overlap).  Lane l holds
// logits l, l+32, l+64, ... of each token in registers.  k rounds of a warp
// arg-max pick the largest remaining logit, ties to the lower expert index
// (a total order: a NaN logit is read as -inf and reported as
// MOE_ERR_BAD_INPUT).  Slot j of the result is the j-th pick.  A token whose
// logits are all -inf has no softmax: it gets zero gates (it contributes
// nothing to the layer) and MOE_ERR_BAD_INPUT.  Also builds this block's
// expert histogram.
template <int VPL>
__global__ void __launch_bounds__(RouteShape<VPL>::THREADS) route_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ topk_idx,
    float* __restrict__ gate, int32_t* __restrict__ block_hist, int nb, int32_t* status) {
  constexpr int NT = RouteShape<VPL>::NT, ILP = RouteShape<VPL>::ILP;
  __shared__ int hist[kMaxE];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int g = 0; g < NT; g += ILP) {
    const int t0 = blockIdx.x * kRouteTokPerBlock + warp * NT + g;
    if (t0 >= T) break;
    float v[ILP][VPL];
    uint32_t taken[ILP];   // bit q: element q*32+lane chosen already or absent
#pragma unroll
    for (int i = 0; i < ILP; ++i) {
      const int t = t0 + i;
      taken[i] = 0;
#pragma unroll
      for (int q = 0; q < VPL; ++q) {
        const int e = q * 32 + lane;
        float x = (e < E && t < T) ? __ldg(logits + (size_t)t * E + e) : 0.f;
        if (x != x) {
          report(status, MOE_ERR_BAD_INPUT);
          x = -INFINITY;
        }
        v[i][q] = x;
        if (e >= E) taken[i] |= 1u << q;
      }
    }
    float sel_v[ILP];
    int sel_e[ILP];
#pragma unroll
    for (int i = 0; i < ILP; ++i) {
      sel_v[i] = 0.f;
      sel_e[i] = 0;
    }
    for (int j = 0; j < k; ++j) {
      float bv[ILP];
      int be[ILP];
#pragma unroll
      for (int i = 0; i < ILP; ++i) {
        bv[i] = -INFINITY;
        be[i] = INT_MAX;
#pragma unroll
        for (int q = 0; q < VPL; ++q) {
          const int e = q * 32 + lane;
          if (!((taken[i] >> q) & 1u) && (v[i][q] > bv[i] || (v[i][q] == bv[i] && e < be[i]))) {
            bv[i] = v[i][q];
            be[i] = e;
          }
        }
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) {
#pragma unroll
        for (int i = 0; i < ILP; ++i) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv[i], off);
          const int oe = __shfl_xor_sync(0xffffffffu, be[i], off);
          if (ov > bv[i] || (ov == bv[i] && oe < be[i])) {
            bv[i] = ov;
            be[i] = oe;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < ILP; ++i) {
        if ((be[i] & 31) == lane) taken[i] |= 1u << (be[i] >> 5);
        if (lane == j) {
          sel_v[i] = bv[i];
          sel_e[i] = be[i];
        }
      }
    }
#pragma unroll
    for (int i = 0; i < ILP; ++i) {
      const int t = t0 + i;
      const float m = __shfl_sync(0xffffffffu, sel_v[i], 0);
      const bool none = !(m > -INFINITY);   // every logit of the token is -inf
      const float w = lane < k && !none ? expf(sel_v[i] - m) : 0.f;
      float sum = w;
#pragma unroll
      for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if (none && t < T && lane == 0) report(status, MOE_ERR_BAD_INPUT);
      if (t < T && lane < k) {
        topk_idx[(size_t)t * k + lane] = sel_e[i];
        gate[(size_t)t * k + lane] = none ? 0.f : w / sum;
        atomicAdd(&hist[sel_e[i]], 1);
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) block_hist[(size_t)e * nb + blockIdx.x] = hist[e];
}

// Single block: per-expert totals and the per-(expert, block) exclusive
// bases (one warp per expert at a time: a shuffle scan over 32 router blocks
// per step), then the exclusive scans over experts (logical and padded).
__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ block_hist, int nb,
                                                    int E, int32_t* __restrict__ block_base,
                                                    int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ padded_offsets) {
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_pad[kMaxE + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int e = warp; e < E; e += nw) {
    const int32_t* h = block_hist + (size_t)e * nb;
    int32_t* bb = block_base + (size_t)e * nb;
    int carry = 0;
    for (int b0 = 0; b0 < nb; b0 += 32) {
      const int b = b0 + lane;
      const int c = b < nb ? h[b] : 0;
      int x = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
      }
      if (b < nb) bb[b] = carry + x - c;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) {
      s_cnt[e] = carry;
      s_pad[e] = (carry + kAlign - 1) / kAlign * kAlign;
      counts[e] = carry;
    }
  }
  __syncthreads();
  // E <= 1024: a warp-parallel scan over 32-expert chunks.
  if (threadIdx.x < 32) {
    int carry_o = 0, carry_p = 0;
    for (int c0 = 0; c0 < E; c0 += 32) {
      const int e = c0 + lane;
      int o = e < E ? s_cnt[e] : 0;
      int p = e < E ? s_pad[e] : 0;
      // inclusive warp scans
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int yo = __shfl_up_sync(0xffffffffu, o, off);
        const int yp = __shfl_up_sync(0xffffffffu, p, off);
        if (lane >= off) {
          o += yo;
          p += yp;
        }
      }
      if (e < E) {
        offsets[e] = carry_o + o - s_cnt[e];
        padded_offsets[e] = carry_p + p - s_pad[e];
      }
      carry_o += __shfl_sync(0xffffffffu, o, 31);
      carry_p += __shfl_sync(0xffffffffu, p, 31);
    }
    if (lane == 0) {
      offsets[E] = carry_o;
      padded_offsets[E] = carry_p;
    }
  }
}

// Blocks [0, nb): stable scatter of this block's assignments (the same
// assignment ranges as the router blocks).  Within a 256-assignment round,
// lanes of a warp with equal experts are ranked by lane (match_any), warps
// take their bases from the running per-expert cursor in warp order, so the
// rank of an assignment inside its expert follows ascending a.
// Blocks [nb, gridDim): mark pad rows and rows past padded_offsets[E] with -1.
__global__ void __launch_bounds__(256) scatter_kernel(
    const int32_t* __restrict__ topk_idx, int n_assign, int E, int k, int nb,
    const int32_t* __restrict__ block_base, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ padded_offsets, int32_t* __restrict__ row_of_assign,
    int32_t* __restrict__ assign_of_row, int64_t max_rows, int32_t* status) {
  __shared__ int run[kMaxE];
  __shared__ int s_base[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((int)blockIdx.x >= nb) {
    const int pb = blockIdx.x - nb, npb = gridDim.x - nb;
    for (int e = pb; e < E; e += npb) {
      const int r1 = padded_offsets[e + 1];
      for (int r = padded_offsets[e] + counts[e] + threadIdx.x; r < r1; r += blockDim.x)
        assign_of_row[r] = -1;
    }
    for (int64_t r = (int64_t)padded_offsets[E] + (int64_t)pb * blockDim.x + threadIdx.x;
         r < max_rows; r += (int64_t)npb * blockDim.x)
      assign_of_row[r] = -1;
    return;
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    run[e] = padded_offsets[e] + block_base[(size_t)e * nb + blockIdx.x];
  __syncthreads();
  const int chunk = kRouteTokPerBlock * k;
  const int a0 = blockIdx.x * chunk;
  const int a1 = min(n_assign, a0 + chunk);
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = a0; base < a1; base += blockDim.x) {
    const int a = base + threadIdx.x;
    int e = a < a1 ? topk_idx[a] : -1;
    if (e >= E || (a < a1 && e < 0)) {
      report(status, MOE_ERR_BAD_INDEX);
      e = -1;
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & lt_mask);
    const int leader = __ffs(same) - 1;
    for (int w = 0; w < 8; ++w) {
      if (warp == w && lane == leader && e >= 0) {
        s_base[w][lane] = run[e];
        run[e] += __popc(same);
      }
      __syncthreads();
    }
    if (e >= 0) {
      const int row = s_base[warp][leader] + rank;
      row_of_assign[a] = row;
      assign_of_row[row] = a;
    }
    __syncthreads();
  }
}

// Router backward: with the selection held fixed, gate_j = exp(l_j) /
// sum_{i in top-k} exp(l_i), so d(logit) of a selected expert i is
// g_i * (dg_i - sum_j g_j dg_j) and zero for every other expert.  One warp
// per token; lane j < k holds slot j; the row of E logits is written once,
// coalesced.
template <int VPL>
__global__ void __launch_bounds__(kBwdThreads) route_backward_kernel(
    const int32_t* __restrict__ topk_idx, const float* __restrict__ gate,
    const float* __restrict__ dgate, int T, int E, int k, float* __restrict__ dlogits,
    int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
    const size_t base = (size_t)t * k;
    const float g = lane < k ? gate[base + lane] : 0.f;
    const float dg = lane < k ? dgate[base + lane] : 0.f;
    int e = lane < k ? topk_idx[base + lane] : -1;
    if (lane < k && (e < 0 || e >= E)) {
      report(status, MOE_ERR_BAD_INDEX);
      e = -1;
    }
    float inner = g * dg;
#pragma unroll
    for (int off = 16; off; off >>= 1) inner += __shfl_xor_sync(0xffffffffu, inner, off);
    const float dl = g * (dg - inner);
    float out[VPL];
#pragma unroll
    for (int q = 0; q < VPL; ++q) out[q] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int ej = __shfl_sync(0xffffffffu, e, j);
      const float dj = __shfl_sync(0xffffffffu, dl, j);
      if (ej >= 0 && (ej & 31) == lane) {
#pragma unroll
        for (int q = 0; q < VPL; ++q)
          if (q == (ej >> 5)) out[q] = dj;
      }
    }
    float* row = dlogits + (size_t)t * E;
#pragma unroll
    for (int q = 0; q < VPL; ++q) {
      const int ee = q * 32 + lane;
      if (ee < E) row[ee] = out[q];
    }
  }
}

}  // namespace

cudaError_t launch_route_backward(const int32_t* topk_idx, const float* gate, const float* dgate,
                                  int T, int E, int k, float* dlogits, int32_t* status,
                                  cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + (kBwdThreads / 32) - 1) / (kBwdThreads / 32);
  const int grid = blocks < 4096 ? blocks : 4096;
  const int vpl = (E + 31) / 32;
  if (vpl <= 1)
    route_backward_kernel<1><<<grid, kBwdThreads, 0, s>>>(topk_idx, gate, dgate, T, E, k, dlogits, status);
  else if (vpl <= 4)
    route_backward_kernel<4><<<grid, kBwdThreads, 0, s>>>(topk_idx, gate, dgate, T, E, k, dlogits, status);
  else if (vpl <= 8)
    route_backward_kernel<8><<<grid, kBwdThreads, 0, s>>>(topk_idx, gate, dgate, T, E, k, dlogits, status);
  else if (vpl <= 16)
    route_backward_kernel<16><<<grid, kBwdThreads, 0, s>>>(topk_idx, gate, dgate, T, E, k, dlogits, status);
  else
    route_backward_kernel<32><<<grid, kBwdThreads, 0, s>>>(topk_idx, gate, dgate, T, E, k, dlogits, status);
  return cudaGetLastError();
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* topk_idx,
                         float* gate, int32_t* block_hist, int32_t* status, cudaStream_t s) {
  const int nb = (T + kRouteTokPerBlock - 1) / kRouteTokPerBlock;
  if (nb == 0) return cudaSuccess;
  const int vpl = (E + 31) / 32;
  if (vpl <= 1)
    route_kernel<1><<<nb, RouteShape<1>::THREADS, 0, s>>>(logits, T, E, k, topk_idx, gate, block_hist, nb, status);
  else if (vpl <= 4)
    route_kernel<4><<<nb, RouteShape<4>::THREADS, 0, s>>>(logits, T, E, k, topk_idx, gate, block_hist, nb, status);
  else if (vpl <= 8)
    route_kernel<8><<<nb, RouteShape<8>::THREADS, 0, s>>>(logits, T, E, k, topk_idx, gate, block_hist, nb, status);
  else if (vpl <= 16)
    route_kernel<16><<<nb, RouteShape<16>::THREADS, 0, s>>>(logits, T, E, k, topk_idx, gate, block_hist, nb, status);
  else
    route_kernel<32><<<nb, RouteShape<32>::THREADS, 0, s>>>(logits, T, E, k, topk_idx, gate, block_hist, nb, status);
  return cudaGetLastError();
}

cudaError_t launch_permute(const int32_t* topk_idx, int T, int E, int k, int64_t max_rows,
                           const int32_t* block_hist, int32_t* block_base, int32_t* counts,
                           int32_t* offsets, int32_t* padded_offsets, int32_t* row_of_assign,
                           int32_t* assign_of_row, int32_t* status, cudaStream_t s) {
  const int nb = (T + kRouteTokPerBlock - 1) / kRouteTokPerBlock;
  scan_kernel<<<1, 1024, 0, s>>>(block_hist, nb, E, block_base, counts, offsets, padded_offsets);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int pad_blocks = 64;
  scatter_kernel<<<nb + pad_blocks, 256, 0, s>>>(topk_idx, T * k, E, k, nb, block_base, counts,
                                                 padded_offsets, row_of_assign, assign_of_row,
                                                 max_rows, status);
  return cudaGetLastError();
}

}  // namespace moe
