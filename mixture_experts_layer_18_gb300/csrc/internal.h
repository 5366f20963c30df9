// internal.h - host-side launchers shared between the C-ABI layer and the
// kernel translation units (not part of the public interface).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "moe.h"

namespace moe {

constexpr int kAlign = 128;        // rows per expert group are padded to this
constexpr int kRouteTokPerBlock = 128;  // tokens per block of the router
constexpr int kMaxE = 1024;
constexpr int kMaxTopK = 32;

// route.cu
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* topk_idx,
                         float* gate, int32_t* block_hist, int32_t* status, cudaStream_t s);
cudaError_t launch_route_backward(const int32_t* topk_idx, const float* gate, const float* dgate,
                                  int T, int E, int k, float* dlogits, int32_t* status,
                                  cudaStream_t s);
cudaError_t launch_permute(const int32_t* topk_idx, int T, int E, int k, int64_t max_rows,
                           const int32_t* block_hist_in, int32_t* block_base, int32_t* counts,
                           int32_t* offsets, int32_t* padded_offsets, int32_t* row_of_assign,
                           int32_t* assign_of_row, int32_t* status, cudaStream_t s);

// gather.cu  (elem_bytes 4: fp32 storage, 2: bf16 storage)
cudaError_t launch_gather_rows(const void* src, void* dst, int H, int elem_bytes, int k,
                               int n_assign, const int32_t* assign_of_row,
                               const int32_t* row_of_assign, const int32_t* padded_offsets,
                               int E, int64_t max_rows, int32_t* status, cudaStream_t s);
cudaError_t launch_gather_grad(const void* dY, void* dY_perm, void* dYg_perm, int H,
                               int elem_bytes, int k, int n_assign, const int32_t* assign_of_row,
                               const float* gate, const int32_t* padded_offsets, int E,
                               int64_t max_rows, int32_t* status, cudaStream_t s);
cudaError_t launch_combine(const void* src_perm, void* out, int T, int H, int elem_bytes, int k,
                           const int32_t* row_of_assign, int64_t max_rows, int32_t* status,
                           cudaStream_t s);
// dst[b][c][r] = src[b][r][c] for fp32 [nb, R, C] (row pitch C) into
// [nb, C, ld_dst] with ld_dst >= R.
cudaError_t launch_transpose_f32(const float* src, float* dst, int nb, int64_t R, int C,
                                 int64_t ld_dst, cudaStream_t s);
cudaError_t launch_dgate_reduce(const float* partial, int nt, int n_assign,
                                const int32_t* row_of_assign, int64_t max_rows, float* dgate,
                                int32_t* status, cudaStream_t s);

// quant.cu  (bf16 source).  layout 0: plain scales [R, C/32] (axis 1) or
// [R/32, C] (axis 0).  layout 1: tensor-core scale atoms, 512 bytes per
// (128 MN indices, 128 K elements); axis 1 = K along columns (MN = rows,
// C % 128 == 0, rows padded to 128), axis 0 = K along rows (MN = columns,
// C % 128 == 0, kgroups = ceil(R/128)).
cudaError_t launch_quantize(const void* src, int R, int C, int ld, int axis,
                            const int32_t* group_offsets, int G, uint8_t* q, uint8_t* scales,
                            int32_t* status, cudaStream_t s, int layout = 0);
// Both layout-1 quantisations (row-wise into qr/sr, column-wise into qc/sc;
// qc == nullptr skips the latter) from one read; R % 32 == 0, C % 128 == 0;
// rows >= *rows_dev (if given) untouched.  With `gather`, output row r is
// token row assign_of_row[r] / k of src (pad rows 0), and with gather->gate
// the column-wise encoding is taken of bf16(gate[a] * row).
struct DualGather {
  const int32_t* assign_of_row;
  int k, n_assign;
  const float* gate;     // optional
  int32_t* status;
};
// Output forms for the block-scaled GEMMs' B operands (192-column tiles,
// K-major B):
//   row_seg > 0   row-wise scales in the 192-column tile slots of segments of
//                 row_seg rows (mx_tile_slot), e.g. W2 [E*I, H] with I;
//   col_ld > 0    column-wise codes stored transposed: column c of input
//                 row r goes to row (r / col_seg) * C + perm(c), column
//                 r % col_seg, of a [.., col_ld] byte matrix (col_seg, a
//                 multiple of 128, is the K extent per segment), scales in
//                 the tile slots of that row; col_perm 1 interleaves 96
//                 gate and 96 up columns per tile (W13 for the gate/up GEMM).
// qr == nullptr skips the row-wise output.
struct DualOut {
  int64_t row_seg;
  int64_t col_ld, col_seg;
  int col_perm;
};
cudaError_t launch_quantize_dual(const void* src, int R, int C, int ld, const int32_t* rows_dev,
                                 uint8_t* qr, uint8_t* sr, uint8_t* qc, uint8_t* sc,
                                 cudaStream_t s, const DualGather* gather = nullptr,
                                 const DualOut* out = nullptr);

// gemm.cu
struct GemmDesc {
  int kind;                    // problem kind (gemm.cu)
  int a_mn, b_mn;              // operand M-/N-major (1) or K-major (0)
  int dep;                     // readiness dependency
  int signal;                  // tiles of this problem bump readiness counters
  const void* a;               // A source tensor
  int64_t a_rows, a_cols;      // its 2-D extent (elements)
  const void* b;               // B source tensor
  int64_t b_rows, b_cols;
  int M, N, K;                 // see GemmProblem
  int b_expert_rows;
  int I;
  void* out;
  int ld_out;
  void* out2;
  int ld_out2;
  const void* aux;
  int ld_aux;
  const float* gate;
  const int32_t* assign_of_row;
  int n_assign;
  float* partial;
  uint8_t* enc_row_q;          // FWD1, MXFP8: A's encodings written by the epilogue
  uint8_t* enc_row_sf;         //   (row-wise; column-wise when enc_col_q is set)
  uint8_t* enc_col_q;
  uint8_t* enc_col_sf;
  int64_t enc_col_kg;          //   128-row groups of the column-wise scale atoms
  int64_t enc_col_ld;          //   > 0: column-wise codes transposed ([col][row], this pitch)
  const uint8_t* sfa;          // MXFP8: scale atoms of A / B (quant.cu layout 1)
  const uint8_t* sfb;
  int64_t sfa_bytes, sfb_bytes;  // size of each scale-atom array (multiple of 512)
  int sfa_kg, sfb_kg;          // K groups of 128 in each operand's 2-D view
  int64_t sfb_seg;             // B scale atoms: MN slots per expert segment (0: one segment)
};

struct EngineLaunch {
  GemmDesc prob[4];
  int nprob;
  int E;
  int elem_bytes;              // 2: bf16 (kind::f16), 4: fp32 (kind::tf32), 1: MXFP8
  int BN;                      // 64, 128 or 256
  const int32_t* padded_offsets;
  const int32_t* counts;       // rows per expert (optional)
  int64_t max_rows;
  int32_t* ready;              // [(max_rows + 127) / 128 + 1] readiness counters
  int ready_target;
  int32_t* status;
  uint64_t wait_ns;
};

cudaError_t launch_engine(const EngineLaunch& L, cudaStream_t s, moe_status* st);

// debug / limits (api.cu)
uint64_t wait_limit_ns();
int debug_flags();

// Identity of the calling thread's current CUDA context (the current
// device's primary context is bound first if none is), unique over the
// process lifetime: a context created after a device reset gets a new one.
cudaError_t current_context_id(unsigned long long* id);

// Host values that belong to a CUDA context (kernel attributes, occupancy,
// device addresses of module variables), cached per context and safe to use
// from several host threads.  get() returns the current context's value,
// computing it with make(&value) the first time the context is seen (only a
// cudaSuccess result is stored); find() only looks.
template <typename V, int N = 32>
class CtxCache {
 public:
  template <typename F>
  cudaError_t get(V* out, F&& make) {
    unsigned long long id = 0;
    cudaError_t e = current_context_id(&id);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu_);
    if (lookup(id, out)) return cudaSuccess;
    V v{};
    e = make(&v);
    if (e != cudaSuccess) return e;
    const int slot = n_ < N ? n_++ : (next_++ % N);   // the oldest entry goes when full
    ids_[slot] = id;
    vals_[slot] = v;
    *out = v;
    return cudaSuccess;
  }
  cudaError_t find(V* out, bool* found) {
    unsigned long long id = 0;
    cudaError_t e = current_context_id(&id);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu_);
    *found = lookup(id, out);
    return cudaSuccess;
  }

 private:
  bool lookup(unsigned long long id, V* out) const {
    for (int i = 0; i < n_; ++i)
      if (ids_[i] == id) {
        *out = vals_[i];
        return true;
      }
    return false;
  }
  std::mutex mu_;
  unsigned long long ids_[N] = {};
  V vals_[N] = {};
  int n_ = 0, next_ = 0;
};

}  // namespace moe
