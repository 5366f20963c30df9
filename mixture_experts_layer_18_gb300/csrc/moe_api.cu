// moe_api.cu - the C ABI declared in include/moe.h: argument checks, buffer
// carving, and the launch sequence of each call on the caller's stream.
#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "mx_encode.cuh"

namespace moe {

namespace {
constexpr int kMaxLaunchEvents = 8;
std::atomic<int> g_debug_flags{0};
std::atomic<long long> g_wait_ns{1000000000LL};   // one second
// one-shot timing events per call kind (forward, backward)
std::atomic<void*> g_ev_start[3] = {nullptr, nullptr, nullptr};
std::atomic<void*> g_ev_stop[3] = {nullptr, nullptr, nullptr};

// one-shot events around each grouped-GEMM launch of the next call of a kind
struct LaunchEvents {
  void* start[kMaxLaunchEvents];
  void* stop[kMaxLaunchEvents];
  int n;
};
LaunchEvents g_launch_ev[3];
std::atomic<int> g_launch_armed[3] = {0, 0, 0};
thread_local const LaunchEvents* t_launch_ev = nullptr;   // the running call's hook
thread_local int t_launch_i = 0;

struct EventScope {   // records the pending hooks' events around a launch group
  cudaEvent_t stop = nullptr;
  cudaStream_t s;
  EventScope(int which, cudaStream_t st) : s(st) {
    void* a = g_ev_start[which].exchange(nullptr);
    void* b = g_ev_stop[which].exchange(nullptr);
    if (a && b) {
      cudaEventRecord(static_cast<cudaEvent_t>(a), s);
      stop = static_cast<cudaEvent_t>(b);
    }
    if (g_launch_armed[which].exchange(0)) {
      t_launch_ev = &g_launch_ev[which];
      t_launch_i = 0;
    }
  }
  void finish() {
    if (stop) cudaEventRecord(stop, s);
    stop = nullptr;
    t_launch_ev = nullptr;
  }
  ~EventScope() { finish(); }
};

// A grouped-GEMM launch, with the running call's per-launch events if any.
cudaError_t engine(const EngineLaunch& L, cudaStream_t s, moe_status* st) {
  const LaunchEvents* h = t_launch_ev;
  const int i = t_launch_i;
  const bool rec = h && i < h->n;
  if (rec) cudaEventRecord(static_cast<cudaEvent_t>(h->start[i]), s);
  const cudaError_t e = launch_engine(L, s, st);
  if (rec) {
    cudaEventRecord(static_cast<cudaEvent_t>(h->stop[i]), s);
    t_launch_i = i + 1;
  }
  return e;
}
}  // namespace

uint64_t wait_limit_ns() { return (uint64_t)g_wait_ns.load(); }
int debug_flags() { return g_debug_flags.load(); }

cudaError_t current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  if (!get_current || !get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) {
    // no context bound to this thread yet: bind the current device's
    // primary context (cudaSetDevice initialises it)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorInitializationError;
  }
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorContextIsDestroyed;
}

namespace {

// Holds its CTA (and the dynamic shared memory it was launched with, which
// it never touches) for `ns` nanoseconds, then returns: the bounded side
// load of moe_debug_occupy.
__global__ void occupy_kernel(uint64_t ns) {
  const uint64_t t0 = global_ns();
  while (global_ns() - t0 < ns) __nanosleep(2000);
}

constexpr int GK_FWD1 = 0, GK_FWD2 = 1, GK_BWD_D = 2, GK_BWD_DX = 3, GK_DW = 4;
constexpr int DEP_NONE = 0, DEP_MBLOCK = 1, DEP_EXPERT = 2;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int elem_bytes(const moe_dims* d) { return d->mode == MOE_F32 ? 4 : 2; }
// MXFP8 GEMMs in the forward (mxfp8) / in the backward (mxfp8, fp8_bwd)
bool mx_fwd(const moe_dims* d) { return d->mode == MOE_MXFP8; }
bool mx_bwd(const moe_dims* d) { return d->mode == MOE_MXFP8 || d->mode == MOE_FP8_BWD; }

bool dims_ok(const moe_dims* d) {
  if (!d) return false;
  if (d->T < 0 || d->E < 1 || d->E > kMaxE) return false;
  if (d->top_k < 1 || d->top_k > kMaxTopK || d->top_k > d->E) return false;
  if (d->H < 64 || d->H % 64 || d->I < 64 || d->I % 64) return false;
  if (d->mode < MOE_F32 || d->mode > MOE_FP8_BWD) return false;
  const int64_t rows = (int64_t)d->T * d->top_k + (int64_t)kAlign * d->E;
  if (rows >= ((int64_t)1 << 31)) return false;
  if ((int64_t)d->E * d->H * 2 * d->I >= ((int64_t)1 << 40)) return false;
  return true;
}

int64_t max_rows(const moe_dims* d) { return (int64_t)d->T * d->top_k + (int64_t)kAlign * d->E; }

bool aligned16(const void* p) { return p && ((uintptr_t)p & 15) == 0; }

// The block-scaled GEMMs run 192-column tiles (96 gate + 96 up columns for
// the gate/up GEMM) and stages of 128 K elements: I (an N of the gate/up
// and D GEMMs, the K of the down GEMM) a multiple of 384, H of 128.
bool mx_shape_ok(const moe_dims* d) { return d->I % 384 == 0 && d->H % 128 == 0; }

// Tile width of the forward gate/up GEMM: BN/2 columns of each half per tile.
int bn_fwd1(const moe_dims* d) {
  if (mx_fwd(d)) return mx_shape_ok(d) ? kMxTileN : 0;
  const int atom = 128 / elem_bytes(d);
  for (int bn : {256, 128, 64})
    if (bn / 2 >= atom && d->I % (bn / 2) == 0) return bn;
  return 0;
}
int bn_div(int n) {
  for (int bn : {256, 128, 64})
    if (n % bn == 0) return bn;
  return 0;
}
int bn_bwd(const moe_dims* d) {
  if (mx_bwd(d)) return mx_shape_ok(d) ? kMxTileN : 0;
  for (int bn : {256, 128, 64})
    if (d->I % bn == 0 && d->H % bn == 0) return bn;
  return 0;
}

// bf16 mode applies the gate to A in the gate/up epilogue (the saved `act`
// is gate * A): the down GEMM then needs no gate, and dW2 = (gate * A)^T
// dY_perm needs no gated copy of dY.
bool gate_on_act(const moe_dims* d) { return d->mode == MOE_BF16; }

// fp32 mode keeps every TF32 operand K-major: the weight operands and the
// token-axis operands of the weight-gradient GEMMs get transposed copies whose
// row pitch is the row capacity rounded up to 32.
int64_t ld_t(const moe_dims* d) { return (max_rows(d) + 31) / 32 * 32; }

// MXFP8: one quantised operand = E4M3 codes + tensor-core scale atoms.
struct MxBuf {
  size_t q, sf, sf_bytes;
};
int64_t rows_pad(const moe_dims* d) { return (max_rows(d) + 127) / 128 * 128; }
// codes of an [R, C] byte matrix (K = C) and the scale atoms of Rp MN slots
// (R padded to 128, or the 192-column tile slots of a B operand)
MxBuf mx_carve(size_t& o, size_t R, size_t Rp, size_t C) {
  MxBuf b;
  b.q = o;
  o += align256(R * C);
  b.sf = o;
  b.sf_bytes = Rp * C / 32;
  o += align256(b.sf_bytes);
  return b;
}

struct FwdWs {
  size_t zg, w13t, w2t, total;
  MxBuf x, w13, a, w2;     // MXFP8 forward operands
};
FwdWs fwd_ws(const moe_dims* d) {
  FwdWs w;
  const size_t rows = (size_t)max_rows(d), es = elem_bytes(d);
  const size_t wsz = (size_t)d->E * d->H * d->I * es;
  size_t o = 0;
  w.zg = o; o += align256(rows * d->H * es);
  const bool t = d->mode == MOE_F32;
  w.w13t = o; o += t ? align256(2 * wsz) : 0;
  w.w2t = o; o += t ? align256(wsz) : 0;
  if (mx_fwd(d)) {
    const size_t rp = (size_t)rows_pad(d), E = d->E, H = d->H, I = d->I;
    w.x = mx_carve(o, rows, rp, H);
    // B operands, K-major: W13 transposed [E*2I, H] (gate / up interleaved per
    // tile) and W2 transposed [E*H, I]
    w.w13 = mx_carve(o, E * 2 * I, E * mx_tile_slots(2 * I), H);
    w.a = mx_carve(o, rows, rp, I);
    w.w2 = mx_carve(o, E * H, E * mx_tile_slots(H), I);
  }
  w.total = o;
  return w;
}

struct BwdWs {
  size_t dy_perm, dyg_perm, dh13, dxp, partial, ready;
  size_t act_t, dyg_t, xp_t, dh13_t, total;
  int nt_d;
  MxBuf dy, w2r, actc, dygc, dh13r, dh13c, w13r, xpc;   // MXFP8 backward operands
};
BwdWs bwd_ws(const moe_dims* d) {
  BwdWs w;
  const size_t rows = (size_t)max_rows(d), es = elem_bytes(d);
  const int bn = bn_bwd(d);
  w.nt_d = bn ? d->I / bn : 1;
  size_t o = 0;
  // dY_perm (bf16, f32) and gate * dY_perm (f32); the MXFP8 backward
  // gathers dY straight into its encodings
  w.dy_perm = o; o += mx_bwd(d) ? 0 : align256(rows * d->H * es);
  w.dyg_perm = o; o += mx_bwd(d) || gate_on_act(d) ? 0 : align256(rows * d->H * es);
  // dh13 in bf16 (the MXFP8 backward keeps only its encodings, dh13r / dh13c)
  w.dh13 = o; o += mx_bwd(d) ? 0 : align256(rows * 2 * d->I * es);
  w.dxp = o; o += align256(rows * d->H * es);
  w.partial = o; o += align256(rows * w.nt_d * sizeof(float));
  w.ready = o; o += align256(((rows + 127) / 128 + 1) * sizeof(int32_t));
  const bool t = d->mode == MOE_F32;
  const size_t lt = (size_t)ld_t(d) * es;
  w.act_t = o; o += t ? align256(lt * d->I) : 0;
  w.dyg_t = o; o += t ? align256(lt * d->H) : 0;
  w.xp_t = o; o += t ? align256(lt * d->H) : 0;
  w.dh13_t = o; o += t ? align256(lt * 2 * d->I) : 0;
  if (mx_bwd(d)) {
    const size_t rp = (size_t)rows_pad(d), E = d->E, H = d->H, I = d->I;
    w.dy = mx_carve(o, rows, rp, H);
    // B operands of the weight gradients, K-major: gate * dY and dh13
    // quantised along tokens, stored transposed ([H, rp], [2I, rp])
    w.dygc = mx_carve(o, H, mx_tile_slots(H), rp);
    w.dh13r = mx_carve(o, rows, rp, 2 * I);
    w.dh13c = mx_carve(o, 2 * I, mx_tile_slots(2 * I), rp);
    if (d->mode != MOE_MXFP8) {   // mxfp8: the forward leaves these in `saved`
      w.w2r = mx_carve(o, E * I, E * mx_tile_slots(I), H);
      w.actc = mx_carve(o, rows, rp, I);
      w.w13r = mx_carve(o, E * H, E * mx_tile_slots(H), 2 * I);
      w.xpc = mx_carve(o, rows, rp, H);
    }
  }
  w.total = o;
  return w;
}

struct RouteWs {
  size_t hist, base, total;
};
RouteWs route_ws(const moe_dims* d) {
  RouteWs w;
  const size_t nb = (size_t)(d->T + kRouteTokPerBlock - 1) / kRouteTokPerBlock;
  const size_t n = nb * d->E * sizeof(int32_t);
  w.hist = 0;
  w.base = align256(n);
  w.total = w.base + align256(n);
  if (w.total == 0) w.total = 256;
  return w;
}

moe_saved_layout saved_layout(const moe_dims* d) {
  moe_saved_layout s;
  memset(&s, 0, sizeof(s));
  const size_t rows = (size_t)max_rows(d), es = elem_bytes(d);
  size_t o = 0;
  // the MXFP8 forward gathers X straight into its encodings (x_col below)
  s.x_perm = o; o += d->mode == MOE_MXFP8 ? 0 : align256(rows * d->H * es);
  s.h13 = o; o += align256(rows * 2 * d->I * es);
  // MXFP8 keeps A only as its encodings (x_col / act_col below, and the
  // forward workspace's row-wise copy)
  s.act = o; o += d->mode == MOE_MXFP8 ? 0 : align256(rows * d->I * es);
  if (d->mode == MOE_MXFP8) {
    const size_t rp = (size_t)rows_pad(d), E = d->E, H = d->H, I = d->I;
    const MxBuf x = mx_carve(o, rows, rp, H), a = mx_carve(o, rows, rp, I);
    const MxBuf w13 = mx_carve(o, E * H, E * mx_tile_slots(H), 2 * I);
    const MxBuf w2 = mx_carve(o, E * I, E * mx_tile_slots(I), H);
    s.x_col_q = x.q; s.x_col_sf = x.sf;
    s.act_col_q = a.q; s.act_col_sf = a.sf;
    s.w13_row_q = w13.q; s.w13_row_sf = w13.sf;
    s.w2_row_q = w2.q; s.w2_row_sf = w2.sf;
  }
  s.total = o;
  return s;
}

// Arrays of T*top_k entries may be NULL when T == 0.
bool route_ok(const moe_route_out* r, int T) {
  if (!r) return false;
  const bool tok = T == 0 || (aligned16(r->topk_idx) && aligned16(r->gate) &&
                              aligned16(r->row_of_assign));
  return tok && aligned16(r->counts) && aligned16(r->offsets) && aligned16(r->padded_offsets) &&
         aligned16(r->assign_of_row);
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                                   \
  do {                                                  \
    cudaError_t _e = (expr);                            \
    if (_e != cudaSuccess) return MOE_ERR_CUDA;         \
  } while (0)


// ---------------------------------------------------------------- MXFP8
// Every GEMM operand is quantised along that GEMM's contraction axis into
// E4M3 codes plus scale atoms laid out for the tensor cores (quant.cu,
// layout 1): token-major activations row-wise (K = columns); weights of the
// forward and token-axis operands of the weight gradients column-wise
// (K = rows, blocks restarting at each expert's 128-aligned start).
struct Mx {
  const void* q;
  const uint8_t* sf;
  int64_t sf_bytes;
};
Mx mx_at(char* base, const MxBuf& b) {
  return Mx{base + b.q, reinterpret_cast<const uint8_t*>(base + b.sf), (int64_t)b.sf_bytes};
}

cudaError_t quant_cols(const void* src, int64_t R, int C, const int32_t* go, int G, const Mx& m,
                       int32_t* st, cudaStream_t s) {
  return launch_quantize(src, (int)R, C, C, 0, go, G, (uint8_t*)m.q, (uint8_t*)m.sf, st, s, 1);
}
// One read of a bf16 [R, C] tensor, two encodings: row-wise into `rw` (if
// given; `row_seg` > 0 puts its scales in the 192-column tile slots of a B
// operand with segments of row_seg rows) and column-wise into `cw` (if
// given; `col` says whether it is stored transposed for a K-major B).  Rows
// at or past *rows_dev (if given) are untouched; with `g`, rows are gathered
// token rows of src (see DualGather).
cudaError_t quant_both(const void* src, int64_t R, int C, const int32_t* rows_dev, const Mx* rw,
                       const Mx* cw, cudaStream_t s, const DualGather* g = nullptr,
                       const DualOut& out = DualOut{}) {
  return launch_quantize_dual(src, (int)R, C, C, rows_dev, rw ? (uint8_t*)rw->q : nullptr,
                              rw ? (uint8_t*)rw->sf : nullptr, cw ? (uint8_t*)cw->q : nullptr,
                              cw ? (uint8_t*)cw->sf : nullptr, s, g, &out);
}
// the backward's operands that the mxfp8 forward writes into `saved`
struct MxSaved {
  Mx x_col, act_col, w13_row, w2_row;
};
MxSaved mx_saved(const moe_dims* d, const moe_saved_layout& sl, char* sv) {
  const int64_t rp = rows_pad(d), E = d->E, H = d->H, I = d->I;
  auto at = [&](size_t q, size_t sf, int64_t sf_bytes) {
    return Mx{sv + q, reinterpret_cast<const uint8_t*>(sv + sf), sf_bytes};
  };
  return MxSaved{at(sl.x_col_q, sl.x_col_sf, rp * H / 32), at(sl.act_col_q, sl.act_col_sf, rp * I / 32),
                 at(sl.w13_row_q, sl.w13_row_sf, E * mx_tile_slots(H) * 2 * I / 32),
                 at(sl.w2_row_q, sl.w2_row_sf, E * mx_tile_slots(I) * H / 32)};
}

// With save_for_backward, each quantisation pass also writes the backward's
// encoding of the same tensor into `saved` (one read, both layouts).
// The dispatch gather is fused into the first quantisation: X_perm exists
// only as its MXFP8 encodings (saved x_perm is not stored in this mode); the
// gate/up epilogue writes A's two encodings itself (A is never stored in
// bf16 in this mode).  B operands are K-major: W13 and W2 are encoded
// transposed (their K = H or I runs along the rows of the stored matrices).
moe_status forward_mx(const moe_dims* d, const void* X, const void* W13, const void* W2,
                      const moe_route_out* r, void* h13, void* zg, char* wsb,
                      const FwdWs& w, const MxSaved& sv, int32_t* dev_status, cudaStream_t s) {
  const int64_t rows = max_rows(d), rp = rows_pad(d);
  const int H = d->H, I = d->I, E = d->E;
  const Mx x = mx_at(wsb, w.x), w13 = mx_at(wsb, w.w13), a = mx_at(wsb, w.a), w2 = mx_at(wsb, w.w2);
  const int32_t* tpad = r->padded_offsets + E;
  const bool both = d->save_for_backward != 0;
  const DualGather gx{r->assign_of_row, d->top_k, d->T * d->top_k, nullptr, dev_status};
  MOE_TRY(quant_both(X, rows, H, tpad, &x, both ? &sv.x_col : nullptr, s, &gx));
  // W13: row-wise for dX (saved), transposed column-wise for the gate/up GEMM
  MOE_TRY(quant_both(W13, (int64_t)E * H, 2 * I, nullptr, both ? &sv.w13_row : nullptr, &w13, s,
                     nullptr, DualOut{H, H, H, 1}));
  moe_status st;
  EngineLaunch L;
  memset(&L, 0, sizeof(L));
  L.nprob = 1;
  L.E = E;
  L.elem_bytes = 1;
  L.BN = kMxTileN;
  L.padded_offsets = r->padded_offsets;
  L.counts = r->counts;
  L.max_rows = rows;
  L.status = dev_status;
  L.wait_ns = wait_limit_ns();
  {
    GemmDesc& g = L.prob[0];
    g = GemmDesc{};
    g.kind = GK_FWD1;
    g.a = x.q; g.a_rows = rows; g.a_cols = H; g.sfa = x.sf; g.sfa_bytes = x.sf_bytes; g.sfa_kg = H / 128;
    g.b = w13.q; g.b_rows = (int64_t)E * 2 * I; g.b_cols = H; g.b_expert_rows = 2 * I;
    g.sfb = w13.sf; g.sfb_bytes = w13.sf_bytes; g.sfb_kg = H / 128; g.sfb_seg = mx_tile_slots(2 * I);
    g.N = 2 * I; g.K = H; g.I = I;
    // A leaves the epilogue as its MXFP8 encodings (row-wise for the down
    // GEMM, column-wise along tokens for dW2), never as bf16
    g.enc_row_q = (uint8_t*)a.q; g.enc_row_sf = (uint8_t*)a.sf;
    if (both) {
      g.enc_col_q = (uint8_t*)sv.act_col.q; g.enc_col_sf = (uint8_t*)sv.act_col.sf;
      g.enc_col_kg = rp / 128;
    }
    g.out2 = d->save_for_backward ? h13 : nullptr; g.ld_out2 = 2 * I;
    MOE_TRY(engine(L, s, &st));
    if (st != MOE_OK) return st;
  }
  // W2: row-wise for D (saved), transposed column-wise for the down GEMM
  MOE_TRY(quant_both(W2, (int64_t)E * I, H, nullptr, both ? &sv.w2_row : nullptr, &w2, s, nullptr,
                     DualOut{I, I, I, 0}));
  {
    GemmDesc& g = L.prob[0];
    g = GemmDesc{};
    g.kind = GK_FWD2;
    g.a = a.q; g.a_rows = rows; g.a_cols = I; g.sfa = a.sf; g.sfa_bytes = a.sf_bytes; g.sfa_kg = I / 128;
    g.b = w2.q; g.b_rows = (int64_t)E * H; g.b_cols = I; g.b_expert_rows = H;
    g.sfb = w2.sf; g.sfb_bytes = w2.sf_bytes; g.sfb_kg = I / 128; g.sfb_seg = mx_tile_slots(H);
    g.N = H; g.K = I;
    g.out = zg; g.ld_out = H;
    g.gate = r->gate; g.assign_of_row = r->assign_of_row; g.n_assign = d->T * d->top_k;
    MOE_TRY(engine(L, s, &st));
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

// Backward with MXFP8 GEMMs (modes mxfp8 and fp8_bwd).  The dSwiGLU epilogue
// writes dh13's two encodings, which dX and dW13 read, so the gradient GEMMs
// run as two launches: {D + dSwiGLU, dW2}, then {dX, dW13}.
// The dY gather is fused into its quantisation: dY_perm and gate * dY_perm
// exist only as their MXFP8 encodings.  The weight gradients' B operands
// (gate * dY and dh13 along tokens) are stored transposed (K-major).
moe_status backward_mx(const moe_dims* d, const void* dY, const void* W13, const void* W2,
                       const moe_route_out* r, const void* x_perm, const void* h13,
                       const void* act, void* dxp,
                       float* partial, void* dW13, void* dW2, char* wsb, const BwdWs& w,
                       const MxSaved& sv, int32_t* dev_status, cudaStream_t s) {
  const int64_t rows = max_rows(d), rp = rows_pad(d);
  const int H = d->H, I = d->I, E = d->E;
  const int kgt = (int)(rp / 128);   // K groups of the token axis
  // mxfp8: X_perm, A, W13 and W2 were quantised for the backward by the
  // forward (saved); fp8_bwd (bf16 forward): quantised here
  const bool saved_mx = d->mode == MOE_MXFP8;
  const Mx dy = mx_at(wsb, w.dy), dygc = mx_at(wsb, w.dygc), dh13r = mx_at(wsb, w.dh13r),
           dh13c = mx_at(wsb, w.dh13c);
  const Mx w2r = saved_mx ? sv.w2_row : mx_at(wsb, w.w2r);
  const Mx actc = saved_mx ? sv.act_col : mx_at(wsb, w.actc);
  const Mx w13r = saved_mx ? sv.w13_row : mx_at(wsb, w.w13r);
  const Mx xpc = saved_mx ? sv.x_col : mx_at(wsb, w.xpc);
  const int32_t* po = r->padded_offsets;
  const DualGather gy{r->assign_of_row, d->top_k, d->T * d->top_k, r->gate, dev_status};
  MOE_TRY(quant_both(dY, rows, H, po + E, &dy, &dygc, s, &gy, DualOut{0, rp, rp, 0}));
  if (!saved_mx) {
    MOE_TRY(quant_both(W2, (int64_t)E * I, H, nullptr, &w2r, nullptr, s, nullptr, DualOut{I, 0, 0, 0}));
    MOE_TRY(quant_cols(act, rows, I, po, E, actc, dev_status, s));
  }
  EngineLaunch L;
  memset(&L, 0, sizeof(L));
  L.E = E;
  L.elem_bytes = 1;
  L.BN = kMxTileN;
  L.padded_offsets = po;
  L.counts = r->counts;
  L.max_rows = rows;
  L.status = dev_status;
  L.wait_ns = wait_limit_ns();
  moe_status st;
  {
    L.nprob = 2;
    GemmDesc& gd = L.prob[0];
    gd = GemmDesc{};
    gd.kind = GK_BWD_D;
    gd.a = dy.q; gd.a_rows = rows; gd.a_cols = H; gd.sfa = dy.sf; gd.sfa_bytes = dy.sf_bytes; gd.sfa_kg = H / 128;
    gd.b = w2r.q; gd.b_rows = (int64_t)E * I; gd.b_cols = H; gd.b_expert_rows = I;
    gd.sfb = w2r.sf; gd.sfb_bytes = w2r.sf_bytes; gd.sfb_kg = H / 128; gd.sfb_seg = mx_tile_slots(I);
    gd.N = I; gd.K = H; gd.I = I;
    // dh13 leaves the dSwiGLU epilogue as its two MXFP8 encodings (row-wise
    // for dX, column-wise along tokens, transposed, for dW13), never as bf16
    gd.enc_row_q = (uint8_t*)dh13r.q; gd.enc_row_sf = (uint8_t*)dh13r.sf;
    gd.enc_col_q = (uint8_t*)dh13c.q; gd.enc_col_sf = (uint8_t*)dh13c.sf;
    gd.enc_col_kg = rp / 128; gd.enc_col_ld = rp;
    gd.aux = h13; gd.ld_aux = 2 * I;
    gd.gate = r->gate; gd.assign_of_row = r->assign_of_row; gd.n_assign = d->T * d->top_k;
    gd.partial = partial;
    GemmDesc& gw2 = L.prob[1];
    gw2 = GemmDesc{};
    gw2.kind = GK_DW;
    gw2.a_mn = 1;
    gw2.a = actc.q; gw2.a_rows = rows; gw2.a_cols = I; gw2.sfa = actc.sf; gw2.sfa_bytes = actc.sf_bytes; gw2.sfa_kg = kgt;
    gw2.b = dygc.q; gw2.b_rows = H; gw2.b_cols = rp; gw2.sfb = dygc.sf; gw2.sfb_bytes = dygc.sf_bytes; gw2.sfb_kg = kgt;
    gw2.M = I; gw2.N = H;
    gw2.out = dW2; gw2.ld_out = H;
    MOE_TRY(engine(L, s, &st));
    if (st != MOE_OK) return st;
  }
  if (!saved_mx) {
    MOE_TRY(quant_both(W13, (int64_t)E * H, 2 * I, nullptr, &w13r, nullptr, s, nullptr,
                       DualOut{H, 0, 0, 0}));
    MOE_TRY(quant_cols(x_perm, rows, H, po, E, xpc, dev_status, s));
  }
  {
    L.nprob = 2;
    GemmDesc& gx = L.prob[0];
    gx = GemmDesc{};
    gx.kind = GK_BWD_DX;
    gx.a = dh13r.q; gx.a_rows = rows; gx.a_cols = 2 * I; gx.sfa = dh13r.sf; gx.sfa_bytes = dh13r.sf_bytes; gx.sfa_kg = 2 * I / 128;
    gx.b = w13r.q; gx.b_rows = (int64_t)E * H; gx.b_cols = 2 * I; gx.b_expert_rows = H;
    gx.sfb = w13r.sf; gx.sfb_bytes = w13r.sf_bytes; gx.sfb_kg = 2 * I / 128; gx.sfb_seg = mx_tile_slots(H);
    gx.N = H; gx.K = 2 * I;
    gx.out = dxp; gx.ld_out = H;
    GemmDesc& gw = L.prob[1];
    gw = GemmDesc{};
    gw.kind = GK_DW;
    gw.a_mn = 1;
    gw.a = xpc.q; gw.a_rows = rows; gw.a_cols = H; gw.sfa = xpc.sf; gw.sfa_bytes = xpc.sf_bytes; gw.sfa_kg = kgt;
    gw.b = dh13c.q; gw.b_rows = 2 * I; gw.b_cols = rp; gw.sfb = dh13c.sf; gw.sfb_bytes = dh13c.sf_bytes; gw.sfb_kg = kgt;
    gw.M = H; gw.N = 2 * I;
    gw.out = dW13; gw.ld_out = 2 * I;
    MOE_TRY(engine(L, s, &st));
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}
}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int64_t moe_max_rows(const moe_dims* d) { return dims_ok(d) ? max_rows(d) : -1; }

size_t moe_workspace_size(const moe_dims* d, int which) {
  if (!dims_ok(d)) return 0;
  switch (which) {
    case MOE_WS_ROUTE: return route_ws(d).total;
    case MOE_WS_FORWARD: return fwd_ws(d).total;
    case MOE_WS_BACKWARD: return bwd_ws(d).total;
  }
  return 0;
}

moe_status moe_saved_layout_of(const moe_dims* d, moe_saved_layout* out) {
  if (!dims_ok(d) || !out) return MOE_ERR_INVALID_ARG;
  *out = saved_layout(d);
  return MOE_OK;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_BAD_INDEX: return "index out of range";
    case MOE_ERR_BAD_INPUT: return "input outside the operation's domain";
  }
  return "unknown status";
}

void moe_set_gemm_events(int which, void* start, void* stop) {
  if (which != MOE_WS_FORWARD && which != MOE_WS_BACKWARD) return;
  g_ev_start[which].store(start && stop ? start : nullptr);
  g_ev_stop[which].store(start && stop ? stop : nullptr);
}

void moe_set_gemm_launch_events(int which, void* const* start, void* const* stop, int n) {
  if (which != MOE_WS_FORWARD && which != MOE_WS_BACKWARD) return;
  g_launch_armed[which].store(0);
  if (!start || !stop || n <= 0) return;
  LaunchEvents& h = g_launch_ev[which];
  h.n = n < kMaxLaunchEvents ? n : kMaxLaunchEvents;
  for (int i = 0; i < h.n; ++i) {
    if (!start[i] || !stop[i]) return;   // incomplete list: stays cancelled
    h.start[i] = start[i];
    h.stop[i] = stop[i];
  }
  g_launch_armed[which].store(1);
}

void moe_set_debug(int flags, int64_t wait_limit_ns) {
  g_debug_flags.store(flags);
  g_wait_ns.store(wait_limit_ns > 0 ? wait_limit_ns : 1000000000LL);
}

moe_status moe_debug_occupy(int ctas, int smem_bytes, int64_t duration_ns, void* stream) {
  if (ctas < 1 || ctas > 4096 || smem_bytes < 0 || smem_bytes > 227 * 1024 || duration_ns <= 0 ||
      duration_ns > 1000000000LL)
    return MOE_ERR_INVALID_ARG;
  static CtxCache<int> attr;
  int done = 0;
  if (attr.get(&done, [](int* v) {
        *v = 1;
        return cudaFuncSetAttribute(occupy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    227 * 1024);
      }) != cudaSuccess)
    return MOE_ERR_CUDA;
  occupy_kernel<<<ctas, 32, smem_bytes, static_cast<cudaStream_t>(stream)>>>(
      (uint64_t)duration_ns);
  return cuda_status(cudaGetLastError());
}

moe_status moe_route(const moe_dims* d, const float* logits, const moe_route_out* out, void* ws,
                     size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (!dims_ok(d) || !route_ok(out, d->T) || !aligned16(ws) || !aligned16(dev_status))
    return MOE_ERR_INVALID_ARG;
  if (d->T > 0 && !aligned16(logits)) return MOE_ERR_INVALID_ARG;
  const RouteWs w = route_ws(d);
  if (ws_bytes < w.total) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* hist = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + w.hist);
  int32_t* base = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + w.base);
  MOE_TRY(launch_route(logits, d->T, d->E, d->top_k, out->topk_idx, out->gate, hist, dev_status, s));
  MOE_TRY(launch_permute(out->topk_idx, d->T, d->E, d->top_k, max_rows(d), hist, base, out->counts,
                         out->offsets, out->padded_offsets, out->row_of_assign,
                         out->assign_of_row, dev_status, s));
  return MOE_OK;
}

moe_status moe_route_backward(const moe_dims* d, const moe_route_out* r, const float* dgate,
                              float* dlogits, int32_t* dev_status, void* stream) {
  if (!dims_ok(d) || !route_ok(r, d->T) || !aligned16(dev_status)) return MOE_ERR_INVALID_ARG;
  if (d->T > 0 && (!aligned16(dgate) || !aligned16(dlogits))) return MOE_ERR_INVALID_ARG;
  MOE_TRY(launch_route_backward(r->topk_idx, r->gate, dgate, d->T, d->E, d->top_k, dlogits,
                                dev_status, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_forward(const moe_dims* d, const void* X, const void* W13, const void* W2,
                       const moe_route_out* r, void* Y, void* saved, size_t saved_bytes,
                       void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (!dims_ok(d) || !route_ok(r, d->T) || !aligned16(W13) || !aligned16(W2) || !aligned16(saved) ||
      !aligned16(ws) || !aligned16(dev_status))
    return MOE_ERR_INVALID_ARG;
  if (d->T > 0 && (!aligned16(X) || !aligned16(Y))) return MOE_ERR_INVALID_ARG;
  const moe_saved_layout sl = saved_layout(d);
  const FwdWs w = fwd_ws(d);
  if (saved_bytes < sl.total || ws_bytes < w.total) return MOE_ERR_INVALID_ARG;
  const int bn1 = bn_fwd1(d), bn2 = bn_div(d->H);
  if (!bn1 || !bn2) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int es = elem_bytes(d);
  const int64_t rows = max_rows(d);
  const int n_assign = d->T * d->top_k;
  char* sv = static_cast<char*>(saved);
  void* x_perm = sv + sl.x_perm;
  void* h13 = sv + sl.h13;
  void* act = sv + sl.act;
  void* zg = static_cast<char*>(ws) + w.zg;

  if (mx_fwd(d)) {
    EventScope timing(MOE_WS_FORWARD, s);
    const moe_status st = forward_mx(d, X, W13, W2, r, h13, zg, static_cast<char*>(ws), w,
                                     mx_saved(d, sl, sv), dev_status, s);
    if (st != MOE_OK) return st;
    timing.finish();
    MOE_TRY(launch_combine(zg, Y, d->T, d->H, es, d->top_k, r->row_of_assign, rows, dev_status, s));
    return MOE_OK;
  }
  const bool f32 = d->mode == MOE_F32;
  const void* w13_src = W13;
  const void* w2_src = W2;
  if (f32) {
    float* w13t = reinterpret_cast<float*>(static_cast<char*>(ws) + w.w13t);
    float* w2t = reinterpret_cast<float*>(static_cast<char*>(ws) + w.w2t);
    MOE_TRY(launch_transpose_f32(static_cast<const float*>(W13), w13t, d->E, d->H, 2 * d->I, d->H, s));
    MOE_TRY(launch_transpose_f32(static_cast<const float*>(W2), w2t, d->E, d->I, d->H, d->I, s));
    w13_src = w13t;
    w2_src = w2t;
  }
  MOE_TRY(launch_gather_rows(X, x_perm, d->H, es, d->top_k, n_assign, r->assign_of_row,
                             r->row_of_assign, r->padded_offsets, d->E, rows, dev_status, s));
  moe_status st;
  EventScope timing(MOE_WS_FORWARD, s);
  EngineLaunch L;
  memset(&L, 0, sizeof(L));
  L.nprob = 1;
  L.E = d->E;
  L.elem_bytes = es;
  L.padded_offsets = r->padded_offsets;
  L.counts = r->counts;
  L.max_rows = rows;
  L.status = dev_status;
  L.wait_ns = wait_limit_ns();
  {
    L.BN = bn1;
    GemmDesc& g = L.prob[0];
    g = GemmDesc{};
    g.kind = GK_FWD1;
    g.a = x_perm; g.a_rows = rows; g.a_cols = d->H;
    if (gate_on_act(d)) {   // A leaves as gate * A (0 on pad rows)
      g.gate = r->gate; g.assign_of_row = r->assign_of_row; g.n_assign = n_assign;
    }
    if (f32) {   // W13^T [E*2I, H], K-major
      g.b = w13_src; g.b_rows = (int64_t)d->E * 2 * d->I; g.b_cols = d->H;
      g.b_expert_rows = 2 * d->I;
    } else {     // W13 [E*H, 2I], N-major
      g.b_mn = 1;
      g.b = w13_src; g.b_rows = (int64_t)d->E * d->H; g.b_cols = 2 * d->I;
      g.b_expert_rows = d->H;
    }
    g.N = 2 * d->I; g.K = d->H; g.I = d->I;
    g.out = act; g.ld_out = d->I;
    g.out2 = d->save_for_backward ? h13 : nullptr; g.ld_out2 = 2 * d->I;
    MOE_TRY(engine(L, s, &st));
    if (st != MOE_OK) return st;
  }
  {
    L.BN = bn2;
    GemmDesc& g = L.prob[0];
    g = GemmDesc{};
    g.kind = GK_FWD2;
    g.a = act; g.a_rows = rows; g.a_cols = d->I;
    if (f32) {   // W2^T [E*H, I], K-major
      g.b = w2_src; g.b_rows = (int64_t)d->E * d->H; g.b_cols = d->I;
      g.b_expert_rows = d->H;
    } else {     // W2 [E*I, H], N-major
      g.b_mn = 1;
      g.b = w2_src; g.b_rows = (int64_t)d->E * d->I; g.b_cols = d->H;
      g.b_expert_rows = d->I;
    }
    g.N = d->H; g.K = d->I;
    g.out = zg; g.ld_out = d->H;
    if (!gate_on_act(d)) {  // Z = gate * (A W2)
      g.gate = r->gate; g.assign_of_row = r->assign_of_row; g.n_assign = n_assign;
    }
    MOE_TRY(engine(L, s, &st));
    if (st != MOE_OK) return st;
  }
  timing.finish();
  MOE_TRY(launch_combine(zg, Y, d->T, d->H, es, d->top_k, r->row_of_assign, rows, dev_status, s));
  return MOE_OK;
}

moe_status moe_backward(const moe_dims* d, const void* dY, const void* W13, const void* W2,
                        const moe_route_out* r, const void* saved, size_t saved_bytes, void* dX,
                        void* dW13, void* dW2, float* dgate, void* ws, size_t ws_bytes,
                        int32_t* dev_status, void* stream) {
  if (!dims_ok(d) || !route_ok(r, d->T) || !aligned16(W13) || !aligned16(W2) || !aligned16(saved) ||
      !aligned16(dW13) || !aligned16(dW2) || !aligned16(ws) || !aligned16(dev_status))
    return MOE_ERR_INVALID_ARG;
  if (d->T > 0 && (!aligned16(dY) || !aligned16(dX) || !aligned16(dgate)))
    return MOE_ERR_INVALID_ARG;
  const moe_saved_layout sl = saved_layout(d);
  const BwdWs w = bwd_ws(d);
  if (saved_bytes < sl.total || ws_bytes < w.total) return MOE_ERR_INVALID_ARG;
  const int bn = bn_bwd(d);
  if (!bn) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int es = elem_bytes(d);
  const int64_t rows = max_rows(d);
  const int n_assign = d->T * d->top_k;
  const char* sv = static_cast<const char*>(saved);
  const void* x_perm = sv + sl.x_perm;
  const void* h13 = sv + sl.h13;
  const void* act = sv + sl.act;
  char* wb = static_cast<char*>(ws);
  void* dy_perm = wb + w.dy_perm;
  void* dyg_perm = wb + w.dyg_perm;
  void* dh13 = wb + w.dh13;
  void* dxp = wb + w.dxp;
  float* partial = reinterpret_cast<float*>(wb + w.partial);
  int32_t* ready = reinterpret_cast<int32_t*>(wb + w.ready);

  if (mx_bwd(d)) {
    EventScope timing(MOE_WS_BACKWARD, s);
    const moe_status st = backward_mx(d, dY, W13, W2, r, x_perm, h13, act, dxp,
                                      partial, dW13, dW2, wb, w,
                                      mx_saved(d, sl, const_cast<char*>(sv)), dev_status, s);
    if (st != MOE_OK) return st;
    timing.finish();
    MOE_TRY(launch_combine(dxp, dX, d->T, d->H, es, d->top_k, r->row_of_assign, rows, dev_status,
                           s));
    MOE_TRY(launch_dgate_reduce(partial, w.nt_d, n_assign, r->row_of_assign, rows, dgate,
                                dev_status, s));
    return MOE_OK;
  }
  if (gate_on_act(d))   // the forward left gate * A in `act`: dY_perm alone
    MOE_TRY(launch_gather_rows(dY, dy_perm, d->H, es, d->top_k, n_assign, r->assign_of_row,
                               r->row_of_assign, r->padded_offsets, d->E, rows, dev_status, s));
  else
    MOE_TRY(launch_gather_grad(dY, dy_perm, dyg_perm, d->H, es, d->top_k, n_assign,
                               r->assign_of_row, r->gate, r->padded_offsets, d->E, rows,
                               dev_status, s));
  // one co-scheduled launch with readiness counters (diagnosis flags only)
  const bool one_launch = d->mode != MOE_F32 &&
                          (debug_flags() & (MOE_DEBUG_ONE_LAUNCH_BACKWARD | MOE_DEBUG_NEVER_READY));
  if (one_launch) MOE_TRY(cudaMemsetAsync(ready, 0, ((rows + 127) / 128 + 1) * sizeof(int32_t), s));
  const bool f32 = d->mode == MOE_F32;
  const int64_t lt = ld_t(d);
  float* act_t = reinterpret_cast<float*>(wb + w.act_t);
  float* dyg_t = reinterpret_cast<float*>(wb + w.dyg_t);
  float* xp_t = reinterpret_cast<float*>(wb + w.xp_t);
  float* dh13_t = reinterpret_cast<float*>(wb + w.dh13_t);

  EngineLaunch L;
  memset(&L, 0, sizeof(L));
  L.E = d->E;
  L.elem_bytes = es;
  L.BN = bn;
  L.padded_offsets = r->padded_offsets;
  L.counts = r->counts;
  L.max_rows = rows;
  L.ready = ready;
  L.ready_target = (debug_flags() & MOE_DEBUG_NEVER_READY) ? 0x7fffffff : d->I / bn;
  L.status = dev_status;
  L.wait_ns = wait_limit_ns();

  // D = dY_perm W2^T with the dSwiGLU / d(gate) epilogue
  GemmDesc gd{};
  gd.kind = GK_BWD_D;
  gd.a = dy_perm; gd.a_rows = rows; gd.a_cols = d->H;
  gd.b = W2; gd.b_rows = (int64_t)d->E * d->I; gd.b_cols = d->H;
  gd.N = d->I; gd.K = d->H; gd.b_expert_rows = d->I; gd.I = d->I;
  gd.out = dh13; gd.ld_out = 2 * d->I;
  gd.aux = h13; gd.ld_aux = 2 * d->I;
  gd.gate = r->gate; gd.assign_of_row = r->assign_of_row; gd.n_assign = n_assign;
  gd.partial = partial;
  // dW2_e = A_e^T (gate * dY)_perm_e = (gate * A)_e^T dY_perm_e, the second
  // form in bf16 mode (`act` holds gate * A); needs nothing from this launch
  GemmDesc gw2{};
  gw2.kind = GK_DW;
  gw2.M = d->I; gw2.N = d->H;
  gw2.out = dW2; gw2.ld_out = d->H;
  // dXp = dh13 W13^T
  GemmDesc gx{};
  gx.kind = GK_BWD_DX;
  gx.a = dh13; gx.a_rows = rows; gx.a_cols = 2 * d->I;
  gx.b = W13; gx.b_rows = (int64_t)d->E * d->H; gx.b_cols = 2 * d->I;
  gx.N = d->H; gx.K = 2 * d->I; gx.b_expert_rows = d->H;
  gx.out = dxp; gx.ld_out = d->H;
  // dW13_e = X_perm_e^T dh13_e
  GemmDesc gw13{};
  gw13.kind = GK_DW;
  gw13.M = d->H; gw13.N = 2 * d->I;
  gw13.out = dW13; gw13.ld_out = 2 * d->I;

  moe_status st;
  EventScope timing(MOE_WS_BACKWARD, s);
  if (!f32) {
    gw2.a_mn = gw2.b_mn = 1;
    gw2.a = act; gw2.a_rows = rows; gw2.a_cols = d->I;
    // dW2 = (gate * A)^T dY_perm (bf16: `act` holds gate * A)
    gw2.b = gate_on_act(d) ? dy_perm : dyg_perm; gw2.b_rows = rows; gw2.b_cols = d->H;
    gw13.a_mn = gw13.b_mn = 1;
    gw13.a = x_perm; gw13.a_rows = rows; gw13.a_cols = d->H;
    gw13.b = dh13; gw13.b_rows = rows; gw13.b_cols = 2 * d->I;
    if (debug_flags() & MOE_DEBUG_SPLIT_BACKWARD) {
      // one launch per gradient GEMM, in dependency order (diagnosis only)
      const GemmDesc parts[4] = {gd, gw2, gx, gw13};
      L.nprob = 1;
      for (const GemmDesc& gp : parts) {
        L.prob[0] = gp;
        MOE_TRY(engine(L, s, &st));
        if (st != MOE_OK) return st;
      }
    } else if (one_launch) {
      // all four in one persistent launch: D tiles publish their m-block,
      // dX tiles wait for their m-block, dW13 tiles for their expert's
      // m-blocks (bounded waits; a cooperative launch, see gemm.cu)
      gd.signal = 1;
      gx.dep = DEP_MBLOCK;
      gw13.dep = DEP_EXPERT;
      L.nprob = 4;
      L.prob[0] = gd;
      L.prob[1] = gw2;
      L.prob[2] = gx;
      L.prob[3] = gw13;
      MOE_TRY(engine(L, s, &st));
      if (st != MOE_OK) return st;
    } else {
      // Co-scheduled in two persistent launches ([OB] "Overlapping Backward
      // Pass": the activation-gradient GEMMs need the weights, not the
      // weight gradients): {D + dSwiGLU, dW2}, then {dX, dW13}, the only
      // dependency (dh13, written by D, read by dX and dW13) ordered by the
      // stream, so no tile waits on another CTA.
      L.nprob = 2;
      L.prob[0] = gd;
      L.prob[1] = gw2;
      MOE_TRY(engine(L, s, &st));
      if (st != MOE_OK) return st;
      L.prob[0] = gx;
      L.prob[1] = gw13;
      MOE_TRY(engine(L, s, &st));
      if (st != MOE_OK) return st;
    }
  } else {
    // TF32 reads K-major operands only: transposed token-axis copies, and the
    // weight-gradient GEMM of W13 runs after dh13 is complete.
    MOE_TRY(launch_transpose_f32(static_cast<const float*>(act), act_t, 1, rows, d->I, lt, s));
    MOE_TRY(launch_transpose_f32(static_cast<const float*>(dyg_perm), dyg_t, 1, rows, d->H, lt, s));
    MOE_TRY(launch_transpose_f32(static_cast<const float*>(x_perm), xp_t, 1, rows, d->H, lt, s));
    gw2.a = act_t; gw2.a_rows = d->I; gw2.a_cols = lt;
    gw2.b = dyg_t; gw2.b_rows = d->H; gw2.b_cols = lt;
    gd.signal = 0;
    L.nprob = 2;
    L.prob[0] = gd;
    L.prob[1] = gw2;
    MOE_TRY(engine(L, s, &st));
    if (st != MOE_OK) return st;
    MOE_TRY(launch_transpose_f32(static_cast<const float*>(dh13), dh13_t, 1, rows, 2 * d->I, lt, s));
    gw13.a = xp_t; gw13.a_rows = d->H; gw13.a_cols = lt;
    gw13.b = dh13_t; gw13.b_rows = 2 * d->I; gw13.b_cols = lt;
    L.nprob = 2;
    L.prob[0] = gx;
    L.prob[1] = gw13;
    MOE_TRY(engine(L, s, &st));
    if (st != MOE_OK) return st;
  }
  timing.finish();
  MOE_TRY(launch_combine(dxp, dX, d->T, d->H, es, d->top_k, r->row_of_assign, rows, dev_status, s));
  MOE_TRY(launch_dgate_reduce(partial, w.nt_d, n_assign, r->row_of_assign, rows, dgate, dev_status,
                              s));
  return MOE_OK;
}

moe_status moe_quantize_mxfp8_dual(const void* src, int R, int C, int ld,
                                   const int32_t* rows_limit, uint8_t* q_row, uint8_t* s_row,
                                   uint8_t* q_col, uint8_t* s_col, int32_t* dev_status,
                                   void* stream) {
  if (R < 0 || C <= 0 || R % 32 || C % 128 || ld < C || ld % 8 || !aligned16(dev_status))
    return MOE_ERR_INVALID_ARG;
  if (R == 0) return MOE_OK;
  if (!aligned16(src) || !aligned16(q_row) || !aligned16(q_col) || !s_row || !s_col)
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(launch_quantize_dual(src, R, C, ld, rows_limit, q_row, s_row, q_col, s_col,
                               static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_quantize_mxfp8(const void* src, int R, int C, int ld, int axis,
                              const int32_t* group_offsets, int G, uint8_t* q, uint8_t* scales,
                              int32_t* dev_status, void* stream) {
  if (R < 0 || C < 0 || ld < C || (axis != 0 && axis != 1)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(dev_status)) return MOE_ERR_INVALID_ARG;
  if (axis == 1 && (C % 32 != 0 || ld % 8 != 0)) return MOE_ERR_INVALID_ARG;
  if (axis == 0 && (R % 32 != 0 || C % 2 != 0 || ld % 2 != 0)) return MOE_ERR_INVALID_ARG;
  if (group_offsets && (axis != 0 || G < 1 || ((uintptr_t)group_offsets & 3)))
    return MOE_ERR_INVALID_ARG;
  if ((int64_t)R * C > 0 && (!aligned16(src) || !aligned16(q) || !scales))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(launch_quantize(src, R, C, ld, axis, group_offsets, G, q, scales, dev_status,
                          static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// moe_route_noalloc: the router and permutation builder for callers that
// cannot allocate device memory (see include/moe.h).  Its scratch (the
// per-block expert histograms and their exclusive bases, 2 * E * ceil(T/128)
// int32) lives in one file-scope device array instead of a caller workspace.
// ---------------------------------------------------------------------------
namespace moe {
namespace {

constexpr int64_t kNoAllocRouteInts = 131072;   // 512 KiB of int32 scratch
__device__ __align__(256) int32_t g_route_scratch[kNoAllocRouteInts];

// In host code g_route_scratch names a host-side stand-in, not the device
// array, so its device address is looked up with the device current, once per
// CUDA context (a context created after a device reset holds a new copy of
// the array and gets a new lookup), and cached.  The lookup is not made while
// the stream is being captured into a graph.
CtxCache<int32_t*> g_scratch_addr;

cudaError_t route_scratch_ptr(cudaStream_t s, int32_t** out) {
  bool found = false;
  cudaError_t e = g_scratch_addr.find(out, &found);
  if (e != cudaSuccess || found) return e;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  if (cs != cudaStreamCaptureStatusNone) return cudaErrorStreamCaptureUnsupported;
  return g_scratch_addr.get(out, [](int32_t** v) {
    void* p = nullptr;
    const cudaError_t r = cudaGetSymbolAddress(&p, g_route_scratch);
    if (r == cudaSuccess) *v = static_cast<int32_t*>(p);
    return r;
  });
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_noalloc(const moe_dims* d, const float* logits,
                                        const moe_route_out* out, int32_t* dev_status,
                                        void* stream) {
  using namespace moe;
  if (!dims_ok(d) || !route_ok(out, d->T) || !aligned16(dev_status)) return MOE_ERR_INVALID_ARG;
  if (d->T > 0 && !aligned16(logits)) return MOE_ERR_INVALID_ARG;
  const int64_t nb = ((int64_t)d->T + kRouteTokPerBlock - 1) / kRouteTokPerBlock;
  if (2 * nb * d->E > kNoAllocRouteInts) return MOE_ERR_INVALID_ARG;   // scratch too small
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* scratch = nullptr;
  if (route_scratch_ptr(s, &scratch) != cudaSuccess) return MOE_ERR_CUDA;
  // Every scratch entry read below is first written by the same call (the
  // router writes all E x nb histogram entries, the scan all bases), so no
  // clearing is needed.
  int32_t* hist = scratch;
  int32_t* base = scratch + nb * d->E;
  MOE_TRY(launch_route(logits, d->T, d->E, d->top_k, out->topk_idx, out->gate, hist, dev_status, s));
  MOE_TRY(launch_permute(out->topk_idx, d->T, d->E, d->top_k, max_rows(d), hist, base, out->counts,
                         out->offsets, out->padded_offsets, out->row_of_assign,
                         out->assign_of_row, dev_status, s));
  return MOE_OK;
}
