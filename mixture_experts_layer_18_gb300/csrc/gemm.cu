// gemm.cu - persistent grouped-GEMM engine for the expert layer (sm_103a:
// tcgen05 MMA with TMEM accumulators, TMA loads, mbarrier pipeline).
//
// "Accelerating dropless MoE in JAX with NVIDIA Transformer Engine",
// "Optimisation 1: grouped GEMM": all expert GEMMs run in one launch over
// each expert's real token count, with the counts kept on the device.  Here
// the per-expert row ranges come from padded_offsets (a device array): every
// 128-row tile belongs to one expert, so the tile list is derived on the GPU
// and nothing is copied to the host.
// "Prime Intellect releases Prime Mega MoE" (MarkTechPost), "How does the
// fused kernel work?": SwiGLU is fused after the first expert linear and the
// combine after the second; the backward is trainable.
// "Prime Intellect Mega MoE" digest, "Overlapping Backward Pass": activation
// gradients need the weights, not the weight gradients, so both kinds of tile
// are co-scheduled in one persistent launch here (readiness counters order
// the dX / dW13 tiles after the dH tiles they read).
//
// Problem kinds (A is M x K, B is K x N, all row-major in HBM):
//   FWD1   h13 = X_perm_e W13_e, epilogue A = silu(u) * v (+ store h13)
//          A: X_perm [rows, H] K-major;  B: W13 as [E*H, 2I] N-major.
//          One MMA tile of N = BN covers BN/2 gate columns and the same BN/2
//          up columns, so the activation needs no second pass.  With a gate
//          vector (bf16) A leaves as gate * A; block-scaled runs write A's
//          MXFP8 encodings instead of bf16.
//   FWD2   Z = gate * (A_e W2_e)  (no gate when FWD1 applied it)
//          A: act [rows, I] K-major;  B: W2 as [E*I, H] N-major.
//   BWD_D  D = dY_perm_e W2_e^T, epilogue dSwiGLU -> dh13, d(gate) partials
//          A: dY_perm [rows, H] K-major;  B: W2 as [E*I, H] K-major.
//          Block-scaled runs write dh13's MXFP8 encodings instead of bf16.
//   BWD_DX dXp = dh13_e W13_e^T
//          A: dh13 [rows, 2I] K-major;  B: W13 as [E*H, 2I] K-major.
//   DW     dW_e = S_e^T G_e over the expert's rows (K = padded rows of e)
//          A: S [rows, M] M-major;  B: G [rows, N] N-major.
// Every operand may instead come K-major from a transposed copy (W13^T
// [E*2I, H], W2^T [E*H, I], S^T [M, rows], G^T [N, rows]); TF32 MMAs read
// K-major operands only, so the fp32 mode uses those copies throughout.
//
// CTA layout (one CTA per SM): warp 0 lane 0 issues TMA loads, warp 1 owns
// TMEM and lane 0 issues tcgen05.mma, warps 2..5 run the epilogue (warp w
// reads TMEM lanes 32*(w%4) .. +31, i.e. tile rows); block-scaled pairs have
// warps 2..9, two per lane quarter, each on half of the tile's columns.
// bf16 problems run on SM pairs (clusters of 2, cta_group::2): one 256-row
// tile per pair, each CTA staging its 128 rows of A and half of B, so a
// pipeline stage is 32 KB per CTA (6 stages) instead of 48 KB (4 stages) and
// each SM's shared-memory traffic per MMA drops by a third.  The leader CTA
// issues the MMAs; its commits signal both CTAs' barriers.  Two
// TMEM accumulators of BN fp32 columns let the epilogue of one tile overlap
// the MMAs of the next.  Every wait is bounded; a wait that runs out records
// MOE_ERR_TIMEOUT, the CTA drains its copies and MMAs, frees TMEM and exits.
#include <climits>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "mx_encode.cuh"

namespace moe {

enum : int { GK_FWD1 = 0, GK_FWD2 = 1, GK_BWD_D = 2, GK_BWD_DX = 3, GK_DW = 4 };
enum : int { DEP_NONE = 0, DEP_MBLOCK = 1, DEP_EXPERT = 2 };

struct GemmProblem {
  CUtensorMap tmA;
  CUtensorMap tmB;
  CUtensorMap tmO;   // bf16 outputs: 32 x 32 boxes, 64-byte swizzle (DW: 3-D [E, M, N])
  CUtensorMap tmO2;  // FWD1: h13
  int kind, dep, signal;
  int a_mn, b_mn;    // operand stored M-/N-major (1) or K-major (0)
  int M, N, K;
  int b_expert_rows;
  int I;
  int nt;            // n-tiles
  int ld_out, ld_out2, ld_aux;
  void* out;
  void* out2;
  const void* aux;
  const float* gate;
  const int32_t* assign_of_row;
  int n_assign;      // valid assignment indices are [0, n_assign)
  float* partial;
  // FWD1 of a block-scaled run: A leaves as its MXFP8 encodings instead of
  // bf16 (codes [rows, I] and tensor-core scale atoms; row-wise blocks along
  // I, and column-wise blocks of 32 rows when enc_col_q is set)
  uint8_t* enc_row_q;
  uint8_t* enc_row_sf;
  uint8_t* enc_col_q;
  uint8_t* enc_col_sf;
  int64_t enc_col_kg;  // 128-row groups of the column-wise scale atoms
  int64_t enc_col_ld;  // > 0: column-wise codes stored transposed with this pitch
  // MXFP8 operands: E8M0 scale atoms (512 B per 128 MN indices x 128 K),
  // read through [atoms * 4, 128]-byte views: atom i is rows 4i .. 4i + 3.
  CUtensorMap tmSFA;
  CUtensorMap tmSFB;
  int sfa_kg, sfb_kg;  // K groups of 128 in each operand's 2-D view
  int64_t sfb_seg;     // B scales: MN slots per expert segment (0: one segment)
};

struct EngineParams {
  GemmProblem prob[4];
  int nprob;
  int E;
  const int32_t* padded_offsets;
  const int32_t* counts;  // rows per expert (optional: weight-gradient K loops stop there)
  int32_t* ready;         // per-m-block counters, then one total at ready_all_index
  int ready_target;       // publications per m-block (n-tiles of the signalling problem)
  int ready_all_index;
  int32_t* status;
  unsigned long long wait_ns;
};

template <typename Elt, int BN_, int PAIR_>
struct Cfg {
  static constexpr bool MX = sizeof(Elt) == 1;    // MXFP8 (E4M3 + E8M0 block scales)
  static constexpr int PAIR = PAIR_;              // CTAs per MMA tile (1, or 2 = SM pair)
  static constexpr int BN = BN_;                  // MMA N = accumulator columns
  static constexpr int BNL = BN / PAIR;           // B columns staged by each CTA
  static constexpr int ES = sizeof(Elt);          // 2: bf16, 4: fp32 read as tf32
  static constexpr int BK = 128 / ES;             // k elements per pipeline stage
  static constexpr int ATOM = 128 / ES;           // MN elements per 128-byte swizzle row
  static constexpr int A_BYTES = 128 * 128;       // 128 rows x 128 bytes
  static constexpr int B_BYTES = BNL * 128;
  static constexpr int ATOM_BYTES = BK * 128;     // one MN-major column block
  // Block-scaled tiles are 192 columns wide (kMxTileN): two accumulators of
  // 192 columns and a scale slot per pipeline stage fit the 512 TMEM
  // columns.  Their B operands come K-major (BNL = 96 rows per CTA of a
  // pair), and the scales of a tile are two whole atoms (mx_tile_pos).
  static_assert(!MX || BN == kMxTileN, "block-scaled tiles are 192 wide");
  // scale atoms per stage: A's 128 rows, and B's scales for all BN columns
  // of the MMA (each CTA of a pair needs every column's scale in its TMEM)
  static constexpr int SFA_BYTES = MX ? 512 : 0;
  static constexpr int SFB_BYTES = MX ? 2 * 512 : 0;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;        // multiple of 1024
  static constexpr int SF_BYTES = SFA_BYTES + SFB_BYTES;       // per stage, own region
  static constexpr int TX_BYTES = (STAGE_BYTES + SF_BYTES) * PAIR;   // bytes per full barrier
  // Epilogue: groups of 4 warps (one per TMEM lane quarter).  Block-scaled
  // tiles take half the MMA time of bf16 tiles of the same K, so they get two
  // groups that take alternate tiles (each group owns one accumulator and
  // has two tiles' worth of MMA time for its epilogue).
  static constexpr int EPI_WARPS = 4;             // warps per group
  static constexpr int EPI_GROUPS = MX ? 2 : 1;
  // Issue work: one thread issuing a stage's TMA loads (and, block-scaled,
  // the three scale copies beside the four MMAs) takes about as long as the
  // stage's MMAs run (384 tensor cycles for block-scaled stages, 512 for
  // bf16), so on SM pairs a second producer warp loads B (and its scales)
  // while warp 0 loads A, and block-scaled runs add a warp that copies the
  // scales into tensor memory.  Measured on GB300 (one thread issuing from
  // ready stages): four 192-column block-scaled MMAs take 384 tensor cycles
  // but the issuing loop ~420 cycles with the scale copies inline, ~480
  // with one barrier wait per stage and ~600 - 640 with two waits and a
  // fence; the copier therefore signals once per SF_GROUP stages.
  static constexpr bool SPLIT_LOAD = PAIR == 2;
  static constexpr bool SPLIT_ISSUE = MX;          // scale-copier warp
  static constexpr int SF_GROUP = 1;               // stages per scale-ready signal
  static constexpr int EXTRA_WARPS = (SPLIT_LOAD ? 1 : 0) + (SPLIT_ISSUE ? 1 : 0);
  static constexpr int THREADS = 64 + 32 * EPI_WARPS * EPI_GROUPS + 32 * EXTRA_WARPS;
  // Block-scaled CTAs put the four single-thread roles (A loader, MMA, B
  // loader, scale copier) in warpgroup 0 and the two epilogue groups in
  // warpgroups 1 and 2, so the roles can hand registers to the epilogues
  // (setmaxnreg: 4 x 32 x ROLE_REGS + 8 x 32 x EPI_REGS <= 384 x 168, the
  // registers the CTA is launched with); other CTAs keep the epilogue at
  // warps 2.. and the B loader after it.
  static constexpr bool REG_SPLIT = MX && PAIR == 2;
  static constexpr int EPI_FIRST = REG_SPLIT ? 4 : 2;     // first epilogue warp
  static constexpr int ROLE_REGS = 64, EPI_REGS = 216;
  static constexpr int STG_BYTES = EPI_WARPS * EPI_GROUPS * 4096;   // staging (2 x 2 KB per warp)
  static constexpr int FIXED_BYTES = STG_BYTES + 1024 /*align*/ + 512 /*bars*/ +
                                     2 * (kMaxE + 1) * 4 + kMaxE * 4 /*counts*/ + 64 + 256;
  static constexpr int STAGES_RAW = (232448 - FIXED_BYTES) / (STAGE_BYTES + SF_BYTES);
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  // TMEM: two accumulators of BN columns (the epilogue of one tile overlaps
  // the MMAs of the next); block-scaled runs add a 16-column scale slot per
  // pipeline stage after them.
  static constexpr int NACC = 2;
  static constexpr int SF_COL0 = 2 * BN;
  static constexpr int TMEM_COLS = MX ? 512 : 2 * BN;
  static constexpr int KSTEPS = 4;                // MMAs per stage (32 bytes of K each)
  static constexpr int MN_KSTEP_BYTES = (32 / ES) * 128;  // MN-major advance per MMA
  static constexpr uint32_t FMT = ES == 2 ? 1u : (ES == 4 ? 2u : 0u);  // BF16 : TF32 : E4M3
  static constexpr int SF_REGION = (STAGES * SF_BYTES + 255) / 256 * 256;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STG_BYTES + SF_REGION +
                                    1024 /*align*/ + 512 /*bars*/ + 2 * (kMaxE + 1) * 4 + kMaxE * 4 + 64;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(STAGE_BYTES % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
  static_assert(!MX || SF_COL0 + STAGES * 16 <= 512, "TMEM scale slots");
  static_assert(!MX || STAGES % SF_GROUP == 0, "scale-ready groups tile the stage ring");
};

// ------------------------------------------------------------ tile decode
// A tile is 128 x BN per CTA.  With PAIR == 2 the two CTAs of a cluster
// compute one 256 x BN tile: CTA rank r owns rows [128 r, 128 r + 128).
struct Tile {
  int p, kind, e, mb, m0, n0, ntile, nk, kbase;
  bool valid;   // this CTA's 128 rows belong to the tile's expert (or M)
};

// last e in [0, E) with arr[e] <= v (entries of empty experts repeat)
__device__ __forceinline__ int last_le(const int* arr, int E, int v) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (arr[mid] <= v) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <class C>
__device__ __forceinline__ Tile decode_tile(const EngineParams& P, const int* cum, const int* s_po,
                                            const int* s_pt, int t, int rank) {
  // s_pt and the per-expert row counts are consecutive arrays of kMaxE + 1
  const int* s_cnt = s_pt + (kMaxE + 1);
  Tile ti;
  int p = 0;
  while (p + 1 < P.nprob && t >= cum[p + 1]) ++p;
  const GemmProblem& g = P.prob[p];
  const int lt = t - cum[p];
  ti.p = p;
  ti.kind = g.kind;
  if (g.kind == GK_DW) {
    const int mslots = ((g.M + 127) / 128 + C::PAIR - 1) / C::PAIR;
    ti.e = lt / (mslots * g.nt);
    const int r = lt - ti.e * mslots * g.nt;
    const int i = r / g.nt;
    ti.ntile = r - i * g.nt;
    ti.mb = i * C::PAIR + rank;
    ti.m0 = ti.mb * 128;
    ti.valid = ti.m0 < g.M;
    ti.kbase = s_po[ti.e];
    // K = the expert's rows; stages past its last real row would only add
    // the zero pad rows, so the loop stops at the stage holding that row
    const int rows_e = s_po[ti.e + 1] - s_po[ti.e];
    const int cnt = s_cnt[ti.e];
    ti.nk = (cnt >= 0 ? min(rows_e, (cnt + C::BK - 1) / C::BK * C::BK) : rows_e) / C::BK;
    ti.n0 = ti.ntile * C::BN;
  } else {
    const int q = lt / g.nt;
    ti.ntile = lt - q * g.nt;
    if (C::PAIR == 1) {
      ti.mb = q;
      ti.e = last_le(s_po, P.E, q * 128);
      ti.valid = true;
    } else {
      ti.e = last_le(s_pt, P.E, q);
      ti.mb = s_po[ti.e] / 128 + 2 * (q - s_pt[ti.e]) + rank;
      ti.valid = ti.mb < s_po[ti.e + 1] / 128;
    }
    ti.m0 = ti.mb * 128;
    ti.kbase = 0;
    ti.nk = g.K / C::BK;
    ti.n0 = ti.ntile * (g.kind == GK_FWD1 ? C::BN / 2 : C::BN);
  }
  return ti;
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ bool wait_counter(const int32_t* ctr, int target, const WaitCtl& c) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (ld_acquire(ctr) >= target) return true;
    if (i == 0) {
      t0 = global_ns();
    } else if ((i & 7) == 0) {
      if (*c.abort) return false;
      if (global_ns() - t0 > c.limit_ns) {
        report(c.status, MOE_ERR_TIMEOUT);
        *c.abort = 1;
        return false;
      }
    }
    __nanosleep(256);
  }
}

// Bounded wait on a barrier that also receives arrivals from the peer CTA.
__device__ __forceinline__ bool wait_bar_cluster(uint64_t* bar, uint32_t parity, const WaitCtl& c) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*c.abort) return false;
      if (global_ns() - t0 > c.limit_ns) {
        report(c.status, MOE_ERR_TIMEOUT);
        *c.abort = 1;
        return false;
      }
    }
  }
}

// Barriers of a CTA pair also receive arrivals / byte counts from the peer
// CTA and from 2-CTA commits, so pair kernels wait with cluster scope.
template <class C>
__device__ __forceinline__ bool wait_bar_p(uint64_t* bar, uint32_t parity, const WaitCtl& c) {
  if constexpr (C::PAIR == 2) return wait_bar_cluster(bar, parity, c);
  else return wait_bar(bar, parity, c);
}

// Wait whose only exit besides success is the time limit (teardown drains).
__device__ __forceinline__ bool wait_bar_drain(uint64_t* bar, uint32_t parity, uint64_t limit) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit) return false;
  return true;
}

template <class C>
__device__ __forceinline__ void tma_load(void* dst, const CUtensorMap* m, int x, int y,
                                         uint64_t* bar, uint32_t bar_cluster) {
  if constexpr (C::PAIR == 2)
    tma_load_2d_pair(dst, m, x, y, bar_cluster);
  else
    tma_load_2d(dst, m, x, y, bar);
}

// ----------------------------------------------------------------- roles
// Producer (one thread per CTA, or two: `part` 0 loads A and its scales and
// arms the full barrier, part 1 loads B and its scales; -1 loads all).  With
// PAIR == 2 both CTAs load their own A rows and their half of B into their
// own shared memory, and both signal the leader CTA's full barrier, which
// the leader arms with the pair's bytes.
template <class C>
__device__ void producer_role(const EngineParams& P, const int* cum, int total, const int* s_po,
                              const int* s_pt, int rank, uint8_t* stages, uint8_t* sfreg,
                              uint64_t* full, uint64_t* empty, const WaitCtl& wc, int part) {
  int it = 0;
  const int cl = blockIdx.x / C::PAIR, ncl = gridDim.x / C::PAIR;
  // ready[nmb] counts every published (m-block, n-tile) of the signalling
  // problem; once it reaches nmb * ready_target all dependencies hold and
  // later tiles skip their per-m-block checks.
  const int nmb = s_po[P.E] / 128;
  int32_t* const ready_all = P.ready + P.ready_all_index;
  bool all_ready = false;
  for (int t = cl; t < total; t += ncl) {
    const Tile ti = decode_tile<C>(P, cum, s_po, s_pt, t, rank);
    const GemmProblem& g = P.prob[ti.p];
    if (g.dep != DEP_NONE && !all_ready) {
      if ((int64_t)ld_acquire(ready_all) >= (int64_t)nmb * P.ready_target) {
        all_ready = true;
      } else if (g.dep == DEP_MBLOCK) {
        if (ti.valid && !wait_counter(P.ready + ti.mb, P.ready_target, wc)) break;
      } else {
        bool ok = true;
        for (int mb = s_po[ti.e] / 128; ok && mb < s_po[ti.e + 1] / 128; ++mb)
          ok = wait_counter(P.ready + mb, P.ready_target, wc);
        if (!ok) break;
      }
      fence_proxy_async_global();
    }
    // B column segments staged by this CTA: (first column or row, count)
    int seg0, seg1 = -1, seglen;
    if (ti.kind == GK_FWD1 && !C::MX) {
      seglen = C::BN / 2;
      if (C::PAIR == 1) {
        seg0 = ti.n0;
        seg1 = g.I + ti.n0;
      } else {
        seg0 = rank ? g.I + ti.n0 : ti.n0;
      }
    } else {
      // (block-scaled gate/up: W13's encoding interleaves 96 gate and 96 up
      // columns per tile, so its B rows are contiguous like the others')
      seglen = C::BNL;
      seg0 = ti.ntile * C::BN + rank * C::BNL;
    }
    bool ok = true;
    for (int kb = 0; kb < ti.nk; ++kb, ++it) {
      const int s = it % C::STAGES;
      const uint32_t par = ((it / C::STAGES) & 1) ^ 1;
      if (!wait_bar_p<C>(&empty[s], par, wc)) { ok = false; break; }
      uint8_t* sA = stages + s * C::STAGE_BYTES;
      uint8_t* sB = sA + C::A_BYTES;
      uint32_t fbar = 0;
      if constexpr (C::PAIR == 2) fbar = mapa_shared(smem_u32(&full[s]), 0);
      if (rank == 0 && part <= 0) mbar_arrive_expect_tx(&full[s], C::TX_BYTES);
      const int k0 = kb * C::BK;
      // A operand: M-major boxes (weight gradients) or one K-major box
      if (part == 1) {
      } else if (g.a_mn) {
#pragma unroll
        for (int j = 0; j < 128 / C::ATOM; ++j)
          tma_load<C>(sA + j * C::ATOM_BYTES, &g.tmA, ti.m0 + j * C::ATOM, ti.kbase + k0, &full[s],
                      fbar);
      } else {
        tma_load<C>(sA, &g.tmA, ti.kbase + k0, ti.m0, &full[s], fbar);
      }
      // B operand
      const int yrow = ti.kind == GK_DW ? 0 : ti.e * g.b_expert_rows;
      const int yb = ti.kind == GK_DW ? ti.kbase + k0 : ti.e * g.b_expert_rows + k0;
      if (part == 0) {
      } else if (!g.b_mn) {
        tma_load<C>(sB, &g.tmB, ti.kbase + k0, yrow + seg0, &full[s], fbar);
        if (seg1 >= 0)
          tma_load<C>(sB + seglen * 128, &g.tmB, ti.kbase + k0, yrow + seg1, &full[s], fbar);
      } else {
        const int na = seglen / C::ATOM;
        for (int j = 0; j < na; ++j)
          tma_load<C>(sB + j * C::ATOM_BYTES, &g.tmB, seg0 + j * C::ATOM, yb, &full[s], fbar);
        if (seg1 >= 0)
          for (int j = 0; j < na; ++j)
            tma_load<C>(sB + (na + j) * C::ATOM_BYTES, &g.tmB, seg1 + j * C::ATOM, yb, &full[s],
                        fbar);
      }
      if constexpr (C::MX) {
        // scale atoms: A's 128 rows x this K block (rows past the expert or
        // M read atom 0: their results are dropped), then B's.
        uint8_t* sSFA = sfreg + s * C::SF_BYTES;
        uint8_t* sSFB = sSFA + C::SFA_BYTES;
        const int amb = ti.valid ? (ti.m0 >> 7) : 0;
        if (part != 1)
          tma_load<C>(sSFA, &g.tmSFA, 0, (amb * g.sfa_kg + ((ti.kbase + k0) >> 7)) * 4, &full[s],
                      fbar);
        // B (K-major): the two atoms of the tile's 192 columns
        const int kidx = ti.kbase + k0;
        const int64_t mn0 = (ti.kind == GK_DW ? 0 : (int64_t)ti.e * g.sfb_seg) + (int64_t)ti.ntile * 256;
        if (part != 0)
#pragma unroll
          for (int j = 0; j < 2; ++j)
            tma_load<C>(sSFB + j * 512, &g.tmSFB, 0,
                        (int)((((mn0 >> 7) + j) * g.sfb_kg + (kidx >> 7)) * 4), &full[s], fbar);
      }
    }
    if (!ok) break;
  }
  // Drain: the latest use of every stage must have landed before exit (the
  // leader owns the full barriers, which also count the peer's bytes and
  // the other part's).
  if (rank == 0 && part <= 0) {
    const int n = it < C::STAGES ? it : C::STAGES;
    for (int q = 1; q <= n; ++q) {
      const int u = it - q;
      wait_bar_drain(&full[u % C::STAGES], (u / C::STAGES) & 1, wc.limit_ns);
    }
  }
}

// MMA issuer: one thread of the (leader) CTA.  Each tcgen05.mma costs the
// issuing thread a large share of the tensor time of a 192-column
// block-scaled MMA, so the loop between MMAs is kept short: operand
// descriptors are built once per tile and advanced by adding offsets, the
// stage ring is walked incrementally, and a stage costs one barrier wait.
// Data landed by TMA needs no tcgen05 fence; block-scaled stages wait only
// for the scale copier's signal, which the copier gives after it saw the
// stage's data land and after its scale copies into TMEM completed (one
// signal per SF_GROUP stages), and fence after it (TMEM written by another
// thread).
template <class C>
__device__ void mma_role(const EngineParams& P, const int* cum, int total, const int* s_po,
                         const int* s_pt, uint8_t* stages, uint64_t* full, uint64_t* empty,
                         uint64_t* tfull, uint64_t* tempty, uint64_t* drain, uint32_t tmem_base,
                         uint64_t* sfready, const WaitCtl& wc) {
  int it = 0, acc = 0;
  int s = 0;            // it % STAGES
  uint32_t ph = 0;      // (it / STAGES) & 1
  uint32_t soff = 0;    // s * STAGE_BYTES in descriptor units (16 bytes)
  const uint32_t sbase = smem_u32(stages);
  const int cl = blockIdx.x / C::PAIR, ncl = gridDim.x / C::PAIR;
  for (int t = cl; t < total; t += ncl) {
    const Tile ti = decode_tile<C>(P, cum, s_po, s_pt, t, 0);
    const int buf = acc % C::NACC;
    if (!wait_bar_p<C>(&tempty[buf], ((acc / C::NACC) & 1) ^ 1, wc)) break;
    tc_fence_after();
    const uint32_t d = tmem_base + buf * C::BN;
    if (ti.nk == 0) {                       // empty expert: nothing to accumulate
      if constexpr (C::PAIR == 2) tc_commit_pair(&tfull[buf], 3); else mbar_arrive(&tfull[buf]);
      ++acc;
      continue;
    }
    const GemmProblem& g = P.prob[ti.p];
    const uint32_t a_mn = g.a_mn ? 1u : 0u;
    const uint32_t b_mn = g.b_mn ? 1u : 0u;
    // instruction descriptor: D fp32 (dense kinds), operand formats, majors,
    // N >> 3, M >> 4; the MXFP8 kind instead carries E8M0 scales (bit 23)
    // and the scale byte of each MMA (bits 4-5 for B, 29-30 for A).
    const uint32_t idesc = (C::MX ? (1u << 23) : (1u << 4)) | (C::FMT << 7) | (C::FMT << 10) |
                           (a_mn << 15) | (b_mn << 16) | ((uint32_t)(C::BN >> 3) << 17) |
                           ((uint32_t)((128 * C::PAIR) >> 4) << 24);
    // stage-0 descriptors of this tile's operand layouts; a stage adds
    // STAGE_BYTES / 16 and an MMA's K step 32 bytes (K-major) or one
    // MN-major column block
    const uint64_t a0 = a_mn ? smem_desc_sw128(sbase, C::ATOM_BYTES, 1024)
                             : smem_desc_sw128(sbase, 16, 1024);
    const uint64_t b0 = b_mn ? smem_desc_sw128(sbase + C::A_BYTES, C::ATOM_BYTES, 1024)
                             : smem_desc_sw128(sbase + C::A_BYTES, 16, 1024);
    const uint32_t ak = a_mn ? C::MN_KSTEP_BYTES >> 4 : 2, bk = b_mn ? C::MN_KSTEP_BYTES >> 4 : 2;
    bool ok = true;
    for (int kb = 0; kb < ti.nk; ++kb) {
      if constexpr (C::MX) {
        if (it % C::SF_GROUP == 0) {
          const int q = it / C::SF_GROUP;
          if (!wait_bar_p<C>(&sfready[q % (C::STAGES / C::SF_GROUP)], ph, wc)) { ok = false; break; }
          tc_fence_after();
        }
      } else {
        if (!wait_bar_p<C>(&full[s], ph, wc)) { ok = false; break; }
      }
      const uint32_t sf_slot = tmem_base + C::SF_COL0 + s * 16;
#pragma unroll
      for (int kk = 0; kk < C::KSTEPS; ++kk) {
        const uint64_t ad = a0 + soff + kk * ak;
        const uint64_t bd = b0 + soff + kk * bk;
        const uint32_t accum = (kb | kk) != 0;
        if constexpr (C::MX && C::PAIR == 2)
          mma_mxf8_pair(d, ad, bd, idesc | ((uint32_t)kk << 4) | ((uint32_t)kk << 29), sf_slot,
                        sf_slot + 4, accum);
        else if constexpr (C::MX)
          mma_mxf8(d, ad, bd, idesc | ((uint32_t)kk << 4) | ((uint32_t)kk << 29), sf_slot,
                   sf_slot + 4, accum);
        else if constexpr (C::PAIR == 2)
          mma_f16_pair(d, ad, bd, idesc, accum);
        else if constexpr (C::ES == 2)
          mma_f16(d, ad, bd, idesc, accum);
        else
          mma_tf32(d, ad, bd, idesc, accum);
      }
      if constexpr (C::PAIR == 2) tc_commit_pair(&empty[s], 3); else tc_commit(&empty[s]);
      ++it;
      if (++s == C::STAGES) {
        s = 0;
        ph ^= 1;
        soff = 0;
      } else {
        soff += C::STAGE_BYTES >> 4;
      }
    }
    if (!ok) break;
    if constexpr (C::PAIR == 2) tc_commit_pair(&tfull[buf], 3); else tc_commit(&tfull[buf]);
    ++acc;
  }
  // Drain every MMA issued by this thread before TMEM is released.
  if constexpr (C::PAIR == 2) tc_commit_pair(drain, 1); else tc_commit(drain);
  wait_bar_drain(drain, 0, wc.limit_ns);
}

// Scale copier (block-scaled runs, one thread of the leader CTA): once a
// stage's operands and scale atoms have landed, copies the scales into that
// stage's TMEM slot (A at +0..3, B at +4..11), and after every SF_GROUP
// stages (and after its last one) signals sfready[group] once those copies
// have completed.  A slot is rewritten only after the stage was refilled,
// i.e. after the MMAs that read its previous scales finished.
template <class C>
__device__ void sf_role(const EngineParams& P, const int* cum, int total, const int* s_po,
                        const int* s_pt, uint8_t* sfreg, uint64_t* full, uint64_t* sfready,
                        uint64_t* drain, uint32_t tmem_base, const WaitCtl& wc) {
  int it = 0;
  const int cl = blockIdx.x / C::PAIR, ncl = gridDim.x / C::PAIR;
  bool ok = true;
  for (int t = cl; ok && t < total; t += ncl) {
    const Tile ti = decode_tile<C>(P, cum, s_po, s_pt, t, 0);
    for (int kb = 0; kb < ti.nk; ++kb, ++it) {
      const int s = it % C::STAGES;
      if (!wait_bar_p<C>(&full[s], (it / C::STAGES) & 1, wc)) { ok = false; break; }
      tc_fence_after();
      const uint32_t slot = tmem_base + C::SF_COL0 + s * 16;
      const uint32_t aS = smem_u32(sfreg) + s * C::SF_BYTES;
#pragma unroll
      for (int j = 0; j < 1 + C::SFB_BYTES / 512; ++j) {
        if constexpr (C::PAIR == 2)
          tmem_cp_32x128b_x4_pair(slot + 4 * j, smem_desc_rows16(aS + 512 * j));
        else
          tmem_cp_32x128b_x4(slot + 4 * j, smem_desc_rows16(aS + 512 * j));
      }
      if (it % C::SF_GROUP == C::SF_GROUP - 1) {
        uint64_t* bar = &sfready[(it / C::SF_GROUP) % (C::STAGES / C::SF_GROUP)];
        if constexpr (C::PAIR == 2) tc_commit_pair(bar, 1); else tc_commit(bar);
      }
    }
  }
  // a last, partial group is signalled too (the MMA issuer waits for it)
  if (ok && it % C::SF_GROUP != 0) {
    uint64_t* bar = &sfready[(it / C::SF_GROUP) % (C::STAGES / C::SF_GROUP)];
    if constexpr (C::PAIR == 2) tc_commit_pair(bar, 1); else tc_commit(bar);
  }
  // every copy completed before TMEM is released
  if constexpr (C::PAIR == 2) tc_commit_pair(drain, 1); else tc_commit(drain);
  wait_bar_drain(drain, 0, wc.limit_ns);
}

// ------------------------------------------------------- epilogue helpers
// MXFP8 encodings of a warp's 32 x 32 block of a result (lane = row, v = its
// 32 columns from col0), from the bf16 values the stored result would hold,
// so the codes equal those of the quantiser kernels on the stored tensor:
// row-wise (one 32-column block per lane) and, when qc is set, column-wise
// (one 32-row block per column: the warp's rows lie in one expert's group,
// whose padded start is a multiple of 128).  `tsm` is 4 KB of this warp's
// shared memory that no copy is reading: lane r writes its values to word
// 32 r + (i ^ r) and lane j reads column j (both without bank conflicts).
// col_ld == 0: column-wise codes at [row][col] (an A operand, M-major);
// col_ld > 0: stored transposed at [col][row] with row pitch col_ld and the
// scales in the 192-column tile slots (a K-major B operand), each lane
// encoding one column.
__device__ __forceinline__ void encode_mx_block(float (&v)[32], int64_t row, int col0, int C,
                                                uint8_t* qr, uint8_t* sr, uint8_t* qc,
                                                uint8_t* sc, int64_t kg_rows, float* tsm,
                                                int lane, int64_t col_ld = 0) {
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) am = fmaxf(am, fabsf(v[i]));
  const int sb = mx_scale_byte(am);
  const float inv = mx_inv_scale(sb);
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    o[i] = (uint32_t)e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv) |
           ((uint32_t)e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv) << 16);
  uint4* dr = reinterpret_cast<uint4*>(qr + (size_t)row * C + col0);
  dr[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dr[1] = make_uint4(o[4], o[5], o[6], o[7]);
  sr[mma_scale_index(row, col0 >> 5, C >> 7)] = (uint8_t)sb;
  if (!qc) return;
  if (col_ld > 0) {
#pragma unroll
    for (int i = 0; i < 32; ++i) tsm[lane * 32 + (i ^ lane)] = v[i];
    __syncwarp();
    float cv[32];                      // column col0 + lane, rows row0 .. row0 + 31
    float cm = 0.f;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      cv[r] = tsm[r * 32 + (lane ^ r)];
      cm = fmaxf(cm, fabsf(cv[r]));
    }
    __syncwarp();                      // reads done before the staging is reused
    const int64_t row0 = row - lane;
    const int sj = mx_scale_byte(cm);
    sc[mma_scale_index(mx_tile_pos(col0 + lane), (int)(row0 >> 5), kg_rows)] = (uint8_t)sj;
    const float invj = mx_inv_scale(sj);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      o[i] = (uint32_t)e4m3x2(cv[4 * i] * invj, cv[4 * i + 1] * invj) |
             ((uint32_t)e4m3x2(cv[4 * i + 2] * invj, cv[4 * i + 3] * invj) << 16);
    uint4* dc = reinterpret_cast<uint4*>(qc + (size_t)(col0 + lane) * col_ld + row0);
    dc[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dc[1] = make_uint4(o[4], o[5], o[6], o[7]);
    return;
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) tsm[lane * 32 + (i ^ lane)] = fabsf(v[i]);
  __syncwarp();
  float cm = 0.f;                      // maximum of column `lane`
#pragma unroll
  for (int r = 0; r < 32; ++r) cm = fmaxf(cm, tsm[r * 32 + (lane ^ r)]);
  __syncwarp();                        // reads done before the staging is reused
  const int sj = mx_scale_byte(cm);
  sc[mma_scale_index(col0 + lane, (int)(row >> 5), kg_rows)] = (uint8_t)sj;
  const float invj = mx_inv_scale(sj);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float i0 = __shfl_sync(0xffffffffu, invj, i), i1 = __shfl_sync(0xffffffffu, invj, i + 1);
    const uint32_t c2 = e4m3x2(v[i] * i0, v[i + 1] * i1);
    if (i & 2) o[i >> 2] |= c2 << 16; else o[i >> 2] = c2;
  }
  uint4* dc = reinterpret_cast<uint4*>(qc + (size_t)row * C + col0);
  dc[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dc[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

template <typename Elt>
__device__ __forceinline__ void store32(Elt* dst, const float (&v)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
  if constexpr (sizeof(Elt) == 2) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      d[q] = make_uint4(pack_bf16(v[8 * q + 0], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                        pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      d[q] = make_uint4(__float_as_uint(v[4 * q + 0]), __float_as_uint(v[4 * q + 1]),
                        __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3]));
  }
}

template <typename Elt>
__device__ __forceinline__ void load32(const Elt* src, float (&v)[32]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  if constexpr (sizeof(Elt) == 2) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = s[q];
      v[8 * q + 0] = bf16_lo(w.x); v[8 * q + 1] = bf16_hi(w.x);
      v[8 * q + 2] = bf16_lo(w.y); v[8 * q + 3] = bf16_hi(w.y);
      v[8 * q + 4] = bf16_lo(w.z); v[8 * q + 5] = bf16_hi(w.z);
      v[8 * q + 6] = bf16_lo(w.w); v[8 * q + 7] = bf16_hi(w.w);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint4 w = s[q];
      v[4 * q + 0] = __uint_as_float(w.x); v[4 * q + 1] = __uint_as_float(w.y);
      v[4 * q + 2] = __uint_as_float(w.z); v[4 * q + 3] = __uint_as_float(w.w);
    }
  }
}

// SiLU pieces for the epilogues, with the fast reciprocal (2 ulp): the
// results are rounded to bf16 right after, so fp32 division rounding is
// irrelevant.  For u below about -88, exp(-u) is +inf and both give 0.
__device__ __forceinline__ float sigmoid_f(float u) { return __fdividef(1.f, 1.f + __expf(-u)); }
__device__ __forceinline__ float silu_f(float u) { return __fdividef(u, 1.f + __expf(-u)); }

// Named barrier of one epilogue group (ids 1, 2, ...).
template <int NTHREADS>
__device__ __forceinline__ void epi_bar(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "n"(NTHREADS) : "memory");
}

// Staging of bf16 results (per epilogue warp: two 2 KB buffers of 32 rows x
// 64 bytes, 64-byte swizzle: 16-byte chunk c of row r sits at chunk
// c ^ ((r >> 1) & 3)), drained by TMA tensor stores.
__device__ __forceinline__ void stage_bf16_row(uint8_t* buf, int r, const float (&v)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(buf + r * 64 + ((c ^ ((r >> 1) & 3)) << 4)) =
        make_uint4(pack_bf16(v[8 * c + 0], v[8 * c + 1]), pack_bf16(v[8 * c + 2], v[8 * c + 3]),
                   pack_bf16(v[8 * c + 4], v[8 * c + 5]), pack_bf16(v[8 * c + 6], v[8 * c + 7]));
}

template <typename Elt, int NV>
__device__ __forceinline__ void load_raw(const Elt* src, uint4 (&d)[NV]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < NV; ++i) d[i] = s[i];
}

template <typename Elt, int NV>
__device__ __forceinline__ void unpack_raw(const uint4 (&d)[NV], float (&v)[32]) {
  if constexpr (sizeof(Elt) == 2) {
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      v[8 * q + 0] = bf16_lo(d[q].x); v[8 * q + 1] = bf16_hi(d[q].x);
      v[8 * q + 2] = bf16_lo(d[q].y); v[8 * q + 3] = bf16_hi(d[q].y);
      v[8 * q + 4] = bf16_lo(d[q].z); v[8 * q + 5] = bf16_hi(d[q].z);
      v[8 * q + 6] = bf16_lo(d[q].w); v[8 * q + 7] = bf16_hi(d[q].w);
    }
  } else {
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      v[4 * q + 0] = __uint_as_float(d[q].x); v[4 * q + 1] = __uint_as_float(d[q].y);
      v[4 * q + 2] = __uint_as_float(d[q].z); v[4 * q + 3] = __uint_as_float(d[q].w);
    }
  }
}

template <class C, typename Elt>
__device__ void epilogue_role(const EngineParams& P, const int* cum, int total, const int* s_po,
                              const int* s_pt, int rank, uint64_t* tfull, uint64_t* tempty,
                              uint32_t tmem_base, volatile int* s_go, uint8_t* stg,
                              const WaitCtl& wc) {
  constexpr bool TS = sizeof(Elt) == 2;      // bf16 results leave through TMA stores
  constexpr int NV = 32 * (int)sizeof(Elt) / 16;   // 16-byte vectors per 32 elements
  constexpr int ET = C::EPI_WARPS * 32;      // threads of an epilogue group
  constexpr int NG = C::EPI_GROUPS;
  static_assert(NG == 1 || NG == C::NACC, "one accumulator per epilogue group");
  const int ew = (threadIdx.x >> 5) - C::EPI_FIRST;   // epilogue warp
  const int grp = ew / C::EPI_WARPS;         // its group: tiles acc with acc % NG == grp
  const int q = (threadIdx.x >> 5) & 3;      // TMEM lane quarter of this warp
  const int lane = threadIdx.x & 31;
  const int r = q * 32 + lane;               // tile row of this thread
  const bool leader = threadIdx.x == 32 * C::EPI_FIRST + grp * ET;   // first thread of the group
  const int cl = blockIdx.x / C::PAIR, ncl = gridDim.x / C::PAIR;
  uint8_t* sb0 = stg + ew * 4096;
  uint8_t* sb1 = sb0 + 2048;
  // write-once results (h13, A, Z, dXp, weight gradients) leave L2 first;
  // dh13, re-read by the dX / dW13 tiles of the same launch, does not
  const uint64_t pol_ef = l2_evict_first_policy();
  // the accumulator is released on the MMA-issuing CTA's barrier
  const uint32_t tempty_cl0 = C::PAIR == 2 ? mapa_shared(smem_u32(&tempty[0]), 0) : 0;
  const uint32_t tempty_cl1 = C::PAIR == 2 ? mapa_shared(smem_u32(&tempty[1]), 0) : 0;
  // staging buffers free again (previous bulk stores have read them)
  auto stage_begin = [&]() {
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
  };
  // this warp's staged rows are visible to the bulk-copy engine
  auto stage_end = [&]() {
    fence_proxy_async_smem();
    __syncwarp();
  };
  int acc = grp;   // this CTA's tile sequence index
  for (int t = cl + grp * ncl; t < total; t += NG * ncl, acc += NG) {
    const Tile ti = decode_tile<C>(P, cum, s_po, s_pt, t, rank);
    const int gs = grp * 2 + ((acc / NG) & 1);   // this group's decision slot
    const GemmProblem& g = P.prob[ti.p];
    const int buf = acc % C::NACC;
    const int yrow = ti.m0 + q * 32;         // first row of this warp's slice
    // accumulator columns [cb, cb + cw) of this warp (FWD1: of each half)
    const int cw = ti.kind == GK_FWD1 ? C::BN / 2 : C::BN;
    const int cb = 0;
    // dSwiGLU inputs: the first chunk of h13 is fetched before the wait
    uint4 pu[NV], pv[NV];
    const Elt* h13a = nullptr;
    if (ti.kind == GK_BWD_D && ti.valid) {
      h13a = static_cast<const Elt*>(g.aux) + (size_t)(ti.m0 + r) * g.ld_aux + ti.n0;
      // the row's u and v columns of this tile reach L2 while its MMAs run
      const int ncol = min(cw, g.I - (ti.n0 + cb));
      const uint32_t pbytes = ncol > 0 ? ((uint32_t)ncol * (uint32_t)sizeof(Elt)) & ~15u : 0u;
      if (pbytes) {
        if ((reinterpret_cast<uintptr_t>(h13a + cb) & 15) == 0) prefetch_l2_bulk(h13a + cb, pbytes);
        if ((reinterpret_cast<uintptr_t>(h13a + g.I + cb) & 15) == 0)
          prefetch_l2_bulk(h13a + g.I + cb, pbytes);
      }
      load_raw<Elt, NV>(h13a + cb, pu);
      load_raw<Elt, NV>(h13a + g.I + cb, pv);
    }
    // One thread waits; the decision is shared so all epilogue threads take
    // the same path through the named barriers below.  (s_go is indexed by
    // the group's tile parity so a slow reader never sees the next decision.)
    if (leader) s_go[gs] = wait_bar_p<C>(&tfull[buf], (acc / C::NACC) & 1, wc) ? 1 : 0;
    epi_bar<ET>(grp);
    if (!s_go[gs]) break;
    tc_fence_after();
    __syncwarp();
    const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + buf * C::BN;
    float v[32], w[32], x[64];
    // 64 results of this thread's row: bf16 through both staging buffers and
    // two bulk stores (3-D [E, M, N] view when z >= 0), fp32 directly
    auto emit64 = [&](const float (&y)[64], Elt* dst, int xc, int yc, int z, bool ok) {
      if constexpr (TS) {
        stage_begin();
        stage_bf16_row(sb0, lane, *reinterpret_cast<const float(*)[32]>(&y[0]));
        stage_bf16_row(sb1, lane, *reinterpret_cast<const float(*)[32]>(&y[32]));
        stage_end();
        if (lane == 0) {
          if (z >= 0) {
            tma_store_3d_ef(&g.tmO, sb0, xc, yc, z, pol_ef);
            tma_store_3d_ef(&g.tmO, sb1, xc + 32, yc, z, pol_ef);
          } else {
            tma_store_2d_ef(&g.tmO, sb0, xc, yc, pol_ef);
            tma_store_2d_ef(&g.tmO, sb1, xc + 32, yc, pol_ef);
          }
          bulk_commit();
        }
      } else if (ok) {
        store32<Elt>(dst, *reinterpret_cast<const float(*)[32]>(&y[0]));
        store32<Elt>(dst + 32, *reinterpret_cast<const float(*)[32]>(&y[32]));
      }
    };
    // gate of a tile row: 1 without a gate vector, 0 on pad rows
    auto row_gate = [&](const GemmProblem& gp, int row) -> float {
      if (!gp.gate) return 1.f;
      int a = gp.assign_of_row[row];
      if (a >= gp.n_assign) {           // corrupted map: treat as a pad row
        report(P.status, MOE_ERR_BAD_INDEX);
        a = -1;
      }
      return a >= 0 ? gp.gate[a] : 0.f;
    };
    if (!ti.valid) {
      // rows past the tile's expert (odd m-block count) or past M: no output
    } else if (ti.kind == GK_FWD1) {
      const int row = ti.m0 + r;
      Elt* outA = static_cast<Elt*>(g.out) + (size_t)row * g.ld_out + ti.n0;
      Elt* h13 = g.out2 ? static_cast<Elt*>(g.out2) + (size_t)row * g.ld_out2 + ti.n0 : nullptr;
      // with a gate vector the activation leaves as gate * A (0 on pad rows)
      const float ga = row_gate(g, row);
      const bool zrow = ga == 0.f;
#pragma unroll 1
      for (int c = cb; c < cb + cw; c += 32) {
        tmem_ld32x2(taddr + c, taddr + C::BN / 2 + c, v, w);   // u: gate half, v: up half
        if (h13) {
          if constexpr (TS) {
            stage_begin();
            stage_bf16_row(sb0, lane, v);
            stage_bf16_row(sb1, lane, w);
            stage_end();
            if (lane == 0) {
              tma_store_2d_ef(&g.tmO2, sb0, ti.n0 + c, yrow, pol_ef);
              tma_store_2d_ef(&g.tmO2, sb1, g.I + ti.n0 + c, yrow, pol_ef);
              bulk_commit();
            }
          } else {
            store32<Elt>(h13 + c, v);
            store32<Elt>(h13 + g.I + c, w);
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = zrow ? 0.f : silu_f(v[i]) * w[i] * ga;
        if (C::MX && g.enc_row_q) {
          if (g.enc_col_q) stage_begin();   // the staging becomes the column-maximum scratch
          encode_mx_block(v, row, ti.n0 + c, g.I, g.enc_row_q, g.enc_row_sf, g.enc_col_q,
                          g.enc_col_sf, g.enc_col_kg, reinterpret_cast<float*>(sb0), lane);
        } else if constexpr (TS) {
          stage_begin();
          stage_bf16_row(sb0, lane, v);
          stage_end();
          if (lane == 0) {
            tma_store_2d_ef(&g.tmO, sb0, ti.n0 + c, yrow, pol_ef);
            bulk_commit();
          }
        } else {
          store32<Elt>(outA + c, v);
        }
      }
    } else if (ti.kind == GK_FWD2) {
      const int row = ti.m0 + r;
      const float gt = row_gate(g, row);
      Elt* out = static_cast<Elt*>(g.out) + (size_t)row * g.ld_out + ti.n0;
#pragma unroll 1
      for (int c = cb; c < cb + cw && ti.n0 + c < g.N; c += 64) {   // a last tile may be ragged
        tmem_ld64(taddr + c, x);
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] *= gt;
        emit64(x, out + c, ti.n0 + c, yrow, -1, true);
      }
    } else if (ti.kind == GK_BWD_D) {
      const int row = ti.m0 + r;
      int a = g.assign_of_row[row];
      if (a >= g.n_assign) {          // corrupted map: treat as a pad row
        report(P.status, MOE_ERR_BAD_INDEX);
        a = -1;
      }
      const float gt = a >= 0 ? g.gate[a] : 0.f;
      Elt* dh = static_cast<Elt*>(g.out) + (size_t)row * g.ld_out + ti.n0;
      float part = 0.f;
      uint32_t src = taddr + cb;               // TMEM columns of the next chunk
#pragma unroll 1
      for (int c = cb; c < cb + cw; c += 32, src += 32) {
        float D[32];
        unpack_raw<Elt, NV>(pu, v);            // u of this chunk
        unpack_raw<Elt, NV>(pv, w);            // v of this chunk
        if (c + 32 < cb + cw) {                // fetch the next chunk while this one runs
          load_raw<Elt, NV>(h13a + c + 32, pu);
          load_raw<Elt, NV>(h13a + g.I + c + 32, pv);
        }
        tmem_ld32(src, D);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float u = v[i], vv = w[i];
          const float sg = sigmoid_f(u);
          const float si = u * sg;
          part += si * vv * D[i];
          const float dA = gt * D[i];
          v[i] = a >= 0 ? dA * vv * sg * (1.f + u * (1.f - sg)) : 0.f;   // du
          w[i] = a >= 0 ? dA * si : 0.f;                                  // dv
        }
        if (C::MX && g.enc_row_q) {
          // block-scaled runs: dh13 leaves as its two MXFP8 encodings,
          // decided from the bf16 values a stored dh13 would hold: row-wise
          // (the dX GEMM's A) and column-wise along tokens, stored
          // transposed (the dW13 GEMM's K-major B)
          stage_begin();   // the staging becomes the encoder's scratch
          encode_mx_block(v, row, ti.n0 + c, 2 * g.I, g.enc_row_q, g.enc_row_sf, g.enc_col_q,
                          g.enc_col_sf, g.enc_col_kg, reinterpret_cast<float*>(sb0), lane,
                          g.enc_col_ld);
          encode_mx_block(w, row, g.I + ti.n0 + c, 2 * g.I, g.enc_row_q, g.enc_row_sf,
                          g.enc_col_q, g.enc_col_sf, g.enc_col_kg, reinterpret_cast<float*>(sb0),
                          lane, g.enc_col_ld);
        } else if constexpr (TS) {
          stage_begin();
          stage_bf16_row(sb0, lane, v);
          stage_bf16_row(sb1, lane, w);
          stage_end();
          if (lane == 0) {
            tma_store_2d(&g.tmO, sb0, ti.n0 + c, yrow);
            tma_store_2d(&g.tmO, sb1, g.I + ti.n0 + c, yrow);
            bulk_commit();
          }
        } else {
          store32<Elt>(dh + c, v);
          store32<Elt>(dh + g.I + c, w);
        }
      }
      g.partial[(size_t)row * g.nt + ti.ntile] = a >= 0 ? part : 0.f;
    } else if (ti.kind == GK_BWD_DX) {
      const int row = ti.m0 + r;
      Elt* out = static_cast<Elt*>(g.out) + (size_t)row * g.ld_out + ti.n0;
#pragma unroll 1
      for (int c = cb; c < cb + cw && ti.n0 + c < g.N; c += 64) {
        tmem_ld64(taddr + c, x);
        emit64(x, out + c, ti.n0 + c, yrow, -1, true);
      }
    } else {  // GK_DW
      const bool valid = ti.m0 + r < g.M;
      Elt* out = static_cast<Elt*>(g.out) + ((size_t)ti.e * g.M + ti.m0 + r) * g.ld_out + ti.n0;
#pragma unroll 1
      for (int c = cb; c < cb + cw && ti.n0 + c < g.N; c += 64) {
        if (ti.nk > 0) {
          tmem_ld64(taddr + c, x);
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) x[i] = 0.f;
        }
        // rows past M are outside the [E, M, N] view: the bulk store clips them
        emit64(x, out + c, ti.n0 + c, ti.m0 + q * 32, ti.e, valid);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if constexpr (C::PAIR == 2) mbar_arrive_cluster(buf ? tempty_cl1 : tempty_cl0);
      else mbar_arrive(&tempty[buf]);
    }
    if (g.signal && ti.valid) {
      // Publish this tile's rows to TMA readers in other CTAs: the bulk
      // stores complete, then a release on the m-block's counter.
      if (TS && lane == 0) bulk_wait_all();
      __syncwarp();
      fence_proxy_async_global();
      __threadfence();
      epi_bar<ET>(grp);
      if (leader) {
        red_release_add(P.ready + ti.mb, 1);
        red_release_add(P.ready + P.ready_all_index, 1);
      }
    }
  }
  if (TS && lane == 0) bulk_wait_all();    // every store done before the CTA exits
  __syncwarp();
}

// ----------------------------------------------------------------- kernel
template <typename In, typename Out, int BN, int PAIR>
__global__ void __launch_bounds__(Cfg<In, BN, PAIR>::THREADS, 1)
    moe_gemm_kernel(const __grid_constant__ EngineParams P) {
  using C = Cfg<In, BN, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* stages = smem;
  uint8_t* stg = smem + C::STAGES * C::STAGE_BYTES;   // 1024-aligned (stage sizes are)
  uint8_t* sfreg = stg + C::STG_BYTES;                 // MXFP8 scale atoms per stage
  uint64_t* bars = reinterpret_cast<uint64_t*>(sfreg + C::SF_REGION);
  uint64_t* full = bars;
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* sfready = drain + 1;        // [STAGES] (block-scaled runs)
  uint64_t* drain2 = sfready + C::STAGES;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain2 + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
  int* s_go = abort_flag + 1;           // [2 per epilogue group]
  int* s_po = reinterpret_cast<int*>(sfreg + C::SF_REGION + 512);   // after the barriers
  int* s_pt = s_po + (kMaxE + 1);       // pair tiles before expert e (PAIR == 2)
  int* s_cnt = s_pt + (kMaxE + 1);      // rows of each expert (weight-gradient K)

  const int warp = threadIdx.x >> 5;
  const int rank = PAIR == 2 ? (int)cluster_ctarank() : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], C::EPI_WARPS * PAIR);  // one arrival per warp of the group, both CTAs
    }
    mbar_init(drain, 1);
    for (int st = 0; st < C::STAGES; ++st) mbar_init(&sfready[st], 1);
    mbar_init(drain2, 1);
    *abort_flag = 0;
    for (int i = 0; i < 2 * C::EPI_GROUPS; ++i) s_go[i] = 0;
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i <= P.E; i += blockDim.x) s_po[i] = P.padded_offsets[i];
  for (int i = threadIdx.x; i < P.E; i += blockDim.x) s_cnt[i] = P.counts ? P.counts[i] : -1;
  if (warp == 1) {
    if constexpr (PAIR == 2) tmem_alloc_pair(tmem_holder, C::TMEM_COLS);
    else tmem_alloc(tmem_holder, C::TMEM_COLS);
  }
  if (threadIdx.x == 0) {
    for (int p = 0; p < P.nprob; ++p) {
      tma_prefetch_desc(&P.prob[p].tmA);
      tma_prefetch_desc(&P.prob[p].tmB);
      if constexpr (C::MX) {
        tma_prefetch_desc(&P.prob[p].tmSFA);
        tma_prefetch_desc(&P.prob[p].tmSFB);
      }
    }
  }
  __syncthreads();
  if constexpr (PAIR == 2) {
    // exclusive scan of ceil(m-blocks / 2) over experts (warp 2)
    if (warp == 2) {
      const int lane = threadIdx.x & 31;
      int carry = 0;
      for (int c0 = 0; c0 < P.E; c0 += 32) {
        const int e = c0 + lane;
        const int v = e < P.E ? ((s_po[e + 1] - s_po[e]) / 128 + 1) / 2 : 0;
        int x = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, off);
          if (lane >= off) x += y;
        }
        if (e < P.E) s_pt[e] = carry + x - v;
        carry += __shfl_sync(0xffffffffu, x, 31);
      }
      if (lane == 0) s_pt[P.E] = carry;
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR == 2) cluster_sync_all();   // peers' barriers exist before use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  // Tile counts per problem (derived from device offsets, no host copy).
  int cum[5];
  cum[0] = 0;
  const int tpad = s_po[P.E];
  for (int p = 0; p < 4; ++p) {
    int n = 0;
    if (p < P.nprob) {
      const GemmProblem& g = P.prob[p];
      if (g.kind == GK_DW)
        n = P.E * (((g.M + 127) / 128 + PAIR - 1) / PAIR) * g.nt;
      else
        n = (PAIR == 2 ? s_pt[P.E] : tpad / 128) * g.nt;
    }
    cum[p + 1] = cum[p] + n;
  }
  const int total = cum[P.nprob];
  const WaitCtl wc{abort_flag, P.status, P.wait_ns};

  if constexpr (C::REG_SPLIT) {
    static_assert(C::THREADS == 384 && C::EPI_WARPS * C::EPI_GROUPS == 8, "three warpgroups");
    static_assert(128 * C::ROLE_REGS + 256 * C::EPI_REGS <= 384 * 168, "register split");
    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::ROLE_REGS));
      if ((threadIdx.x & 31) == 0) {
        if (warp == 0)
          producer_role<C>(P, cum, total, s_po, s_pt, rank, stages, sfreg, full, empty, wc, 0);
        else if (warp == 1 && rank == 0)
          mma_role<C>(P, cum, total, s_po, s_pt, stages, full, empty, tfull, tempty, drain,
                      tmem_base, sfready, wc);
        else if (warp == 2)
          producer_role<C>(P, cum, total, s_po, s_pt, rank, stages, sfreg, full, empty, wc, 1);
        else if (warp == 3 && rank == 0)
          sf_role<C>(P, cum, total, s_po, s_pt, sfreg, full, sfready, drain2, tmem_base, wc);
      }
      __syncwarp();
    } else {
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::EPI_REGS));
      epilogue_role<C, Out>(P, cum, total, s_po, s_pt, rank, tfull, tempty, tmem_base, s_go, stg, wc);
    }
  } else {
    constexpr int EPI_END = 2 + C::EPI_WARPS * C::EPI_GROUPS;   // first warp after the epilogue
    if (warp == 0) {
      if ((threadIdx.x & 31) == 0)
        producer_role<C>(P, cum, total, s_po, s_pt, rank, stages, sfreg, full, empty, wc,
                         C::SPLIT_LOAD ? 0 : -1);
      __syncwarp();
    } else if (warp == 1) {
      if ((threadIdx.x & 31) == 0 && rank == 0)
        mma_role<C>(P, cum, total, s_po, s_pt, stages, full, empty, tfull, tempty, drain,
                    tmem_base, sfready, wc);
      __syncwarp();
    } else if (warp < EPI_END) {
      epilogue_role<C, Out>(P, cum, total, s_po, s_pt, rank, tfull, tempty, tmem_base, s_go, stg, wc);
    } else if (C::SPLIT_LOAD && warp == EPI_END) {
      if ((threadIdx.x & 31) == 0)
        producer_role<C>(P, cum, total, s_po, s_pt, rank, stages, sfreg, full, empty, wc, 1);
      __syncwarp();
    } else if constexpr (C::SPLIT_ISSUE) {
      if ((threadIdx.x & 31) == 0 && rank == 0)
        sf_role<C>(P, cum, total, s_po, s_pt, sfreg, full, sfready, drain2, tmem_base, wc);
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR == 2) {
    // After an abort, copies issued by either CTA of the pair may still be
    // in flight towards the other; give them time to land before the pair
    // leaves (they complete in microseconds).
    if (threadIdx.x == 0 && *abort_flag) {
      const uint64_t t0 = global_ns();
      while (global_ns() - t0 < 200000) __nanosleep(1000);
    }
    __syncthreads();
    cluster_sync_all();
  }
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR == 2) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------- host
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major [rows, cols] tensor, 128-byte swizzled boxes of
// box_cols x box_rows elements.
bool make_tmap(CUtensorMap* m, const void* base, int elem_bytes, int64_t rows, int64_t cols,
               int box_cols, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  const CUtensorMapDataType dt =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                      : (elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT8);
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * elem_bytes};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 output views for the epilogue's bulk stores: 32 x 32 boxes, 64-byte
// swizzle (matching the staging layout).  2-D [rows, cols] or 3-D [E, M, N].
bool make_tmap_out(CUtensorMap* m, void* base, int64_t rows, int64_t cols) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MXFP8 scale atoms as a [bytes / 128, 128] uint8 tensor, boxes of one
// 512-byte atom (4 x 128), no swizzle.
bool make_tmap_sf(CUtensorMap* m, const void* base, int64_t bytes) {
  auto enc = encode_fn();
  if (!enc || bytes <= 0 || bytes % 512) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)(bytes / 128)};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, 4};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_out3(CUtensorMap* m, void* base, int64_t E, int64_t M, int64_t N) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)E};
  cuuint64_t strides[2] = {(cuuint64_t)N * 2, (cuuint64_t)(M * N * 2)};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
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

// `gang`: tiles of this launch wait on tiles of other CTAs, so it is made a
// cooperative launch: the GPU starts it only once every CTA of the grid can
// be resident, instead of starting the CTAs that fit while other work (a
// kernel on another stream) holds the rest of the SMs, whose tiles the
// started ones would then wait for.
template <typename In, typename Out, int BN, int PAIR>
cudaError_t launch_typed(const EngineParams& P, int64_t tile_bound, bool gang, cudaStream_t s) {
  using C = Cfg<In, BN, PAIR>;
  auto kern = moe_gemm_kernel<In, Out, BN, PAIR>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (PAIR == 2) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = PAIR;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  // Per context: the shared-memory opt-in, and for pairs the number of
  // clusters resident at once (tiles wait on other tiles, so the grid never
  // exceeds it).
  static CtxCache<int> resident;
  int max_units = 0;
  cudaError_t e = resident.get(&max_units, [&](int* v) {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (r != cudaSuccess) return r;
    if constexpr (PAIR == 1) {
      *v = sm_count();
      return cudaSuccess;
    } else {
      cudaLaunchConfig_t q = cfg;
      q.gridDim = dim3(2 * (sm_count() / 2), 1, 1);
      int n = 0;
      r = cudaOccupancyMaxActiveClusters(&n, kern, &q);
      if (r == cudaSuccess && n < 1) r = cudaErrorInvalidConfiguration;
      *v = n;
      return r;
    }
  });
  if (e != cudaSuccess) return e;
  int64_t units = max_units;
  if (tile_bound < units) units = tile_bound < 1 ? 1 : tile_bound;
  cfg.gridDim = dim3((unsigned)(PAIR * units), 1, 1);
  if (gang) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    cfg.numAttrs = ++na;
  }
  return cudaLaunchKernelEx(&cfg, kern, P);
}

}  // namespace

cudaError_t launch_engine(const EngineLaunch& L, cudaStream_t s, moe_status* st) {
  *st = MOE_OK;
  EngineParams P;
  memset(&P, 0, sizeof(P));
  P.nprob = L.nprob;
  P.E = L.E;
  P.padded_offsets = L.padded_offsets;
  P.counts = L.counts;
  P.ready = L.ready;
  P.ready_target = L.ready_target;
  P.ready_all_index = (int)((L.max_rows + 127) / 128);
  P.status = L.status;
  P.wait_ns = L.wait_ns;
  const int es = L.elem_bytes;
  const int BK = 128 / es, ATOM = 128 / es;
  // bf16 and MXFP8 run 256-row tiles over an SM pair (B split in halves of
  // >= 64 columns); TF32 and narrow tiles run on single CTAs.
  const int pair = (es == 2 || es == 1) && L.BN >= 128 && !(debug_flags() & MOE_DEBUG_SINGLE_CTA)
                       ? 2 : 1;
  int64_t tile_bound = 0;
  bool gang = false;
  const int64_t mblocks_max = (L.max_rows + 127) / 128;
  for (int p = 0; p < L.nprob; ++p) {
    const GemmDesc& d = L.prob[p];
    GemmProblem& g = P.prob[p];
    g.kind = d.kind;
    g.a_mn = d.a_mn;
    g.b_mn = d.b_mn;
    g.dep = d.dep;
    g.signal = d.signal;
    gang = gang || d.dep != DEP_NONE;
    g.M = d.M;
    g.N = d.N;
    g.K = d.K;
    g.b_expert_rows = d.b_expert_rows;
    g.I = d.I;
    g.ld_out = d.ld_out;
    g.ld_out2 = d.ld_out2;
    g.ld_aux = d.ld_aux;
    g.out = d.out;
    g.out2 = d.out2;
    g.aux = d.aux;
    g.gate = d.gate;
    g.assign_of_row = d.assign_of_row;
    g.n_assign = d.n_assign;
    g.partial = d.partial;
    g.sfa_kg = d.sfa_kg;
    g.sfb_kg = d.sfb_kg;
    g.enc_row_q = d.enc_row_q;
    g.enc_row_sf = d.enc_row_sf;
    g.enc_col_q = d.enc_col_q;
    g.enc_col_sf = d.enc_col_sf;
    g.enc_col_kg = d.enc_col_kg;
    g.enc_col_ld = d.enc_col_ld;
    g.sfb_seg = d.sfb_seg;
    if (es == 1 && !(make_tmap_sf(&g.tmSFA, d.sfa, d.sfa_bytes) &&
                     make_tmap_sf(&g.tmSFB, d.sfb, d.sfb_bytes))) {
      *st = MOE_ERR_INVALID_ARG;
      return cudaSuccess;
    }
    const bool a_mn = d.a_mn != 0;
    const bool b_mn = d.b_mn != 0;
    if ((a_mn || b_mn) && es == 4) { *st = MOE_ERR_UNSUPPORTED; return cudaSuccess; }  // TF32: K-major only
    if (a_mn && d.kind != GK_DW) { *st = MOE_ERR_UNSUPPORTED; return cudaSuccess; }
    if (b_mn && es == 1) { *st = MOE_ERR_UNSUPPORTED; return cudaSuccess; }  // 192-wide tiles: K-major B
    const int n_per_tile = d.kind == GK_FWD1 ? L.BN / 2 : L.BN;
    const int n_total = d.kind == GK_FWD1 ? d.N / 2 : d.N;
    // the gate/up and D epilogues need whole tiles; the others store through
    // views that clip a ragged last tile
    const bool whole = d.kind == GK_FWD1 || d.kind == GK_BWD_D;
    if (n_total % n_per_tile != 0 && (whole || es != 1)) { *st = MOE_ERR_UNSUPPORTED; return cudaSuccess; }
    g.nt = (n_total + n_per_tile - 1) / n_per_tile;
    bool ok = a_mn ? make_tmap(&g.tmA, d.a, es, d.a_rows, d.a_cols, ATOM, BK)
                   : make_tmap(&g.tmA, d.a, es, d.a_rows, d.a_cols, BK, 128);
    ok = ok && (b_mn ? make_tmap(&g.tmB, d.b, es, d.b_rows, d.b_cols, ATOM, BK)
                     : make_tmap(&g.tmB, d.b, es, d.b_rows, d.b_cols, BK,
                                 d.kind == GK_FWD1 && es != 1 ? L.BN / 2 : L.BN / pair));
    if (es != 4) {   // bf16 results: bulk-store views of the outputs
      // every bf16 result leaves through a view built here; the results
      // that may be absent are FWD1's A and BWD_D's dh13 when the epilogue
      // encodes them instead
      if (!d.out && !((d.kind == GK_FWD1 || d.kind == GK_BWD_D) && d.enc_row_q)) {
        *st = MOE_ERR_INVALID_ARG;
        return cudaSuccess;
      }
      if (d.kind == GK_DW) {
        if (d.ld_out != d.N) { *st = MOE_ERR_UNSUPPORTED; return cudaSuccess; }
        ok = make_tmap_out3(&g.tmO, d.out, L.E, d.M, d.N);
      } else {
        if (d.out) ok = make_tmap_out(&g.tmO, d.out, L.max_rows, d.ld_out);
        if (ok && d.out2) ok = make_tmap_out(&g.tmO2, d.out2, L.max_rows, d.ld_out2);
      }
    }
    if (!ok) { *st = MOE_ERR_CUDA; return cudaSuccess; }
    tile_bound += d.kind == GK_DW ? (int64_t)L.E * ((d.M + 127) / 128) * g.nt : mblocks_max * g.nt;
  }
  if (es == 2 && pair == 2) {
    switch (L.BN) {
      case 256: return launch_typed<__nv_bfloat16, __nv_bfloat16, 256, 2>(P, tile_bound, gang, s);
      case 128: return launch_typed<__nv_bfloat16, __nv_bfloat16, 128, 2>(P, tile_bound, gang, s);
    }
  } else if (es == 2) {
    switch (L.BN) {
      case 256: return launch_typed<__nv_bfloat16, __nv_bfloat16, 256, 1>(P, tile_bound, gang, s);
      case 128: return launch_typed<__nv_bfloat16, __nv_bfloat16, 128, 1>(P, tile_bound, gang, s);
      case 64: return launch_typed<__nv_bfloat16, __nv_bfloat16, 64, 1>(P, tile_bound, gang, s);
    }
  } else if (es == 1) {   // MXFP8 operands, bf16 outputs
    if (L.BN == kMxTileN && pair == 2)
      return launch_typed<uint8_t, __nv_bfloat16, kMxTileN, 2>(P, tile_bound, gang, s);
    if (L.BN == kMxTileN) return launch_typed<uint8_t, __nv_bfloat16, kMxTileN, 1>(P, tile_bound, gang, s);
  } else if (es == 4) {
    switch (L.BN) {
      case 256: return launch_typed<float, float, 256, 1>(P, tile_bound, gang, s);
      case 128: return launch_typed<float, float, 128, 1>(P, tile_bound, gang, s);
      case 64: return launch_typed<float, float, 64, 1>(P, tile_bound, gang, s);
    }
  }
  *st = MOE_ERR_UNSUPPORTED;
  return cudaSuccess;
}

}  // namespace moe
