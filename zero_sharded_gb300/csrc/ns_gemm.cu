// Newton-Schulz GEMMs on the 5th-generation tensor cores (sm_103a).
//
// One kernel template over the product it runs and over the tile geometry.  All
// products are D = A * B^T with bf16 operands and an fp32 accumulator in TMEM,
// grouped over every owned tensor of the shard (tensors of one shape form a
// batched "problem"; a launch carries up to kMaxProblems of them):
//   Gram    A  = X X^T                  operands X rows, X rows      (K = n, both K-major)
//   Poly    B' = a I + b A + c A A^T    operands A rows, A rows      (K = m), A symmetric
//   Update  X' <- B' X                  operands B' rows (K-major), X (MN-major: K = m
//                                       rows of n contiguous columns)
// a X + B X = (a I + B) X, so the a X term rides in the Poly output and the
// Update epilogue reads no operand.  X is kept only in its m x n orientation, in
// two buffers: the Update reads one and writes the other (tiles of one column
// block read every row of X).  Step 1 folds the Frobenius normalisation in as
// scalars: A_1 = s^2 X~X~^T and X_1 = s B'_1 X~, s = 1/(||u||_F + eps).  The last
// Update instead runs the apply epilogue: W <- W - lr*sqrt(max(1,rows/cols)) * X_K
// in fp32, the bf16 parameter copy, and (optionally) the applied delta.
//
// Launches: one per product (PHASE = kGram .. kApply), each unit walking its
// range of an LPT-assigned tile list; or one for every product of every step
// (kFused), each unit walking the host's dependency-aware schedule (or the
// per-(step, product) lists), with per-(matrix, step, product) completion
// counters ordering the stages of each matrix.
//
// Structure of a unit: by default a CTA pair (cluster of 2, tcgen05 cta_group::2)
// computes a 256 x 256 tile; CZ_NS_PAIR=0 gives one CTA per 128 x 256 tile.  Per CTA:
//   warp 0      TMA producer (one lane): its 128 rows of the A side and its share of
//               the B side per 64-wide k-block, 128-byte swizzle, an mbarrier ring
//   warp 1      TMEM allocation (512 columns: two 256-column fp32 accumulators) and,
//               in the even CTA, the one lane that issues tcgen05.mma (M = 256 across
//               the pair, N = 256, K = 16) and its commits
//   warps 2..   epilogue, one or two warps per TMEM lane quarter: tcgen05.ld 32
//               columns at a time, the phase's math, then each 32 x 32 block is
//               staged in smem (as is and, above the diagonal of a symmetric
//               product, transposed) and written with TMA bulk tensor stores,
//               which clip at the tensor's edges; the apply updates W directly.
//               The global operands an epilogue chunk needs (A for Poly, W for
//               the apply) are loaded one chunk ahead.
// The TMEM double buffer lets the epilogue of tile i overlap the main loop of
// i + 1.  For the symmetric products only tiles touching the upper triangle are
// computed.  Every wait is bounded (see ptx.cuh).

#include <cuda_bf16.h>

#include <cstdlib>

#include "ptx.cuh"
#include "step_kernels.h"

namespace cz {

namespace {

// Threads of a launch of phase P: producer warp, MMA warp, epilogue warps.
__host__ __device__ constexpr int threads_of(int phase) { return 64 + 32 * epi_warps(phase); }
// Limit of the drain waits at exit (in-flight TMA copies and MMAs must finish
// before shared memory and TMEM are released); independent of p.timeout_ns.
constexpr int64_t kDrainTimeoutNs = 2000000000LL;
constexpr uint32_t kTmemCols = 512;

// Geometry of the two variants: one CTA per 128 x 256 tile, or a CTA pair per
// 256 x 256 tile (cta_group::2: each CTA holds 128 rows of A and 128 of the 256
// B rows per stage, and receives its 128 x 256 half of the accumulator).
template <bool PAIR>
struct Cfg {
  static constexpr int kStages = PAIR ? 6 : 4;
  static constexpr int kTileM = PAIR ? 256 : 128;
  static constexpr int kRowsB = PAIR ? 128 : 256;
  static constexpr int kBytesA = 128 * kBK * 2;
  static constexpr int kBytesB = kRowsB * kBK * 2;
  static constexpr int kStageBytes = kBytesA + kBytesB;
};
static_assert(Cfg<true>::kStages * Cfg<true>::kStageBytes <= kStages * (kStageBytesA + kStageBytesB), "smem");
static_assert(Cfg<false>::kStages * Cfg<false>::kStageBytes <= kStages * (kStageBytesA + kStageBytesB), "smem");

struct Smem {
  uint8_t* a;              // kStages A tiles (1024-byte aligned)
  uint8_t* b;              // kStages B tiles
  __nv_bfloat16* epi;      // kEpiWarps x (direct + transposed 32 x 32 bf16 staging blocks)
  uint64_t* full;          // [kStages]
  uint64_t* empty;         // [kStages]
  uint64_t* tfull;         // [2]
  uint64_t* tempty;        // [2]
  uint64_t* drain;         // [1]
  uint32_t* tmem_holder;
  int* abort;
};

template <bool PAIR>
__device__ __forceinline__ Smem carve(uint8_t* raw) {
  using C = Cfg<PAIR>;
  Smem s;
  const uint32_t base = smem_u32(raw);
  uint8_t* p = raw + ((1024u - (base & 1023u)) & 1023u);
  s.a = p;
  p += C::kStages * C::kBytesA;
  s.b = p;
  p += C::kStages * C::kBytesB;
  s.epi = reinterpret_cast<__nv_bfloat16*>(p);
  p += kEpiWarps * kEpiBytesPerWarp;
  uint64_t* bars = reinterpret_cast<uint64_t*>(p);
  s.full = bars;
  s.empty = bars + C::kStages;
  s.tfull = bars + 2 * C::kStages;
  s.tempty = bars + 2 * C::kStages + 2;
  s.drain = bars + 2 * C::kStages + 4;
  s.tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 5);
  s.abort = reinterpret_cast<int*>(bars + 2 * C::kStages + 6);
  return s;
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Operands one epilogue chunk needs from global memory, loaded ahead of use.
struct Pre {
  uint4 x[4];     // 32 bf16 of A in this row (Poly: the b A term)
  float4 w[8];    // 32 fp32 master weights (Apply)
};

// Component c of v, c known at compile time after unrolling (keeps Pre in registers).
__device__ __forceinline__ float& f4(float4& v, int c) {
  return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

template <int PHASE>
__device__ __forceinline__ void prefetch(Pre& pre, const GemmParams& p, const GemmProblem& pr, int mat,
                                         const MatInfo& mi, int rbase, int lane, int col0) {
  if constexpr (PHASE == kPoly) {
    // A[row][col0 .. col0+31] of this lane's row
    const int row = rbase + lane;
    const __nv_bfloat16* aux = reinterpret_cast<const __nv_bfloat16*>(pr.aux) + (int64_t)mat * pr.ms_aux +
                               (int64_t)row * pr.ld_aux + col0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      pre.x[q] = (row < pr.M && col0 + q * 8 < pr.N) ? *reinterpret_cast<const uint4*>(aux + q * 8)
                                                      : make_uint4(0u, 0u, 0u, 0u);
  }
  if constexpr (PHASE == kApply) {
    if (mi.rows > mi.cols && mi.vec_ok) {
      // tall W = X^T, in the coalesced layout of apply_chunk: entry 4h+k holds W row col0 + 8k + lane/4
      // (D column), W columns rbase + 16h + 4(lane%4) .. +3 (D rows)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = col0 + 8 * k + (lane >> 2);
          const int c = rbase + 16 * h + 4 * (lane & 3);
          if (j < pr.N && c < pr.M)
            pre.w[4 * h + k] = *reinterpret_cast<const float4*>(p.W + mi.w_off + (int64_t)j * mi.cols + c);
        }
      return;
    }
    if (mi.rows > mi.cols) {
      // tall W = X^T: this lane's D row is W column rbase + lane; entry q holds W row col0 + q
      const int i = rbase + lane;
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int j = col0 + q;
        f4(pre.w[q >> 2], q & 3) = (i < pr.M && j < pr.N) ? p.W[mi.w_off + (int64_t)j * mi.cols + i] : 0.f;
      }
      return;
    }
    // W in the coalesced layout of apply_chunk: entry 4h+i holds row rbase + 8i + lane/4,
    // columns col0 + 16h + 4(lane%4) .. +3
    if (mi.vec_ok) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = rbase + i * 8 + (lane >> 2);
          const int c = col0 + 16 * h + (lane & 3) * 4;
          if (r < pr.M && c < pr.N)
            pre.w[4 * h + i] = *reinterpret_cast<const float4*>(p.W + mi.w_off + (int64_t)r * mi.cols + c);
        }
    }
  }
}

// Writes the warp's 32 x 32 block (lane L holds row L) into dense smem staging:
// D[L][c] for the direct store and, if wanted, T[c][L] for the transposed one.
__device__ __forceinline__ void stage_block(__nv_bfloat16* D, __nv_bfloat16* T, const float* v, int lane,
                                            bool want_t) {
  uint4* d = reinterpret_cast<uint4*>(D + lane * 32);
#pragma unroll
  for (int q = 0; q < 4; ++q) d[q] = pack8(v + 8 * q);
  if (want_t) {
#pragma unroll
    for (int c = 0; c < 32; ++c) T[c * 32 + lane] = __float2bfloat16_rn(v[c]);
  }
}

// Apply epilogue of one 32-column chunk of the warp's 32 rows.  The fp32 delta
// lrs * v goes through a padded smem block (lane = row) so that W is read,
// updated and written with lanes across columns: each instruction touches 8 rows
// x 64 contiguous bytes instead of 32 rows x 16 bytes.  W was prefetched in the
// same layout (prefetch<kApply>).  In the parameter's rows x cols layout:
// W <- W - delta, bf16 copy = RNE(W), optional debug delta.  A tall parameter
// holds X^T: its chunk goes through smem transposed, so W is again updated with
// lanes across its columns (or, when W rows are not 16-byte aligned, written
// column by column straight from the lanes).
constexpr int kApplyPitch = 20;   // floats per staged row (16 + 4): conflict-free v4 writes

__device__ __forceinline__ void apply_chunk(const GemmParams& p, const GemmProblem& pr, const MatInfo& mi, int rbase,
                                            int col0, const float* v, Pre& pre, float* stage, int lane) {
  const float lrs = lr_times_scale(p.lr_dev ? __ldg(p.lr_dev) : p.lr, mi.scale);
  if (mi.rows > mi.cols && mi.vec_ok) {
    // tall W = X^T with 16-byte W access: the chunk's delta goes through smem transposed (W row jj =
    // D column, 32 floats per row; 4-float groups XOR-swizzled by the row's parity, so both the
    // column writes and the float4 row reads are free of bank conflicts), then W is updated with
    // lanes across its columns in the layout prefetch<kApply> loaded
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 32; ++q)
      stage[q * 32 + ((((lane >> 2) ^ ((q & 1) << 2)) << 2) | (lane & 3))] = __fmul_rn(lrs, v[q]);
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int jj = 8 * k + (lane >> 2);
        const int g4 = 4 * h + (lane & 3);
        const int j = col0 + jj, c = rbase + 4 * g4;
        if (j >= pr.N || c >= pr.M) continue;   // cols % 4 == 0: the 4 columns are in range together
        const float4 d = *reinterpret_cast<const float4*>(stage + jj * 32 + ((g4 ^ ((jj & 1) << 2)) << 2));
        const int64_t idx = mi.w_off + (int64_t)j * mi.cols + c;
        float4 w = pre.w[4 * h + k];
        w.x = __fsub_rn(w.x, d.x); w.y = __fsub_rn(w.y, d.y); w.z = __fsub_rn(w.z, d.z); w.w = __fsub_rn(w.w, d.w);
        *reinterpret_cast<float4*>(p.W + idx) = w;
        if (p.Wb)
          *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.Wb) + idx) =
              make_uint2(pack_bf16x2(w.x, w.y), pack_bf16x2(w.z, w.w));
        if (p.dbg) *reinterpret_cast<float4*>(p.dbg + idx) = d;
      }
    return;
  }
  if (mi.rows > mi.cols) {
    // tall W (n x m) = X^T: D element (row i, column j) is W[j][i]; the lanes (rows i)
    // cover 32 consecutive W columns, so each column q of the chunk is one 128-byte access
    const int i = rbase + lane;
#pragma unroll
    for (int q = 0; q < 32; ++q) {
      const int j = col0 + q;
      if (i < pr.M && j < pr.N) {
        const float d = __fmul_rn(lrs, v[q]);   // two roundings, as the wide path (no contraction)
        const int64_t idx = mi.w_off + (int64_t)j * mi.cols + i;
        const float w = __fsub_rn(f4(pre.w[q >> 2], q & 3), d);
        p.W[idx] = w;
        if (p.Wb) reinterpret_cast<__nv_bfloat16*>(p.Wb)[idx] = __float2bfloat16_rn(w);
        if (p.dbg) p.dbg[idx] = d;
      }
    }
    return;
  }
  const bool vec = mi.vec_ok != 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    __syncwarp();
    float4* srow = reinterpret_cast<float4*>(stage + lane * kApplyPitch);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      srow[q] = make_float4(lrs * v[16 * h + 4 * q], lrs * v[16 * h + 4 * q + 1], lrs * v[16 * h + 4 * q + 2],
                            lrs * v[16 * h + 4 * q + 3]);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = i * 8 + (lane >> 2);
      const int c4 = (lane & 3) * 4;
      const int row = rbase + r;
      const int col = col0 + 16 * h + c4;
      if (row >= pr.M || col >= pr.N) continue;
      const float4 d = *reinterpret_cast<const float4*>(stage + r * kApplyPitch + c4);
      const int64_t idx = mi.w_off + (int64_t)row * mi.cols + col;
      if (vec) {   // cols % 4 == 0 and w_off % 4 == 0: the 4 columns are in range and 16-byte aligned
        float4 w = pre.w[4 * h + i];
        w.x -= d.x; w.y -= d.y; w.z -= d.z; w.w -= d.w;
        *reinterpret_cast<float4*>(p.W + idx) = w;
        if (p.Wb)
          *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.Wb) + idx) =
              make_uint2(pack_bf16x2(w.x, w.y), pack_bf16x2(w.z, w.w));
        if (p.dbg) *reinterpret_cast<float4*>(p.dbg + idx) = d;
      } else {
        const float dd[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (col + e < pr.N) {
            const float w = p.W[idx + e] - dd[e];
            p.W[idx + e] = w;
            if (p.Wb) reinterpret_cast<__nv_bfloat16*>(p.Wb)[idx + e] = __float2bfloat16_rn(w);
            if (p.dbg) p.dbg[idx + e] = dd[e];
          }
        }
      }
    }
  }
}

// The tiles a unit (CTA or CTA pair) processes, in order.  A per-phase launch
// walks its own range of p.tiles.  The fused launch walks the unit's sequence of
// the host's schedule (p.sched) when there is one; otherwise, for every
// Newton-Schulz step, the unit's ranges of the Gram, Poly and Update (Apply in the
// last step) lists.  All three roles see the same sequence either way.
template <int PHASE>
struct Walker {
  const GemmParams& p;
  const int unit;
  int it = 0, slot = 0, j = 0, j_end = 0;
  bool open = false;
  __device__ Walker(const GemmParams& p_, int unit_) : p(p_), unit(unit_) {}
  __device__ int list_of(int i, int sl) const {
    return sl == 0 ? (i & 1) : sl == 1 ? 2 : (i + 1 == p.ns_steps ? 5 : 3) + (i & 1);
  }
  // Next tile: its entry, global problem index, Newton-Schulz step and slot.
  __device__ bool next(int4& tl, int& prob, int& iter, int& sl) {
    if constexpr (!is_fused(PHASE)) {
      if (!open) {
        j = p.cta_first[unit];
        j_end = p.cta_first[unit + 1];
        open = true;
      }
      if (j >= j_end) return false;
      tl = p.tiles[j++];
      prob = tl.x;
      iter = 0;
      sl = 0;
      return true;
    } else {
      if (p.sched) {
        // the host's dependency-aware schedule: this unit's tiles of every step, in order
        if (!open) {
          j = p.sched_first[unit];
          j_end = p.sched_first[unit + 1];
          open = true;
        }
        if (j >= j_end) return false;
        tl = p.sched[j++];
        prob = tl.x & 0xFF;
        iter = tl.x >> 8;
        sl = p.prob[prob].slot;
        return true;
      }
      while (true) {
        const TileList& L = p.lists[list_of(it, slot)];
        if (!open) {
          j = L.cta_first[unit];
          j_end = L.cta_first[unit + 1];
          open = true;
        }
        if (j < j_end) {
          tl = L.tiles[j++];
          prob = L.prob_off + tl.x;
          iter = it;
          sl = slot;
          return true;
        }
        open = false;
        if (++slot == 3) {
          slot = 0;
          if (++it == p.ns_steps) return false;
        }
      }
    }
  }
};

// Whether a tile's B operand is read MN-major: fixed by the phase where it can be
// (Gram and Poly never, Update and Apply always), else per problem.
template <int PHASE>
__device__ __forceinline__ bool b_operand_mn(const GemmProblem& pr) {
  if constexpr (PHASE == kGram || PHASE == kPoly) return false;
  else if constexpr (PHASE == kUpdate || PHASE == kApply) return true;
  else return pr.b_mn != 0;
}

// Completion counter and arrivals of the stage a fused tile depends on
// (previous slot of the same Newton-Schulz step, or the last slot of the step before).
__device__ __forceinline__ bool fused_dependency(const GemmParams& p, int gm, int iter, int sl, const int** ctr,
                                                 int* target) {
  if (iter == 0 && sl == 0) return false;
  const int ps = sl == 0 ? 2 : sl - 1;
  const int pit = sl == 0 ? iter - 1 : iter;
  *ctr = p.done + (size_t)(pit * 3 + ps) * p.n_mats + gm;
  *target = p.expect[gm * 3 + ps];
  return true;
}

struct EpiCtx {
  uint64_t* tfull;
  uint64_t* tempty;
  volatile int* abort;
  uint32_t tmem_base, lane_field;
  int quad, half, lane;
  uint32_t rank;
  __nv_bfloat16* stD;
  __nv_bfloat16* stT;
  bool pending;           // bulk stores in flight from the staging blocks
};

// Epilogue of one tile in phase PH: prefetch the first chunk's operands, wait for
// the accumulator, then per 32-column chunk read TMEM, apply the phase math and
// store; the accumulator is handed back after its last read.  Symmetric outputs
// (Gram, Poly) are written by aligned 32 x 32 blocks: a block above the diagonal
// directly and mirrored, a diagonal block directly, a block below not at all (its
// mirror comes from the block above), so each element is written exactly once.
// Returns false if the wait for the accumulator ran out.
template <int PH, bool PAIR, int EW>
__device__ __forceinline__ bool epilogue_tile(const GemmParams& p, EpiCtx& e, const GemmProblem& pr, int prob,
                                              int mat, int tile_m, int tile_n, bool first, uint32_t acc,
                                              uint32_t acc_phase) {
  using C = Cfg<PAIR>;
  constexpr bool kSym = PH == kGram || PH == kPoly;
  const int lane = e.lane;
  const int gm = pr.mat_base + mat;
  const int rbase = tile_m * C::kTileM + (int)e.rank * 128 + e.quad * 32;
  constexpr int kChunks = 32 / EW;            // 32-column chunks per warp (the lane quarter's 8, shared by EW/4 warps)
  const int ch_first = e.half * kChunks;
  const int col_first = tile_n * kBN + ch_first * 32;
  auto release = [&]() {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(smem_u32(&e.tempty[acc]), 0));
      else mbar_arrive(&e.tempty[acc]);
    }
  };
  // chunks this warp reads from TMEM (warp-uniform bit mask)
  uint32_t need = 0;
  if (rbase < pr.M) {
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const int col0 = col_first + c * 32;
      if (col0 < pr.N && (!kSym || rbase <= col0)) need |= 1u << c;
    }
  }
  const int last = need ? 31 - __clz(need) : -1;
  float s = 1.f;
  if (first) {
    const float sg = p.sigma[gm];
    s = (PH == kGram) ? sg * sg : sg;
  }
  MatInfo mi{};
  if constexpr (PH == kApply) mi = p.mats[gm];
  Pre cur;
  const int first_c = need ? __ffs(need) - 1 : 0;
  if constexpr (PH == kApply) {
    // the master weights of this warp's whole share of the tile into L2 while the MMAs run:
    // 32 D rows x (32 kChunks) D columns = 32 kChunks lines of 128 bytes, kChunks per lane
    if (need) {
      const bool tall = mi.rows > mi.cols;
#pragma unroll
      for (int q = 0; q < kChunks; ++q) {
        int wr, wc;                                   // W row and first W column of the line
        if (tall) { wr = col_first + lane * kChunks + q; wc = rbase; }   // W rows = D columns
        else { wr = rbase + lane; wc = col_first + q * 32; }             // kChunks lines per D row
        if (wr < mi.rows && wc < mi.cols)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(p.W + mi.w_off + (int64_t)wr * mi.cols + wc));
      }
    }
  }
  if (need) prefetch<PH>(cur, p, pr, mat, mi, rbase, lane, col_first + first_c * 32);
  const bool w = mbar_wait(&e.tfull[acc], acc_phase, e.abort, p.status, p.timeout_ns);
  if (!__all_sync(0xffffffffu, w)) return false;
  tc_fence_after();
  const uint32_t tbase = e.tmem_base + acc * (uint32_t)kBN + e.lane_field;
  if (last < 0) release();
  for (int c = first_c; c <= last; ++c) {
    if (!((need >> c) & 1u)) continue;
    const int col0 = col_first + c * 32;
    Pre nxt;
    const uint32_t later = need >> (c + 1);
    if (later) prefetch<PH>(nxt, p, pr, mat, mi, rbase, lane, col0 + 32 * __ffs(later));
    float v[32];
    tmem_ld32(tbase + (uint32_t)((ch_first + c) * 32), v);
    if (c == last) release();     // accumulator no longer needed: let the MMA reuse it
    if constexpr (PH == kApply) {
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] *= s;
      apply_chunk(p, pr, mi, rbase, col0, v, cur, reinterpret_cast<float*>(e.stD), lane);
    } else {
      if constexpr (PH == kPoly) {
        // B' = a I + b A + c (A A)
        float a[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) unpack8(cur.x[q], a + 8 * q);
        const bool diag = rbase == col0;
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] = fmaf(p.b, a[q], p.c * v[q]) + ((diag && q == lane) ? p.a : 0.f);
      } else {
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] *= s;   // Gram: s = sigma^2; Update: s = sigma (step 1)
      }
      const bool do_t = kSym && rbase < col0;     // the mirror of a block above the diagonal
      if (lane == 0 && e.pending) bulk_wait_read_all();
      __syncwarp();
      stage_block(e.stD, e.stT, v, lane, do_t);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&p.tmO[prob], e.stD, col0, rbase, mat);
        if (do_t) tma_store_3d(&p.tmOT[prob], e.stT, rbase, col0, mat);
        bulk_commit();
        e.pending = true;
      }
    }
    cur = nxt;
  }
  return true;
}

// Per-product launches run 10 warps: two of the four SM sub-partitions hold 3 warps,
// so a thread gets at most 16384 / 96 registers (168 after rounding).  The fused
// launch runs 6 warps (at most 2 per sub-partition: up to 255 registers).
template <int PHASE, bool PAIR>
__global__ void __launch_bounds__(threads_of(PHASE), 1) ns_gemm_kernel(const __grid_constant__ GemmParams p) {
  constexpr int EW = epi_warps(PHASE);
  using C = Cfg<PAIR>;
  extern __shared__ uint8_t smem_raw[];
  Smem sm = carve<PAIR>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort = sm.abort;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;     // 0: the CTA that issues the MMAs
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.tfull[i], 1);
      mbar_init(&sm.tempty[i], EW * (PAIR ? 2 : 1));   // one arrival per epilogue warp
    }
    mbar_init(sm.drain, 1);
    *sm.abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    if constexpr (PAIR) tmem_alloc_pair(sm.tmem_holder, kTmemCols);
    else tmem_alloc(sm.tmem_holder, kTmemCols);
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync();   // the peer's barriers exist before any remote arrival
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_holder;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer (both CTAs of a pair)
    // One thread runs the whole loop (TMA copies are single-thread instructions).
    if (lane == 0) {
      for (int i = 0; i < p.n_prob; ++i) {
        tma_prefetch_desc(&p.tmA[i]);
        tma_prefetch_desc(&p.tmB[i]);
        if (PHASE != kApply && p.prob[i].phase != kApply) {   // Apply problems store no tiles
          tma_prefetch_desc(&p.tmO[i]);
          if (p.prob[i].phase != kUpdate) tma_prefetch_desc(&p.tmOT[i]);
        }
      }
      uint32_t stage = 0, phase = 0, issued = 0, last_par = 0;   // bit s: parity of stage s's last fill
      bool ok = true;
      Walker<PHASE> walk(p, unit);
      int4 tl;
      int prob, iter, sl;
      int issued_tiles = 0;   // tiles whose loads this unit has issued (wave pacing)
      while (ok && walk.next(tl, prob, iter, sl)) {
        const GemmProblem& pr = p.prob[prob];
        if constexpr (!is_fused(PHASE)) {
          // wave pacing: this tile starts once every unit has issued as many tiles as this
          // one (the even CTA paces; the odd one follows through the shared stage ring)
          if (p.pace && rank == 0 && issued_tiles > 0 && issued_tiles < p.pace_tiles &&
              !counter_wait(p.pace, issued_tiles * p.grid, abort, p.status, p.timeout_ns))
            break;
        }
        if constexpr (is_fused(PHASE)) {
          // the matrix's previous stage must be complete (and visible) before its data is loaded
          const int* ctr;
          int target;
          if (fused_dependency(p, pr.mat_base + tl.y, iter, sl, &ctr, &target) &&
              !counter_wait(ctr, target, abort, p.status, p.timeout_ns))
            break;
        }
        const int nk = ceil_div(pr.K, kBK);
        const CUtensorMap* ma = &p.tmA[prob];
        const CUtensorMap* mb = &p.tmB[prob];
        const int arow = tl.z * C::kTileM + (int)rank * 128;
        const int brow = tl.w * kBN + (int)rank * C::kRowsB;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          uint8_t* da = sm.a + stage * C::kBytesA;
          uint8_t* db = sm.b + stage * C::kBytesB;
          // A: one box of its rows x 64 k; B the same when K-major, else 64 x 64 boxes
          // (64 N columns x 64 k rows, 8 KB each) side by side
          if constexpr (PAIR) {
            // both CTAs' copies complete on the even CTA's full barrier
            const uint32_t fb = mapa_shared(smem_u32(&sm.full[stage]), 0);
            if (rank == 0) mbar_arrive_expect_tx(&sm.full[stage], 2 * C::kStageBytes);
            tma_load_3d_pair(da, ma, fb, kb * kBK, arow, tl.y);
            if (b_operand_mn<PHASE>(pr)) {
              for (int j = 0; j < C::kRowsB / 64; ++j)
                tma_load_3d_pair(db + j * 8192, mb, fb, brow + 64 * j, kb * kBK, tl.y);
            } else {
              tma_load_3d_pair(db, mb, fb, kb * kBK, brow, tl.y);
            }
          } else {
            mbar_arrive_expect_tx(&sm.full[stage], C::kStageBytes);
            tma_load_3d(da, ma, &sm.full[stage], kb * kBK, arow, tl.y);
            if (b_operand_mn<PHASE>(pr)) {
              for (int j = 0; j < C::kRowsB / 64; ++j)
                tma_load_3d(db + j * 8192, mb, &sm.full[stage], brow + 64 * j, kb * kBK, tl.y);
            } else {
              tma_load_3d(db, mb, &sm.full[stage], kb * kBK, brow, tl.y);
            }
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if constexpr (!is_fused(PHASE)) {
          if (ok && p.pace && rank == 0) atomicAdd(p.pace, 1);
        }
        ++issued_tiles;
      }
      // every issued copy must land before the CTA may exit; a pair's copies are
      // counted on the even CTA's barriers, and the odd CTA waits for the even one
      // at the final cluster barrier
      if (rank == 0) {
        for (int s = 0; s < C::kStages; ++s)
          if (issued & (1u << s)) mbar_wait(&sm.full[s], (last_par >> s) & 1u, nullptr, p.status, kDrainTimeoutNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer (even CTA only)
    // One thread runs the whole issue loop: tcgen05.mma is single-thread, and keeping
    // the other lanes out removes a warp shuffle and a warp barrier from every k-block.
    if (rank == 0 && lane == 0) {
      constexpr uint32_t idesc_kk = idesc_bf16_f32(C::kTileM, kBN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      Walker<PHASE> walk(p, unit);
      int4 tl;
      int prob, iter, sl;
      while (ok && walk.next(tl, prob, iter, sl)) {
        const GemmProblem& pr = p.prob[prob];
        const int nk = ceil_div(pr.K, kBK);
        const bool b_mn = b_operand_mn<PHASE>(pr);
        // MN-major B: bit 16 of the instruction descriptor
        const uint32_t idesc = idesc_kk | (b_mn ? (1u << 16) : 0u);
        // descriptors of stage 0, K step 0; a stage adds its byte offset, a K = 16 step
        // adds 32 bytes (K-major) or 16 rows = 2048 bytes (MN-major; boxes 8192 apart),
        // all in the 16-byte units of the start-address field (addresses < 256 KB: no carry)
        const uint64_t da0 = sdesc_kmajor_sw128(smem_u32(sm.a));
        const uint64_t db0 = b_mn ? sdesc_mnmajor_sw128(smem_u32(sm.b), 8192, 1024) : sdesc_kmajor_sw128(smem_u32(sm.b));
        const uint32_t a_step = 32 / 16, b_step = b_mn ? 2048 / 16 : 32 / 16;
        if (!mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, abort, p.status, p.timeout_ns)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * (uint32_t)kBN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&sm.full[stage], phase, abort, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t as = da0 + stage * (uint32_t)(C::kBytesA / 16);
          const uint64_t bs = db0 + stage * (uint32_t)(C::kBytesB / 16);
#pragma unroll
          for (int s = 0; s < kBK / 16; ++s) {
            const uint64_t ad = as + s * a_step, bd = bs + s * b_step;
            if constexpr (PAIR) umma_bf16_pair(d, ad, bd, idesc, (kb | s) != 0 ? 1u : 0u);
            else umma_bf16(d, ad, bd, idesc, (kb | s) != 0 ? 1u : 0u);
          }
          if constexpr (PAIR) umma_commit_pair(&sm.empty[stage], 0x3);   // frees the stage in both CTAs
          else umma_commit(&sm.empty[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (PAIR) umma_commit_pair(&sm.tfull[acc], 0x3);     // both halves of the accumulator
        else umma_commit(&sm.tfull[acc]);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // wait until every issued MMA has completed (TMEM is released below)
      if constexpr (PAIR) umma_commit_pair(sm.drain, 0x1);
      else umma_commit(sm.drain);
      mbar_wait(sm.drain, 0, nullptr, p.status, kDrainTimeoutNs);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue (both CTAs of a pair)
    const int ew = warp - 2;                    // 0 .. EW-1
    EpiCtx e;
    e.tfull = sm.tfull;
    e.tempty = sm.tempty;
    e.abort = abort;
    e.tmem_base = tmem_base;
    e.quad = warp & 3;                          // TMEM lane quarter this warp may access
    e.half = ew >> 2;                           // which share of the 256 accumulator columns
    e.lane = lane;
    e.rank = rank;
    e.lane_field = (uint32_t)(e.quad * 32) << 16;
    e.stD = sm.epi + ew * (kEpiBytesPerWarp / 2);
    e.stT = e.stD + 32 * 32;
    e.pending = false;
    uint32_t acc = 0, acc_phase = 0;
    Walker<PHASE> walk(p, unit);
    int4 tl;
    int prob, iter, sl;
    while (walk.next(tl, prob, iter, sl)) {
      const GemmProblem& pr = p.prob[prob];
      bool ok;
      if constexpr (is_fused(PHASE)) {
        const bool first = iter == 0;
        switch (pr.phase) {
          case kGram: ok = epilogue_tile<kGram, PAIR, EW>(p, e, pr, prob, tl.y, tl.z, tl.w, first, acc, acc_phase); break;
          case kPoly: {
            // the Poly epilogue reads A directly: acquire the Gram stage it depends on
            const int* ctr;
            int target;
            if (fused_dependency(p, pr.mat_base + tl.y, iter, sl, &ctr, &target))
              counter_wait(ctr, target, abort, p.status, p.timeout_ns);
            ok = epilogue_tile<kPoly, PAIR, EW>(p, e, pr, prob, tl.y, tl.z, tl.w, first, acc, acc_phase);
            break;
          }
          case kUpdate:
            ok = epilogue_tile<kUpdate, PAIR, EW>(p, e, pr, prob, tl.y, tl.z, tl.w, first, acc, acc_phase);
            break;
          default: ok = epilogue_tile<kApply, PAIR, EW>(p, e, pr, prob, tl.y, tl.z, tl.w, first, acc, acc_phase); break;
        }
        // publish this warp's part of the tile once its stores are complete; the
        // last step's Apply has no successor
        if (ok && !(sl == 2 && iter + 1 == p.ns_steps)) {
          if (lane == 0) {
            if (e.pending) {
              bulk_wait_all();
              e.pending = false;
            }
            counter_release_add(p.done + (size_t)(iter * 3 + sl) * p.n_mats + pr.mat_base + tl.y, 1);
          }
          __syncwarp();
        }
      } else {
        ok = epilogue_tile<PHASE, PAIR, EW>(p, e, pr, prob, tl.y, tl.z, tl.w, p.first != 0, acc, acc_phase);
      }
      if (!ok) break;
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0 && e.pending) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  if constexpr (PAIR) cluster_sync();   // the even CTA's MMAs (which read both CTAs' smem) are done
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

// The fused launch is cooperative unless CZ_NS_COOPERATIVE=0 or a CUDA tool is
// attached to the process: Nsight Compute (it sets NV_COMPUTE_PROFILER_PERFWORKS_DIR
// and NV_NSIGHT_INJECTION_TRANSPORT_TYPE in the target) or a tool injected through
// CUDA_INJECTION64_PATH.  Nsight Compute's kernel profiling fails a cooperative
// cluster launch with LaunchFailed and then shuts the application down; such tools
// serialise launches, so the units of the fused grid (the occupancy limit) are
// co-resident there without the attribute.
bool cooperative_fused() {
  static const bool on = [] {
    const char* e = std::getenv("CZ_NS_COOPERATIVE");
    if (e && e[0] == '0') return false;
    for (const char* v : {"NV_COMPUTE_PROFILER_PERFWORKS_DIR", "NV_NSIGHT_INJECTION_TRANSPORT_TYPE",
                          "CUDA_INJECTION64_PATH"}) {
      const char* t = std::getenv(v);
      if (t && t[0]) return false;
    }
    return true;
  }();
  return on;
}

template <int PHASE, bool PAIR>
cudaError_t launch_phase(const GemmParams& p, cudaStream_t s) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(ns_gemm_kernel<PHASE, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kGemmSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  // The fused launch's units wait on one another's completion counters, so it is a
  // cooperative launch: the runtime guarantees that every CTA is resident at once
  // (or refuses the launch) even when other work shares the GPU.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((PAIR ? 2 : 1) * p.grid, 1, 1);
  cfg.blockDim = dim3(threads_of(PHASE), 1, 1);
  cfg.dynamicSmemBytes = kGemmSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n_attr = 0;
  if constexpr (PAIR) {
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = 2;
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr].val.clusterDim.z = 1;
    ++n_attr;
  }
  // The fused launch's units wait on one another's completion counters and paced
  // units on one another's progress, so those launches are cooperative.
  if (is_fused(PHASE) || p.pace) {
    if (cooperative_fused()) {
      attr[n_attr].id = cudaLaunchAttributeCooperative;
      attr[n_attr].val.cooperative = 1;
      ++n_attr;
    }
  }
  cfg.attrs = attr;
  cfg.numAttrs = n_attr;
  return cudaLaunchKernelEx(&cfg, ns_gemm_kernel<PHASE, PAIR>, p);
}

}  // namespace

cudaError_t launch_ns_gemm(int phase, bool pair, const GemmParams& p, cudaStream_t s) {
  if (p.n_tiles <= 0) return cudaSuccess;
  switch (phase * 2 + (pair ? 1 : 0)) {
    case kGram * 2: return launch_phase<kGram, false>(p, s);
    case kGram * 2 + 1: return launch_phase<kGram, true>(p, s);
    case kPoly * 2: return launch_phase<kPoly, false>(p, s);
    case kPoly * 2 + 1: return launch_phase<kPoly, true>(p, s);
    case kUpdate * 2: return launch_phase<kUpdate, false>(p, s);
    case kUpdate * 2 + 1: return launch_phase<kUpdate, true>(p, s);
    case kApply * 2: return launch_phase<kApply, false>(p, s);
    case kApply * 2 + 1: return launch_phase<kApply, true>(p, s);
    case kFused * 2: return launch_phase<kFused, false>(p, s);
    case kFused * 2 + 1: return launch_phase<kFused, true>(p, s);
    case kFusedLatency * 2: return launch_phase<kFusedLatency, false>(p, s);
    case kFusedLatency * 2 + 1: return launch_phase<kFusedLatency, true>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

int gemm_max_units(bool pair) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) return 1;
  if (!pair) return sms;
  // CTA pairs that can be resident at once (clusters of 2 need two SMs of one GPC)
  if (cudaFuncSetAttribute(ns_gemm_kernel<kUpdate, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kGemmSmemBytes) != cudaSuccess)
    return sms / 2 > 0 ? sms / 2 : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sms / 2 > 0 ? sms / 2 : 1), 1, 1);
  cfg.blockDim = dim3(threads_of(kUpdate), 1, 1);
  cfg.dynamicSmemBytes = kGemmSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, ns_gemm_kernel<kUpdate, true>, &cfg) != cudaSuccess || clusters < 1) {
    cudaGetLastError();
    return sms / 2 > 0 ? sms / 2 : 1;
  }
  return clusters;
}

}  // namespace cz
