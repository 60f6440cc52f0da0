// Launch interface between the host orchestration of the Muon step
// (muon_step.cpp) and the CUDA kernels (momentum.cu, ns_gemm.cu).
// Plain structs with device pointers; bf16 buffers are uint16_t on the host side.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace cz {

// ------------------------------------------------------------------ momentum pass
// Momentum tiles are 64 rows x kMomTileCols columns (fp32 gradients) or 64 x
// kMomTileColsBf16 (bf16 gradients): 8 columns a thread, so each thread moves two
// 16-byte vectors of momentum and one (bf16) or two (fp32) of gradient per row.
constexpr int kMomTileCols = 128;
constexpr int kMomTileColsBf16 = 128;

// One tile of one owned tensor (rows x cols layout of the parameter).
struct MomTile {
  int32_t mat;     // index into MomMat
  int32_t r0, c0;  // tile origin (element row / column)
  int32_t pad;
};

struct MomMat {
  int64_t off;            // element offset of the tensor in the flat buffers
  int32_t rows, cols;     // parameter layout (rows x cols, row-major)
  uint16_t* direct;       // bf16 buffer receiving u in rows x cols orientation, or null
  uint16_t* trans;        // bf16 buffer receiving u^T (cols x rows), or null
  int64_t ld_direct;      // element pitch of `direct` rows
  int64_t ld_trans;       // element pitch of `trans` rows
  int32_t tile_first;     // first tile of this tensor (its partial sums are contiguous)
  int32_t tile_count;
};

struct MomParams {
  float* mom;             // flat fp32 momentum
  const void* grad;       // flat fp32 or bf16 gradient
  int32_t grad_bf16;
  int32_t nesterov;
  float mu;
  float eps;
  const MomTile* tiles;
  int32_t n_tiles;
  const MomMat* mats;
  int32_t n_mats;
  float* partial;         // per tile: sum of u^2 over the tile
  float* sigma;           // per tensor: 1 / (||u||_F + eps)
  int* tile_done;         // per tensor: tiles finished in this launch (zero at launch, reset by the last)
  int* status;
};

cudaError_t launch_momentum(const MomParams& p, cudaStream_t s);

// Copies a step program's tables (tile lists, per-tensor descriptors, zeroed
// counters) from page-locked, device-mapped host memory into the workspace with
// a kernel: no copy-engine transfer, so the copy neither synchronises the host
// with the stream (as a pageable upload may) nor queues behind the caller's own
// host-to-device copies.  src and dst 16-byte aligned, bytes a multiple of 16.
cudaError_t launch_tables_copy(const void* src, void* dst, int64_t bytes, cudaStream_t s);

// ------------------------------------------------------------------ NS GEMM
constexpr int kBM = 128;        // UMMA M (TMEM lanes)
constexpr int kBN = 256;        // UMMA N (TMEM columns per accumulator)
constexpr int kBK = 64;         // 64 bf16 = one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kMaxProblems = 32;
constexpr int kMaxGrid = 1024;  // upper bound on the persistent grid (SM count)

enum Phase : int32_t {
  kGram = 0,     // A = s^2 X X^T                   (symmetric output)
  kPoly = 1,     // B' = a I + b A + c A A          (symmetric output)
  kUpdate = 2,   // X' <- s B' X into the other X buffer (= s (a X + B X))
  kApply = 3,    // last step: W <- W - lr*scale*s B' X, transposed for a tall W (+ bf16 copy, debug delta)
  kFused = 4,    // every product of all ns_steps in one launch, per-matrix dependencies
  kFusedLatency = 5,   // the same with twice the epilogue warps (shards with fewer tiles per product than units)
};
__host__ __device__ constexpr bool is_fused(int phase) { return phase == kFused || phase == kFusedLatency; }

// One batched GEMM: `count` matrices of the same M x N x K, operands read by
// the two tensor maps of the same index (A side: M rows, B side: N rows), output
// written by the epilogue of the launch's phase.  The A operand is K-major (rows of
// K elements, 64 x 128-row boxes); the B operand too (64 x 128- or 256-row boxes)
// unless b_mn is set: then it is stored with N contiguous (X, read by the Update
// and the Apply) and loaded as 64 (N) x 64 (K) boxes.
struct GemmProblem {
  int32_t M, N, K, count;
  int32_t b_mn;           // B operand read MN-major
  int32_t pad;
  int32_t mat_base;       // global index (sigma / MatInfo) of matrix 0 of this problem
  int32_t phase;          // kGram .. kApply (read by the fused launch)
  int32_t slot;           // position in a Newton-Schulz step: 0 Gram, 1 Poly, 2 Update/Apply
  const uint16_t* aux;   int64_t ld_aux, ms_aux;     // kPoly: A (for the b A term)
};

// Per global matrix: where its parameter lives (for the apply epilogue).  The
// learning rate is a launch parameter, so the tables hold only the shape scale.
struct MatInfo {
  int64_t w_off;          // element offset in the flat parameter buffers
  double scale;           // sqrt(max(1, rows/cols)), in double
  int32_t rows, cols;     // parameter layout
  int32_t vec_ok;         // w_off and cols are multiples of 4 (16-byte fp32 vectors)
  int32_t pad;
};

#ifdef __CUDACC__
// The apply's coefficient lr * sqrt(max(1, rows/cols)): the product formed in
// double and rounded to fp32 once, as the host forms it for the standalone apply.
__device__ __forceinline__ float lr_times_scale(float lr, double scale) {
  return __double2float_rn(__dmul_rn((double)lr, scale));
}
#endif

// One phase's tile list inside a fused launch.
struct TileList {
  const int4* tiles;          // {problem (index within the list's problems), matrix, tile_m, tile_n}
  const int32_t* cta_first;   // grid+1 entries, as GemmParams::cta_first
  int32_t prob_off;           // the list's problem 0 in GemmParams::prob
  int32_t pad;
};
constexpr int kFusedLists = 7;  // Gram (X buffer 0), Gram (1), Poly, Update (0), Update (1), Apply (0), Apply (1)

struct GemmParams {
  CUtensorMap tmA[kMaxProblems];    // A-side operand loads (128-byte swizzle)
  CUtensorMap tmB[kMaxProblems];    // B-side operand loads
  CUtensorMap tmO[kMaxProblems];    // output stores, 32 x 32 boxes (Gram/Poly: A or B'; Update: X')
  CUtensorMap tmOT[kMaxProblems];   // mirrored-output stores of the symmetric products (same matrix)
  GemmProblem prob[kMaxProblems];
  int32_t n_prob;
  int32_t n_tiles;
  int32_t grid;           // units (CTAs, or CTA pairs) the tile assignment was made for
  const int4* tiles;      // {problem, matrix, tile_m, tile_n}, grouped by CTA
  const int32_t* cta_first;   // grid+1 entries: unit b runs tiles [cta_first[b], cta_first[b+1])
  const float* sigma;     // per global matrix
  const MatInfo* mats;    // per global matrix
  float a, b, c;
  float lr;               // learning rate (kApply)
  const float* lr_dev;    // or null: the learning rate in device memory, read in place of lr
  int32_t first;          // 1: Newton-Schulz step 1 (scale by sigma)
  float* W;               // fp32 master (kApply)
  uint16_t* Wb;           // bf16 copy or null (kApply)
  float* dbg;             // debug delta or null (kApply)
  int* status;
  int64_t timeout_ns;
  // one-product launches: null, or a counter of the tiles whose operand loads the
  // units have issued.  A unit starts its j-th tile, j < pace_tiles, once every unit
  // has issued j tiles (j * grid), so each wave of tiles starts together and the
  // tiles sharing an operand read it at the same k (cooperative launch).  Every unit
  // has at least pace_tiles - 1 tiles, so the least advanced unit never waits.
  int* pace;
  int32_t pace_tiles;
  int32_t pad_pace;
  // fused launch (kFused) only
  int32_t ns_steps;
  int32_t n_mats;
  TileList lists[kFusedLists];
  int* done;              // (3 * ns_steps) x n_mats completion counters, zero at launch
  const int* expect;      // n_mats x 3: arrivals that complete (matrix, slot)
  // or null: every unit's tiles of all steps in one scheduled sequence, in place of
  // the per-(step, product) lists: entry {problem | step << 8, matrix, tile_m, tile_n},
  // unit b runs entries [sched_first[b], sched_first[b+1])
  const int4* sched;
  const int32_t* sched_first;
};

// Dynamic shared memory of the GEMM kernel.
// Epilogue warps: two per TMEM lane quarter for the one-product launches (the apply's
// master-weight traffic wants the memory parallelism), one per quarter for the fused
// launch (fewer warps competing with the producer and MMA threads for issue slots;
// measured faster there, slower for the per-product Poly and Apply).  A shard whose
// products all have fewer tiles than there are units waits on each stage's epilogue
// (its matrices' stage chains are the whole launch): there the fused launch runs two
// epilogue warps per quarter as well (kFusedLatency; six small matrices and one
// 256 x 256 one: 0.157 -> 0.142 ms per step; on the Qwen3-1.7B layer, 8 warps were
// 2.7% slower than 4).
constexpr int kEpiWarps = 8;                                  // the most any variant uses (shared memory)
constexpr int kFusedEpiWarps = 4;
__host__ __device__ constexpr int epi_warps(int phase) { return phase == kFused ? kFusedEpiWarps : kEpiWarps; }
constexpr int kStageBytesA = kBM * kBK * 2;
constexpr int kStageBytesB = kBN * kBK * 2;
constexpr int kEpiBlockBytes = 32 * 32 * 2;                   // one dense 32 x 32 bf16 block
constexpr int kEpiBytesPerWarp = 2 * kEpiBlockBytes;          // direct + transposed staging
constexpr int kGemmSmemBytes = 1024 /*align slack*/ + kStages * (kStageBytesA + kStageBytesB) +
                               kEpiWarps * kEpiBytesPerWarp + 256 /*barriers*/;

// pair: 256 x 256 tiles on CTA pairs (tcgen05 cta_group::2), else 128 x 256 tiles
// on single CTAs.  p.grid counts units (pairs or CTAs).
cudaError_t launch_ns_gemm(int phase, bool pair, const GemmParams& p, cudaStream_t s);
int gemm_max_units(bool pair);   // units that can be resident at once (persistent grid bound)

// ------------------------------------------------------------------ small-matrix Newton-Schulz
// Matrices with m <= kSmallMaxM and n <= kSmallMaxN run every Newton-Schulz step
// in one CTA with X, A and B' resident in shared memory and the accumulators
// in TMEM (one CTA per matrix, one launch for all of them).  Matrices with
// kSmallMaxM < m <= kSmallPairMaxM and n <= kSmallMaxN do the same on a CTA pair
// (one cluster of two CTAs per matrix, half of every iterate's rows each).
constexpr int kSmallMaxM = 128;
constexpr int kSmallMaxN = 256;
constexpr int kSmallPairMaxM = 256;

struct SmallMat {
  const uint16_t* x;      // bf16 X (m x n), row pitch ldx (written by the momentum pass)
  int32_t ldx;
  int32_t pad0;
  int32_t m, n;
  int32_t mat;            // global matrix index (sigma, MatInfo)
  int32_t pad;
};

struct SmallParams {
  const SmallMat* mats;
  int32_t n_mats;
  int32_t ns_steps;
  const float* sigma;     // per global matrix
  const MatInfo* info;    // per global matrix
  float a, b, c;
  float lr;               // learning rate
  const float* lr_dev;    // or null: the learning rate in device memory, read in place of lr
  float* W;               // fp32 master
  uint16_t* Wb;           // bf16 copy or null
  float* dbg;             // debug delta or null
  int* status;
  int64_t timeout_ns;
};

cudaError_t launch_ns_small(const SmallParams& p, cudaStream_t s);
cudaError_t launch_ns_small_pair(const SmallParams& p, cudaStream_t s);   // p.mats: CTA-pair matrices

}  // namespace cz
