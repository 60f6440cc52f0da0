// Newton-Schulz GEMMs on the 5th-generation tensor cores (sm_103a).
//
// One kernel template, one launch per Newton-Schulz product, grouped over every
// owned tensor of the shard (tensors of the same shape form one batched
// "problem"; a launch carries up to kMaxProblems of them and a flat tile list).
// All products are D = A * B^T with both operands K-major bf16 and an fp32
// accumulator in TMEM:
//   Gram    A_t = X X^T                 operands X rows, X rows      (K = n)
//   Poly    B_t = b A + c A A^T         operands A rows, A rows      (K = m), A symmetric
//   Update  X  <- a X + B X = a X + B (X^T)^T   operands B rows, X^T rows (K = m)
// The update also writes X^T for the next step, so no MN-major operand is needed.
// Step 1 folds the Frobenius normalisation in as scalars: A_1 = s^2 X~X~^T and
// X_1 = s (a X~ + B_1 X~), s = 1/(||u||_F + eps).  The last update instead runs
// the apply epilogue: W <- W - lr*sqrt(max(1,rows/cols)) * X_K in fp32, the bf16
// parameter copy, and (optionally) the applied delta.
//
// Structure (one CTA per SM, persistent over a static round-robin tile list):
//   warp 0      TMA producer: 128x64 (A side) and 256x64 (B side) bf16 tiles,
//               128-byte swizzle, kStages-deep mbarrier ring
//   warp 1      TMEM allocation (512 columns = two 128x256 fp32 accumulators)
//               and the single thread that issues tcgen05.mma (M=128, N=256, K=16)
//   warps 2..5  epilogue: tcgen05.ld 32 columns at a time from its TMEM lane
//               quarter, phase-specific math, bf16/fp32 stores; a per-warp smem
//               transpose writes the mirrored (symmetric) or X^T copy.
// The TMEM double buffer lets the epilogue of tile i overlap the mainloop of i+1.
// For the symmetric products only tiles touching the upper triangle are
// computed; each element (i <= j) is written once directly and once mirrored.

#include <cuda_bf16.h>

#include "ptx.cuh"
#include "step_kernels.h"

namespace cz {

namespace {

constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;

struct Smem {
  uint8_t* a[kStages];
  uint8_t* b[kStages];
  __nv_bfloat16* epi;      // 4 warps x 32 x kEpiPitch
  uint64_t* full;          // [kStages]
  uint64_t* empty;         // [kStages]
  uint64_t* tfull;         // [2]
  uint64_t* tempty;        // [2]
  uint64_t* drain;         // [1]
  uint32_t* tmem_holder;
  int* abort;
};

__device__ __forceinline__ Smem carve(uint8_t* raw) {
  Smem s;
  const uint32_t base = smem_u32(raw);
  uint8_t* p = raw + ((1024u - (base & 1023u)) & 1023u);
  for (int i = 0; i < kStages; ++i) s.a[i] = p + i * kStageBytesA;
  p += kStages * kStageBytesA;
  for (int i = 0; i < kStages; ++i) s.b[i] = p + i * kStageBytesB;
  p += kStages * kStageBytesB;
  s.epi = reinterpret_cast<__nv_bfloat16*>(p);
  p += 4 * kEpiBytesPerWarp;
  uint64_t* bars = reinterpret_cast<uint64_t*>(p);
  s.full = bars;
  s.empty = bars + kStages;
  s.tfull = bars + 2 * kStages;
  s.tempty = bars + 2 * kStages + 2;
  s.drain = bars + 2 * kStages + 4;
  s.tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
  s.abort = reinterpret_cast<int*>(bars + 2 * kStages + 6);
  return s;
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ uint4 pack8(const float* v) {
  uint4 r;
  __nv_bfloat162 t;
  t = __floats2bfloat162_rn(v[0], v[1]); r.x = *reinterpret_cast<uint32_t*>(&t);
  t = __floats2bfloat162_rn(v[2], v[3]); r.y = *reinterpret_cast<uint32_t*>(&t);
  t = __floats2bfloat162_rn(v[4], v[5]); r.z = *reinterpret_cast<uint32_t*>(&t);
  t = __floats2bfloat162_rn(v[6], v[7]); r.w = *reinterpret_cast<uint32_t*>(&t);
  return r;
}

__device__ __forceinline__ void unpack8(uint4 r, float* v) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 t = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    v[2 * i] = __low2float(t);
    v[2 * i + 1] = __high2float(t);
  }
}

// 32 bf16 of row `row`, columns [col0, col0+32) of a bf16 matrix (row pitch ld);
// vectors starting at or beyond `ncols` read as zero.
__device__ __forceinline__ void load_row32(const __nv_bfloat16* base, int64_t ld, int row, int col0, int ncols,
                                           float* v) {
  const __nv_bfloat16* p = base + (int64_t)row * ld + col0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (col0 + q * 8 < ncols) {
      unpack8(*reinterpret_cast<const uint4*>(p + q * 8), v + q * 8);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[q * 8 + e] = 0.f;
    }
  }
}

// Direct store of 32 values at (row, col0..col0+31).  SYM: only elements with
// col >= row are stored (the upper triangle incl. the diagonal).
template <bool SYM>
__device__ __forceinline__ void store_row32(__nv_bfloat16* base, int64_t ld, int row, int col0, int ncols,
                                            const float* v) {
  __nv_bfloat16* p = base + (int64_t)row * ld + col0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int c8 = col0 + q * 8;
    if (c8 >= ncols) continue;
    if (!SYM || c8 >= row) {
      *reinterpret_cast<uint4*>(p + q * 8) = pack8(v + q * 8);
    } else if (c8 + 7 >= row) {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (c8 + e >= row && c8 + e < ncols) p[q * 8 + e] = __float2bfloat16_rn(v[q * 8 + e]);
    }
  }
}

// Transposed store through the warp's smem scratch: the warp holds rows
// [rbase, rbase+32) x columns [col0, col0+32); lane L writes row col0+L of the
// target, columns [rbase, rbase+32).  SYM: only source elements with row < col
// (their mirror lies strictly below the diagonal).  nrows/ncols bound the
// source tile; the caller guarantees col0 < ncols.
template <bool SYM>
__device__ __forceinline__ void store_transposed32(__nv_bfloat16* scratch, __nv_bfloat16* base, int64_t ld,
                                                   int rbase, int col0, int nrows, int ncols, const float* v,
                                                   int lane) {
#pragma unroll
  for (int q = 0; q < 32; ++q) scratch[q * kEpiPitch + lane] = __float2bfloat16_rn(v[q]);
  __syncwarp();
  const int trow = col0 + lane;          // target row = source column
  if (trow < ncols) {
    __nv_bfloat16* p = base + (int64_t)trow * ld + rbase;
    const __nv_bfloat16* s = scratch + lane * kEpiPitch;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r8 = rbase + q * 8;      // source rows r8..r8+7
      if (r8 >= nrows) continue;
      const bool full = !SYM || (r8 + 7 < trow);
      if (full) {
        *reinterpret_cast<uint4*>(p + q * 8) = *reinterpret_cast<const uint4*>(s + q * 8);
      } else if (r8 < trow) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (r8 + e < trow && r8 + e < nrows) p[q * 8 + e] = s[q * 8 + e];
      }
    }
  }
  __syncwarp();
}

template <int PHASE>
__device__ __forceinline__ void epilogue_chunk(const GemmParams& p, const GemmProblem& pr, int mat, int row,
                                               int rbase, int col0, float* v, __nv_bfloat16* scratch,
                                               int lane) {
  const int gm = pr.mat_base + mat;
  const bool row_ok = row < pr.M;
  if (PHASE == kGram) {
    float s2 = 1.f;
    if (p.first) {
      const float s = p.sigma[gm];
      s2 = s * s;
    }
#pragma unroll
    for (int q = 0; q < 32; ++q) v[q] *= s2;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(pr.out) + (int64_t)mat * pr.ms_out;
    if (row_ok) store_row32<true>(out, pr.ld_out, row, col0, pr.N, v);
    store_transposed32<true>(scratch, out, pr.ld_out, rbase, col0, pr.M, pr.N, v, lane);
  } else if (PHASE == kPoly) {
    float a[32];
    const __nv_bfloat16* aux = reinterpret_cast<const __nv_bfloat16*>(pr.aux) + (int64_t)mat * pr.ms_aux;
    if (row_ok) {
      load_row32(aux, pr.ld_aux, row, col0, pr.N, a);
    } else {
#pragma unroll
      for (int q = 0; q < 32; ++q) a[q] = 0.f;
    }
#pragma unroll
    for (int q = 0; q < 32; ++q) v[q] = fmaf(p.b, a[q], p.c * v[q]);
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(pr.out) + (int64_t)mat * pr.ms_out;
    if (row_ok) store_row32<true>(out, pr.ld_out, row, col0, pr.N, v);
    store_transposed32<true>(scratch, out, pr.ld_out, rbase, col0, pr.M, pr.N, v, lane);
  } else {
    // X_new = s * (a X + acc)
    float x[32];
    const __nv_bfloat16* aux = reinterpret_cast<const __nv_bfloat16*>(pr.aux) + (int64_t)mat * pr.ms_aux;
    if (row_ok) {
      load_row32(aux, pr.ld_aux, row, col0, pr.N, x);
    } else {
#pragma unroll
      for (int q = 0; q < 32; ++q) x[q] = 0.f;
    }
    const float s = p.first ? p.sigma[gm] : 1.f;
#pragma unroll
    for (int q = 0; q < 32; ++q) v[q] = s * fmaf(p.a, x[q], v[q]);
    if (PHASE == kUpdate) {
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(pr.out) + (int64_t)mat * pr.ms_out;
      if (row_ok) store_row32<false>(out, pr.ld_out, row, col0, pr.N, v);
      __nv_bfloat16* outt = reinterpret_cast<__nv_bfloat16*>(pr.out_t) + (int64_t)mat * pr.ms_out_t;
      store_transposed32<false>(scratch, outt, pr.ld_out_t, rbase, col0, pr.M, pr.N, v, lane);
    } else {
      // apply: the output orientation is the parameter's rows x cols layout
      if (!row_ok) return;
      const MatInfo mi = p.mats[gm];
      const int64_t wrow = mi.w_off + (int64_t)row * mi.cols;
      float* W = p.W + wrow + col0;
      const float lrs = mi.lrs;
      if (mi.vec_ok && col0 + 32 <= pr.N) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 w = *reinterpret_cast<const float4*>(W + 4 * q);
          float d0 = lrs * v[4 * q], d1 = lrs * v[4 * q + 1], d2 = lrs * v[4 * q + 2], d3 = lrs * v[4 * q + 3];
          w.x -= d0; w.y -= d1; w.z -= d2; w.w -= d3;
          *reinterpret_cast<float4*>(W + 4 * q) = w;
          v[4 * q] = w.x; v[4 * q + 1] = w.y; v[4 * q + 2] = w.z; v[4 * q + 3] = w.w;
          if (p.dbg) *reinterpret_cast<float4*>(p.dbg + wrow + col0 + 4 * q) = make_float4(d0, d1, d2, d3);
        }
        if (p.Wb) {
          __nv_bfloat16* wb = reinterpret_cast<__nv_bfloat16*>(p.Wb) + wrow + col0;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 pk = pack8(v + 8 * q);
            // 8-byte stores: wrow + col0 is a multiple of 4 elements
            reinterpret_cast<uint2*>(wb + 8 * q)[0] = make_uint2(pk.x, pk.y);
            reinterpret_cast<uint2*>(wb + 8 * q)[1] = make_uint2(pk.z, pk.w);
          }
        }
      } else {
        for (int q = 0; q < 32; ++q) {
          if (col0 + q >= pr.N) break;
          const float d = lrs * v[q];
          const float w = W[q] - d;
          W[q] = w;
          if (p.dbg) p.dbg[wrow + col0 + q] = d;
          if (p.Wb) reinterpret_cast<__nv_bfloat16*>(p.Wb)[wrow + col0 + q] = __float2bfloat16_rn(w);
        }
      }
    }
  }
}

template <int PHASE>
__global__ void __launch_bounds__(kThreads, 1) ns_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem sm = carve(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort = sm.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.tfull[i], 1);
      mbar_init(&sm.tempty[i], 128);
    }
    mbar_init(sm.drain, 1);
    *sm.abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(sm.tmem_holder, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_holder;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      for (int i = 0; i < p.n_prob; ++i) {
        tma_prefetch_desc(&p.tmA[i]);
        tma_prefetch_desc(&p.tmB[i]);
      }
    }
    uint32_t stage = 0, phase = 0, issued = 0;
    uint32_t last_par[kStages] = {0, 0, 0, 0};
    bool ok = true;
    for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x) {
      const int4 tl = p.tiles[t];
      const int nk = ceil_div(p.prob[tl.x].K, kBK);
      const CUtensorMap* ma = &p.tmA[tl.x];
      const CUtensorMap* mb = &p.tmB[tl.x];
      for (int kb = 0; kb < nk; ++kb) {
        bool w = true;
        if (lane == 0) {
          w = mbar_wait(&sm.empty[stage], phase ^ 1u, abort, p.status, p.timeout_ns);
          if (w) {
            mbar_arrive_expect_tx(&sm.full[stage], kStageBytesA + kStageBytesB);
            tma_load_3d(sm.a[stage], ma, &sm.full[stage], kb * kBK, tl.z * kBM, tl.y);
            tma_load_3d(sm.b[stage], mb, &sm.full[stage], kb * kBK, tl.w * kBN, tl.y);
            issued |= 1u << stage;
            last_par[stage] = phase;
          }
        }
        if (!__shfl_sync(0xffffffffu, (int)w, 0)) {
          ok = false;
          break;
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // every issued copy must land before the CTA may exit
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if (issued & (1u << s)) mbar_wait(&sm.full[s], last_par[s], nullptr, p.status, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x) {
      const int4 tl = p.tiles[t];
      const int nk = ceil_div(p.prob[tl.x].K, kBK);
      bool w = true;
      if (lane == 0) w = mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, abort, p.status, p.timeout_ns);
      if (!__shfl_sync(0xffffffffu, (int)w, 0)) break;
      tc_fence_after();
      const uint32_t d = tmem_base + acc * (uint32_t)kBN;
      for (int kb = 0; kb < nk; ++kb) {
        if (lane == 0) w = mbar_wait(&sm.full[stage], phase, abort, p.status, p.timeout_ns);
        if (!__shfl_sync(0xffffffffu, (int)w, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = smem_u32(sm.a[stage]);
          const uint32_t b0 = smem_u32(sm.b[stage]);
#pragma unroll
          for (int s = 0; s < kBK / 16; ++s) {
            umma_bf16(d, sdesc_kmajor_sw128(a0 + s * 32), sdesc_kmajor_sw128(b0 + s * 32), idesc,
                      (kb | s) != 0 ? 1u : 0u);
          }
          umma_commit(&sm.empty[stage]);
        }
        __syncwarp();
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(&sm.tfull[acc]);
      __syncwarp();
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    // wait until every issued MMA has completed (TMEM is released below)
    if (lane == 0) {
      umma_commit(sm.drain);
      mbar_wait(sm.drain, 0, nullptr, p.status, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int quad = warp & 3;                  // TMEM lane quarter this warp may access
    __nv_bfloat16* scratch = sm.epi + (warp - 2) * (32 * kEpiPitch);
    uint32_t acc = 0, acc_phase = 0;
    for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x) {
      const int4 tl = p.tiles[t];
      const bool w = mbar_wait(&sm.tfull[acc], acc_phase, abort, p.status, p.timeout_ns);
      if (!__all_sync(0xffffffffu, w)) break;
      tc_fence_after();
      const GemmProblem& pr = p.prob[tl.x];
      const int rbase = tl.z * kBM + quad * 32;
      const int row = rbase + lane;
      for (int ch = 0; ch < kBN / 32; ++ch) {
        const int col0 = tl.w * kBN + ch * 32;
        if (col0 >= pr.N) break;
        float v[32];
        tmem_ld32(tmem_base + acc * (uint32_t)kBN + ch * 32 + ((uint32_t)(quad * 32) << 16), v);
        epilogue_chunk<PHASE>(p, pr, tl.y, row, rbase, col0, v, scratch, lane);
      }
      tc_fence_before();
      mbar_arrive(&sm.tempty[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int PHASE>
cudaError_t launch_phase(const GemmParams& p, int grid, cudaStream_t s) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(ns_gemm_kernel<PHASE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  ns_gemm_kernel<PHASE><<<grid, kThreads, kGemmSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ns_gemm(int phase, const GemmParams& p, int grid, cudaStream_t s) {
  if (p.n_tiles <= 0) return cudaSuccess;
  if (grid > p.n_tiles) grid = p.n_tiles;
  switch (phase) {
    case kGram: return launch_phase<kGram>(p, grid, s);
    case kPoly: return launch_phase<kPoly>(p, grid, s);
    case kUpdate: return launch_phase<kUpdate>(p, grid, s);
    case kApply: return launch_phase<kApply>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

int gemm_max_grid() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return sms > 0 ? sms : 1;
}

}  // namespace cz
