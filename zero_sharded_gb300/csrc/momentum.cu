// Momentum pass of the Muon step: one streaming kernel over the owned tensors.
//
// Per element:  m <- mu*m + g  (fp32, stored);  u = g + mu*m  (Nesterov) or u = m;
// u is written as bf16 in the Newton-Schulz orientation X (min x max): as is for
// a wide tensor, transposed (through shared memory) for a tall one; and sum(u^2)
// is reduced per tensor for the Frobenius
// normalisation, deterministically (fixed shuffle tree per tile, then a
// fixed-order per-tensor sum of the tile partials in double), so results do not
// depend on timing.  The per-tensor sum is done by whichever block finishes the
// tensor's last tile (a per-tensor arrival counter), inside the same launch.
//
// HBM traffic per element: read g (4 or 2 B) and m (4 B), write m (4 B) and the
// bf16 copy (2 B).

#include <cuda_bf16.h>

#include "ptx.cuh"
#include "step_kernels.h"

namespace cz {

namespace {

constexpr int kTileRows = 64;
constexpr int kThreads = 256;
constexpr int kTrPitch = 65;   // odd pitch: the transposed smem writes are bank-conflict free

// NQ consecutive gradient values at idx as floats (q >= n_ok: 0).
template <int NQ>
__device__ __forceinline__ void load_grad(const void* grad, int64_t idx, bool bf16, bool vec, int n_ok, float* g) {
  if (bf16) {
    const __nv_bfloat16* gp = static_cast<const __nv_bfloat16*>(grad) + idx;
    if (vec) {
      if constexpr (NQ == 8) {
        const uint4 raw = *reinterpret_cast<const uint4*>(gp);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) { g[2 * k] = bf16_lo(w[k]); g[2 * k + 1] = bf16_hi(w[k]); }
      } else {
        const uint2 raw = *reinterpret_cast<const uint2*>(gp);
        g[0] = bf16_lo(raw.x); g[1] = bf16_hi(raw.x);
        g[2] = bf16_lo(raw.y); g[3] = bf16_hi(raw.y);
      }
    } else {
#pragma unroll
      for (int q = 0; q < NQ; ++q) g[q] = q < n_ok ? __bfloat162float(gp[q]) : 0.f;
    }
  } else {
    const float* gp = static_cast<const float*>(grad) + idx;
    if (vec) {
#pragma unroll
      for (int k = 0; k < NQ / 4; ++k) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(gp) + k);
        g[4 * k] = v.x; g[4 * k + 1] = v.y; g[4 * k + 2] = v.z; g[4 * k + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < NQ; ++q) g[q] = q < n_ok ? gp[q] : 0.f;
    }
  }
}

// One block per tile of 64 rows x CW columns of one owned tensor: 16 threads per
// row, NQ = CW/16 consecutive columns each, four passes of 16 rows.  CW = 128: a
// thread moves 8 columns per row, so each pass keeps 48 (bf16 gradients) or 64
// (fp32) bytes in flight per thread (measured: 64 x 64 tiles were 4% slower with
// fp32 gradients, 11% with bf16).
// At most 32 registers a thread (no spills): eight blocks per SM (six, at 40
// registers, measured 8% slower with bf16 gradients).
template <int CW>
__global__ void __launch_bounds__(kThreads, 8) momentum_kernel(const MomParams p) {
  constexpr int NQ = CW / 16;
  __shared__ __nv_bfloat16 trT[CW * kTrPitch];   // trT[c][r]: the tile, transposed
  __shared__ float warp_sum[kThreads / 32];

  const MomTile t = p.tiles[blockIdx.x];
  const MomMat mm = p.mats[t.mat];
  const int tid = threadIdx.x;
  const bool row_vec = ((mm.off % NQ) == 0) && ((mm.cols % NQ) == 0);
  const int cq = (tid & 15) * NQ;
  const int rsub = tid >> 4;
  const float mu = p.mu;
  float ss = 0.f;

#pragma unroll
  for (int pass = 0; pass < kTileRows / 16; ++pass) {
    const int r = rsub + pass * 16;
    const int gr = t.r0 + r;
    const int gc = t.c0 + cq;
    float u[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) u[q] = 0.f;
    if (gr < mm.rows && gc < mm.cols) {
      const int n_ok = min(NQ, mm.cols - gc);
      const int64_t idx = mm.off + (int64_t)gr * mm.cols + gc;
      const bool vec = row_vec && n_ok == NQ;
      float g[NQ], m[NQ];
      load_grad<NQ>(p.grad, idx, p.grad_bf16 != 0, vec, n_ok, g);
      float* mp = p.mom + idx;
      if (vec) {
#pragma unroll
        for (int k = 0; k < NQ / 4; ++k) {
          const float4 v = reinterpret_cast<const float4*>(mp)[k];
          m[4 * k] = v.x; m[4 * k + 1] = v.y; m[4 * k + 2] = v.z; m[4 * k + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < NQ; ++q) m[q] = q < n_ok ? mp[q] : 0.f;
      }
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const float mn = __fadd_rn(__fmul_rn(mu, m[q]), g[q]);
        m[q] = mn;
        u[q] = p.nesterov ? __fadd_rn(g[q], __fmul_rn(mu, mn)) : mn;
        if (q >= n_ok) u[q] = 0.f;
      }
      if (vec) {
#pragma unroll
        for (int k = 0; k < NQ / 4; ++k)
          reinterpret_cast<float4*>(mp)[k] = make_float4(m[4 * k], m[4 * k + 1], m[4 * k + 2], m[4 * k + 3]);
      } else {
        for (int q = 0; q < n_ok; ++q) mp[q] = m[q];
      }
      // rows x cols orientation; a partial tail vector lands in the row padding
      // (the pitch is the column count rounded up to 8)
      if (mm.direct) {
        uint16_t* xp = mm.direct + (int64_t)gr * mm.ld_direct + gc;
        if constexpr (NQ == 8)
          *reinterpret_cast<uint4*>(xp) = make_uint4(pack_bf16x2(u[0], u[1]), pack_bf16x2(u[2], u[3]),
                                                     pack_bf16x2(u[4], u[5]), pack_bf16x2(u[6], u[7]));
        else
          *reinterpret_cast<uint2*>(xp) = make_uint2(pack_bf16x2(u[0], u[1]), pack_bf16x2(u[2], u[3]));
      }
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      ss = fmaf(u[q], u[q], ss);
      trT[(cq + q) * kTrPitch + r] = __float2bfloat16_rn(u[q]);
    }
  }
  __syncthreads();
  // transposed orientation: rows of u^T are columns of the tile; 16 threads per
  // u^T row, 4 tile rows (8 bytes) each
#pragma unroll
  for (int pass = 0; pass < CW / 16; ++pass) {
    const int c = rsub + pass * 16;
    const int rq = (tid & 15) * 4;
    const int gc = t.c0 + c;
    const int gr = t.r0 + rq;
    if (mm.trans && gc < mm.cols && gr < mm.rows) {
      const __nv_bfloat16* s = trT + c * kTrPitch + rq;
      __nv_bfloat162 lo = __halves2bfloat162(s[0], s[1]);
      __nv_bfloat162 hi = __halves2bfloat162(s[2], s[3]);
      uint2 v;
      v.x = *reinterpret_cast<uint32_t*>(&lo);
      v.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(mm.trans + (int64_t)gc * mm.ld_trans + gr) = v;
    }
  }

  // deterministic block reduction of sum(u^2)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) warp_sum[tid >> 5] = ss;
  __syncthreads();
  __shared__ int last;
  if (tid == 0) {
    float s = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) s += warp_sum[w];
    p.partial[blockIdx.x] = s;
    // arrival with acq_rel at GPU scope: this partial is visible before the count
    // moves, and the last arrival sees every other tile's partial
    int prev;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(p.tile_done + t.mat) : "memory");
    last = prev == mm.tile_count - 1;
  }
  __syncthreads();
  if (last) {
    // every tile of the tensor has arrived (the barrier orders these reads after
    // thread 0's acquire): sigma = 1 / (||u||_F + eps) from the tile partials,
    // summed in double in a fixed order: thread-strided with 4 loads in flight,
    // shuffle tree per warp, warps in index order
    __shared__ double wsum[kThreads / 32];
    double d = 0.0;
    for (int i0 = tid; i0 < mm.tile_count; i0 += 4 * kThreads) {
      float v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + q * kThreads;
        v[q] = i < mm.tile_count ? __ldcg(p.partial + mm.tile_first + i) : 0.f;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) d += (double)v[q];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if ((tid & 31) == 0) wsum[tid >> 5] = d;
    __syncthreads();
    if (tid == 0) {
      double tot = 0.0;
      for (int w = 0; w < kThreads / 32; ++w) tot += wsum[w];
      p.sigma[t.mat] = (float)(1.0 / (sqrt(tot) + (double)p.eps));
      p.tile_done[t.mat] = 0;                               // ready for the next launch
    }
  }
}

}  // namespace

// A step program's tables, copied from page-locked host memory: 16-byte loads
// over the host link with kTablesVec in flight per thread.  The copy is
// latency-bound (a few hundred KB); with every load issued before the first
// store it takes about one round trip.
constexpr int kTablesVec = 4;

__global__ void __launch_bounds__(kThreads) tables_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                               int64_t n) {
  const int64_t i0 = (int64_t)blockIdx.x * (kThreads * kTablesVec) + threadIdx.x;
  uint4 v[kTablesVec];
#pragma unroll
  for (int q = 0; q < kTablesVec; ++q) {
    const int64_t i = i0 + (int64_t)q * kThreads;
    if (i < n) v[q] = src[i];
  }
#pragma unroll
  for (int q = 0; q < kTablesVec; ++q) {
    const int64_t i = i0 + (int64_t)q * kThreads;
    if (i < n) dst[i] = v[q];
  }
}

cudaError_t launch_tables_copy(const void* src, void* dst, int64_t bytes, cudaStream_t s) {
  if (bytes <= 0) return cudaSuccess;
  if ((bytes & 15) || (reinterpret_cast<uintptr_t>(src) & 15) || (reinterpret_cast<uintptr_t>(dst) & 15))
    return cudaErrorInvalidValue;
  const int64_t n = bytes >> 4;
  const int64_t per_block = (int64_t)kThreads * kTablesVec;
  const int64_t blocks = (n + per_block - 1) / per_block;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  tables_copy_kernel<<<(unsigned)blocks, kThreads, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n);
  return cudaGetLastError();
}

cudaError_t launch_momentum(const MomParams& p, cudaStream_t s) {
  if (p.n_tiles <= 0) return cudaSuccess;
  if (p.grad_bf16) momentum_kernel<kMomTileColsBf16><<<p.n_tiles, kThreads, 0, s>>>(p);
  else momentum_kernel<kMomTileCols><<<p.n_tiles, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace cz
