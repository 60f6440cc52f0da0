// Newton-Schulz for small matrices, entirely on chip (sm_103a).
//
// A matrix whose Newton-Schulz orientation X (m x n, m = min(rows, cols)) has
// m <= 128 and n <= 256 is handled by one CTA from the first Gram product to the
// apply: X, A and B' live in shared memory as 128-byte-swizzled bf16 operands,
// the three accumulators live in TMEM, and nothing but the starting X (written
// by the momentum pass) and the parameter itself is touched in global memory.  Per step (Canzona summary page, section 2, the
// Muon update with its quintic Newton-Schulz iteration):
//   Gram    A  = s^2 X X^T                 M = 128, N = 128, K = n_pad   (TMEM cols   0..127)
//   Poly    B' = a I + b A + c A A         M = 128, N = 128, K = 128     (TMEM cols 128..255)
//   Update  X <- s B' X                    M = 128, N = n_pad, K = 128   (TMEM cols 256..)
// X is stored once, rows of 64 consecutive columns (128 bytes): read K-major by
// the Gram product (K = n) and MN-major by the Update (N = n, K = m), so no X^T
// is formed.
// with s = 1/(||u||_F + eps) in step 1 and 1 afterwards, the same folding and
// the same bf16 rounding points as the tiled kernels.  Rows m..127 and columns
// n..n_pad-1 are zero and stay zero (B' is a on the padded diagonal, applied to
// zero rows).  The last step writes W <- W - lr*sqrt(max(1, rows/cols)) * X_K,
// the bf16 copy and the optional debug delta, staged through shared memory so
// the parameter is read and written along its rows.
//
// 128 threads: thread t owns TMEM lane t (row t of every accumulator); thread 0
// also issues the tcgen05.mma.  One CTA per matrix, one launch for all of them.

#include <cuda_bf16.h>

#include "ptx.cuh"
#include "step_kernels.h"

namespace cz {

namespace {

constexpr int kSmThreads = 128;
constexpr int kBlk = 128 * 128;                               // one 64-wide K block of 128 rows, bytes
constexpr int kOffX = 0;                                      // X: 128 rows x n_pad columns
constexpr int kOffA = kOffX + (kSmallMaxN / 64) * kBlk;       // A: 128 rows, K = 128
constexpr int kOffB = kOffA + 2 * kBlk;                       // B': 128 rows, K = 128
// The fp32 apply staging (m rows x (n_pad + 1) floats) reuses X, A and B' (all
// consumed by then) and a little slack behind them.
constexpr int kStageEnd = kSmallMaxM * (kSmallMaxN + 1) * 4;
constexpr int kOffBar = ((kOffB + 2 * kBlk > kStageEnd ? kOffB + 2 * kBlk : kStageEnd) + 1023) & ~1023;
constexpr int kSmallSmemBytes = 1024 /*align slack*/ + kOffBar + 64;
constexpr uint32_t kSmallTmemCols = 512;
constexpr int64_t kSmallDrainNs = 2000000000LL;
static_assert(kSmallSmemBytes <= 227 * 1024, "shared memory");

// Byte offset of element (row, k) in a K-major operand of `rows` rows stored as
// 64-wide K blocks of rows x 128 bytes with the 128-byte swizzle (16-byte chunk
// index XOR row % 8), the layout TMA writes and the UMMA descriptor reads.
__device__ __forceinline__ uint32_t sw128(int rows, int row, int k) {
  return (uint32_t)((k >> 6) * rows * 128 + row * 128 + ((((k >> 3) & 7) ^ (row & 7)) << 4) + ((k & 7) << 1));
}

// Keeps the first `keep` (1..7) bf16 of a 16-byte chunk, zeroes the rest.
__device__ __forceinline__ uint4 keep_first(uint4 v, int keep) {
  auto m = [keep](int e0) -> uint32_t {
    return e0 + 1 < keep ? 0xFFFFFFFFu : (e0 < keep ? 0x0000FFFFu : 0u);
  };
  return make_uint4(v.x & m(0), v.y & m(2), v.z & m(4), v.w & m(6));
}

__global__ void __launch_bounds__(kSmThreads, 1) ns_small_kernel(const SmallParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + kOffBar);
  uint32_t* holder = reinterpret_cast<uint32_t*>(base + kOffBar + 8);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const SmallMat sm = p.mats[blockIdx.x];
  const int m = sm.m, n = sm.n;
  const int n_pad = (n + 63) & ~63;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(holder, kSmallTmemCols);

  // starting X (m x n), zero padded to 128 x n_pad;
  // 8 chunks per thread in flight (all loads of a batch before its smem stores)
  constexpr int kBatch = 8;
  const int xch = n_pad >> 3;
  for (int i0 = tid; i0 < kSmallMaxM * xch; i0 += kSmThreads * kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * kSmThreads;
      const int r = i / xch, k0 = (i - r * xch) * 8;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (i < kSmallMaxM * xch && r < m && k0 < n) {
        v[u] = *reinterpret_cast<const uint4*>(sm.x + (int64_t)r * sm.ldx + k0);   // pitch ldx: n rounded to 8
        if (k0 + 8 > n) v[u] = keep_first(v[u], n - k0);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * kSmThreads;
      const int r = i / xch, k0 = (i - r * xch) * 8;
      if (i < kSmallMaxM * xch) *reinterpret_cast<uint4*>(base + kOffX + sw128(kSmallMaxM, r, k0)) = v[u];
    }
  }
  {
    // the parameter is read only by the apply at the end: bring it into L2 now
    const MatInfo& wi = p.info[sm.mat];
    const char* w0 = reinterpret_cast<const char*>(p.W + wi.w_off);
    const int64_t bytes = (int64_t)wi.rows * wi.cols * 4;
    for (int64_t o = (int64_t)tid * 128; o < bytes; o += (int64_t)kSmThreads * 128)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(w0 + o));
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = *holder;
  const uint32_t lrow = (uint32_t)(warp * 32) << 16;     // this warp's TMEM lane quarter
  const uint32_t tA = tmem, tP = tmem + 128, tX = tmem + 256;
  const uint32_t sX = smem_u32(base + kOffX);
  const uint32_t sA = smem_u32(base + kOffA), sB = smem_u32(base + kOffB);
  const float sg = p.sigma[sm.mat];
  const MatInfo mi = p.info[sm.mat];
  uint32_t ph = 0;
  bool ok = true;

  for (int it = 0; it < p.ns_steps; ++it) {
    const bool first = it == 0, last = it + 1 == p.ns_steps;
    // ---------------------------------------------------------------- Gram
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16_f32(128, 128);
      for (int kb = 0; kb < (n_pad >> 6); ++kb)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t d = sdesc_kmajor_sw128(sX + kb * kBlk + 32 * k);
          umma_bf16(tA, d, d, id, (kb | k) != 0);
        }
      umma_commit(bar);
    }
    ok = __syncthreads_and(mbar_wait(bar, ph, nullptr, p.status, p.timeout_ns));
    if (!ok) break;
    ph ^= 1;
    tc_fence_after();
    {
      const float s2 = first ? sg * sg : 1.f;
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        float v[32];
        tmem_ld32(tA + lrow + 32 * j, v);
        if (first) {
#pragma unroll
          for (int q = 0; q < 32; ++q) v[q] *= s2;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(base + kOffA + sw128(128, tid, 32 * j + 8 * q)) = pack8(v + 8 * q);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---------------------------------------------------------------- Poly
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16_f32(128, 128);
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t d = sdesc_kmajor_sw128(sA + kb * kBlk + 32 * k);
          umma_bf16(tP, d, d, id, (kb | k) != 0);
        }
      umma_commit(bar);
    }
    ok = __syncthreads_and(mbar_wait(bar, ph, nullptr, p.status, p.timeout_ns));
    if (!ok) break;
    ph ^= 1;
    tc_fence_after();
#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
      float v[32], a[32];
      tmem_ld32(tP + lrow + 32 * j, v);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        unpack8(*reinterpret_cast<const uint4*>(base + kOffA + sw128(128, tid, 32 * j + 8 * q)), a + 8 * q);
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] = fmaf(p.b, a[q], p.c * v[q]) + ((32 * j + q == tid) ? p.a : 0.f);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(base + kOffB + sw128(128, tid, 32 * j + 8 * q)) = pack8(v + 8 * q);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---------------------------------------------------------------- Update
    if (tid == 0) {
      tc_fence_after();
      // B operand X, MN-major: 64-column blocks kBlk apart, 8-row groups 1024 apart;
      // each K = 16 step takes the next 16 rows (2048 bytes)
      const uint32_t id = idesc_bf16_f32_bmn(128, n_pad);
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_bf16(tX, sdesc_kmajor_sw128(sB + kb * kBlk + 32 * k),
                    sdesc_mnmajor_sw128(sX + (kb * 4 + k) * 2048, kBlk, 1024), id, (kb | k) != 0);
      umma_commit(bar);
    }
    ok = __syncthreads_and(mbar_wait(bar, ph, nullptr, p.status, p.timeout_ns));
    if (!ok) break;
    ph ^= 1;
    tc_fence_after();
    const float s = first ? sg : 1.f;
    if (!last) {
      // X of the next step
#pragma unroll 1
      for (int j = 0; j < (n_pad >> 5); ++j) {
        float v[32];
        tmem_ld32(tX + lrow + 32 * j, v);
        if (first) {
#pragma unroll
          for (int q = 0; q < 32; ++q) v[q] *= s;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(base + kOffX + sw128(kSmallMaxM, tid, 32 * j + 8 * q)) = pack8(v + 8 * q);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
    } else {
      // apply: delta = lrs * s * X_K staged as fp32 rows of pitch n_pad + 1 (odd:
      // conflict-free both along rows and down columns), then W updated along its rows
      float* S = reinterpret_cast<float*>(base);
      const int pitch = n_pad + 1;
      const float lrs = lr_times_scale(p.lr_dev ? __ldg(p.lr_dev) : p.lr, mi.scale);
#pragma unroll 1
      for (int j = 0; j < (n_pad >> 5); ++j) {
        float v[32];
        tmem_ld32(tX + lrow + 32 * j, v);
        if (tid < m) {
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            if (first) v[q] *= s;
            S[tid * pitch + 32 * j + q] = lrs * v[q];
          }
        }
      }
      tc_fence_before();
      __syncthreads();
      // 8 rows per lane in flight: the loads of a batch are issued before any store
      const bool tall = mi.rows > mi.cols;
      constexpr int kRowsInFlight = 8;
      constexpr int kWarps = kSmThreads / 32;
      for (int pr0 = warp; pr0 < mi.rows; pr0 += kWarps * kRowsInFlight) {
        for (int pc = lane; pc < mi.cols; pc += 32) {
          float w[kRowsInFlight];
#pragma unroll
          for (int u = 0; u < kRowsInFlight; ++u) {
            const int pr = pr0 + u * kWarps;
            if (pr < mi.rows) w[u] = p.W[mi.w_off + (int64_t)pr * mi.cols + pc];
          }
#pragma unroll
          for (int u = 0; u < kRowsInFlight; ++u) {
            const int pr = pr0 + u * kWarps;
            if (pr >= mi.rows) continue;
            const float d = tall ? S[pc * pitch + pr] : S[pr * pitch + pc];
            const int64_t idx = mi.w_off + (int64_t)pr * mi.cols + pc;
            const float wn = w[u] - d;
            p.W[idx] = wn;
            if (p.Wb) reinterpret_cast<__nv_bfloat16*>(p.Wb)[idx] = __float2bfloat16_rn(wn);
            if (p.dbg) p.dbg[idx] = d;
          }
        }
      }
    }
  }
  if (!ok) {
    // a product did not complete in time: wait (bounded) for it before TMEM is released
    mbar_wait(bar, ph, nullptr, nullptr, kSmallDrainNs);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kSmallTmemCols);
  }
}

}  // namespace

cudaError_t launch_ns_small(const SmallParams& p, cudaStream_t s) {
  if (p.n_mats <= 0) return cudaSuccess;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(ns_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmallSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  ns_small_kernel<<<p.n_mats, kSmThreads, kSmallSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace cz
