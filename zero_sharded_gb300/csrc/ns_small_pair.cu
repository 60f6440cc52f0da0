// Newton-Schulz for matrices of 128 < m <= 256, n <= 256, entirely on chip, on a
// CTA pair (sm_103a, tcgen05 cta_group::2).
//
// One matrix per cluster of two CTAs.  CTA q (its rank in the cluster) holds row
// half q of every m x m or m x n iterate (rows 128q .. 128q + 127, zero beyond m),
// and each product is one M = 256 pair MMA issued by CTA 0 that reads both CTAs'
// shared memory.  Per step (Canzona summary page, section 2, the Muon update with
// its quintic Newton-Schulz iteration), with s = 1/(||u||_F + eps) in step 1 and 1
// afterwards:
//   Gram    A  = s^2 X X^T         A operand X rows (K-major), B operand X rows again
//   Poly    B' = a I + b A + c A A A operand A rows, B operand A rows (A is symmetric)
//   Update  X <- s B' X            A operand B' rows, B operand X read MN-major
// In a pair MMA the B operand's N extent is split between the CTAs: for the Gram
// and the Poly product that is again the CTA's own row half (the outputs are
// symmetric), but the Update needs X split by COLUMNS (N = n).  So every CTA keeps
// two copies of X: its rows (Xr, K-major, read by the Gram product) and, for all
// m rows, its half of the columns (Xc, MN-major, read by the Update).  The Update's
// epilogue writes each new X row into the local Xr and, through distributed shared
// memory, into the Xc of the CTA that owns each column half.
// n is padded to 256 and m to 256 with zeros that stay zero (B' is a on the padded
// diagonal, applied to zero rows), so every product is 256 x 256 x 256.  The bf16
// rounding points, the K order of the accumulation and the apply's two roundings
// are those of the tiled kernels: the result is bit-identical to them.
//
// 256 threads per CTA: warp w reads TMEM lane quarter w % 4 (rows 128q + 32 (w % 4)
// .. + 31 of every accumulator) and column half w / 4, so the two warps of a lane
// quarter share each epilogue; thread 0 of CTA 0 also issues the MMAs.  Every wait is bounded, and
// a CTA whose wait failed still takes part in every cluster barrier (no early
// exit), so neither CTA can be left waiting for the other.

#include <cuda_bf16.h>

#include "ptx.cuh"
#include "step_kernels.h"

namespace cz {

namespace {

constexpr int kPThreads = 256;
constexpr int kPRows = 128;                                   // rows of an iterate per CTA
constexpr int kPN = 256;                                      // padded n (and m)
constexpr int kKBlk = kPRows * 128;                           // one 64-wide K block of 128 rows, bytes
constexpr int kCBlk = kPN * 128;                              // one 64-column block of Xc (256 rows), bytes
constexpr int kOffXr = 0;                                     // Xr: 128 rows x 256 columns, K-major
constexpr int kOffAB = kOffXr + (kPN / 64) * kKBlk;           // A, then B' in place: 128 rows, K = 256
constexpr int kOffXc = kOffAB + (kPN / 64) * kKBlk;           // Xc: 256 rows x 128 columns, MN-major
constexpr int kOffBar = kOffXc + 2 * kCBlk;                   // 196608
constexpr int kPairSmemBytes = 1024 /*align slack*/ + kOffBar + 64;
constexpr uint32_t kPairTmemCols = 512;                       // cols 0..255: Gram, Update; 256..511: Poly
constexpr int64_t kPairDrainNs = 2000000000LL;
constexpr int kStagePitch = kPN + 1;                          // fp32 apply staging, floats per row
static_assert(kPRows * kStagePitch * 4 <= kOffBar, "apply staging fits in the consumed operands");
static_assert(kPairSmemBytes <= 227 * 1024, "shared memory");

// Byte offset of element (row, k) of a 128-byte-swizzled operand stored as 64-wide
// blocks of `rows` rows x 128 bytes (16-byte chunk index XOR row % 8): the layout
// the UMMA descriptors read, K-major (k = K index) or MN-major (k = N index).
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

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Ends an epilogue: its shared-memory writes (local and remote) are made visible
// to the tensor cores of both CTAs before the next pair MMA is issued.
__device__ __forceinline__ void pair_handoff() {
  asm volatile("fence.proxy.async;" ::: "memory");
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
}

// Loads 128-row or 256-row slabs of the starting X (m x n, pitch ldx) into a
// swizzled operand, zero beyond m rows and n columns: rows [r0, r0 + rows),
// columns [c0, c0 + cols).  8 chunks per thread in flight.
__device__ __forceinline__ void load_x(uint8_t* dst, int rows_layout, const uint16_t* x, int ldx, int m, int n,
                                       int r0, int rows, int c0, int cols, int tid) {
  constexpr int kBatch = 8;
  const int xch = cols >> 3;
  const int total = rows * xch;
  for (int i0 = tid; i0 < total; i0 += kPThreads * kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * kPThreads;
      const int r = i / xch, k = (i - r * xch) * 8;
      const int gr = r0 + r, gk = c0 + k;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (i < total && gr < m && gk < n) {
        v[u] = *reinterpret_cast<const uint4*>(x + (int64_t)gr * ldx + gk);   // pitch ldx: n rounded to 8
        if (gk + 8 > n) v[u] = keep_first(v[u], n - gk);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * kPThreads;
      const int r = i / xch, k = (i - r * xch) * 8;
      if (i < total) *reinterpret_cast<uint4*>(dst + sw128(rows_layout, r, k)) = v[u];
    }
  }
}

__global__ void __launch_bounds__(kPThreads, 1) ns_small_pair_kernel(const SmallParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + kOffBar);         // products
  uint64_t* drain = reinterpret_cast<uint64_t*>(base + kOffBar + 8);    // error path: every issued MMA done
  uint32_t* holder = reinterpret_cast<uint32_t*>(base + kOffBar + 16);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t q = cluster_ctarank();
  const SmallMat sm = p.mats[blockIdx.x >> 1];
  const int m = sm.m, n = sm.n;
  const int row = (warp & 3) * 32 + lane;                     // this thread's row of the CTA's half
  const int grow = (int)q * kPRows + row;                     // ... of every iterate
  const int chalf = warp >> 2;                                // its column half (epilogues)

  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc_pair(holder, kPairTmemCols);

  // starting X: this CTA's rows (Xr) and, for all rows, its half of the columns (Xc)
  load_x(base + kOffXr, kPRows, sm.x, sm.ldx, m, n, (int)q * kPRows, kPRows, 0, kPN, tid);
  load_x(base + kOffXc, kPN, sm.x, sm.ldx, m, n, 0, kPN, (int)q * kPRows, kPRows, tid);
  const MatInfo mi = p.info[sm.mat];
  {
    // the parameter is read only by the apply at the end: bring this CTA's half into L2 now
    const char* w0 = reinterpret_cast<const char*>(p.W + mi.w_off);
    const int64_t bytes = (int64_t)mi.rows * mi.cols * 4;
    for (int64_t o = ((int64_t)q * kPThreads + tid) * 128; o < bytes; o += (int64_t)2 * kPThreads * 128)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(w0 + o));
  }
  fence_proxy_async_smem();
  tc_fence_before();
  cluster_sync();               // both CTAs' barriers, TMEM and operands exist before the first MMA
  tc_fence_after();

  const uint32_t tmem = *holder;
  const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16;    // this warp's TMEM lane quarter
  const uint32_t tA = tmem, tP = tmem + 256, tX = tmem;
  const uint32_t sXr = smem_u32(base + kOffXr), sAB = smem_u32(base + kOffAB), sXc = smem_u32(base + kOffXc);
  const float sg = p.sigma[sm.mat];
  const bool issuer = q == 0 && tid == 0;
  constexpr uint32_t kId = idesc_bf16_f32(256, kPN);
  constexpr uint32_t kIdMN = idesc_bf16_f32_bmn(256, kPN);
  uint32_t ph = 0;
  bool ok = true;

  // Waits for this CTA's half of the product just issued; false (the status word
  // records the timeout) if it did not complete in time.
  auto product_done = [&]() -> bool {
    const bool done = __syncthreads_and(ok && mbar_wait(bar, ph, nullptr, p.status, p.timeout_ns));
    if (done) ph ^= 1u;
    tc_fence_after();
    return done;
  };

  for (int it = 0; it < p.ns_steps; ++it) {
    const bool first = it == 0, last = it + 1 == p.ns_steps;
    // ---------------------------------------------------------------- Gram
    if (ok && issuer) {
#pragma unroll 1
      for (int kb = 0; kb < kPN / 64; ++kb)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t d = sdesc_kmajor_sw128(sXr + kb * kKBlk + 32 * k);
          umma_bf16_pair(tA, d, d, kId, (kb | k) != 0);
        }
      umma_commit_pair(bar, 0x3);
    }
    ok = product_done();
    if (ok) {
      const float s2 = first ? sg * sg : 1.f;
#pragma unroll 1
      for (int j = 4 * chalf; j < 4 * chalf + 4; ++j) {
        float v[32];
        tmem_ld32(tA + lrow + 32 * j, v);
        if (first) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= s2;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4*>(base + kOffAB + sw128(kPRows, row, 32 * j + 8 * i)) = pack8(v + 8 * i);
      }
    }
    pair_handoff();
    // ---------------------------------------------------------------- Poly
    if (ok && issuer) {
#pragma unroll 1
      for (int kb = 0; kb < kPN / 64; ++kb)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t d = sdesc_kmajor_sw128(sAB + kb * kKBlk + 32 * k);
          umma_bf16_pair(tP, d, d, kId, (kb | k) != 0);
        }
      umma_commit_pair(bar, 0x3);
    }
    ok = product_done();
    if (ok) {
      // B' overwrites A in place: the product that read A (in both CTAs) is complete,
      // and each element is read and written by the same thread
#pragma unroll 1
      for (int j = 4 * chalf; j < 4 * chalf + 4; ++j) {
        float v[32], a[32];
        tmem_ld32(tP + lrow + 32 * j, v);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          unpack8(*reinterpret_cast<const uint4*>(base + kOffAB + sw128(kPRows, row, 32 * j + 8 * i)), a + 8 * i);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = fmaf(p.b, a[i], p.c * v[i]) + ((32 * j + i == grow) ? p.a : 0.f);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4*>(base + kOffAB + sw128(kPRows, row, 32 * j + 8 * i)) = pack8(v + 8 * i);
      }
    }
    pair_handoff();
    // ---------------------------------------------------------------- Update
    if (ok && issuer) {
      // B operand Xc, MN-major: 64-column blocks kCBlk apart, 8-row groups 1024 apart;
      // each K = 16 step takes the next 16 rows (2048 bytes)
#pragma unroll 1
      for (int kb = 0; kb < kPN / 64; ++kb)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_bf16_pair(tX, sdesc_kmajor_sw128(sAB + kb * kKBlk + 32 * k),
                         sdesc_mnmajor_sw128(sXc + (kb * 4 + k) * 2048, kCBlk, 1024), kIdMN, (kb | k) != 0);
      umma_commit_pair(bar, 0x3);
    }
    ok = product_done();
    const float s = first ? sg : 1.f;
    if (!last) {
      if (ok) {
        // X of the next step: this CTA's rows into Xr, and the thread's column half
        // of them into the Xc of the CTA that owns that half (both Xc were read by
        // the product just completed)
        const uint32_t xc = mapa_shared(sXc, (uint32_t)chalf);
#pragma unroll 1
        for (int j = 4 * chalf; j < 4 * chalf + 4; ++j) {
          float v[32];
          tmem_ld32(tX + lrow + 32 * j, v);
          if (first) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= s;
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int col = 32 * j + 8 * i;
            const uint4 w = pack8(v + 8 * i);
            *reinterpret_cast<uint4*>(base + kOffXr + sw128(kPRows, row, col)) = w;
            st_cluster_v4(xc + sw128(kPN, grow, col & (kPRows - 1)), w);
          }
        }
      }
      pair_handoff();
    } else {
      // apply: delta = lrs * s * X_K staged as fp32 rows of pitch 257 (odd: conflict-free
      // both along rows and down columns), then W updated along its rows.  Only this
      // CTA's operands are overwritten, and the peer no longer reads them.
      float* S = reinterpret_cast<float*>(base);
      if (ok) {
        const float lrs = lr_times_scale(p.lr_dev ? __ldg(p.lr_dev) : p.lr, mi.scale);
#pragma unroll 1
        for (int j = 4 * chalf; j < 4 * chalf + 4; ++j) {
          float v[32];
          tmem_ld32(tX + lrow + 32 * j, v);
          if (grow < m) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (first) v[i] *= s;
              S[row * kStagePitch + 32 * j + i] = lrs * v[i];
            }
          }
        }
      }
      tc_fence_before();
      __syncthreads();
      if (ok) {
        // this CTA's rows of X are rows of W (wide) or columns of W (tall)
        const bool tall = mi.rows > mi.cols;
        const int lo = (int)q * kPRows, hi = min(m, lo + kPRows);
        const int r_lo = tall ? 0 : lo, r_hi = tall ? mi.rows : hi;
        const int c_lo = tall ? lo : 0, c_hi = tall ? hi : mi.cols;
        constexpr int kRowsInFlight = 8;
        constexpr int kWarps = kPThreads / 32;
        for (int pr0 = r_lo + warp; pr0 < r_hi; pr0 += kWarps * kRowsInFlight) {
          for (int pc = c_lo + lane; pc < c_hi; pc += 32) {
            float w[kRowsInFlight];
#pragma unroll
            for (int u = 0; u < kRowsInFlight; ++u) {
              const int pr = pr0 + u * kWarps;
              if (pr < r_hi) w[u] = p.W[mi.w_off + (int64_t)pr * mi.cols + pc];
            }
#pragma unroll
            for (int u = 0; u < kRowsInFlight; ++u) {
              const int pr = pr0 + u * kWarps;
              if (pr >= r_hi) continue;
              const float d = tall ? S[(pc - lo) * kStagePitch + pr] : S[(pr - lo) * kStagePitch + pc];
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
  }
  if (!ok && issuer) {
    // a product did not complete in time: wait (bounded) for every issued MMA before
    // TMEM is released
    umma_commit_pair(drain, 0x1);
    mbar_wait(drain, 0, nullptr, nullptr, kPairDrainNs);
  }
  tc_fence_before();
  cluster_sync();               // the pair MMAs (which read both CTAs' shared memory) are done
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kPairTmemCols);
  }
}

}  // namespace

cudaError_t launch_ns_small_pair(const SmallParams& p, cudaStream_t s) {
  if (p.n_mats <= 0) return cudaSuccess;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(ns_small_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.n_mats, 1, 1);
  cfg.blockDim = dim3(kPThreads, 1, 1);
  cfg.dynamicSmemBytes = kPairSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ns_small_pair_kernel, p);
}

}  // namespace cz
