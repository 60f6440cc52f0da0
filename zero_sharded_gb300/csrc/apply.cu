// Standalone scale-and-apply of an update that is already in the parameters'
// layout (the apply the Muon step otherwise fuses into its last Newton-Schulz
// epilogue).
//
// Canzona summary page (paper-graph-ui), section 3.4: the update rule
// W_{t+1} = W_t - eta * MatrixOp(W_t, grad W_t) ("The Atomicity Constraint and
// Why Standard Approaches Fail"), and stage 4 of the TP micro-group lifecycle
// ("The TP Task Abstraction"): every rank adds the update shards it receives to
// its local parameter shards, P_local <- P_local + Delta W_local, a purely
// element-wise operation.
//
// Per tensor i (elements [off_i, off_i + rows_i*cols_i) of the flat buffers):
//   coef_i = lr * sqrt(max(1, rows_i/cols_i))   (or lr when shape_scale = 0),
//            computed in double and rounded to fp32 once, as the fused apply does;
//   d = fp32(coef_i * U);  W <- fp32(W - d);  bf16 copy = RNE(W)  (optional).
// Two roundings, written explicitly (no contraction), so that the result equals
// the fused apply's for the same delta.
//
// HBM traffic per element: read W 4 + U 4, write W 4 (+ bf16 copy 2).  One block
// per 4096-element chunk of one tensor; 16-byte vectors when the tensor's offset
// and the base pointers allow it, scalar accesses otherwise.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <stdint.h>
#include <utility>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "cz.h"

namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;
constexpr int kChunk = kThreads * kVecPerThread * 4;   // 4096 elements per block
constexpr int kMaxSeg = 256;                            // tensors per launch (kernel parameter space)

struct Segments {
  int64_t off[kMaxSeg];        // element offset of the tensor in the flat buffers
  int64_t n[kMaxSeg];          // its element count
  int32_t blk_first[kMaxSeg + 1];   // first block of each tensor (+ end)
  float coef[kMaxSeg];
  int32_t vec[kMaxSeg];        // 16-byte vector path allowed
  int32_t n_seg;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThreads) apply_kernel(float* __restrict__ W, __nv_bfloat16* __restrict__ Wb,
                                                         const float* __restrict__ U,
                                                         const __grid_constant__ Segments s) {
  // the tensor this block works on: the last segment whose first block <= blockIdx.x
  const int b = blockIdx.x;
  int lo = 0, hi = s.n_seg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.blk_first[mid] <= b) lo = mid; else hi = mid - 1;
  }
  const int seg = lo;
  const int64_t c0 = (int64_t)(b - s.blk_first[seg]) * kChunk;   // chunk start within the tensor
  const int64_t len = min((int64_t)kChunk, s.n[seg] - c0);
  const int64_t base = s.off[seg] + c0;
  const float coef = s.coef[seg];

  if (s.vec[seg]) {
    const int nv = (int)(len >> 2);
    float4 w[kVecPerThread], u[kVecPerThread];
#pragma unroll
    for (int q = 0; q < kVecPerThread; ++q) {
      const int j = threadIdx.x + q * kThreads;
      if (j < nv) {
        w[q] = *reinterpret_cast<const float4*>(W + base + 4 * j);
        u[q] = __ldcs(reinterpret_cast<const float4*>(U + base + 4 * j));
      }
    }
#pragma unroll
    for (int q = 0; q < kVecPerThread; ++q) {
      const int j = threadIdx.x + q * kThreads;
      if (j < nv) {
        float4 r;
        r.x = __fsub_rn(w[q].x, __fmul_rn(coef, u[q].x));
        r.y = __fsub_rn(w[q].y, __fmul_rn(coef, u[q].y));
        r.z = __fsub_rn(w[q].z, __fmul_rn(coef, u[q].z));
        r.w = __fsub_rn(w[q].w, __fmul_rn(coef, u[q].w));
        *reinterpret_cast<float4*>(W + base + 4 * j) = r;
        if (Wb)
          *reinterpret_cast<uint2*>(Wb + base + 4 * j) = make_uint2(pack_bf16x2(r.x, r.y), pack_bf16x2(r.z, r.w));
      }
    }
    // a ragged tail (fewer than 4 elements) at the tensor's end
    for (int64_t e = 4 * (int64_t)nv + threadIdx.x; e < len; e += kThreads) {
      const float r = __fsub_rn(W[base + e], __fmul_rn(coef, U[base + e]));
      W[base + e] = r;
      if (Wb) Wb[base + e] = __float2bfloat16_rn(r);
    }
  } else {
    for (int64_t e = threadIdx.x; e < len; e += kThreads) {
      const float r = __fsub_rn(W[base + e], __fmul_rn(coef, U[base + e]));
      W[base + e] = r;
      if (Wb) Wb[base + e] = __float2bfloat16_rn(r);
    }
  }
}

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CZ_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return CZ_ERR_CUDA;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return CZ_ERR_CUDA;
  if (major != 10 || minor != 3) return CZ_ERR_UNSUPPORTED;
  return CZ_OK;
}

}  // namespace

extern "C" int cz_apply_update(float* flat_param, void* param_bf16, const float* flat_update, const int64_t* offsets,
                               const int64_t* shapes, int64_t n_tensors, float lr, int32_t shape_scale, void* stream) {
  if (n_tensors < 0 || !std::isfinite(lr) || (shape_scale != 0 && shape_scale != 1)) return CZ_ERR_INVALID;
  if (n_tensors == 0) return CZ_OK;
  if (!flat_param || !flat_update || !offsets || !shapes) return CZ_ERR_INVALID;
  const uintptr_t pa = reinterpret_cast<uintptr_t>(flat_param), ua = reinterpret_cast<uintptr_t>(flat_update),
                  ba = reinterpret_cast<uintptr_t>(param_bf16);
  if ((pa & 3) || (ua & 3) || (ba & 1)) return CZ_ERR_INVALID;
  std::vector<std::pair<int64_t, int64_t>> iv((size_t)n_tensors);
  for (int64_t i = 0; i < n_tensors; ++i) {
    const int64_t r = shapes[2 * i], c = shapes[2 * i + 1];
    if (r <= 0 || c <= 0 || r > (1LL << 30) || c > (1LL << 30) || offsets[i] < 0) return CZ_ERR_INVALID;
    iv[(size_t)i] = {offsets[i], offsets[i] + r * c};
  }
  std::sort(iv.begin(), iv.end());
  for (size_t i = 1; i < iv.size(); ++i)
    if (iv[i].first < iv[i - 1].second) return CZ_ERR_INVALID;   // overlapping tensors would race
  const int st = check_device();
  if (st != CZ_OK) return st;
  nvtxRangePushA("cz/apply_update");

  // 16-byte vectors need the fp32 buffers 16-byte aligned at the tensor's start and the
  // bf16 copy 8-byte aligned there
  const bool vec_base = (pa & 15) == 0 && (ua & 15) == 0 && (ba & 7) == 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Segments seg;
  int64_t i = 0;
  while (i < n_tensors) {
    seg.n_seg = 0;
    int64_t blocks = 0;
    while (i < n_tensors && seg.n_seg < kMaxSeg) {
      const int64_t r = shapes[2 * i], c = shapes[2 * i + 1], n = r * c;
      const int64_t nb = (n + kChunk - 1) / kChunk;
      if (nb > (int64_t)INT32_MAX) {
        nvtxRangePop();
        return CZ_ERR_INVALID;
      }
      if (blocks + nb > (int64_t)INT32_MAX && seg.n_seg > 0) break;
      const int k = seg.n_seg++;
      seg.off[k] = offsets[i];
      seg.n[k] = n;
      seg.blk_first[k] = (int32_t)blocks;
      const double scale = shape_scale ? std::sqrt(std::max(1.0, (double)r / (double)c)) : 1.0;
      seg.coef[k] = (float)((double)lr * scale);
      seg.vec[k] = vec_base && (offsets[i] & 3) == 0;
      blocks += nb;
      ++i;
    }
    seg.blk_first[seg.n_seg] = (int32_t)blocks;
    apply_kernel<<<(unsigned)blocks, kThreads, 0, s>>>(flat_param, static_cast<__nv_bfloat16*>(param_bf16),
                                                      flat_update, seg);
    if (cudaGetLastError() != cudaSuccess) {
      nvtxRangePop();
      return CZ_ERR_CUDA;
    }
  }
  nvtxRangePop();
  return CZ_OK;
}
