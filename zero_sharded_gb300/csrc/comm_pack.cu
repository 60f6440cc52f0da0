// Bucket <-> padded shard blocks for the variable-size collectives around the step.
//
// Canzona summary page, section 3.4, "Runtime Static-Layout Enforcement": the
// gradients of bucket B_i are reduce-scattered and the updated parameters
// all-gathered with per-rank sizes S_{i,r} = s_{i,r} - s_{i,r-1} (element cuts of
// the partition map).  Collective primitives that need equal counts per rank take
// R blocks of max_r S_{i,r} elements: pack copies rank r's interval of the bucket
// into block r and zero-fills the tail; unpack copies block r's first S_{i,r}
// elements back into the bucket.  Pure data movement (HBM-bound): bit-exact.

#include <cuda_runtime.h>

#include <algorithm>
#include <stdint.h>

#include "cz.h"

namespace {

constexpr int kMaxRanks = 1024;

struct Cuts {
  int64_t c[kMaxRanks + 1];
};

// One grid row per rank (blockIdx.y = r): copy S_r elements between the bucket
// interval and block r, in 16-byte vectors when both sides share their
// alignment modulo 16 (head and tail bytes copied singly), and zero-fill the
// padding of block r when packing.
template <typename U>
__device__ __noinline__ void copy_units(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t nbytes,
                                        int64_t tid, int64_t nthr) {
  const U* s = reinterpret_cast<const U*>(src);
  U* d = reinterpret_cast<U*>(dst);
  const int64_t n = nbytes / (int64_t)sizeof(U);
  for (int64_t i = tid; i < n; i += nthr) d[i] = s[i];
}

// n bytes of elements of eb bytes; both pointers are eb-aligned.
__device__ __forceinline__ void copy_bytes(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t n,
                                           int eb) {
  const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  const uintptr_t sa = reinterpret_cast<uintptr_t>(src), da = reinterpret_cast<uintptr_t>(dst);
  if ((sa & 15) == (da & 15)) {
    const int64_t head = (int64_t)((16 - (sa & 15)) & 15) < n ? (int64_t)((16 - (sa & 15)) & 15) : n;
    for (int64_t i = tid; i < head; i += nthr) dst[i] = src[i];
    const int64_t nv = (n - head) >> 4;
    const uint4* sv = reinterpret_cast<const uint4*>(src + head);
    uint4* dv = reinterpret_cast<uint4*>(dst + head);
    // four vectors per thread in flight (loads issued before the stores), then the rest one at a time
    int64_t i = tid;
#pragma unroll 1
    for (; i + 3 * nthr < nv; i += 4 * nthr) {
      const uint4 v0 = sv[i], v1 = sv[i + nthr], v2 = sv[i + 2 * nthr], v3 = sv[i + 3 * nthr];
      dv[i] = v0;
      dv[i + nthr] = v1;
      dv[i + 2 * nthr] = v2;
      dv[i + 3 * nthr] = v3;
    }
#pragma unroll 1
    for (; i < nv; i += nthr) dv[i] = sv[i];
    for (int64_t e = head + (nv << 4) + tid; e < n; e += nthr) dst[e] = src[e];
  } else {   // different alignment modulo 16: element-wide copies
    switch (eb) {
      case 8: copy_units<uint64_t>(src, dst, n, tid, nthr); break;
      case 4: copy_units<uint32_t>(src, dst, n, tid, nthr); break;
      case 2: copy_units<uint16_t>(src, dst, n, tid, nthr); break;
      default: copy_units<uint8_t>(src, dst, n, tid, nthr); break;
    }
  }
}

__device__ __forceinline__ void zero_bytes(uint8_t* __restrict__ dst, int64_t n) {
  const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  const uintptr_t da = reinterpret_cast<uintptr_t>(dst);
  const int64_t head = (int64_t)((16 - (da & 15)) & 15) < n ? (int64_t)((16 - (da & 15)) & 15) : n;
  for (int64_t i = tid; i < head; i += nthr) dst[i] = 0;
  const int64_t nv = (n - head) >> 4;
  uint4* dv = reinterpret_cast<uint4*>(dst + head);
  for (int64_t i = tid; i < nv; i += nthr) dv[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t i = head + (nv << 4) + tid; i < n; i += nthr) dst[i] = 0;
}

__global__ void pack_kernel(const uint8_t* __restrict__ bucket, const __grid_constant__ Cuts cuts, int eb,
                            int64_t block, uint8_t* __restrict__ padded) {
  const int r = blockIdx.y;
  const int64_t lo = cuts.c[r], n = cuts.c[r + 1] - lo;
  uint8_t* dst = padded + (int64_t)r * block * eb;
  copy_bytes(bucket + lo * eb, dst, n * eb, eb);
  zero_bytes(dst + n * eb, (block - n) * eb);
}

__global__ void unpack_kernel(const uint8_t* __restrict__ padded, const __grid_constant__ Cuts cuts, int eb,
                              int64_t block, uint8_t* __restrict__ bucket) {
  const int r = blockIdx.y;
  const int64_t lo = cuts.c[r], n = cuts.c[r + 1] - lo;
  copy_bytes(padded + (int64_t)r * block * eb, bucket + lo * eb, n * eb, eb);
}

int check(const void* a, const void* b, int32_t elem_bytes, const int64_t* cuts, int32_t R, int64_t block,
          Cuts& out) {
  if (!a || !b || !cuts || R < 1 || R > kMaxRanks || block < 0) return CZ_ERR_INVALID;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8) return CZ_ERR_INVALID;
  if (cuts[0] != 0) return CZ_ERR_INVALID;
  for (int r = 0; r < R; ++r) {
    if (cuts[r + 1] < cuts[r] || cuts[r + 1] - cuts[r] > block) return CZ_ERR_INVALID;
  }
  for (int r = 0; r <= R; ++r) out.c[r] = cuts[r];
  return CZ_OK;
}

template <bool PACK>
int launch(const void* src, void* dst, int32_t elem_bytes, const Cuts& c, int32_t R, int64_t block, void* stream) {
  if (block == 0) return CZ_OK;
  const int threads = 256;
  // enough CTAs per rank row to cover the largest interval with 16-byte vectors,
  // and about 8 CTAs per SM over all rows
  const int64_t per_row_vec = (block * elem_bytes + 15) / 16;
  const int64_t want = std::max<int64_t>(1, std::min<int64_t>((per_row_vec + threads - 1) / threads,
                                                              std::max<int64_t>(1, 152 * 8 / R)));
  dim3 grid((unsigned)want, (unsigned)R, 1);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (PACK)
    pack_kernel<<<grid, threads, 0, s>>>(static_cast<const uint8_t*>(src), c, elem_bytes, block,
                                         static_cast<uint8_t*>(dst));
  else
    unpack_kernel<<<grid, threads, 0, s>>>(static_cast<const uint8_t*>(src), c, elem_bytes, block,
                                           static_cast<uint8_t*>(dst));
  return cudaGetLastError() == cudaSuccess ? CZ_OK : CZ_ERR_CUDA;
}

}  // namespace

extern "C" int cz_bucket_pack(const void* bucket, int32_t elem_bytes, const int64_t* elem_cuts, int32_t R,
                              int64_t block, void* padded, void* stream) {
  Cuts c;
  int st = check(bucket, padded, elem_bytes, elem_cuts, R, block, c);
  if (st != CZ_OK) return st;
  return launch<true>(bucket, padded, elem_bytes, c, R, block, stream);
}

extern "C" int cz_bucket_unpack(const void* padded, int32_t elem_bytes, const int64_t* elem_cuts, int32_t R,
                                int64_t block, void* bucket, void* stream) {
  Cuts c;
  int st = check(padded, bucket, elem_bytes, elem_cuts, R, block, c);
  if (st != CZ_OK) return st;
  return launch<false>(padded, bucket, elem_bytes, c, R, block, stream);
}
