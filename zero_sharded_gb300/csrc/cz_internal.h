// Internal declarations shared by the host planner, the step orchestration and
// the CUDA kernels of libcz.  Not part of the C-ABI (see include/cz.h).
#pragma once

#include <stdint.h>

#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "cz.h"

struct cz_plan {};   // the opaque handle type of the C-ABI; cz::Plan derives from it

namespace cz {

// An NVTX range ("cz/..."), open for the object's lifetime: profilers that record
// NVTX (Nsight Systems, ncu --nvtx) show the library's host phases by name.  The
// NVTX3 header is self-contained; with no tool attached a push/pop costs a few ns.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Process-unique id for plans and step programs: caches key on it, never on
// an address that a later allocation could reuse.
uint64_t next_uid();

struct Plan : cz_plan {
  uint64_t uid = next_uid();
  int32_t R = 1;
  int64_t n_params = 0, n_buckets = 0;
  int kind = 0;              // 0: Algorithm 1, 1: Eq. 1 start-index split
  double alpha = 0.0;
  std::vector<int64_t> numels, costs, bucket_sizes;   // costs = W(p) (numels unless given)
  std::vector<int64_t> bucket_first;   // first parameter of each bucket (+ end)
  std::vector<int64_t> phi_first;      // start of each bucket's prefixes in `phi`/`cphi` (+ end)
  std::vector<int64_t> phi;            // element prefix per bucket, u = 0..n_i, concatenated
  std::vector<int64_t> cphi;           // cost prefix Phi_i(u), same layout
  std::vector<int64_t> param_cuts;     // n_buckets*(R+1)
  std::vector<int64_t> elem_cuts;      // n_buckets*(R+1)
  std::vector<int32_t> owner;          // n_params
  std::vector<int64_t> rank_load;      // R, in cost units
  std::vector<int64_t> rank_elems;     // R, elements
  double r_lb = 0, j_dp = 0, j_comm = 0;
};

// The Muon step behind cz_muon_step_ex and cz_muon_step_noalloc.  pin_ok: a new
// step program may keep its tables in page-locked host memory (copied into the
// workspace by a kernel on every call); false keeps them in pageable memory
// (uploaded by cudaMemcpyAsync), for callers that must not page-lock memory.
int muon_step(const cz_plan* plan, int32_t rank, float* flat_param, const void* flat_grad, float* flat_mom,
              const int64_t* offsets, const int64_t* shapes, float lr, float mu, int32_t ns_steps, void* stream,
              const cz_step_opts* opts, bool pin_ok);

// Device address of cz_muon_step_noalloc's static scratch on the current device,
// or null if no such call has set it up there; cz_device_status(stream, NULL)
// reads and clears its status word.
void* noalloc_scratch_if_set_up();

}  // namespace cz
