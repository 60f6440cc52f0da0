// Host orchestration of the local Muon step (cz_muon_step / cz_muon_step_ex).
//
// Canzona summary page, section 3.4, "Runtime Static-Layout Enforcement",
// phase 2: rank r updates exactly the parameters inside its intervals
// [s_{i,r-1}, s_{i,r}) of every bucket, with no communication, because each
// owned tensor is whole on the rank.  This file selects the owned tensors from
// the plan, groups them by Newton-Schulz shape (m = min, n = max of rows/cols),
// lays out the device workspace, and builds once per (plan, rank, buffers) a step
// program: TMA tensor maps, LPT-assigned tile lists in L2-friendly order, and,
// for shards whose iterate fits the L2, the fused launch's dependency-aware
// schedule.  Every call then enqueues, on the caller's stream: the copy of the
// program's tables into the workspace -> the momentum pass (with the per-tensor
// norm) -> either one fused launch for every Newton-Schulz product of every step,
// or ns_steps x (Gram, Poly, Update) launches, the last Update fused with the
// apply; small matrices run all their steps on chip, beside the tiled ones.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <queue>
#include <string>
#include <tuple>
#include <vector>

#include "cz_internal.h"
#include "fused_schedule.h"
#include "step_kernels.h"

namespace cz {
namespace {

constexpr int64_t kAlign = 256;
constexpr int64_t kDefaultTimeoutNs = 1000000000LL;   // 1 s per device-side wait
constexpr int64_t kMaxNsSteps = 64;
// The fused launch's dependency-aware schedule covers up to this many Newton-Schulz
// steps, for shards whose bf16 iterate is at most kSchedMaxXBytes (above any L2
// size: the fused launch only runs shards whose iterate fits the L2).
constexpr int64_t kSchedMaxSteps = 16;
constexpr int64_t kSchedMaxXBytes = 256LL << 20;

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct OwnedMat {
  int64_t param;      // parameter index
  int64_t off;        // element offset
  int32_t rows, cols;
  int32_t m, n;       // NS orientation: m = min, n = max
  bool tall;          // rows > cols: X = u^T
  int32_t group;
  int32_t idx;        // index inside the group
};

struct Group {
  int32_t m, n, count = 0;
  int32_t mat_base = 0;        // global matrix index of the group's first matrix
  int64_t ldx = 0, ldm = 0;    // element pitches: X rows (n), A / B' rows (m)
  int64_t off_x[2] = {0, 0}, off_a = 0, off_b = 0;   // workspace byte offsets (X ping-pong, A, B')
  bool has_wide = false, has_tall = false;
  bool small = false;          // every Newton-Schulz step on chip (ns_small), no tiled GEMMs
  bool small_pair = false;     // ... on a CTA pair (128 < m <= 256): ns_small_pair
};

struct Layout {
  std::vector<OwnedMat> mats;      // global matrix order (grouped)
  std::vector<Group> groups;
  int64_t n_mom_tiles = 0;
  int64_t off_status = 0, off_sigma = 0, off_partial = 0, off_momtiles = 0, off_mommats = 0, off_matinfo = 0;
  int64_t off_small = 0;           // SmallMat per matrix of the small groups
  int64_t off_tiledone = 0;        // momentum pass: per-tensor tile arrival counters (int32, zero)
  int32_t n_small = 0;             // single-CTA and CTA-pair small matrices (SmallMat entries)
  int64_t off_tiles = 0;           // all GEMM tile lists
  int64_t n_gemm_tiles = 0;
  int64_t off_cta = 0;             // per launch: grid+1 tile offsets (int32)
  int64_t n_cta_entries = 0;
  int64_t off_expect = 0;          // fused launch: n_mats x 3 expected arrivals (int32)
  int64_t off_done = 0;            // fused launch: 3 x kMaxNsSteps x n_mats counters (int32), zero in the tables
  int64_t off_sched_first = 0;     // fused launch schedule: kMaxGrid + 1 offsets (int32)
  int64_t off_sched = 0;           // and its entries (int4), room for kSchedMaxSteps steps
  int64_t sched_per_step = 0;      // tiles of one Newton-Schulz step (Gram + Poly + Update)
  int64_t sched_cap = 0;           // entries the schedule region holds (0: no schedule)
  int64_t bytes = 0;
};

// Small groups (m <= 128, n <= 256: one CTA; 128 < m <= 256, n <= 256: a CTA pair)
// take the on-chip kernels (default); CZ_NS_SMALL=0 sends them through the tiled
// GEMMs like every other group.
bool use_small() {
  static const bool small = [] {
    const char* e = std::getenv("CZ_NS_SMALL");
    return !(e && e[0] == '0');
  }();
  return small;
}

int validate_shapes(const Plan* p, const int64_t* shapes) {
  for (int64_t i = 0; i < p->n_params; ++i) {
    const int64_t r = shapes[2 * i], c = shapes[2 * i + 1];
    if (r <= 0 || c <= 0 || r > (1LL << 30) || c > (1LL << 30)) return CZ_ERR_INVALID;
    if (r * c != p->numels[i]) return CZ_ERR_PLAN_MISMATCH;
  }
  return CZ_OK;
}

// Owned tensors grouped by (m, n), groups in order of first appearance.
int build_layout(const Plan* p, int32_t rank, const int64_t* offsets, const int64_t* shapes, Layout& L) {
  std::map<std::pair<int32_t, int32_t>, int32_t> gid;
  std::vector<std::vector<OwnedMat>> per_group;
  for (int64_t i = 0; i < p->n_params; ++i) {
    if (p->owner[i] != rank) continue;
    OwnedMat om;
    om.param = i;
    om.off = offsets ? offsets[i] : 0;
    om.rows = (int32_t)shapes[2 * i];
    om.cols = (int32_t)shapes[2 * i + 1];
    om.tall = om.rows > om.cols;
    om.m = std::min(om.rows, om.cols);
    om.n = std::max(om.rows, om.cols);
    auto key = std::make_pair(om.m, om.n);
    auto it = gid.find(key);
    if (it == gid.end()) {
      it = gid.emplace(key, (int32_t)per_group.size()).first;
      per_group.emplace_back();
      Group g;
      g.m = om.m;
      g.n = om.n;
      L.groups.push_back(g);
    }
    om.group = it->second;
    per_group[it->second].push_back(om);
  }
  int32_t base = 0;
  for (size_t g = 0; g < per_group.size(); ++g) {
    Group& G = L.groups[g];
    G.count = (int32_t)per_group[g].size();
    G.mat_base = base;
    for (int32_t j = 0; j < G.count; ++j) {
      OwnedMat om = per_group[g][j];
      om.idx = j;
      G.has_tall |= om.tall;
      G.has_wide |= !om.tall;
      L.mats.push_back(om);
    }
    G.small = use_small() && G.m <= kSmallPairMaxM && G.n <= kSmallMaxN;
    G.small_pair = G.small && G.m > kSmallMaxM;
    if (G.small) L.n_small += G.count;
    base += G.count;
  }
  // workspace layout
  const int64_t n_mats = (int64_t)L.mats.size();
  // momentum tiles: 64 rows x kMomTileCols (kMomTileColsBf16 with bf16 gradients); sized for the narrower
  const int64_t mom_cw = std::min(kMomTileCols, kMomTileColsBf16);
  for (const OwnedMat& om : L.mats) L.n_mom_tiles += ceil_div64(om.rows, 64) * ceil_div64(om.cols, mom_cw);
  int64_t off = 0;
  L.off_status = off;  off += kAlign;
  L.off_sigma = off;   off = align_up(off + 4 * std::max<int64_t>(n_mats, 1), kAlign);
  L.off_momtiles = off; off = align_up(off + (int64_t)sizeof(MomTile) * std::max<int64_t>(L.n_mom_tiles, 1), kAlign);
  L.off_mommats = off; off = align_up(off + (int64_t)sizeof(MomMat) * std::max<int64_t>(n_mats, 1), kAlign);
  L.off_matinfo = off; off = align_up(off + (int64_t)sizeof(MatInfo) * std::max<int64_t>(n_mats, 1), kAlign);
  L.off_small = off;   off = align_up(off + (int64_t)sizeof(SmallMat) * std::max<int64_t>(L.n_small, 1), kAlign);
  // inside the tables region: the zeros of the host image reset them on every call
  L.off_tiledone = off; off = align_up(off + 4 * std::max<int64_t>(n_mats, 1), kAlign);
  // GEMM tiles: Gram + Poly (same count), and two ping-pong copies each of the
  // Update and Apply lists (a tall tensor's Apply tiles cover n x m)
  int64_t nt = 0;
  for (const Group& G : L.groups) {
    if (G.small) continue;
    const int64_t tm = ceil_div64(G.m, kBM), tn = ceil_div64(G.m, kBN);
    int64_t sym = 0;
    for (int64_t a = 0; a < tm; ++a)
      for (int64_t b = 0; b < tn; ++b)
        if (a * kBM <= b * kBN + kBN - 1) ++sym;
    const int64_t upd = ceil_div64(G.m, kBM) * ceil_div64(G.n, kBN);
    const int64_t app_t = ceil_div64(G.n, kBM) * ceil_div64(G.m, kBN);
    nt += G.count * (3 * sym + 2 * upd + 2 * std::max(upd, app_t));   // Gram x2, Poly, Update x2, Apply x2
  }
  L.n_gemm_tiles = nt;
  L.off_tiles = off; off = align_up(off + 16 * std::max<int64_t>(nt, 1), kAlign);
  // launches per step program: Gram + Poly (one per chunk of kMaxProblems groups),
  // two Update and two Apply lists (Apply: up to two problems per group)
  const int64_t G = (int64_t)L.groups.size();
  const int64_t n_launch = 3 * ceil_div64(std::max<int64_t>(G, 1), kMaxProblems) +
                           2 * ceil_div64(std::max<int64_t>(G, 1), kMaxProblems) +
                           2 * ceil_div64(std::max<int64_t>(2 * G, 1), kMaxProblems);
  L.n_cta_entries = n_launch * (kMaxGrid + 1);
  L.off_cta = off; off = align_up(off + 4 * L.n_cta_entries, kAlign);
  L.off_expect = off; off = align_up(off + 4 * 3 * std::max<int64_t>(n_mats, 1), kAlign);
  L.off_done = off; off = align_up(off + 4 * 3 * kMaxNsSteps * std::max<int64_t>(n_mats, 1), kAlign);
  // the fused launch's schedule, for shards small enough to take it
  {
    int64_t per_step = 0, xb = 0;
    for (const Group& G : L.groups) {
      if (G.small) continue;
      // counted with 128-row tiles, which cover the CTA-pair variant's 256-row tiles too
      int64_t sym = 0;
      for (int64_t a = 0; a < ceil_div64(G.m, kBM); ++a)
        for (int64_t b = 0; b < ceil_div64(G.m, kBN); ++b)
          if (a * kBM <= b * kBN + kBN - 1) ++sym;
      per_step += G.count * (2 * sym + ceil_div64(G.m, kBM) * ceil_div64(G.n, kBN));
      xb += 2 * (int64_t)G.m * G.n * G.count;
    }
    L.sched_per_step = per_step;
    L.sched_cap = xb <= kSchedMaxXBytes ? kSchedMaxSteps * per_step : 0;
  }
  L.off_sched_first = off; off = align_up(off + 4 * (kMaxGrid + 1), kAlign);
  L.off_sched = off; off = align_up(off + 16 * std::max<int64_t>(L.sched_cap, 1), kAlign);
  // per-tile partial sums of the momentum pass: written before they are read, so outside the tables
  // that are copied in on every call
  L.off_partial = off; off = align_up(off + 4 * std::max<int64_t>(L.n_mom_tiles, 1), kAlign);
  for (Group& G : L.groups) {
    G.ldx = align_up(G.n, 8);
    G.ldm = align_up(G.m, 8);
    const int64_t c = G.count;
    G.off_x[0] = off;  off = align_up(off + 2 * c * G.m * G.ldx, kAlign);
    if (!G.small) {    // the on-chip kernel keeps its iterates in shared memory
      G.off_x[1] = off;  off = align_up(off + 2 * c * G.m * G.ldx, kAlign);
    }
    G.off_a = off;     off = align_up(off + 2 * c * G.m * G.ldm, kAlign);
    G.off_b = off;     off = align_up(off + 2 * c * G.m * G.ldm, kAlign);
  }
  L.bytes = off;
  return CZ_OK;
}

// Newton-Schulz GEMM variant: CTA pairs (tcgen05 cta_group::2, 256 x 256 tiles)
// by default; CZ_NS_PAIR=0 selects single-CTA 128 x 256 tiles.
bool use_pair() {
  static const bool pair = [] {
    const char* e = std::getenv("CZ_NS_PAIR");
    return !(e && e[0] == '0');
  }();
  return pair;
}

// All Newton-Schulz products of a step in one persistent launch with per-matrix
// dependencies (default); CZ_NS_FUSED=0 launches each product separately.
bool use_fused() {
  static const bool fused = [] {
    const char* e = std::getenv("CZ_NS_FUSED");
    return !(e && e[0] == '0');
  }();
  return fused;
}

// One-product launches start each wave of tiles together (default): tiles that
// share an operand then read it at the same k, while it is in the L2.  On the
// Qwen3-32B shard Gram's DRAM reads fell 27% per matrix; the step went from 53.40 to
// 52.98 ms on one box, from 54.57 to 53.85 on another, and did not move on a third.
// A launch whose tiles differ in K is paced over the waves every unit has (its
// heaviest K): the Qwen3-14B micro-group went from 173.3 to 170.2 ms.  Tiles of
// fewer than kPaceMinKBlocks k-blocks are not paced: waiting for the slowest unit at
// every short tile cost more than it saved (the Qwen3-1.7B x 28 set's Poly, 32
// k-blocks, went from 4.81 to 5.00 ms per step).  Letting units run up to 1, 2 or 4
// waves apart did not help.  CZ_NS_PACE=0 turns it off.
constexpr int64_t kPaceMinKBlocks = 64;
bool use_pace() {
  static const bool on = [] {
    const char* e = std::getenv("CZ_NS_PACE");
    return !(e && e[0] == '0');
  }();
  return on;
}

// The fused launch walks the host's dependency-aware schedule (default);
// CZ_NS_SCHED=0 walks the per-(step, product) tile lists instead.
bool use_sched() {
  static const bool on = [] {
    const char* e = std::getenv("CZ_NS_SCHED");
    return !(e && e[0] == '0');
  }();
  return on;
}

// L2 size of the current device, in bytes (0 if it cannot be read).
int64_t l2_bytes() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return 0;
  return v;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D bf16 map over `count` matrices of `rows` x `inner` (row pitch ld elements,
// matrix stride ms elements).  Operand loads: box 64 (inner) x box_rows, 128-byte
// swizzle.  Output stores (store = true): box 32 x 32, no swizzle (dense smem block).
bool encode_map(CUtensorMap* map, void* base, int64_t inner, int64_t rows, int64_t count, int64_t ld, int64_t ms,
                uint32_t box_rows, bool store = false) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)count};
  cuuint64_t strides[2] = {(cuuint64_t)(ld * 2), (cuuint64_t)(ms * 2)};
  cuuint32_t box[3] = {store ? 32u : (cuuint32_t)kBK, store ? 32u : box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, store ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct Launch {
  int phase;
  int first;
  int cur;                          // X buffer read (Gram, Update, Apply)
  int32_t pace_tiles = 0;           // wave pacing of each unit's first pace_tiles tiles (0: none)
  GemmParams params;
};

// Everything that depends only on (plan, rank, shapes, offsets, buffers, the
// gradient dtype).  The step's scalars (lr, mu, eps, Nesterov, the Newton-Schulz
// coefficients) are launch parameters, set on every call.
struct Program {
  uint64_t uid = next_uid();
  bool pair = true;
  bool fused_ok = false;
  int32_t fused_phase = kFused;  // kFusedLatency when every product has fewer tiles than units
  int32_t sched_steps = 0;      // the fused launch's schedule is for this many steps (0: none)
  GemmParams fused{};
  Layout L;
  std::vector<uint8_t> host_tables;   // image of the workspace's [tables_begin, tables_end)
  int64_t tables_begin = 0, tables_end = 0;
  // The same image in page-locked, device-mapped host memory (null when that
  // allocation failed: the pageable image is uploaded instead), and an event
  // recorded after every copy out of it, waited on before it is freed.
  uint8_t* pinned = nullptr;
  const void* pinned_dev = nullptr;
  cudaEvent_t copied = nullptr;
  // Used inside a stream capture: a CUDA graph may replay the copy out of the
  // page-locked image at any later time, so the image is never freed.
  bool captured = false;
  // The small-matrix launches run on a side stream, beside the tiled products
  // (or the single-CTA one beside the CTA-pair one when no tiled product is left),
  // when both sides fit on the GPU at once (forked after the momentum pass, joined
  // before the call's work ends); events of this program.
  bool fork_small = false;
  bool tiled = false;           // some matrices take the tiled products
  cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
  MomParams mom{};
  std::vector<Launch> gram[2], poly, update[2], apply[2];   // [cur]: X buffer read
  SmallParams small{};          // single-CTA matrices (m <= 128)
  SmallParams small_pair{};     // CTA-pair matrices (128 < m <= 256), SmallMat entries after the single ones

  Program() = default;
  Program(const Program&) = delete;
  Program& operator=(const Program&) = delete;
  ~Program() {
    if (copied) {
      cudaEventSynchronize(copied);
      cudaEventDestroy(copied);
    }
    if (pinned && !captured) cudaFreeHost(pinned);
    if (fork_ev) cudaEventDestroy(fork_ev);
    if (join_ev) cudaEventDestroy(join_ev);
  }
};

// Moves the program's table image into page-locked, device-mapped host memory.
// On failure the program keeps the pageable image (and the upload by copy).
void pin_tables(Program& P) {
  const size_t bytes = P.host_tables.size();
  if (bytes == 0) return;
  void* h = nullptr;
  if (cudaHostAlloc(&h, bytes, cudaHostAllocPortable | cudaHostAllocMapped) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  void* d = nullptr;
  cudaEvent_t ev = nullptr;
  if (cudaHostGetDevicePointer(&d, h, 0) != cudaSuccess ||
      cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    cudaFreeHost(h);
    return;
  }
  std::memcpy(h, P.host_tables.data(), bytes);
  P.pinned = static_cast<uint8_t*>(h);
  P.pinned_dev = d;
  P.copied = ev;
  std::vector<uint8_t>().swap(P.host_tables);
}

struct Key {
  uint64_t plan; int32_t rank; int dev;
  const void *param, *grad, *mom, *pbf16, *dbg, *ws;
  int32_t grad_bf16;
  std::vector<int64_t> offsets, shapes;
  bool operator<(const Key& o) const {
    return std::tie(plan, rank, dev, param, grad, mom, pbf16, dbg, ws, grad_bf16, offsets, shapes) <
           std::tie(o.plan, o.rank, o.dev, o.param, o.grad, o.mom, o.pbf16, o.dbg, o.ws, o.grad_bf16, o.offsets,
                    o.shapes);
  }
};

// ---------------------------------------------------------------- tracing
struct ProfRec { int kind; cudaEvent_t a, b; };
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;

// Last CUDA error behind a CZ_ERR_CUDA of this thread (cz_last_cuda_error).
thread_local cudaError_t t_last_cuda = cudaSuccess;

cudaError_t note(cudaError_t e) {
  if (e != cudaSuccess) t_last_cuda = e;
  return e;
}

// NVTX names of the kernel kinds (numbering of cz_profile_read).
const char* const kKindNames[CZ_KERNEL_KINDS] = {"cz/momentum", "cz/tables",    "cz/ns_gram",  "cz/ns_poly",
                                                 "cz/ns_update", "cz/ns_update_apply", "cz/ns_fused", "cz/ns_small"};

// Launches `fn` on stream s inside an NVTX range named by its kind, bracketed by
// events when tracing is on.
// Set while a call enqueues into a stream that is being captured: no timing
// events are recorded then (a captured event record is not a timing point).
thread_local bool t_capturing = false;

template <class F>
cudaError_t traced(int kind, cudaStream_t s, F&& fn) {
  NvtxRange range(kKindNames[kind]);
  if (!g_prof_on || t_capturing) return note(fn());
  ProfRec r{kind, nullptr, nullptr};
  if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return note(cudaGetLastError());
  cudaEventRecord(r.a, s);
  cudaError_t e = fn();
  cudaEventRecord(r.b, s);
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof.push_back(r);
  return note(e);
}

std::mutex g_mu;
std::map<Key, std::shared_ptr<Program>> g_cache;
int64_t g_programs_built = 0;   // under g_mu
struct DevWs { void* ptr = nullptr; size_t bytes = 0; };
std::map<int, DevWs> g_ws;

template <class T>
T* at(std::vector<uint8_t>& img, int64_t base, int64_t off) {
  return reinterpret_cast<T*>(img.data() + (off - base));
}

// Tile lists for one phase: {problem, matrix, tile_m, tile_n}, sorted so the
// longest K goes first (LPT), then chunked into launches of <= kMaxProblems problems.
struct ProbDesc {
  GemmProblem gp;
  CUtensorMap ta, tb, to, tot;
  std::vector<int4> tiles;
};

// Tiles go to CTAs by the LPT rule (Graham): heaviest tile first, each to the
// currently least-loaded CTA (ties: lower CTA index).  Cost of a tile = its
// k-blocks plus a constant for the epilogue.  Each CTA's tiles are stored
// contiguously, heaviest first; cta_first gives the ranges.
struct TileRef { int4 t; int64_t cost; };

// Tiles of one matrix's Update (B' X, B' m x m, X m x n) in an L2-friendly order.
// Consecutive entries run at the same time, one per unit, so a wave of `units`
// entries reads the B' row blocks and the X column blocks of its tiles.  Each X
// column block is read by one wave only, while B' is read again by every wave, so
// B' must stay in the L2 from wave to wave.  At m = 5120 (B' 52 MB) it did not: the
// Update read 4.5x its algorithmic bytes from DRAM.  B' rows are therefore split
// into parts of at most kUpdateBBytes each; a wave covers one part's row blocks and
// as many X column blocks as fill the units, and X is swept once per part.  Two
// parts at m = 5120: DRAM reads -22% and the Qwen3-32B shard's step 55.18 ->
// 54.41 ms (the step runs at the power cap, where less DRAM traffic means clock);
// three parts read X once more than they save.
constexpr int64_t kUpdateBBytes = 32LL << 20;
constexpr int64_t kSymBlock = 8;   // tiles per side of a block of the symmetric products' tile order

void update_tiles(std::vector<int4>& out, int mat, int64_t m, int64_t TM, int64_t TN, int64_t units) {
  const int64_t parts = std::min<int64_t>(TM, std::max<int64_t>(1, ceil_div64(2 * m * m, kUpdateBBytes)));
  for (int64_t sp = 0; sp < parts; ++sp) {
    const int64_t a_lo = sp * TM / parts, a_hi = (sp + 1) * TM / parts;
    const int64_t group = std::max<int64_t>(1, ceil_div64(units, a_hi - a_lo));
    for (int64_t b0 = 0; b0 < TN; b0 += group)
      for (int64_t a = a_lo; a < a_hi; ++a)
        for (int64_t b = b0; b < std::min(TN, b0 + group); ++b) out.push_back(make_int4(0, mat, (int)a, (int)b));
  }
}

// carry: null, or per-unit loads that the assignment starts from and adds to (a
// list that fits one launch only), so that consecutive lists balance their sum.
bool make_launches(int phase, std::vector<ProbDesc>& probs, int4* dev_tiles, int4* host_tiles, int64_t& tile_cursor,
                   int32_t* dev_cta, int32_t* host_cta, int64_t& cta_cursor, int max_grid, const GemmParams& common,
                   std::vector<Launch>& out, int first, int cur, std::vector<int64_t>* carry) {
  if (carry && probs.size() > (size_t)kMaxProblems) carry = nullptr;
  for (size_t c0 = 0; c0 < probs.size(); c0 += kMaxProblems) {
    const size_t c1 = std::min(probs.size(), c0 + (size_t)kMaxProblems);
    std::vector<TileRef> tl;
    for (size_t i = c0; i < c1; ++i) {
      const int64_t cost = ceil_div64(probs[i].gp.K, kBK) + 2;
      for (int4 t : probs[i].tiles) tl.push_back({make_int4((int)(i - c0), t.y, t.z, t.w), cost});
    }
    if (tl.empty()) continue;
    std::stable_sort(tl.begin(), tl.end(), [](const TileRef& x, const TileRef& y) { return x.cost > y.cost; });
    // every list of a program uses the same unit count, so a fused launch can walk them all
    const int grid = std::min(max_grid, kMaxGrid);
    std::vector<std::vector<int4>> per(grid);
    {
      // min-heap of (load, cta)
      std::vector<std::pair<int64_t, int>> heap;
      if (carry) carry->resize((size_t)grid, 0);
      for (int b = 0; b < grid; ++b) heap.push_back({carry ? (*carry)[(size_t)b] : 0, b});
      auto gt = [](const std::pair<int64_t, int>& x, const std::pair<int64_t, int>& y) { return x > y; };
      std::make_heap(heap.begin(), heap.end(), gt);
      for (const TileRef& r : tl) {
        std::pop_heap(heap.begin(), heap.end(), gt);
        auto& top = heap.back();
        per[top.second].push_back(r.t);
        top.first += r.cost;
        std::push_heap(heap.begin(), heap.end(), gt);
      }
      if (carry)
        for (const auto& e : heap) (*carry)[(size_t)e.second] = e.first;
    }
    Launch ln;
    ln.phase = phase;
    ln.first = first;
    ln.cur = cur;
    // Wave pacing covers the tiles every unit has: the shortest list's length, plus
    // the next tile (it waits only for tiles every unit issues).  LPT deals the
    // heaviest tiles first, round-robin, so those waves hold tiles of one K.  Only
    // launches whose heaviest tiles have at least kPaceMinKBlocks k-blocks are paced.
    {
      size_t mn = per[0].size();
      for (int b = 1; b < grid; ++b) mn = std::min(mn, per[b].size());
      ln.pace_tiles = (tl.front().cost - 2 >= kPaceMinKBlocks && mn >= 1) ? (int32_t)mn + 1 : 0;
    }
    std::memset(&ln.params, 0, sizeof(GemmParams));
    ln.params = common;
    ln.params.n_prob = (int)(c1 - c0);
    for (size_t i = c0; i < c1; ++i) {
      ln.params.tmA[i - c0] = probs[i].ta;
      ln.params.tmB[i - c0] = probs[i].tb;
      ln.params.tmO[i - c0] = probs[i].to;
      ln.params.tmOT[i - c0] = probs[i].tot;
      ln.params.prob[i - c0] = probs[i].gp;
    }
    ln.params.first = first;
    ln.params.n_tiles = (int)tl.size();
    ln.params.grid = grid;
    ln.params.tiles = dev_tiles + tile_cursor;
    ln.params.cta_first = dev_cta + cta_cursor;
    int32_t pos = 0;
    for (int b = 0; b < grid; ++b) {
      host_cta[cta_cursor + b] = pos;
      for (const int4& t : per[b]) host_tiles[tile_cursor + pos++] = t;
    }
    host_cta[cta_cursor + grid] = pos;
    tile_cursor += (int64_t)tl.size();
    cta_cursor += grid + 1;
    out.push_back(ln);
  }
  return true;
}

int build_program(const Plan* plan, int32_t rank, float* flat_param, const void* flat_grad, float* flat_mom,
                  const int64_t* offsets, const int64_t* shapes, float lr, float mu, int32_t ns_steps,
                  const cz_step_opts& o, uint8_t* ws, Program& P) {
  Layout& L = P.L;
  int st = build_layout(plan, rank, offsets, shapes, L);
  if (st != CZ_OK) return st;
  const int64_t n_mats = (int64_t)L.mats.size();
  P.tables_begin = L.off_sigma;
  // through the fused launch's completion counters, which the image's zeros reset on every call
  P.tables_end = align_up(L.off_done + 4 * 3 * kMaxNsSteps * (int64_t)std::max<size_t>(L.mats.size(), 1), 16);
  P.host_tables.assign((size_t)(P.tables_end - P.tables_begin), 0);
  auto& img = P.host_tables;
  const int64_t tb = P.tables_begin;

  // momentum pass tables
  MomTile* mt = at<MomTile>(img, tb, L.off_momtiles);
  MomMat* mm = at<MomMat>(img, tb, L.off_mommats);
  MatInfo* mi = at<MatInfo>(img, tb, L.off_matinfo);
  int64_t tcur = 0;
  for (int64_t g = 0; g < n_mats; ++g) {
    const OwnedMat& om = L.mats[g];
    const Group& G = L.groups[om.group];
    uint16_t* X = reinterpret_cast<uint16_t*>(ws + G.off_x[0]) + (int64_t)om.idx * G.m * G.ldx;
    MomMat& d = mm[g];
    d.off = om.off;
    d.rows = om.rows;
    d.cols = om.cols;
    if (!om.tall) {          // X = u (rows x cols)
      d.direct = X; d.ld_direct = G.ldx;
      d.trans = nullptr; d.ld_trans = 0;
    } else {                 // X = u^T
      d.direct = nullptr; d.ld_direct = 0;
      d.trans = X; d.ld_trans = G.ldx;
    }
    d.tile_first = (int32_t)tcur;
    // momentum tiles: 64 rows x kMomTileCols columns (kMomTileColsBf16 with bf16 gradients)
    const int64_t cw = o.grad_is_bf16 ? kMomTileColsBf16 : kMomTileCols;
    const int64_t tr = ceil_div64(om.rows, 64), tc = ceil_div64(om.cols, cw);
    d.tile_count = (int32_t)(tr * tc);
    for (int64_t a = 0; a < tr; ++a)
      for (int64_t b = 0; b < tc; ++b) {
        MomTile& t = mt[tcur++];
        t.mat = (int32_t)g;
        t.r0 = (int32_t)(a * 64);
        t.c0 = (int32_t)(b * cw);
        t.pad = 0;
      }
    MatInfo& m = mi[g];
    m.w_off = om.off;
    m.rows = om.rows;
    m.cols = om.cols;
    m.scale = std::sqrt(std::max(1.0, (double)om.rows / (double)om.cols));
    m.vec_ok = ((om.off & 3) == 0 && (om.cols & 3) == 0) ? 1 : 0;
    m.pad = 0;
  }
  MomParams& mp = P.mom;
  mp.mom = flat_mom;
  mp.grad = flat_grad;
  mp.grad_bf16 = o.grad_is_bf16 ? 1 : 0;
  mp.nesterov = o.nesterov ? 1 : 0;
  mp.mu = mu;
  mp.eps = o.eps;
  mp.tiles = reinterpret_cast<const MomTile*>(ws + L.off_momtiles);
  mp.n_tiles = (int32_t)tcur;   // <= L.n_mom_tiles, the count the workspace holds
  mp.mats = reinterpret_cast<const MomMat*>(ws + L.off_mommats);
  mp.n_mats = (int32_t)n_mats;
  mp.partial = reinterpret_cast<float*>(ws + L.off_partial);
  mp.sigma = reinterpret_cast<float*>(ws + L.off_sigma);
  mp.tile_done = reinterpret_cast<int*>(ws + L.off_tiledone);
  mp.status = reinterpret_cast<int*>(ws + L.off_status);

  // GEMM problems
  GemmParams common;
  std::memset(&common, 0, sizeof(common));
  common.sigma = mp.sigma;
  common.mats = reinterpret_cast<const MatInfo*>(ws + L.off_matinfo);
  common.a = o.a;
  common.b = o.b;
  common.c = o.c;
  common.lr = lr;
  common.W = flat_param;
  common.Wb = reinterpret_cast<uint16_t*>(o.param_bf16);
  common.dbg = o.debug_update_out;
  common.status = mp.status;
  common.timeout_ns = kDefaultTimeoutNs;

  int4* dev_tiles = reinterpret_cast<int4*>(ws + L.off_tiles);
  int4* host_tiles = at<int4>(img, tb, L.off_tiles);
  int32_t* dev_cta = reinterpret_cast<int32_t*>(ws + L.off_cta);
  int32_t* host_cta = at<int32_t>(img, tb, L.off_cta);
  int64_t cursor = 0, cta_cursor = 0;
  const bool pair = P.pair = use_pair();
  const int tm_rows = pair ? 256 : kBM;          // output rows per tile
  const uint32_t b_box = pair ? 128 : kBN;       // B-side rows each CTA loads per stage
  const int max_grid = gemm_max_units(pair);
  std::vector<ProbDesc> gram[2], poly, upd[2], app[2];
  SmallMat* smt = at<SmallMat>(img, tb, L.off_small);
  int32_t n_small = 0, n_small_single = 0;
  for (int pass = 0; pass < 2; ++pass) {        // the single-CTA matrices first, then the CTA-pair ones
    for (const Group& G : L.groups) {
      if (!G.small || G.small_pair != (pass == 1)) continue;
      for (int j = 0; j < G.count; ++j) {
        SmallMat& e = smt[n_small++];
        e.x = reinterpret_cast<const uint16_t*>(ws + G.off_x[0]) + (int64_t)j * G.m * G.ldx;
        e.ldx = (int32_t)G.ldx;
        e.pad0 = 0;
        e.m = G.m;
        e.n = G.n;
        e.mat = G.mat_base + j;
        e.pad = 0;
      }
    }
    if (pass == 0) n_small_single = n_small;
  }
  for (const Group& G : L.groups) {
    if (G.small) continue;
    uint16_t* X[2] = {reinterpret_cast<uint16_t*>(ws + G.off_x[0]), reinterpret_cast<uint16_t*>(ws + G.off_x[1])};
    uint16_t* A = reinterpret_cast<uint16_t*>(ws + G.off_a);
    uint16_t* B = reinterpret_cast<uint16_t*>(ws + G.off_b);
    const int64_t msx = (int64_t)G.m * G.ldx, msa = (int64_t)G.m * G.ldm;
    const int c = G.count;
    // symmetric tiles of an m x m output: the tiles touching the upper triangle, in
    // blocks of kSymBlock x kSymBlock tiles, so that a wave of consecutive tiles reads
    // fewer row blocks of its operand (Qwen3-32B shard: 54.12 -> 53.90 ms per step,
    // Gram DRAM reads -1.5%, Poly -15%; row by row, column by column and diagonal
    // bands read as much or more)
    std::vector<int4> sym;
    {
      const int64_t TA = ceil_div64(G.m, tm_rows), TB = ceil_div64(G.m, kBN);
      for (int j = 0; j < c; ++j)
        for (int64_t i0 = 0; i0 < TA; i0 += kSymBlock)
          for (int64_t j0 = 0; j0 < TB; j0 += kSymBlock)
            for (int64_t a = i0; a < std::min(TA, i0 + kSymBlock); ++a)
              for (int64_t b = j0; b < std::min(TB, j0 + kSymBlock); ++b)
                if (a * tm_rows <= b * kBN + kBN - 1) sym.push_back(make_int4(0, j, (int)a, (int)b));
    }
    for (int cur = 0; cur < 2; ++cur) {
      // Gram: A = s^2 X X^T from X buffer `cur`, stored with its mirror into A
      ProbDesc d{};
      d.gp.M = G.m; d.gp.N = G.m; d.gp.K = G.n; d.gp.count = c; d.gp.mat_base = G.mat_base;
      d.gp.phase = kGram; d.gp.slot = 0;
      if (!encode_map(&d.ta, X[cur], G.n, G.m, c, G.ldx, msx, kBM) ||
          !encode_map(&d.tb, X[cur], G.n, G.m, c, G.ldx, msx, b_box) ||
          !encode_map(&d.to, A, G.m, G.m, c, G.ldm, msa, 0, true))
        return CZ_ERR_CUDA;
      d.tot = d.to;
      d.tiles = sym;
      gram[cur].push_back(d);
    }
    {
      // Poly: B' = a I + b A + c A A, stored with its mirror into B
      ProbDesc d{};
      d.gp.M = G.m; d.gp.N = G.m; d.gp.K = G.m; d.gp.count = c; d.gp.mat_base = G.mat_base;
      d.gp.phase = kPoly; d.gp.slot = 1;
      d.gp.aux = A; d.gp.ld_aux = G.ldm; d.gp.ms_aux = msa;
      if (!encode_map(&d.ta, A, G.m, G.m, c, G.ldm, msa, kBM) || !encode_map(&d.tb, A, G.m, G.m, c, G.ldm, msa, b_box) ||
          !encode_map(&d.to, B, G.m, G.m, c, G.ldm, msa, 0, true))
        return CZ_ERR_CUDA;
      d.tot = d.to;
      d.tiles = sym;
      poly.push_back(d);
    }
    for (int cur = 0; cur < 2; ++cur) {
      // update: X[cur ^ 1] (m x n) <- s B' X[cur]; operands B' rows (K = m) and
      // X[cur] read MN-major (64 x 64 boxes: 64 columns of n, 64 rows of K = m)
      ProbDesc d{};
      d.gp.M = G.m; d.gp.N = G.n; d.gp.K = G.m; d.gp.count = c; d.gp.mat_base = G.mat_base;
      d.gp.phase = kUpdate; d.gp.slot = 2;
      d.gp.b_mn = 1;
      if (!encode_map(&d.ta, B, G.m, G.m, c, G.ldm, msa, kBM) ||
          !encode_map(&d.tb, X[cur], G.n, G.m, c, G.ldx, msx, 64) ||
          !encode_map(&d.to, X[cur ^ 1], G.n, G.m, c, G.ldx, msx, 0, true))
        return CZ_ERR_CUDA;
      d.tot = d.to;
      // update tiles: B' (m x m) is the small operand, X (m x n) the large one
      const int64_t TMu = ceil_div64(G.m, tm_rows), TNu = ceil_div64(G.n, kBN);
      for (int j = 0; j < c; ++j) update_tiles(d.tiles, j, G.m, TMu, TNu, max_grid);
      upd[cur].push_back(d);
      // apply: the same product, the epilogue writes W (X for a wide tensor, X^T for a tall one)
      ProbDesc e = d;
      e.gp.phase = kApply;
      app[cur].push_back(e);
    }
  }
  // Units of every GEMM launch: no more than the most tiles of any one product
  // list, so that a shard of a few small tiles leaves the rest of the GPU free.
  int64_t most = 1;
  for (auto* v : {&gram[0], &poly, &upd[0], &app[0]}) {
    int64_t t = 0;
    for (const ProbDesc& d : *v) t += (int64_t)d.tiles.size();
    most = std::max(most, t);
  }
  const int units = (int)std::min<int64_t>(max_grid, most);
  // Gram with first=0/1 share one tile list: build first, copy for the other flag.
  auto ml = [&](int phase, std::vector<ProbDesc>& probs, std::vector<Launch>& out, int cur,
                std::vector<int64_t>* carry) {
    make_launches(phase, probs, dev_tiles, host_tiles, cursor, dev_cta, host_cta, cta_cursor, units, common, out,
                  0, cur, carry);
  };
  // The fused launch walks a step's Gram, Poly and Update (or Apply) lists on every
  // unit, so when it will run, each list's assignment starts from the loads the
  // previous list left: the units' totals per step are balanced, not each list
  // alone (balancing each alone leaves the same low-index units heavier in every
  // list, since ties go to the lower index).  One launch per product keeps each
  // list balanced on its own.
  bool fused_candidate = use_fused();
  {
    int64_t xb = 0;
    for (const Group& G : L.groups)
      if (!G.small) xb += 2 * (int64_t)G.m * G.n * G.count;
    size_t np = 0;
    for (auto* v : {&gram[0], &gram[1], &poly, &upd[0], &upd[1], &app[0], &app[1]}) np += v->size();
    fused_candidate = fused_candidate && np <= (size_t)kMaxProblems && xb <= l2_bytes();
  }
  std::vector<int64_t> c_gram, c_poly;
  std::vector<int64_t>* cg = fused_candidate ? &c_gram : nullptr;
  ml(kGram, gram[0], P.gram[0], 0, cg);
  c_poly = c_gram;                 // the Poly list starts where Gram left the units
  if (cg) c_gram.assign(c_gram.size(), 0);
  ml(kGram, gram[1], P.gram[1], 1, cg);   // the same tiles from the same start: the same assignment
  ml(kPoly, poly, P.poly, 0, fused_candidate ? &c_poly : nullptr);
  for (int cur = 0; cur < 2; ++cur) {
    std::vector<int64_t> cu = c_poly, ca = c_poly;
    ml(kUpdate, upd[cur], P.update[cur], cur, fused_candidate ? &cu : nullptr);
    ml(kApply, app[cur], P.apply[cur], cur, fused_candidate ? &ca : nullptr);
  }
  SmallParams& sp = P.small;
  sp.mats = reinterpret_cast<const SmallMat*>(ws + L.off_small);
  sp.n_mats = n_small_single;
  sp.ns_steps = 0;                // set per call
  sp.sigma = mp.sigma;
  sp.info = common.mats;
  sp.a = o.a;
  sp.b = o.b;
  sp.c = o.c;
  sp.lr = lr;
  sp.W = flat_param;
  sp.Wb = common.Wb;
  sp.dbg = o.debug_update_out;
  sp.status = mp.status;
  sp.timeout_ns = kDefaultTimeoutNs;
  P.small_pair = sp;
  P.small_pair.mats = sp.mats + n_small_single;
  P.small_pair.n_mats = n_small - n_small_single;
  // cannot happen: both regions are sized by build_layout
  if (cursor > L.n_gemm_tiles || cta_cursor > L.n_cta_entries) return CZ_ERR_NOMEM;

  // the fused launch's variant: a shard whose products all have fewer tiles than the
  // units waits on every stage's epilogue, so it runs twice the epilogue warps
  P.fused_phase = most < max_grid ? kFusedLatency : kFused;
  // expected arrivals per (matrix, slot): tiles of the matrix x epilogue warps per unit
  const int arrivals = epi_warps(P.fused_phase) * (pair ? 2 : 1);
  int32_t* expect = at<int32_t>(img, tb, L.off_expect);
  for (auto& pd : gram[0])
    for (const int4& t : pd.tiles) expect[(pd.gp.mat_base + t.y) * 3 + 0] += arrivals;
  for (auto& pd : poly)
    for (const int4& t : pd.tiles) expect[(pd.gp.mat_base + t.y) * 3 + 1] += arrivals;
  for (auto& pd : upd[0])
    for (const int4& t : pd.tiles) expect[(pd.gp.mat_base + t.y) * 3 + 2] += arrivals;

  // fused launch: one problem table over the seven lists, each list walked per unit
  const std::vector<Launch>* lists[kFusedLists] = {&P.gram[0], &P.gram[1], &P.poly,     &P.update[0],
                                                   &P.update[1], &P.apply[0], &P.apply[1]};
  bool ok_fused = true;
  int total = 0;
  for (auto* v : lists) {
    if (v->size() != 1) ok_fused = false;
    else total += (*v)[0].params.n_prob;
  }
  // The fused launch runs the products of all matrices side by side, so it pays only
  // while the shard's bf16 iterate fits the L2: larger shards keep their L2 reuse
  // better with one launch per product in grouped raster order.
  int64_t x_bytes = 0;
  for (const Group& G : L.groups)
    if (!G.small) x_bytes += 2 * (int64_t)G.m * G.n * G.count;
  if (ok_fused && total <= kMaxProblems && x_bytes <= l2_bytes()) {
    GemmParams& F = P.fused;
    F = common;
    int off = 0;
    for (int li = 0; li < kFusedLists; ++li) {
      const GemmParams& q = (*lists[li])[0].params;
      for (int i = 0; i < q.n_prob; ++i) {
        F.tmA[off + i] = q.tmA[i];
        F.tmB[off + i] = q.tmB[i];
        F.tmO[off + i] = q.tmO[i];
        F.tmOT[off + i] = q.tmOT[i];
        F.prob[off + i] = q.prob[i];
      }
      F.lists[li].tiles = q.tiles;
      F.lists[li].cta_first = q.cta_first;
      F.lists[li].prob_off = off;
      F.grid = q.grid;
      off += q.n_prob;
    }
    F.n_prob = total;
    F.n_tiles = 1;   // non-zero: the launch is not skipped
    F.n_mats = (int32_t)n_mats;
    F.expect = reinterpret_cast<const int*>(ws + L.off_expect);
    F.done = reinterpret_cast<int*>(ws + L.off_done);
    P.fused_ok = true;
    // the dependency-aware schedule for the step count of this first call (other
    // step counts walk the per-(step, product) lists)
    if (use_sched() && ns_steps >= 1 && ns_steps <= kSchedMaxSteps && F.grid <= kMaxGrid) {
      static_assert(kSchedLists == kFusedLists, "the schedule walks the fused lists");
      const std::vector<ProbDesc>* const pl[kFusedLists] = {&gram[0], &gram[1], &poly,  &upd[0],
                                                             &upd[1],  &app[0],  &app[1]};
      std::vector<SchedTile> st[kFusedLists];
      for (int li = 0; li < kFusedLists; ++li)
        for (size_t i = 0; i < pl[li]->size(); ++i) {
          const ProbDesc& pd = (*pl[li])[i];
          for (const int4& t : pd.tiles)
            st[li].push_back({F.lists[li].prob_off + (int32_t)i, t.y, t.z, t.w, pd.gp.mat_base + t.y,
                              ceil_div64(pd.gp.K, kBK)});
        }
      std::vector<std::vector<SchedEntry>> per_unit;
      const bool scheduled = schedule_fused(st, ns_steps, F.grid, (int)n_mats, per_unit);
      int64_t entries = 0;
      for (const auto& v : per_unit) entries += (int64_t)v.size();
      if (scheduled && entries <= L.sched_cap) {
        const int64_t end = align_up(L.off_sched + 16 * entries, 16);
        if (end > P.tables_end) {
          P.tables_end = end;
          img.resize((size_t)(P.tables_end - tb), 0);
        }
        int32_t* sf = at<int32_t>(img, tb, L.off_sched_first);
        int4* se = at<int4>(img, tb, L.off_sched);
        int32_t pos = 0;
        for (int u = 0; u < F.grid; ++u) {
          sf[u] = pos;
          for (const SchedEntry& e : per_unit[(size_t)u]) se[pos++] = make_int4(e.x, e.y, e.z, e.w);
        }
        sf[F.grid] = pos;
        F.sched = reinterpret_cast<const int4*>(ws + L.off_sched);
        F.sched_first = reinterpret_cast<const int32_t*>(ws + L.off_sched_first);
        P.sched_steps = ns_steps;
      }
    }
  }
  // The small-matrix CTAs beside the other side's work: beside the tiled products'
  // units (the side stream runs the single-CTA launch, then the CTA-pair one) or,
  // with no tiled product, the single-CTA launch beside the CTA-pair one; only when
  // both sides fit on the GPU at once (then neither waits for the other's SMs).
  bool tiled = false;
  for (const Group& G : L.groups) tiled |= !G.small;
  P.tiled = tiled;
  const int64_t pair_ctas = 2 * (int64_t)(n_small - n_small_single);
  int64_t need = -1;
  if (tiled && n_small > 0)
    need = (int64_t)units * (pair ? 2 : 1) + std::max<int64_t>(n_small_single, pair_ctas);
  else if (!tiled && n_small_single > 0 && pair_ctas > 0)
    need = n_small_single + pair_ctas;
  int dev = 0, sms = 0;
  if (need >= 0 && cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && need <= sms) {
    if (cudaEventCreateWithFlags(&P.fork_ev, cudaEventDisableTiming) == cudaSuccess &&
        cudaEventCreateWithFlags(&P.join_ev, cudaEventDisableTiming) == cudaSuccess)
      P.fork_small = true;
    else
      cudaGetLastError();
  }
  return CZ_OK;
}

// The library's side stream for the caller's stream `s` on the current device
// (non-blocking, never destroyed).  One per caller stream: a side stream shared
// by several caller streams would order their work behind one another and could
// close a wait cycle that the caller's own event waits do not have.
cudaStream_t side_stream(cudaStream_t s) {
  static std::map<std::pair<int, cudaStream_t>, cudaStream_t> streams;   // callers hold g_mu
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  const auto key = std::make_pair(dev, s);
  auto it = streams.find(key);
  if (it != streams.end()) return it->second;
  cudaStream_t st = nullptr;
  if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  streams.emplace(key, st);
  return st;
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

int get_internal_ws(size_t need, void** out, bool capturing) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CZ_ERR_CUDA;
  DevWs& w = g_ws[dev];
  if (w.bytes < need) {
    if (capturing) return CZ_ERR_INVALID;   // growing it synchronises and allocates
    if (w.ptr) {
      cudaDeviceSynchronize();
      cudaFree(w.ptr);
      w.ptr = nullptr;
      w.bytes = 0;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, need) != cudaSuccess) {
      cudaGetLastError();
      return CZ_ERR_NOMEM;
    }
    if (cudaMemset(p, 0, kAlign) != cudaSuccess) return CZ_ERR_CUDA;
    w.ptr = p;
    w.bytes = need;
  }
  *out = w.ptr;
  return CZ_OK;
}

}  // namespace
}  // namespace cz

using namespace cz;

extern "C" {

void cz_step_opts_default(cz_step_opts* o) {
  if (!o) return;
  std::memset(o, 0, sizeof(*o));
  o->nesterov = 1;
  o->eps = 1e-7f;
  o->a = 3.4445f;
  o->b = -4.7750f;
  o->c = 2.0315f;
}

int cz_workspace_size(const cz_plan* plan, int32_t rank, const int64_t* shapes, size_t* bytes) {
  if (!plan || !shapes || !bytes) return CZ_ERR_INVALID;
  const Plan* p = static_cast<const Plan*>(plan);
  if (rank < 0 || rank >= p->R) return CZ_ERR_INVALID;
  int st = validate_shapes(p, shapes);
  if (st != CZ_OK) return st;
  Layout L;
  st = build_layout(p, rank, nullptr, shapes, L);
  if (st != CZ_OK) return st;
  *bytes = (size_t)L.bytes;
  return CZ_OK;
}

int cz_muon_step(const cz_plan* plan, int32_t rank, float* flat_param, const void* flat_grad, float* flat_mom,
                 const int64_t* offsets, const int64_t* shapes, float lr, float mu, int32_t ns_steps, void* stream) {
  cz_step_opts o;
  cz_step_opts_default(&o);
  return cz_muon_step_ex(plan, rank, flat_param, flat_grad, flat_mom, offsets, shapes, lr, mu, ns_steps, stream, &o);
}

}  // extern "C"

namespace cz {

int muon_step(const cz_plan* plan, int32_t rank, float* flat_param, const void* flat_grad, float* flat_mom,
              const int64_t* offsets, const int64_t* shapes, float lr, float mu, int32_t ns_steps, void* stream,
              const cz_step_opts* opts, bool pin_ok) {
  if (!plan || !flat_param || !flat_grad || !flat_mom || !offsets || !shapes || !opts) return CZ_ERR_INVALID;
  const Plan* p = static_cast<const Plan*>(plan);
  NvtxRange range("cz/muon_step");
  if (rank < 0 || rank >= p->R || ns_steps < 1 || ns_steps > 64) return CZ_ERR_INVALID;
  if (!std::isfinite(lr) || !std::isfinite(mu) || !std::isfinite(opts->eps) || opts->eps < 0.f) return CZ_ERR_INVALID;
  // the kernels move the flat buffers in 16-byte vectors (8 bytes for bf16 ones): their base
  // addresses must be aligned as any allocation is (a view at an odd element offset is rejected)
  auto aligned = [](const void* q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) & (a - 1)) == 0; };
  if (!aligned(flat_param, 16) || !aligned(flat_mom, 16) || !aligned(flat_grad, opts->grad_is_bf16 ? 8 : 16) ||
      !aligned(opts->param_bf16, 8) || !aligned(opts->debug_update_out, 16) || !aligned(opts->lr_device, 4))
    return CZ_ERR_INVALID;
  int st = validate_shapes(p, shapes);
  if (st != CZ_OK) return st;
  // parameters must not overlap in the flat layout
  {
    std::vector<std::pair<int64_t, int64_t>> iv(p->n_params);
    for (int64_t i = 0; i < p->n_params; ++i) {
      if (offsets[i] < 0) return CZ_ERR_INVALID;
      iv[i] = {offsets[i], offsets[i] + p->numels[i]};
    }
    std::sort(iv.begin(), iv.end());
    for (size_t i = 1; i < iv.size(); ++i)
      if (iv[i].first < iv[i - 1].second) return CZ_ERR_PLAN_MISMATCH;
  }
  bool any = false;
  for (int64_t i = 0; i < p->n_params; ++i) any |= (p->owner[i] == rank);
  if (!any) return CZ_OK;   // an empty shard: nothing to do
  st = check_device();
  if (st != CZ_OK) return st;

  size_t need = 0;
  st = cz_workspace_size(plan, rank, shapes, &need);
  if (st != CZ_OK) return st;

  std::lock_guard<std::mutex> lock(g_mu);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Inside a stream capture the call may only enqueue: no table build, no
  // allocation, no pageable upload (none of them can be captured).
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (note(cudaStreamIsCapturing(s, &cap)) != cudaSuccess) return CZ_ERR_CUDA;
  const bool capturing = cap != cudaStreamCaptureStatusNone;
  struct CaptureFlag {
    explicit CaptureFlag(bool on) { t_capturing = on; }
    ~CaptureFlag() { t_capturing = false; }
  } capture_flag(capturing);
  void* ws = opts->workspace;
  if (ws) {
    if (opts->workspace_bytes < need) return CZ_ERR_NOMEM;
    if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return CZ_ERR_INVALID;
  } else {
    st = get_internal_ws(need, &ws, capturing);
    if (st != CZ_OK) return st;
  }
  int dev = 0;
  cudaGetDevice(&dev);

  Key k;
  k.plan = p->uid; k.rank = rank; k.dev = dev;
  k.param = flat_param; k.grad = flat_grad; k.mom = flat_mom;
  k.pbf16 = opts->param_bf16; k.dbg = opts->debug_update_out; k.ws = ws;
  k.grad_bf16 = opts->grad_is_bf16 ? 1 : 0;
  k.offsets.assign(offsets, offsets + p->n_params);
  k.shapes.assign(shapes, shapes + 2 * p->n_params);
  std::shared_ptr<Program> prog;
  auto it = g_cache.find(k);
  if (it != g_cache.end()) {
    prog = it->second;
  } else {
    if (capturing) return CZ_ERR_INVALID;   // the first call for these buffers must run outside the capture
    prog = std::make_shared<Program>();
    st = build_program(p, rank, flat_param, flat_grad, flat_mom, offsets, shapes, lr, mu, ns_steps, *opts,
                       static_cast<uint8_t*>(ws), *prog);
    if (st != CZ_OK) return st;
    ++g_programs_built;
    if (pin_ok) pin_tables(*prog);
    if (g_cache.size() > 64) g_cache.clear();
    g_cache.emplace(k, prog);
  }
  // The tables (tile lists, per-tensor descriptors, zeroed counters) are copied
  // into the workspace on every call: the caller may have reused the workspace
  // memory for something else since the last call, even at the same address.
  const int64_t tbytes = prog->tables_end - prog->tables_begin;
  uint8_t* tdst = static_cast<uint8_t*>(ws) + prog->tables_begin;
  if (capturing && !prog->pinned) return CZ_ERR_INVALID;   // a pageable upload cannot be captured
  if (prog->pinned) {
    if (traced(1, s, [&] { return launch_tables_copy(prog->pinned_dev, tdst, tbytes, s); }) != cudaSuccess)
      return CZ_ERR_CUDA;
    if (capturing) prog->captured = true;
    else if (cudaEventRecord(prog->copied, s) != cudaSuccess) return CZ_ERR_CUDA;
  } else if (cudaMemcpyAsync(tdst, prog->host_tables.data(), (size_t)tbytes, cudaMemcpyHostToDevice, s) !=
             cudaSuccess) {
    return CZ_ERR_CUDA;
  }

  const Program& P = *prog;
  MomParams mp = P.mom;
  mp.nesterov = opts->nesterov ? 1 : 0;
  mp.mu = mu;
  mp.eps = opts->eps;
  if (traced(0, s, [&] { return launch_momentum(mp, s); }) != cudaSuccess) return CZ_ERR_CUDA;
  // joins the side stream back into s on every return path once it has been forked
  struct Join {
    cudaStream_t s = nullptr;
    cudaEvent_t ev = nullptr;
    ~Join() {
      if (ev) cudaStreamWaitEvent(s, ev, 0);
    }
  } join;
  if (P.small.n_mats > 0 || P.small_pair.n_mats > 0) {
    SmallParams sp = P.small, spp = P.small_pair;
    for (SmallParams* x : {&sp, &spp}) {
      x->ns_steps = ns_steps;
      x->a = opts->a; x->b = opts->b; x->c = opts->c; x->lr = lr; x->lr_dev = opts->lr_device;
    }
    auto single = [&](cudaStream_t st) {
      return sp.n_mats > 0 ? traced(7, st, [&] { return launch_ns_small(sp, st); }) : cudaSuccess;
    };
    auto pairs = [&](cudaStream_t st) {
      return spp.n_mats > 0 ? traced(7, st, [&] { return launch_ns_small_pair(spp, st); }) : cudaSuccess;
    };
    cudaStream_t side = (P.fork_small && !capturing) ? side_stream(s) : nullptr;
    if (side) {
      // side: the single-CTA launch, and the CTA-pair one too when tiled products
      // take s; otherwise the CTA-pair launch runs on s beside it
      if (cudaEventRecord(P.fork_ev, s) != cudaSuccess || cudaStreamWaitEvent(side, P.fork_ev, 0) != cudaSuccess)
        return CZ_ERR_CUDA;
      cudaError_t e = single(side);
      if (e == cudaSuccess && P.tiled) e = pairs(side);
      if (cudaEventRecord(P.join_ev, side) != cudaSuccess) return CZ_ERR_CUDA;
      join.s = s;
      join.ev = P.join_ev;
      if (e != cudaSuccess) return CZ_ERR_CUDA;
      if (!P.tiled && pairs(s) != cudaSuccess) return CZ_ERR_CUDA;
    } else if (single(s) != cudaSuccess || pairs(s) != cudaSuccess) {
      return CZ_ERR_CUDA;
    }
  }
  GemmParams gp;
  auto scalars = [&](GemmParams& g) {
    g.a = opts->a; g.b = opts->b; g.c = opts->c; g.lr = lr; g.lr_dev = opts->lr_device;
  };
  auto refused = [](cudaError_t e) {
    return e == cudaErrorCooperativeLaunchTooLarge || e == cudaErrorLaunchOutOfResources ||
           e == cudaErrorNotSupported || e == cudaErrorInvalidConfiguration;
  };
  if (P.fused_ok && use_fused() && ns_steps <= kMaxNsSteps) {
    gp = P.fused;
    gp.ns_steps = ns_steps;
    if (ns_steps != P.sched_steps) {   // the schedule is for another step count
      gp.sched = nullptr;
      gp.sched_first = nullptr;
    }
    scalars(gp);
    const cudaError_t e = traced(6, s, [&] { return launch_ns_gemm(P.fused_phase, P.pair, gp, s); });
    if (e == cudaSuccess) return CZ_OK;
    // The runtime refused the launch (e.g. it cannot guarantee that all units are
    // resident at once): clear the error and run one launch per product instead.
    if (e != cudaErrorCooperativeLaunchTooLarge && e != cudaErrorLaunchOutOfResources &&
        e != cudaErrorNotSupported && e != cudaErrorInvalidConfiguration)
      return CZ_ERR_CUDA;
    cudaGetLastError();
  }
  // One launch of a product.  A launch with pace_tiles >= 2 (make_launches: the
  // waves every unit has, heaviest tiles of at least kPaceMinKBlocks k-blocks) is
  // paced by a counter of its own, one per (step, product) in the fused launch's
  // completion counters (zeroed by every call's table copy; the fused launch does not
  // run in a call that takes this path).  The least advanced unit never waits, so the
  // pacing cannot deadlock once every unit is resident, which the cooperative
  // attribute guarantees; a refused cooperative launch runs again unpaced.
  int* pace_base = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + P.L.off_done);
  const size_t pace_stride = (size_t)std::max<size_t>(P.L.mats.size(), 1);
  auto run = [&](const Launch& ln, int phase, int kind, int first, int t, int slot) -> cudaError_t {
    gp = ln.params;
    gp.first = first;
    scalars(gp);
    gp.pace = (use_pace() && ln.pace_tiles >= 2) ? pace_base + (size_t)(t * 3 + slot) * pace_stride : nullptr;
    gp.pace_tiles = ln.pace_tiles;
    cudaError_t e = traced(kind, s, [&] { return launch_ns_gemm(phase, P.pair, gp, s); });
    if (e != cudaSuccess && gp.pace && refused(e)) {
      cudaGetLastError();
      gp.pace = nullptr;
      e = traced(kind, s, [&] { return launch_ns_gemm(phase, P.pair, gp, s); });
    }
    return e;
  };
  for (int t = 0; t < ns_steps; ++t) {
    const int first = t == 0 ? 1 : 0;
    const int cur = t & 1;
    for (const Launch& ln : P.gram[cur])
      if (run(ln, kGram, 2, first, t, 0) != cudaSuccess) return CZ_ERR_CUDA;
    for (const Launch& ln : P.poly)
      if (run(ln, kPoly, 3, 0, t, 1) != cudaSuccess) return CZ_ERR_CUDA;
    const bool final_step = t + 1 == ns_steps;
    const std::vector<Launch>& last = final_step ? P.apply[cur] : P.update[cur];
    for (const Launch& ln : last)
      if (run(ln, ln.phase, final_step ? 5 : 4, first, t, 2) != cudaSuccess) return CZ_ERR_CUDA;
  }
  return CZ_OK;
}

}  // namespace cz

extern "C" {

int cz_muon_step_ex(const cz_plan* plan, int32_t rank, float* flat_param, const void* flat_grad, float* flat_mom,
                    const int64_t* offsets, const int64_t* shapes, float lr, float mu, int32_t ns_steps, void* stream,
                    const cz_step_opts* opts) {
  return cz::muon_step(plan, rank, flat_param, flat_grad, flat_mom, offsets, shapes, lr, mu, ns_steps, stream, opts,
                       true);
}

int cz_step_programs_built(int64_t* count) {
  if (!count) return CZ_ERR_INVALID;
  std::lock_guard<std::mutex> lock(g_mu);
  *count = g_programs_built;
  return CZ_OK;
}

int cz_device_status(void* stream, void* workspace, int* status_out) {
  if (!status_out) return CZ_ERR_INVALID;
  *status_out = CZ_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return CZ_ERR_CUDA;
  // the status words to read: the caller's workspace, or every library-owned
  // scratch of the current device (the cached workspace of cz_muon_step(_ex) and
  // the static array of cz_muon_step_noalloc, where each has been set up)
  void* words[2] = {workspace, nullptr};
  if (!workspace) {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CZ_ERR_CUDA;
    auto it = g_ws.find(dev);
    words[0] = (it == g_ws.end()) ? nullptr : it->second.ptr;
    words[1] = noalloc_scratch_if_set_up();
  }
  for (void* ws : words) {
    if (!ws) continue;
    int v = 0;
    if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CZ_ERR_CUDA;
    if (v != 0 && cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return CZ_ERR_CUDA;
    if (*status_out == CZ_OK) *status_out = v;   // the first error found is reported; every word is cleared
  }
  return CZ_OK;
}

int cz_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = on != 0;
  return CZ_OK;
}

int cz_profile_read(double* ms, int64_t* launches, int32_t n_kinds) {
  if (!ms || !launches || n_kinds < 0 || n_kinds > CZ_KERNEL_KINDS) return CZ_ERR_INVALID;
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    recs.swap(g_prof);
  }
  for (int i = 0; i < n_kinds; ++i) {
    ms[i] = 0.0;
    launches[i] = 0;
  }
  int st = CZ_OK;
  for (ProfRec& r : recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) st = CZ_ERR_CUDA;
    if (r.kind < n_kinds) {
      ms[r.kind] += t;
      launches[r.kind] += 1;
    }
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  return st;
}

const char* cz_status_string(int status) {
  switch (status) {
    case CZ_OK: return "ok";
    case CZ_ERR_INVALID: return "invalid argument";
    case CZ_ERR_CUDA: return "CUDA call failed";
    case CZ_ERR_NOMEM: return "out of memory / workspace too small";
    case CZ_ERR_PLAN_MISMATCH: return "offsets/shapes do not match the plan";
    case CZ_ERR_TIMEOUT: return "device-side wait timed out";
    case CZ_ERR_DEVICE_CHECK: return "device-side check failed";
    case CZ_ERR_UNSUPPORTED: return "unsupported device or feature";
    default: return "unknown status";
  }
}

const char* cz_version(void) { return "cz 0.1 sm_103a"; }

const char* cz_last_cuda_error(void) {
  thread_local std::string msg;
  msg = std::string(cudaGetErrorName(t_last_cuda)) + ": " + cudaGetErrorString(t_last_cuda);
  return msg.c_str();
}

}  // extern "C"
