// Host runtime and C ABI of the Muon step (declared in include/muon.h).
//
// A call validates its descriptors on the host, finds or builds the plan for
// its matrix shapes (grouping by oriented shape, workspace, tensor maps, tile
// lists), then queues the kernels on the caller's stream:
//
//   muon_step:          momentum+norm -> scale/orient -> k x (Gram, combine) -> update
//   muon_orthogonalize: norm          -> scale/orient -> k x (Gram, combine) -> copy out
//
// With c != 0 each iteration runs a second Gram pass (A A, with b A added in
// its epilogue) between the two.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <queue>
#include <utility>
#include <memory>
#include <string>
#include <vector>

#include "../../include/muon.h"
#include "elementwise.cuh"
#include "ns_fused.cuh"
#include "ns_gemm.cuh"

using namespace muon;

namespace {

// Paired-SM MMAs (tcgen05 cta_group::2): each CTA holds half of B, so a stage is 32 KB and five fit
// beside the 64 KB of epilogue staging.
constexpr int kGramBN = 256, kGramStages = 5;
constexpr int kCombBN = 256, kCombStages = 5;
// Kernel parameters are limited to 32764 bytes.
static_assert(sizeof(GemmArgs) + sizeof(FinalArgs<kMaxFinal>) <= 32764, "GEMM parameter block too large");
using GramShape = GemmShape<true, kGramBN, kGramStages>;
using CombShape = GemmShape<false, kCombBN, kCombStages>;
// The persistent launch running every iteration (ns_fused.cuh).
constexpr int kFusedStages = 5;
using FusedShape = GemmShape<true, 256, kFusedStages>;
static_assert(sizeof(FusedArgs) + sizeof(FinalArgs<kMaxFinal>) <= 32764, "fused parameter block too large");
// The persistent schedule's model, in units of one 64-wide k-block of a 256 x 256 tile (512
// tensor-core cycles of the pair):
// matrix state (both X buffers, B, A) admitted at once. Larger budgets schedule better: with
// 150 MB the GPT-2 124M step took 1.0906 ms, with 512 MB 1.0867 ms and with 2 GB 1.0708 ms, so the
// cap matters only for batches far larger than that set;
constexpr double kFusedL2Budget = 512e6;
// what a tile occupies its cluster for beyond its MMAs;
constexpr int kFusedTileOverhead = 3;
// from a tile's last MMA until the next stage of its matrix can use the result (epilogue drain,
// store, counter, first operand loads). Planned with 32, the lists left the producers waiting on
// counters about 7% of the kernel on the GPT-2 124M step; with 0, 44%.
constexpr double kFusedLatency = 32.0;

constexpr int64_t kMaxDim = 1 << 20;          // rows or cols
constexpr int64_t kMaxShort = 32768;          // min(rows, cols): the n x n Gram lives in workspace
constexpr int64_t kMaxElems = 1ll << 32;      // rows * cols
constexpr int kMaxSteps = 100000;

const char* kKernelNames[MUON_KERNEL_KINDS] = {"momentum_norm", "norm",   "scale_orient", "gram_xxt",
                                               "gram_aa",       "combine_ax_bx", "update", "copy_out",
                                               "newton_schulz"};

enum Kind { K_MOMENTUM = 0, K_NORM = 1, K_SCALE = 2, K_GRAM = 3, K_GRAM_AA = 4, K_COMBINE = 5, K_UPDATE = 6,
            K_COPY = 7, K_FUSED = 8 };

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
int64_t ceil_div(int64_t x, int64_t m) { return (x + m - 1) / m; }

size_t elem_size(int32_t dt) { return dt == MUON_F32 ? 4 : 2; }

void put_msg(char* msg, int len, const char* fmt, ...) {
  if (!msg || len <= 0) return;
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(msg, static_cast<size_t>(len), fmt, ap);
  va_end(ap);
}

bool dims_ok(const muon_matrix& m, const char* what, int j, char* msg, int len) {
  if (m.rows < 0 || m.cols < 0 || m.rows > kMaxDim || m.cols > kMaxDim) {
    put_msg(msg, len, "%s[%d]: shape %lld x %lld out of range", what, j, (long long)m.rows, (long long)m.cols);
    return false;
  }
  if (m.dtype != MUON_F32 && m.dtype != MUON_BF16) {
    put_msg(msg, len, "%s[%d]: unknown dtype %d", what, j, (int)m.dtype);
    return false;
  }
  if (m.rows == 0 || m.cols == 0) return true;
  if (std::min(m.rows, m.cols) > kMaxShort || m.rows * m.cols > kMaxElems) {
    put_msg(msg, len, "%s[%d]: shape %lld x %lld too large", what, j, (long long)m.rows, (long long)m.cols);
    return false;
  }
  if (m.ld < m.cols) {
    put_msg(msg, len, "%s[%d]: ld %lld < cols %lld", what, j, (long long)m.ld, (long long)m.cols);
    return false;
  }
  if (m.ptr == nullptr) {
    put_msg(msg, len, "%s[%d]: null pointer", what, j);
    return false;
  }
  return true;
}

struct Range {
  uintptr_t lo, hi;
  int who;
};

// Byte range touched by a matrix: [ptr, ptr + ((rows-1)*ld + cols) * size).
Range range_of(const muon_matrix& m, int who) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(m.ptr);
  const uintptr_t n = static_cast<uintptr_t>((m.rows - 1) * m.ld + m.cols) * elem_size(m.dtype);
  return {lo, lo + n, who};
}

bool any_overlap(std::vector<Range> r, int* a, int* b) {
  std::sort(r.begin(), r.end(), [](const Range& x, const Range& y) { return x.lo < y.lo; });
  uintptr_t hi = 0;
  int hi_who = -1;
  for (size_t i = 0; i < r.size(); ++i) {
    if (i > 0 && r[i].lo < hi) {
      *a = hi_who;
      *b = r[i].who;
      return true;
    }
    if (r[i].hi > hi) {
      hi = r[i].hi;
      hi_who = r[i].who;
    }
  }
  return false;
}

// ------------------------------------------------------------------ plan

struct MatInfo {
  int64_t rows = 0, cols = 0;
  bool skip = false;     // zero-sized
  bool transposed = false;
  int group = -1, idx = -1;  // shape group and position within it
  int64_t n = 0, m = 0;      // oriented shape
  int64_t nchunks = 0;       // norm partials: blocks of the flat or the transposed-tile decomposition
  int64_t partial_off = 0;
  int gslot = -1;            // index in group order (group's first slot + idx)
};

struct Group {
  int64_t n = 0, m = 0;
  int count = 0;
  int first_slot = 0;  // the group's first matrix in group order
  int64_t ld_x = 0, ld_p = 0;
  size_t x_off[2] = {0, 0}, p_off = 0, a_off = 0;  // byte offsets in the workspace
  size_t lo_off[2] = {0, 0};  // precise carry: low parts of X, laid out like X (allocated only then)
};

struct GemmBatch {           // up to kMaxGroups groups served by one launch
  int first_group = 0, num_groups = 0;
  int4* gram_tiles = nullptr;
  int* gram_begin = nullptr;
  int num_gram_tiles = 0, gram_grid = 0;
  int4* comb_tiles = nullptr;
  int* comb_begin = nullptr;
  int num_comb_tiles = 0, comb_grid = 0;
  GemmArgs gram[2];          // X_t -> b A in the B buffer, t parity
  GemmArgs gram_to_a[2];     // X_t -> A in the A buffer (c != 0)
  GemmArgs gram_aa;          // A -> c A A + b A
  GemmArgs comb[2];          // (B, X_t) -> X_{t+1}
};

struct Plan {
  std::vector<std::pair<int64_t, int64_t>> key;
  bool carry = false;  // X carried as bf16 hi + lo: low-part buffers exist and the kernels use them
  std::vector<MatInfo> mats;
  std::vector<Group> groups;
  std::vector<GemmBatch> batches;
  uint8_t* ws = nullptr;
  size_t ws_bytes = 0;
  size_t dev_bytes = 0;  // device memory this plan holds (workspace and tile schedules)
  float* partial = nullptr;
  int* tickets = nullptr;
  float* inv = nullptr;
  float* post = nullptr;   // group order: scale folded into the first iteration's products
  int4* tiles_dev = nullptr;
  int* begin_dev = nullptr;
  uint64_t last_use = 0;
  // Writing the last combine's result straight into the caller's matrices: tensor maps of the
  // caller's matrices (re-encoded when a pointer or ld changes) and one argument block per batch.
  struct UserMap {
    const void* ptr = nullptr;
    int64_t ld = -1;
    CUtensorMap map;
  };
  std::vector<UserMap> user_maps;
  std::vector<std::unique_ptr<FinalArgs<kMaxFinal>>> fin;
  // The persistent launch: tensor maps [group][role] and group table in device memory, per-matrix
  // stage counters and the finish ticket in the workspace, and one item schedule per
  // (iteration count, c != 0), built on first use.
  CUtensorMap* maps_dev = nullptr;
  NsGroup* groups_dev = nullptr;
  int* counters = nullptr;
  unsigned int* done = nullptr;
  struct FusedSchedule {
    int4* items = nullptr;
    int* begin = nullptr;
    int grid = 0;      // clusters
    size_t bytes = 0;
  };
  std::map<std::pair<int, int>, FusedSchedule> fused;
  std::unique_ptr<FinalArgs<kMaxFinal>> fin_slots;  // the last combine's caller maps, by matrix slot
};

}  // namespace

struct muon_ctx {
  int device = 0;
  int num_sms = 0;
  int max_lists = 0;  // GEMM tile lists run at once: co-resident clusters (or CTAs)
  muon_config cfg{};
  int* err_dev = nullptr;            // 256 bytes: the error flag at 0, the profiling clock sums at 64
  unsigned long long* clk_dev = nullptr;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  // Plans by (matrix shapes, precise carry).
  std::map<std::pair<std::vector<std::pair<int64_t, int64_t>>, bool>, std::unique_ptr<Plan>> plans;
  uint64_t use_clock = 0;
  std::string last_error;
  // profiling
  bool profiling = false;
  struct Rec {
    int kind;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> event_pool;
  // Device memory held by the plans, and the cap on it (0: none; muon_set_workspace_limit).
  size_t plan_bytes = 0;
  size_t plan_limit = 0;
  int launch_mode = MUON_PERSISTENT_AUTO;  // muon_config.persistent
};

namespace {

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

muon_status fail(muon_handle h, muon_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (h) h->last_error = buf;
  return s;
}

muon_status cuda_fail(muon_handle h, cudaError_t e, const char* where) {
  return fail(h, MUON_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

cudaEvent_t pooled_event(muon_handle h) {
  if (!h->event_pool.empty()) {
    cudaEvent_t e = h->event_pool.back();
    h->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

struct ProfScope {
  muon_handle h;
  int kind;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  ProfScope(muon_handle h_, int kind_, cudaStream_t s_) : h(h_), kind(kind_), s(s_) {
    if (h->profiling) {
      a = pooled_event(h);
      cudaEventRecord(a, s);
    }
  }
  ~ProfScope() {
    if (h->profiling && a) {
      cudaEvent_t b = pooled_event(h);
      cudaEventRecord(b, s);
      h->recs.push_back({kind, a, b});
    }
  }
};

bool encode_map(muon_handle h, CUtensorMap* map, void* base, int64_t inner, int64_t rows, int64_t count,
                int64_t ld, int box_inner, int box_rows, bool swizzle = true) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(count)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2), static_cast<cuuint64_t>(rows * ld * 2)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = h->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                               CU_TENSOR_MAP_INTERLEAVE_NONE,
                               swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Groups matrices by oriented shape (n <= m), in order of first appearance.
void group_shapes(const std::vector<std::pair<int64_t, int64_t>>& shapes, std::vector<MatInfo>& mats,
                  std::vector<Group>& groups) {
  mats.assign(shapes.size(), MatInfo{});
  std::map<std::pair<int64_t, int64_t>, int> gid;
  for (size_t j = 0; j < shapes.size(); ++j) {
    MatInfo& mi = mats[j];
    mi.rows = shapes[j].first;
    mi.cols = shapes[j].second;
    if (mi.rows == 0 || mi.cols == 0) {
      mi.skip = true;
      continue;
    }
    mi.transposed = mi.rows > mi.cols;
    mi.n = std::min(mi.rows, mi.cols);
    mi.m = std::max(mi.rows, mi.cols);
    auto it = gid.find({mi.n, mi.m});
    if (it == gid.end()) {
      it = gid.emplace(std::make_pair(mi.n, mi.m), static_cast<int>(groups.size())).first;
      Group g;
      g.n = mi.n;
      g.m = mi.m;
      g.ld_x = round_up(mi.m, 8);
      g.ld_p = round_up(mi.n, 8);
      groups.push_back(g);
    }
    mi.group = it->second;
    mi.idx = groups[mi.group].count++;
    mi.nchunks = std::max(ceil_div(mi.rows * mi.cols, kFlatChunk), ceil_div(mi.rows, 128) * ceil_div(mi.cols, kTile));
  }
  int slot = 0;
  for (Group& g : groups) {
    g.first_slot = slot;
    slot += g.count;
  }
  for (MatInfo& mi : mats)
    if (!mi.skip) mi.gslot = groups[mi.group].first_slot + mi.idx;
}

// One GEMM launch's schedule: tiles grouped by CTA, and CTA b's range
// [begin[b], begin[b+1]) in `tiles`.
struct Schedule {
  std::vector<int4> tiles;
  std::vector<int> begin;
};

// Longest-processing-time-first assignment: tiles sorted by contraction
// length, each given to the CTA with the least work so far. Every CTA's list
// stays in decreasing-cost order.
Schedule lpt_schedule(std::vector<std::pair<int4, int64_t>> work, int max_lists) {
  std::stable_sort(work.begin(), work.end(),
                   [](const std::pair<int4, int64_t>& x, const std::pair<int4, int64_t>& y) { return x.second > y.second; });
  Schedule sc;
  const int ctas = static_cast<int>(std::min<size_t>(work.size(), static_cast<size_t>(std::max(1, max_lists))));
  std::vector<std::vector<int4>> per(ctas);
  using Load = std::pair<int64_t, int>;
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int b = 0; b < ctas; ++b) heap.push({0, b});
  for (const auto& w : work) {
    Load l = heap.top();
    heap.pop();
    per[l.second].push_back(w.first);
    heap.push({l.first + w.second, l.second});
  }
  sc.begin.push_back(0);
  for (int b = 0; b < ctas; ++b) {
    sc.tiles.insert(sc.tiles.end(), per[b].begin(), per[b].end());
    sc.begin.push_back(static_cast<int>(sc.tiles.size()));
  }
  return sc;
}

// Gram and combine schedules of one batch of groups. A tile's cost is its
// number of k-blocks times its width in 128-column units. Gram tiles are
// 128 x 256 and cover the upper triangle: tile row I <= 2J + 1 in tile column J.
// Within a matrix both run column by column, so the tiles that run at once (one
// per cluster, in list order) share their B operand block: for a combine, the
// 256 columns of X every row pair of the column multiplies. Row-major order would
// put 74 different column blocks of X in flight at once; on a 4096 x 16384
// matrix that read X from DRAM once per row pair (1.84 GB per launch).
void build_tiles(const std::vector<Group>& groups, int g0, int ng, int max_lists, Schedule& gram, Schedule& comb) {
  std::vector<std::pair<int4, int64_t>> gt, ct;
  for (int gi = 0; gi < ng; ++gi) {
    const Group& g = groups[g0 + gi];
    const int nt = static_cast<int>(ceil_div(g.n, 128));
    const int gt2 = static_cast<int>(ceil_div(g.n, kGramBN));
    const int mt = static_cast<int>(ceil_div(g.m, kCombBN));
    // With clusters, an entry is the first tile row of a group of kCluster consecutive rows.
    for (int b = 0; b < g.count; ++b) {
      for (int J = 0; J < gt2; ++J)
        for (int I = 0; I < std::min(2 * J + 2, nt); I += kCluster)
          gt.push_back({make_int4(gi, b, I, J), 2 * ceil_div(g.m, 64)});
      for (int J = 0; J < mt; ++J)
        for (int I = 0; I < nt; I += kCluster) ct.push_back({make_int4(gi, b, I, J), 2 * ceil_div(g.n, 64)});
    }
  }
  gram = lpt_schedule(std::move(gt), max_lists);
  comb = lpt_schedule(std::move(ct), max_lists);
}

void free_plan(muon_handle h, Plan* p) {
  if (!p) return;
  if (p->ws) cudaFree(p->ws);
  if (p->tiles_dev) cudaFree(p->tiles_dev);
  if (p->begin_dev) cudaFree(p->begin_dev);
  if (p->maps_dev) cudaFree(p->maps_dev);
  for (auto& kv : p->fused)  // items and list offsets share one allocation
    if (kv.second.items) cudaFree(kv.second.items);
  p->fused.clear();
  p->ws = nullptr;
  p->tiles_dev = nullptr;
  p->begin_dev = nullptr;
  p->maps_dev = nullptr;
  p->groups_dev = nullptr;
  h->plan_bytes -= p->dev_bytes;
  p->dev_bytes = 0;
}

// cudaMalloc for plan memory. Past the handle's cap it fails the way an exhausted device does
// (cudaErrorMemoryAllocation), so both take the same out-of-memory path.
cudaError_t plan_malloc(muon_handle h, Plan& P, void** ptr, size_t bytes) {
  if (h->plan_limit != 0 && h->plan_bytes + bytes > h->plan_limit) return cudaErrorMemoryAllocation;
  const cudaError_t e = cudaMalloc(ptr, bytes);
  if (e == cudaSuccess) {
    P.dev_bytes += bytes;
    h->plan_bytes += bytes;
  }
  return e;
}

muon_status build_plan(muon_handle h, const std::vector<std::pair<int64_t, int64_t>>& key, bool carry, Plan** out) {
  auto plan = std::make_unique<Plan>();
  Plan& P = *plan;
  P.key = key;
  P.carry = carry;
  group_shapes(key, P.mats, P.groups);

  // Workspace: per group X ping/pong [count][n][ld_x], B and A [count][n][ld_p];
  // then per matrix partial sums, tickets and the inverse norm.
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = static_cast<size_t>(round_up(static_cast<int64_t>(off + bytes), 256));
    return o;
  };
  for (Group& g : P.groups) {
    const size_t xb = static_cast<size_t>(g.count) * g.n * g.ld_x * 2;
    const size_t pb = static_cast<size_t>(g.count) * g.n * g.ld_p * 2;
    g.x_off[0] = take(xb);
    g.x_off[1] = take(xb);
    g.p_off = take(pb);
    g.a_off = take(pb);
    if (P.carry) {
      g.lo_off[0] = take(xb);
      g.lo_off[1] = take(xb);
    }
  }
  int64_t nparts = 0;
  for (MatInfo& mi : P.mats) {
    mi.partial_off = nparts;
    nparts += mi.nchunks;
  }
  const size_t part_off = take(static_cast<size_t>(std::max<int64_t>(nparts, 1)) * 4);
  const size_t tick_off = take(P.mats.size() * 4 + 4);
  const size_t inv_off = take(P.mats.size() * 4 + 4);
  const size_t post_off = take(P.mats.size() * 4 + 4);
  const size_t cnt_off = take(P.mats.size() * 4 + 4);
  const size_t done_off = take(16);
  P.ws_bytes = off;

  cudaError_t e = plan_malloc(h, P, reinterpret_cast<void**>(&P.ws), P.ws_bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    free_plan(h, &P);
    return fail(h, MUON_ERR_NOMEM, "workspace of %zu bytes: %s", P.ws_bytes, cudaGetErrorString(e));
  }
  P.partial = reinterpret_cast<float*>(P.ws + part_off);
  P.tickets = reinterpret_cast<int*>(P.ws + tick_off);
  P.inv = reinterpret_cast<float*>(P.ws + inv_off);
  P.post = reinterpret_cast<float*>(P.ws + post_off);
  P.counters = reinterpret_cast<int*>(P.ws + cnt_off);
  P.done = reinterpret_cast<unsigned int*>(P.ws + done_off);
  e = cudaMemset(P.ws, 0, P.ws_bytes);
  if (e != cudaSuccess) {
    free_plan(h, &P);
    return cuda_fail(h, e, "workspace clear");
  }

  // GEMM batches and their schedules.
  std::vector<int4> all_tiles;
  std::vector<int> all_begin;
  struct Offs {
    size_t gt, gb, ct, cb;
  };
  std::vector<Offs> offs;
  for (int g0 = 0; g0 < static_cast<int>(P.groups.size()); g0 += kMaxGroups) {
    GemmBatch B;
    B.first_group = g0;
    B.num_groups = std::min<int>(kMaxGroups, static_cast<int>(P.groups.size()) - g0);
    Schedule gs, cs;
    build_tiles(P.groups, g0, B.num_groups, h->max_lists, gs, cs);
    B.num_gram_tiles = static_cast<int>(gs.tiles.size());
    B.gram_grid = static_cast<int>(gs.begin.size()) - 1;
    B.num_comb_tiles = static_cast<int>(cs.tiles.size());
    B.comb_grid = static_cast<int>(cs.begin.size()) - 1;
    Offs o{all_tiles.size(), all_begin.size(), 0, 0};
    all_tiles.insert(all_tiles.end(), gs.tiles.begin(), gs.tiles.end());
    all_begin.insert(all_begin.end(), gs.begin.begin(), gs.begin.end());
    o.ct = all_tiles.size();
    o.cb = all_begin.size();
    all_tiles.insert(all_tiles.end(), cs.tiles.begin(), cs.tiles.end());
    all_begin.insert(all_begin.end(), cs.begin.begin(), cs.begin.end());
    offs.push_back(o);
    P.batches.push_back(B);
  }
  if (!all_tiles.empty()) {
    e = plan_malloc(h, P, reinterpret_cast<void**>(&P.tiles_dev), all_tiles.size() * sizeof(int4));
    cudaError_t e2 = e != cudaSuccess ? e
                                      : plan_malloc(h, P, reinterpret_cast<void**>(&P.begin_dev),
                                                    all_begin.size() * sizeof(int));
    if (e != cudaSuccess || e2 != cudaSuccess) {
      cudaGetLastError();
      free_plan(h, &P);
      return fail(h, MUON_ERR_NOMEM, "tile schedule: %s", cudaGetErrorString(e != cudaSuccess ? e : e2));
    }
    e = cudaMemcpy(P.tiles_dev, all_tiles.data(), all_tiles.size() * sizeof(int4), cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
      e = cudaMemcpy(P.begin_dev, all_begin.data(), all_begin.size() * sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      free_plan(h, &P);
      return cuda_fail(h, e, "tile schedule upload");
    }
  }

  for (size_t bi = 0; bi < P.batches.size(); ++bi) {
    GemmBatch& B = P.batches[bi];
    B.gram_tiles = P.tiles_dev + offs[bi].gt;
    B.gram_begin = P.begin_dev + offs[bi].gb;
    B.comb_tiles = P.tiles_dev + offs[bi].ct;
    B.comb_begin = P.begin_dev + offs[bi].cb;
    GemmArgs base;
    memset(&base, 0, sizeof(base));
    base.num_groups = B.num_groups;
    base.err = h->err_dev;
    for (int t = 0; t < 2; ++t) {
      B.gram[t] = base;
      B.comb[t] = base;
      B.gram[t].tiles = B.gram_tiles;
      B.gram[t].cta_begin = B.gram_begin;
      B.gram[t].num_tiles = B.num_gram_tiles;
      B.gram[t].grid = B.gram_grid;
      B.comb[t].tiles = B.comb_tiles;
      B.comb[t].cta_begin = B.comb_begin;
      B.comb[t].num_tiles = B.num_comb_tiles;
      B.comb[t].grid = B.comb_grid;
    }
    B.gram_aa = B.gram[0];
    B.gram_to_a[0] = B.gram[0];
    B.gram_to_a[1] = B.gram[1];
    for (int gi = 0; gi < B.num_groups; ++gi) {
      const Group& g = P.groups[B.first_group + gi];
      uint8_t* xb[2] = {P.ws + g.x_off[0], P.ws + g.x_off[1]};
      uint16_t* pbuf = reinterpret_cast<uint16_t*>(P.ws + g.p_off);
      uint16_t* abuf = reinterpret_cast<uint16_t*>(P.ws + g.a_off);
      bool ok = true;
      for (int t = 0; t < 2; ++t) {
        // Gram on X_t: both operands are rows of X_t (K-major), output n x n.
        ok &= encode_map(h, &B.gram[t].map_a[gi], xb[t], g.m, g.n, g.count, g.ld_x, 64, 128);
        B.gram[t].map_b[gi] = B.gram[t].map_a[gi];
        ok &= encode_map(h, &B.gram[t].map_out[gi], pbuf, g.n, g.n, g.count, g.ld_p, 64, 128);
        ok &= encode_map(h, &B.gram[t].map_mirror[gi], pbuf, g.n, g.n, g.count, g.ld_p, 128, 64, false);
        B.gram[t].grp[gi] = GemmGroup{nullptr, nullptr, g.n * g.ld_p, static_cast<int>(g.n), static_cast<int>(g.n),
                                      static_cast<int>(g.ld_p), static_cast<int>(ceil_div(g.m, 64))};
        // The same Gram writing A = X X^T into the A buffer (first pass when c != 0).
        B.gram_to_a[t].map_a[gi] = B.gram[t].map_a[gi];
        B.gram_to_a[t].map_b[gi] = B.gram[t].map_b[gi];
        B.gram_to_a[t].grp[gi] = B.gram[t].grp[gi];
        ok &= encode_map(h, &B.gram_to_a[t].map_out[gi], abuf, g.n, g.n, g.count, g.ld_p, 64, 128);
        ok &= encode_map(h, &B.gram_to_a[t].map_mirror[gi], abuf, g.n, g.n, g.count, g.ld_p, 128, 64, false);
        // Combine: A operand = B (n x n, K-major), B operand = X_t MN-major, out = X_{1-t}, addend X_t.
        ok &= encode_map(h, &B.comb[t].map_a[gi], pbuf, g.n, g.n, g.count, g.ld_p, 64, 128);
        ok &= encode_map(h, &B.comb[t].map_b[gi], xb[t], g.m, g.n, g.count, g.ld_x, 64, 64);
        ok &= encode_map(h, &B.comb[t].map_out[gi], xb[1 - t], g.m, g.n, g.count, g.ld_x, 64, 128);
        ok &= encode_map(h, &B.comb[t].map_e[gi], xb[t], g.m, g.n, g.count, g.ld_x, 64, 128);
        B.comb[t].grp[gi] = GemmGroup{reinterpret_cast<uint16_t*>(xb[t]), nullptr, g.n * g.ld_x, static_cast<int>(g.n),
                                      static_cast<int>(g.m), static_cast<int>(g.ld_x),
                                      static_cast<int>(ceil_div(g.n, 64))};
        if (P.carry) {  // addend and output low parts, laid out like X
          uint8_t* lb[2] = {P.ws + g.lo_off[0], P.ws + g.lo_off[1]};
          ok &= encode_map(h, &B.comb[t].map_e_lo[gi], lb[t], g.m, g.n, g.count, g.ld_x, 64, 128);
          ok &= encode_map(h, &B.comb[t].map_out_lo[gi], lb[1 - t], g.m, g.n, g.count, g.ld_x, 64, 128);
          B.comb[t].carry = 1;
        }
      }
      // A A pass: operands are rows of A (symmetric), addend A, output B.
      ok &= encode_map(h, &B.gram_aa.map_a[gi], abuf, g.n, g.n, g.count, g.ld_p, 64, 128);
      B.gram_aa.map_b[gi] = B.gram_aa.map_a[gi];
      ok &= encode_map(h, &B.gram_aa.map_out[gi], pbuf, g.n, g.n, g.count, g.ld_p, 64, 128);
      ok &= encode_map(h, &B.gram_aa.map_mirror[gi], pbuf, g.n, g.n, g.count, g.ld_p, 128, 64, false);
      ok &= encode_map(h, &B.gram_aa.map_e[gi], abuf, g.n, g.n, g.count, g.ld_p, 64, 128);
      B.gram_aa.grp[gi] = GemmGroup{abuf, nullptr, g.n * g.ld_p, static_cast<int>(g.n), static_cast<int>(g.n),
                                    static_cast<int>(g.ld_p), static_cast<int>(ceil_div(g.n, 64))};
      if (!ok) {
        free_plan(h, &P);
        return fail(h, MUON_ERR_CUDA, "cuTensorMapEncodeTiled failed for group %lld x %lld", (long long)g.n,
                    (long long)g.m);
      }
    }
  }
  // Tensor maps and group table of the persistent launch.
  if (!P.groups.empty()) {
    const size_t ng = P.groups.size();
    std::vector<CUtensorMap> maps(ng * kNumRoles);
    std::vector<NsGroup> gt(ng);
    for (size_t gi = 0; gi < ng; ++gi) {
      const Group& g = P.groups[gi];
      CUtensorMap* m = &maps[gi * kNumRoles];
      uint8_t* xb[2] = {P.ws + g.x_off[0], P.ws + g.x_off[1]};
      uint8_t* pbuf = P.ws + g.p_off;
      uint8_t* abuf = P.ws + g.a_off;
      bool ok = true;
      for (int t = 0; t < 2; ++t) {
        ok &= encode_map(h, &m[kRoleX0 + t], xb[t], g.m, g.n, g.count, g.ld_x, 64, 128);
        ok &= encode_map(h, &m[kRoleXmn0 + t], xb[t], g.m, g.n, g.count, g.ld_x, 64, 64);
        // Without the precise carry the low-part roles are never used; they hold valid maps of X.
        uint8_t* lb = P.carry ? P.ws + g.lo_off[t] : xb[t];
        ok &= encode_map(h, &m[kRoleLo0 + t], lb, g.m, g.n, g.count, g.ld_x, 64, 128);
      }
      ok &= encode_map(h, &m[kRoleP], pbuf, g.n, g.n, g.count, g.ld_p, 64, 128);
      ok &= encode_map(h, &m[kRolePm], pbuf, g.n, g.n, g.count, g.ld_p, 128, 64, false);
      ok &= encode_map(h, &m[kRoleA], abuf, g.n, g.n, g.count, g.ld_p, 64, 128);
      ok &= encode_map(h, &m[kRoleAm], abuf, g.n, g.n, g.count, g.ld_p, 128, 64, false);
      if (!ok) {
        free_plan(h, &P);
        return fail(h, MUON_ERR_CUDA, "cuTensorMapEncodeTiled failed for group %lld x %lld", (long long)g.n,
                    (long long)g.m);
      }
      gt[gi] = NsGroup{static_cast<int>(g.n), static_cast<int>(g.m), g.count, g.first_slot,
                       static_cast<int>(ceil_div(g.m, 64)), static_cast<int>(ceil_div(g.n, 64))};
    }
    const size_t mb = maps.size() * sizeof(CUtensorMap), gb = gt.size() * sizeof(NsGroup);
    e = plan_malloc(h, P, reinterpret_cast<void**>(&P.maps_dev), mb + gb);
    if (e != cudaSuccess) {
      cudaGetLastError();
      free_plan(h, &P);
      return fail(h, MUON_ERR_NOMEM, "tensor maps: %s", cudaGetErrorString(e));
    }
    P.groups_dev = reinterpret_cast<NsGroup*>(reinterpret_cast<uint8_t*>(P.maps_dev) + mb);
    e = cudaMemcpy(P.maps_dev, maps.data(), mb, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(P.groups_dev, gt.data(), gb, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      free_plan(h, &P);
      return cuda_fail(h, e, "tensor map upload");
    }
  }
  // The clear above ran on the legacy stream; the caller's stream may not be ordered after it.
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    free_plan(h, &P);
    return cuda_fail(h, e, "plan synchronize");
  }
  *out = plan.get();
  h->plans[std::make_pair(key, carry)] = std::move(plan);
  return MUON_OK;
}

muon_status get_plan(muon_handle h, const std::vector<std::pair<int64_t, int64_t>>& key, bool carry, Plan** out) {
  auto it = h->plans.find(std::make_pair(key, carry));
  if (it != h->plans.end()) {
    it->second->last_use = ++h->use_clock;
    *out = it->second.get();
    return MUON_OK;
  }
  if (h->plans.size() >= 16) {  // drop the least recently used plan
    auto victim = h->plans.begin();
    for (auto i = h->plans.begin(); i != h->plans.end(); ++i)
      if (i->second->last_use < victim->second->last_use) victim = i;
    cudaDeviceSynchronize();
    free_plan(h, victim->second.get());
    h->plans.erase(victim);
  }
  muon_status s = build_plan(h, key, carry, out);
  if (s == MUON_OK) (*out)->last_use = ++h->use_clock;
  return s;
}

// Where matrix mi's X_t (t = 0, 1: the ping-pong pair) lives in the workspace.
uint16_t* x_slot(const Plan& P, const MatInfo& mi, int t) {
  const Group& g = P.groups[mi.group];
  return reinterpret_cast<uint16_t*>(P.ws + g.x_off[t]) + static_cast<int64_t>(mi.idx) * g.n * g.ld_x;
}

// Where matrix mi's low parts of X_t live (precise carry), or nullptr without the carry.
uint16_t* lo_slot(const Plan& P, const MatInfo& mi, int t) {
  const Group& g = P.groups[mi.group];
  if (g.lo_off[t] == 0) return nullptr;
  return reinterpret_cast<uint16_t*>(P.ws + g.lo_off[t]) + static_cast<int64_t>(mi.idx) * g.n * g.ld_x;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ launches

// Launches with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream finishes, and waits for it in-kernel
// (griddepcontrol.wait) before touching its outputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(block), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The result of one launch: its own return code (an error left over from an unrelated earlier
// call is not this launch's failure), then the launch error state, which it clears.
muon_status launch_checked(muon_handle h, cudaError_t launch, const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (launch != cudaSuccess) return cuda_fail(h, launch, what);
  (void)e;
  return MUON_OK;
}

// Norm pass (kStep = false: u = input, nothing written) or momentum + norm (kStep = true:
// u written in the Newton-Schulz orientation into the first X buffer, unscaled; the scale is
// folded into the first iteration, or applied in place by the kernel for norms outside the fold range).
template <bool kStep>
muon_status launch_momentum(muon_handle h, const Plan& P, const muon_matrix* src, const muon_matrix* buf, float beta,
                            int nesterov, int force_rescale, cudaStream_t s) {
  const bool f32 = [&] {
    for (size_t j = 0; j < P.mats.size(); ++j)
      if (!P.mats[j].skip) return src[j].dtype == MUON_F32;
    return false;
  }();
  MomArgs a;
  memset(&a, 0, sizeof(a));
  a.beta = beta;
  a.nesterov = nesterov ? 1 : 0;
  a.eps = h->cfg.eps;
  a.force_rescale = force_rescale;
  int blocks = 0;
  auto flush = [&]() -> muon_status {
    if (a.count == 0) return MUON_OK;
    ProfScope ps(h, kStep ? K_MOMENTUM : K_NORM, s);
    const cudaError_t e = f32 ? launch_pdl(momentum_norm_kernel<kStep, true>, blocks, kEwThreads, 0, s, a)
                              : launch_pdl(momentum_norm_kernel<kStep, false>, blocks, kEwThreads, 0, s, a);
    a.count = 0;
    blocks = 0;
    return launch_checked(h, e, "momentum/norm kernel");
  };
  for (size_t j = 0; j < P.mats.size(); ++j) {
    const MatInfo& mi = P.mats[j];
    if (mi.skip) continue;
    const Group& g = P.groups[mi.group];
    MomMat& M = a.m[a.count];
    M.g = src[j].ptr;
    M.ld_g = src[j].ld;
    M.buf = kStep ? static_cast<float*>(buf[j].ptr) : nullptr;
    M.ld_buf = kStep ? buf[j].ld : 0;
    M.u = kStep ? x_slot(P, mi, 0) : nullptr;
    M.u_lo = kStep ? lo_slot(P, mi, 0) : nullptr;
    M.ld_u = g.ld_x;
    M.rows = static_cast<int>(mi.rows);
    M.cols = static_cast<int>(mi.cols);
    M.transposed = (kStep && mi.transposed) ? 1 : 0;
    bool vec = aligned16(src[j].ptr) && (!kStep || aligned16(buf[j].ptr));
    int nblk;
    if (M.transposed) {
      vec = vec && src[j].ld % 8 == 0 && buf[j].ld % 8 == 0;
      M.tiles_c = static_cast<int>(ceil_div(mi.cols, kTile));
      nblk = static_cast<int>(ceil_div(mi.rows, 128) * M.tiles_c);
    } else {
      vec = vec && mi.cols % 8 == 0 && src[j].ld == mi.cols && (!kStep || (buf[j].ld == mi.cols && g.ld_x == mi.cols));
      M.tiles_c = 0;
      nblk = static_cast<int>(ceil_div(mi.rows * mi.cols, kFlatChunk));
    }
    M.vec_ok = vec ? 1 : 0;
    M.block_begin = blocks;
    M.nchunks = nblk;
    M.partial = P.partial + mi.partial_off;
    M.ticket = P.tickets + j;
    M.inv = P.inv + j;
    M.post = kStep ? P.post + mi.gslot : nullptr;
    blocks += nblk;
    if (++a.count == kEwMax) {
      muon_status st = flush();
      if (st != MUON_OK) return st;
    }
  }
  return flush();
}

// One map launch family: chooses the template by dtypes and mode.
template <int kMode>
muon_status launch_map_dispatch(muon_handle h, const MapArgs& a, int blocks, bool src_f32, bool dst_f32,
                                cudaStream_t s, int kind) {
  ProfScope ps(h, kind, s);
  // Only the scale pass reads the caller's (possibly fp32) matrices; the others read the bf16 workspace.
  cudaError_t e;
  if constexpr (kMode == kScale) {
    e = src_f32 ? launch_pdl(map_kernel<kMode, true, false>, blocks, kEwThreads, 0, s, a)
                : launch_pdl(map_kernel<kMode, false, false>, blocks, kEwThreads, 0, s, a);
  } else {
    e = dst_f32 ? launch_pdl(map_kernel<kMode, false, true>, blocks, kEwThreads, 0, s, a)
                : launch_pdl(map_kernel<kMode, false, false>, blocks, kEwThreads, 0, s, a);
  }
  return launch_checked(h, e, "map kernel");
}

// kMode = kScale: src = the caller's input (orthogonalize), dst = X0 slot, oriented.
// kMode = kUpdate / kCopy: src = X_k slot (oriented), dst = params / out in the caller's orientation.
template <int kMode>
muon_status launch_map(muon_handle h, const Plan& P, const muon_matrix* user, int xk, float lr,
                       cudaStream_t s, int kind) {
  bool user_f32 = false;
  for (size_t j = 0; user && j < P.mats.size(); ++j)
    if (!P.mats[j].skip) {
      user_f32 = user[j].dtype == MUON_F32;
      break;
    }
  MapArgs a;
  memset(&a, 0, sizeof(a));
  a.keep = (kMode == kUpdate) ? 1.0f - lr * h->cfg.weight_decay : 1.0f;
  int blocks = 0;
  bool src_f32 = false, dst_f32 = false;
  auto flush = [&]() -> muon_status {
    if (a.count == 0) return MUON_OK;
    muon_status st = launch_map_dispatch<kMode>(h, a, blocks, src_f32, dst_f32, s, kind);
    a.count = 0;
    blocks = 0;
    return st;
  };
  for (size_t j = 0; j < P.mats.size(); ++j) {
    const MatInfo& mi = P.mats[j];
    if (mi.skip) continue;
    const Group& g = P.groups[mi.group];
    MapMat& M = a.m[a.count];
    M.transposed = mi.transposed ? 1 : 0;
    if (kMode == kScale) {
      M.src = user[j].ptr;  // the caller's input (muon_orthogonalize)
      M.ld_src = user[j].ld;
      src_f32 = user_f32;
      M.dst = x_slot(P, mi, 0);
      M.dst_lo = lo_slot(P, mi, 0);
      M.ld_dst = g.ld_x;
      M.sr = static_cast<int>(mi.rows);
      M.sc = static_cast<int>(mi.cols);
      dst_f32 = false;
      M.inv = P.inv + j;
    } else {
      M.src = x_slot(P, mi, xk);
      M.src_lo = lo_slot(P, mi, xk);
      M.ld_src = g.ld_x;
      M.dst = user[j].ptr;
      M.ld_dst = user[j].ld;
      M.sr = static_cast<int>(mi.n);
      M.sc = static_cast<int>(mi.m);
      src_f32 = false;
      dst_f32 = user_f32;
      const double sc = h->cfg.scale_lr_by_shape ? std::sqrt(std::max(1.0, double(mi.rows) / double(mi.cols))) : 1.0;
      M.scale = static_cast<float>(double(lr) * sc);
    }
    const bool aligned = aligned16(M.src) && aligned16(M.dst);
    const bool vec = M.transposed ? (aligned && M.ld_src % 8 == 0 && M.ld_dst % 8 == 0)
                                  : (aligned && M.sc % 8 == 0 && M.ld_src == M.sc && M.ld_dst == M.sc);
    M.vec_ok = vec ? 1 : 0;
    M.block_begin = blocks;
    if (M.transposed) {
      M.tiles_c = static_cast<int>(ceil_div(M.sc, kTile));
      blocks += static_cast<int>(ceil_div(M.sr, kTileRows) * M.tiles_c);
    } else {
      M.tiles_c = 0;
      blocks += static_cast<int>(ceil_div(static_cast<int64_t>(M.sr) * M.sc, kFlatChunk));
    }
    if (++a.count == kEwMax) {
      muon_status st = flush();
      if (st != MUON_OK) return st;
    }
  }
  return flush();
}

template <bool kGram, int kBN, int kStages>
cudaLaunchConfig_t gemm_config(int lists, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(lists * kCluster), 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = GemmShape<kGram, kBN, kStages>::SMEM_BYTES;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

template <bool kGram, int kBN, int kStages, bool kFinal = false>
muon_status launch_gemm(muon_handle h, const GemmArgs& a, const FinalArgs<kFinal ? kMaxFinal : 1>& f, cudaStream_t s,
                        int kind) {
  if (a.num_tiles == 0) return MUON_OK;
  ProfScope ps(h, kind, s);
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = gemm_config<kGram, kBN, kStages>(a.grid, s, attr);
  cudaError_t e;
  if (h->profiling) {
    GemmArgs ap = a;
    ap.clk = h->clk_dev;
    e = cudaLaunchKernelEx(&cfg, ns_gemm_kernel<kGram, kBN, kStages, kFinal>, ap, f);
  } else {
    e = cudaLaunchKernelEx(&cfg, ns_gemm_kernel<kGram, kBN, kStages, kFinal>, a, f);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(h, e, "tcgen05 GEMM launch");
  }
  return launch_checked(h, cudaSuccess, "tcgen05 GEMM kernel");
}

const FinalArgs<1> kNoFinal = {};

// Fills the per-batch argument blocks that let the last combine write into the caller's
// matrices `user` (update: W <- W - lr*s*X_k; else out <- X_k). Returns false, leaving the
// separate update / copy kernel to do it, when a matrix is not bf16, not 16-byte aligned, its
// ld is not a multiple of 8 elements, or a batch holds more than kMaxFinal matrices.
bool prepare_final(muon_handle h, Plan& P, const muon_matrix* user, bool update, float lr) {
  for (size_t j = 0; j < P.mats.size(); ++j) {
    if (P.mats[j].skip) continue;
    const muon_matrix& u = user[j];
    if (u.dtype != MUON_BF16 || !aligned16(u.ptr) || u.ld % 8 != 0) return false;
  }
  if (P.fin.size() != P.batches.size()) {
    P.fin.clear();
    for (size_t b = 0; b < P.batches.size(); ++b) P.fin.push_back(std::make_unique<FinalArgs<kMaxFinal>>());
  }
  if (P.user_maps.size() != P.mats.size()) P.user_maps.assign(P.mats.size(), Plan::UserMap{});
  for (size_t b = 0; b < P.batches.size(); ++b) {
    FinalArgs<kMaxFinal>& F = *P.fin[b];
    int running = 0;
    for (int gi = 0; gi < P.batches[b].num_groups; ++gi) {
      F.first[gi] = running;
      running += P.groups[P.batches[b].first_group + gi].count;
    }
    if (running > kMaxFinal) return false;
    F.update = update ? 1 : 0;
    F.keep = update ? 1.0f - lr * h->cfg.weight_decay : 1.0f;
  }
  for (size_t j = 0; j < P.mats.size(); ++j) {
    const MatInfo& mi = P.mats[j];
    if (mi.skip) continue;
    const muon_matrix& u = user[j];
    Plan::UserMap& um = P.user_maps[j];
    if (um.ptr != u.ptr || um.ld != u.ld) {
      // 128 rows x 64 columns swizzled as the combine's tiles; transposed matrices take the
      // transposed box, 64 rows x 128 columns, unswizzled.
      const bool ok = mi.transposed
                          ? encode_map(h, &um.map, u.ptr, mi.cols, mi.rows, 1, u.ld, 128, 64, false)
                          : encode_map(h, &um.map, u.ptr, mi.cols, mi.rows, 1, u.ld, 64, 128, true);
      if (!ok) {
        um.ptr = nullptr;
        return false;
      }
      um.ptr = u.ptr;
      um.ld = u.ld;
    }
    FinalArgs<kMaxFinal>& F = *P.fin[mi.group / kMaxGroups];
    const int slot = F.first[mi.group % kMaxGroups] + mi.idx;
    F.map[slot] = um.map;
    F.trans[slot] = mi.transposed ? 1 : 0;
    const double sc = h->cfg.scale_lr_by_shape ? std::sqrt(std::max(1.0, double(mi.rows) / double(mi.cols))) : 1.0;
    F.scale[slot] = update ? static_cast<float>(double(lr) * sc) : 0.f;
  }
  return true;
}

// k Newton-Schulz iterations on X0 (buffer 0). Returns the buffer holding X_k.
// With `final_into_user`, the last combine writes into the caller's matrices (prepare_final).
// With `folded_scale`, X0 holds u unscaled and the first iteration's Gram and combine apply
// the per-matrix scale (P.post).
muon_status run_iterations(muon_handle h, const Plan& P, int steps, float a, float b, float c, cudaStream_t s,
                           int* xk, bool final_into_user = false, bool folded_scale = false) {
  int t = 0;
  for (int it = 0; it < steps; ++it) {
    for (size_t bi = 0; bi < P.batches.size(); ++bi) {
      const GemmBatch& B = P.batches[bi];
      muon_status st;
      const bool first = folded_scale && it == 0;
      auto with_post = [&](GemmArgs& ga) {
        if (!first) return;
        for (int gi = 0; gi < ga.num_groups; ++gi) ga.grp[gi].post = P.post + P.groups[B.first_group + gi].first_slot;
      };
      if (c == 0.0f) {
        GemmArgs g = B.gram[t];
        with_post(g);
        g.s_acc = b;
        g.s_e = 0.f;
        st = launch_gemm<true, kGramBN, kGramStages>(h, g, kNoFinal, s, K_GRAM);
      } else {
        GemmArgs g = B.gram_to_a[t];  // A = X X^T into the A buffer
        with_post(g);
        g.s_acc = 1.f;
        g.s_e = 0.f;
        st = launch_gemm<true, kGramBN, kGramStages>(h, g, kNoFinal, s, K_GRAM);
        if (st != MUON_OK) return st;
        GemmArgs g2 = B.gram_aa;
        g2.s_acc = c;
        g2.s_e = b;
        st = launch_gemm<true, kGramBN, kGramStages>(h, g2, kNoFinal, s, K_GRAM_AA);
      }
      if (st != MUON_OK) return st;
      GemmArgs cb = B.comb[t];
      with_post(cb);
      cb.s_acc = 1.f;
      cb.s_e = a;
      if (final_into_user && it == steps - 1)
        st = launch_gemm<false, kCombBN, kCombStages, true>(h, cb, *P.fin[bi], s, K_COMBINE);
      else
        st = launch_gemm<false, kCombBN, kCombStages>(h, cb, kNoFinal, s, K_COMBINE);
      if (st != MUON_OK) return st;
    }
    t ^= 1;
  }
  *xk = t;
  return MUON_OK;
}

// ------------------------------------------------------------------ persistent launch

// Iterations one persistent launch covers at most; longer runs take several launches. Even, so every
// launch starts with X in buffer 0 or an even iteration's buffer, as its items assume.
constexpr int kFusedMaxIters = 16;
// Shape groups one persistent launch can name (10 bits of a work item); more take the per-phase launches.
constexpr size_t kFusedMaxGroups = 1024;
// MUON_PERSISTENT_AUTO takes the per-phase launches once one iteration gives every cluster this many
// 64-wide k-blocks of 256 x 256 pair tiles or more. Measured in one process (20-step bursts, ms per
// step, persistent / per-phase): GPT-2 124M step (350 per cluster) 1.023 / 1.052, its quintic (420)
// 1.508 / 1.588, 64 x 1024^2 (360) 0.904 / 0.956, GPT-2 350M step (1619) 4.665 / 4.652, 4096 x 16384
// with k = 10 (1356) 6.078 / 5.827: where each phase already streams hundreds of k-blocks per cluster,
// the per-phase launches' ramps and tails cost less than the persistent launch's item changes.
constexpr double kAutoPerPhaseKblocks = 800.0;

// 64-wide k-blocks of one Newton-Schulz iteration of every matrix, per cluster: the Gram's upper
// triangle of 256 x 256 pair tiles (K = m), the A A pass when c != 0 (K = n), the combine (K = n).
double iteration_kblocks_per_cluster(const std::vector<Group>& groups, bool c_nz, int clusters) {
  double kb = 0.0;
  for (const Group& g : groups) {
    const int64_t nt = ceil_div(g.n, 128), gt2 = ceil_div(g.n, 256), mt = ceil_div(g.m, 256);
    const int64_t nk_m = ceil_div(g.m, 64), nk_n = ceil_div(g.n, 64);
    int64_t gram_pairs = 0;
    for (int64_t J = 0; J < gt2; ++J) gram_pairs += ceil_div(std::min<int64_t>(2 * J + 2, nt), 2);
    const int64_t comb_pairs = ceil_div(nt, 2) * mt;
    kb += static_cast<double>(g.count) *
          static_cast<double>(gram_pairs * nk_m + (c_nz ? gram_pairs * nk_n : 0) + comb_pairs * nk_n);
  }
  return kb / std::max(1, clusters);
}

// Whether a call runs one launch per phase instead of the persistent launch.
bool per_phase_launches(const std::vector<Group>& groups, int mode, bool c_nz, int clusters) {
  if (groups.size() > kFusedMaxGroups || mode == 0) return true;
  if (mode == 1) return false;
  return iteration_kblocks_per_cluster(groups, c_nz, clusters) >= kAutoPerPhaseKblocks;
}

struct SimMatrix {
  int slot = 0;
  double bytes = 0.0, work = 0.0;
  std::vector<std::vector<std::pair<int4, int>>> stages;  // per stage: (item, modelled cost)
  std::vector<double> path;  // per stage: the longest chain from its start to the matrix's end
};

// The items of `iters` iterations of every matrix, in the order a list-scheduling simulation of
// `clusters` clusters takes them. A matrix's stages are, per iteration: the Gram tiles (upper
// triangle, 256 x 256 pairs), the A A tiles when c != 0, the combine tiles. A stage may start once
// its matrix's previous stage has ended (the item's counter target is the number of epilogue halves
// of the earlier stages). Matrices enter in decreasing order of work, and a new one enters only
// while the state of those in flight (both X buffers, B, A) fits kFusedL2Budget, or when nothing
// else can run. A free cluster takes the item that can start soonest (the earliest admitted
// matrix on ties). Each cluster's list keeps the simulation's order, which every dependency
// respects: an item's stage begins only after all items of the stage before it were placed.
void fused_schedule(const Plan& P, bool carry, int iters, bool c_nz, int clusters, std::vector<int4>& items,
                    std::vector<int>& begin) {
  std::vector<SimMatrix> mats;
  for (size_t gi = 0; gi < P.groups.size(); ++gi) {
    const Group& g = P.groups[gi];
    const int nt = static_cast<int>(ceil_div(g.n, 128)), gt2 = static_cast<int>(ceil_div(g.n, 256));
    const int mt = static_cast<int>(ceil_div(g.m, 256));
    const int nk_m = static_cast<int>(ceil_div(g.m, 64)), nk_n = static_cast<int>(ceil_div(g.n, 64));
    for (int b = 0; b < g.count; ++b) {
      SimMatrix M;
      M.slot = g.first_slot + b;
      M.bytes = 2.0 * static_cast<double>(g.n * g.ld_x) * 2.0 * (carry ? 2.0 : 1.0) +
                static_cast<double>(g.n * g.ld_p) * 2.0 * (c_nz ? 2.0 : 1.0);
      int halves = 0;  // epilogue halves of the stages placed so far
      for (int it = 0; it < iters; ++it) {
        const int flags = (it == 0 ? kNsFirst : 0) | (it == iters - 1 ? kNsLast : 0) | ((it & 1) ? kNsOdd : 0);
        auto gram_stage = [&](int kind, int nk) {
          std::vector<std::pair<int4, int>> st;
          for (int J = 0; J < gt2; ++J)
            for (int I = 0; I < std::min(2 * J + 2, nt); I += kCluster)
              st.push_back({ns_item(kind, static_cast<int>(gi), flags, b, I, J, halves), nk + kFusedTileOverhead});
          halves += 4 * static_cast<int>(st.size());
          M.stages.push_back(std::move(st));
        };
        gram_stage(kNsGram, nk_m);
        if (c_nz) gram_stage(kNsGramAA, nk_n);
        std::vector<std::pair<int4, int>> st;
        for (int J = 0; J < mt; ++J)  // column by column, as in build_tiles
          for (int I = 0; I < nt; I += kCluster)
            st.push_back({ns_item(kNsComb, static_cast<int>(gi), flags, b, I, J, halves), nk_n + kFusedTileOverhead});
        halves += 4 * static_cast<int>(st.size());
        M.stages.push_back(std::move(st));
      }
      for (const auto& st : M.stages)
        for (const auto& x : st) M.work += x.second;
      M.path.assign(M.stages.size() + 1, 0.0);
      for (size_t q = M.stages.size(); q-- > 0;) {
        int longest = 0;
        for (const auto& x : M.stages[q]) longest = std::max(longest, x.second);
        M.path[q] = M.path[q + 1] + longest + kFusedLatency;
      }
      mats.push_back(std::move(M));
    }
  }
  std::vector<int> order(mats.size());
  for (size_t j = 0; j < mats.size(); ++j) order[j] = static_cast<int>(j);
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return mats[x].work > mats[y].work; });

  const int C = std::max(1, clusters);
  using Ev = std::pair<double, int>;
  std::priority_queue<Ev, std::vector<Ev>, std::greater<Ev>> freeq;
  for (int c = 0; c < C; ++c) freeq.push({0.0, c});
  std::vector<std::vector<int4>> per(static_cast<size_t>(C));
  struct State {
    size_t stage = 0, next = 0;
    double ready = 0.0, end = 0.0;
    bool finished = false;
  };
  std::vector<State> st(mats.size());
  std::vector<int> active;
  size_t admitted = 0, finished = 0;
  double act_bytes = 0.0;
  while (finished < mats.size()) {
    const Ev top = freeq.top();
    freeq.pop();
    const double t = top.first;
    // Among the items that can start now, the one with the longest chain still ahead of its matrix;
    // if none can, the same among those that must wait.
    int best = -1;
    double best_start = 0.0;
    bool best_now = false;
    for (int j : active) {
      if (st[j].finished) continue;
      const double start = std::max(t, st[j].ready);
      const bool now = start <= t;
      if (best < 0 || (now && !best_now) ||
          (now == best_now && mats[j].path[st[j].stage] > mats[best].path[st[best].stage])) {
        best = j;
        best_start = start;
        best_now = now;
      }
    }
    if ((best < 0 || best_start > t) && admitted < order.size() &&
        (best < 0 || act_bytes + mats[order[admitted]].bytes <= kFusedL2Budget)) {
      const int j = order[admitted++];
      active.push_back(j);
      act_bytes += mats[j].bytes;
      freeq.push(top);
      continue;
    }
    SimMatrix& M = mats[best];
    State& s = st[best];
    const auto& stage = M.stages[s.stage];
    const auto& x = stage[s.next++];
    const double end = best_start + x.second;
    per[top.second].push_back(x.first);
    // The cluster is free at `end`, but the item's result lands (and its matrix's next stage may
    // start) only once the epilogue has drained it and the next item's operands have arrived.
    s.end = std::max(s.end, end + kFusedLatency);
    if (s.next == stage.size()) {
      s.ready = s.end;
      ++s.stage;
      s.next = 0;
      if (s.stage == M.stages.size()) {
        s.finished = true;
        ++finished;
        act_bytes -= M.bytes;
      }
    }
    freeq.push({end, top.second});
  }
  items.clear();
  begin.assign(1, 0);
  for (const auto& l : per) {
    items.insert(items.end(), l.begin(), l.end());
    begin.push_back(static_cast<int>(items.size()));
  }
}

// Fills the caller-matrix maps of the last combine by matrix slot (group order). False when a
// matrix is not bf16, 16-byte aligned with ld a multiple of 8, or the batch has more than
// kMaxFinal matrices: the separate update / copy kernel then writes the caller's matrices.
bool prepare_final_slots(muon_handle h, Plan& P, const muon_matrix* user, bool update, float lr) {
  int slots = 0;
  for (const Group& g : P.groups) slots += g.count;
  if (slots > kMaxFinal) return false;
  for (size_t j = 0; j < P.mats.size(); ++j) {
    if (P.mats[j].skip) continue;
    const muon_matrix& u = user[j];
    if (u.dtype != MUON_BF16 || !aligned16(u.ptr) || u.ld % 8 != 0) return false;
  }
  if (!P.fin_slots) P.fin_slots = std::make_unique<FinalArgs<kMaxFinal>>();
  if (P.user_maps.size() != P.mats.size()) P.user_maps.assign(P.mats.size(), Plan::UserMap{});
  FinalArgs<kMaxFinal>& F = *P.fin_slots;
  F.update = update ? 1 : 0;
  F.keep = update ? 1.0f - lr * h->cfg.weight_decay : 1.0f;
  for (size_t j = 0; j < P.mats.size(); ++j) {
    const MatInfo& mi = P.mats[j];
    if (mi.skip) continue;
    const muon_matrix& u = user[j];
    Plan::UserMap& um = P.user_maps[j];
    if (um.ptr != u.ptr || um.ld != u.ld) {
      const bool ok = mi.transposed
                          ? encode_map(h, &um.map, u.ptr, mi.cols, mi.rows, 1, u.ld, 128, 64, false)
                          : encode_map(h, &um.map, u.ptr, mi.cols, mi.rows, 1, u.ld, 64, 128, true);
      if (!ok) {
        um.ptr = nullptr;
        return false;
      }
      um.ptr = u.ptr;
      um.ld = u.ld;
    }
    F.map[mi.gslot] = um.map;
    F.trans[mi.gslot] = mi.transposed ? 1 : 0;
    const double sc = h->cfg.scale_lr_by_shape ? std::sqrt(std::max(1.0, double(mi.rows) / double(mi.cols))) : 1.0;
    F.scale[mi.gslot] = update ? static_cast<float>(double(lr) * sc) : 0.f;
  }
  return true;
}

cudaLaunchConfig_t fused_config(int clusters, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * kCluster), 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = FusedShape::SMEM_BYTES;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// k Newton-Schulz iterations on X0 (buffer 0) in persistent launches of up to kFusedMaxIters
// iterations each. Returns the buffer holding X_k. With `final_into_user` the last combine writes
// the caller's matrices (prepare_final_slots); with `folded_scale` the first iteration applies the
// per-matrix scale P.post.
muon_status run_iterations_fused(muon_handle h, Plan& P, int steps, float a, float b, float c, cudaStream_t s,
                                 int* xk, bool final_into_user, bool folded_scale) {
  const bool c_nz = c != 0.0f;
  int slots = 0;
  for (const Group& g : P.groups) slots += g.count;
  for (int i0 = 0; i0 < steps; i0 += kFusedMaxIters) {
    const int iters = std::min(kFusedMaxIters, steps - i0);
    const auto key = std::make_pair(iters, c_nz ? 1 : 0);
    auto it = P.fused.find(key);
    if (it == P.fused.end()) {
      std::vector<int4> items;
      std::vector<int> begin;
      fused_schedule(P, P.carry, iters, c_nz, h->max_lists, items, begin);
      Plan::FusedSchedule fs;
      fs.grid = static_cast<int>(begin.size()) - 1;
      const size_t ib = items.size() * sizeof(int4), bb = begin.size() * sizeof(int);
      void* buf = nullptr;
      cudaError_t e = plan_malloc(h, P, &buf, ib + bb);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(h, MUON_ERR_NOMEM, "persistent schedule of %zu bytes: %s", ib + bb, cudaGetErrorString(e));
      }
      fs.items = static_cast<int4*>(buf);
      fs.begin = reinterpret_cast<int*>(static_cast<uint8_t*>(buf) + ib);
      fs.bytes = ib + bb;
      e = cudaMemcpy(fs.items, items.data(), ib, cudaMemcpyHostToDevice);
      if (e == cudaSuccess) e = cudaMemcpy(fs.begin, begin.data(), bb, cudaMemcpyHostToDevice);
      if (e != cudaSuccess) {
        cudaFree(buf);
        P.dev_bytes -= ib + bb;
        h->plan_bytes -= ib + bb;
        return cuda_fail(h, e, "persistent schedule upload");
      }
      it = P.fused.emplace(key, fs).first;
    }
    const Plan::FusedSchedule& fs = it->second;
    FusedArgs fa;
    memset(&fa, 0, sizeof(fa));
    fa.maps = P.maps_dev;
    fa.groups = P.groups_dev;
    fa.items = fs.items;
    fa.begin = fs.begin;
    fa.counters = P.counters;
    fa.done = P.done;
    fa.post = (folded_scale && i0 == 0) ? P.post : nullptr;
    fa.num_slots = slots;
    fa.num_groups = static_cast<int>(P.groups.size());
    fa.c_nonzero = c_nz ? 1 : 0;
    fa.a = a;
    fa.b = b;
    fa.c = c;
    fa.carry = P.carry ? 1 : 0;
    fa.final_mode = (final_into_user && i0 + iters == steps) ? 1 : 0;
    fa.err = h->err_dev;
    fa.clk = h->profiling ? h->clk_dev : nullptr;
    static const FinalArgs<kMaxFinal> kNoFinalSlots = {};
    const FinalArgs<kMaxFinal>& fin = fa.final_mode ? *P.fin_slots : kNoFinalSlots;
    ProfScope ps(h, K_FUSED, s);
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = fused_config(fs.grid, s, attr);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, ns_fused_kernel<kFusedStages>, fa, fin);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return cuda_fail(h, e, "persistent Newton-Schulz launch");
    }
  }
  *xk = steps & 1;
  return MUON_OK;
}

// Failure-detection self-test: one thread waits, through the GEMMs' bounded
// wait, on a barrier that nothing arrives at.
__global__ void wait_selftest_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, err, limit_ns);
  __syncthreads();
}

std::vector<std::pair<int64_t, int64_t>> shape_key(const muon_matrix* m, int count) {
  std::vector<std::pair<int64_t, int64_t>> k(static_cast<size_t>(count));
  for (int j = 0; j < count; ++j) k[j] = {m[j].rows, m[j].cols};
  return k;
}

// Whether a call with coefficient c carries X as bf16 hi + lo (muon_config.precise_carry).
bool uses_carry(const muon_config& cfg, float c) {
  return cfg.precise_carry == 1 || (cfg.precise_carry == MUON_CARRY_WHEN_C && c != 0.0f);
}

bool all_skipped(const muon_matrix* m, int count) {
  for (int j = 0; j < count; ++j)
    if (m[j].rows > 0 && m[j].cols > 0) return false;
  return true;
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

void muon_default_config(muon_config* cfg) {
  if (!cfg) return;
  cfg->steps = 5;
  cfg->a = 1.5f;
  cfg->b = -0.5f;
  cfg->c = 0.0f;
  cfg->eps = 1e-7f;
  cfg->scale_lr_by_shape = 1;
  cfg->weight_decay = 0.0f;
  cfg->precise_carry = MUON_CARRY_WHEN_C;
  cfg->persistent = MUON_PERSISTENT_AUTO;
}

const char* muon_status_string(muon_status s) {
  switch (s) {
    case MUON_OK: return "MUON_OK";
    case MUON_ERR_INVALID: return "MUON_ERR_INVALID";
    case MUON_ERR_CUDA: return "MUON_ERR_CUDA";
    case MUON_ERR_NOMEM: return "MUON_ERR_NOMEM";
    case MUON_ERR_UNSUPPORTED: return "MUON_ERR_UNSUPPORTED";
    case MUON_ERR_TIMEOUT: return "MUON_ERR_TIMEOUT";
  }
  return "MUON_ERR_UNKNOWN";
}

const char* muon_kernel_name(int kind) {
  if (kind < 0 || kind >= MUON_KERNEL_KINDS) return "unknown";
  return kKernelNames[kind];
}

const char* muon_last_error(muon_handle h) {
  if (!h) return "null handle";
  return h->last_error.c_str();
}

muon_status muon_check_orthogonalize(const muon_matrix* in, const muon_matrix* out, int count, int steps, char* msg,
                                     int msg_len) {
  if (count < 0) {
    put_msg(msg, msg_len, "count %d < 0", count);
    return MUON_ERR_INVALID;
  }
  if (steps < 0 || steps > kMaxSteps) {
    put_msg(msg, msg_len, "steps %d out of range", steps);
    return MUON_ERR_INVALID;
  }
  if (count == 0) return MUON_OK;
  if (!in || !out) {
    put_msg(msg, msg_len, "null descriptor array");
    return MUON_ERR_INVALID;
  }
  int in_dt = -1, out_dt = -1;
  std::vector<Range> outs;
  for (int j = 0; j < count; ++j) {
    if (!dims_ok(in[j], "in", j, msg, msg_len) || !dims_ok(out[j], "out", j, msg, msg_len)) return MUON_ERR_INVALID;
    if (in[j].rows != out[j].rows || in[j].cols != out[j].cols) {
      put_msg(msg, msg_len, "in[%d] and out[%d] differ in shape", j, j);
      return MUON_ERR_INVALID;
    }
    if (in[j].rows == 0 || in[j].cols == 0) continue;
    if (in_dt < 0) in_dt = in[j].dtype;
    if (out_dt < 0) out_dt = out[j].dtype;
    if (in[j].dtype != in_dt || out[j].dtype != out_dt) {
      put_msg(msg, msg_len, "matrix %d: all inputs must share one dtype and all outputs another", j);
      return MUON_ERR_INVALID;
    }
    outs.push_back(range_of(out[j], j));
  }
  int x, y;
  if (any_overlap(outs, &x, &y)) {
    put_msg(msg, msg_len, "out[%d] and out[%d] overlap", x, y);
    return MUON_ERR_INVALID;
  }
  return MUON_OK;
}

muon_status muon_check_step(const muon_matrix* params, const muon_matrix* grads, const muon_matrix* momentum,
                            int count, char* msg, int msg_len) {
  if (count < 0) {
    put_msg(msg, msg_len, "count %d < 0", count);
    return MUON_ERR_INVALID;
  }
  if (count == 0) return MUON_OK;
  if (!params || !grads || !momentum) {
    put_msg(msg, msg_len, "null descriptor array");
    return MUON_ERR_INVALID;
  }
  int p_dt = -1, g_dt = -1;
  std::vector<Range> ranges;
  for (int j = 0; j < count; ++j) {
    if (!dims_ok(params[j], "params", j, msg, msg_len) || !dims_ok(grads[j], "grads", j, msg, msg_len) ||
        !dims_ok(momentum[j], "momentum", j, msg, msg_len))
      return MUON_ERR_INVALID;
    if (grads[j].rows != params[j].rows || grads[j].cols != params[j].cols ||
        momentum[j].rows != params[j].rows || momentum[j].cols != params[j].cols) {
      put_msg(msg, msg_len, "matrix %d: params, grads and momentum differ in shape", j);
      return MUON_ERR_INVALID;
    }
    if (params[j].rows == 0 || params[j].cols == 0) continue;
    if (momentum[j].dtype != MUON_F32) {
      put_msg(msg, msg_len, "momentum[%d]: must be F32", j);
      return MUON_ERR_INVALID;
    }
    if (p_dt < 0) p_dt = params[j].dtype;
    if (g_dt < 0) g_dt = grads[j].dtype;
    if (params[j].dtype != p_dt || grads[j].dtype != g_dt) {
      put_msg(msg, msg_len, "matrix %d: all params must share one dtype and all grads another", j);
      return MUON_ERR_INVALID;
    }
    ranges.push_back(range_of(params[j], j));
    ranges.push_back(range_of(grads[j], count + j));
    ranges.push_back(range_of(momentum[j], 2 * count + j));
  }
  int x, y;
  if (any_overlap(ranges, &x, &y)) {
    const char* names[3] = {"params", "grads", "momentum"};
    put_msg(msg, msg_len, "%s[%d] and %s[%d] overlap", names[x / count], x % count, names[y / count], y % count);
    return MUON_ERR_INVALID;
  }
  return MUON_OK;
}

muon_status muon_plan_stats(const int64_t* rows, const int64_t* cols, int count, int with_c, int* groups,
                            int64_t* gram_tiles, int64_t* combine_tiles, double* flops_per_iter) {
  if (count < 0 || (count > 0 && (!rows || !cols))) return MUON_ERR_INVALID;
  std::vector<std::pair<int64_t, int64_t>> key(static_cast<size_t>(count));
  for (int j = 0; j < count; ++j) {
    if (rows[j] < 0 || cols[j] < 0) return MUON_ERR_INVALID;
    key[j] = {rows[j], cols[j]};
  }
  std::vector<MatInfo> mats;
  std::vector<Group> grps;
  group_shapes(key, mats, grps);
  int64_t gt = 0, ct = 0;
  for (const Group& g : grps) {
    const int64_t nt = ceil_div(g.n, 128);
    for (int64_t J = 0; J < ceil_div(g.n, kGramBN); ++J) gt += g.count * std::min<int64_t>(2 * J + 2, nt);
    ct += g.count * nt * ceil_div(g.m, kCombBN);
  }
  double fl = 0.0;
  for (const MatInfo& mi : mats) {
    if (mi.skip) continue;
    const double n = double(mi.n), m = double(mi.m);
    fl += n * (n + 1.0) * m + 2.0 * n * n * m;
    if (with_c) fl += n * n * (n + 1.0);
  }
  if (groups) *groups = static_cast<int>(grps.size());
  if (gram_tiles) *gram_tiles = gt * (with_c ? 2 : 1);
  if (combine_tiles) *combine_tiles = ct;
  if (flops_per_iter) *flops_per_iter = fl;
  return MUON_OK;
}

muon_status muon_launch_choice(const int64_t* rows, const int64_t* cols, int count, int with_c, int clusters,
                               int persistent, int* use_persistent, double* kblocks_per_cluster) {
  if (count < 0 || (count > 0 && (!rows || !cols)) || clusters < 1 || persistent < 0 || persistent > 2)
    return MUON_ERR_INVALID;
  std::vector<std::pair<int64_t, int64_t>> key(static_cast<size_t>(count));
  for (int j = 0; j < count; ++j) {
    if (rows[j] < 0 || cols[j] < 0) return MUON_ERR_INVALID;
    key[j] = {rows[j], cols[j]};
  }
  std::vector<MatInfo> mats;
  std::vector<Group> grps;
  group_shapes(key, mats, grps);
  if (use_persistent) *use_persistent = per_phase_launches(grps, persistent, with_c != 0, clusters) ? 0 : 1;
  if (kblocks_per_cluster) *kblocks_per_cluster = iteration_kblocks_per_cluster(grps, with_c != 0, clusters);
  return MUON_OK;
}

muon_status muon_persistent_schedule(const int64_t* rows, const int64_t* cols, int count, int steps, int with_c,
                                     int clusters, int32_t* items, int64_t items_cap, int32_t* begin,
                                     int64_t* num_items) {
  if (count < 0 || (count > 0 && (!rows || !cols)) || steps < 1 || steps > kFusedMaxIters || clusters < 1 ||
      !num_items || items_cap < 0)
    return MUON_ERR_INVALID;
  std::vector<std::pair<int64_t, int64_t>> key(static_cast<size_t>(count));
  for (int j = 0; j < count; ++j) {
    if (rows[j] < 0 || cols[j] < 0) return MUON_ERR_INVALID;
    key[j] = {rows[j], cols[j]};
  }
  Plan P;
  group_shapes(key, P.mats, P.groups);
  if (P.groups.size() > kFusedMaxGroups) return MUON_ERR_UNSUPPORTED;
  std::vector<int4> it;
  std::vector<int> bg;
  fused_schedule(P, false, steps, with_c != 0, clusters, it, bg);
  *num_items = static_cast<int64_t>(it.size());
  if (!items && !begin) return MUON_OK;
  if (!items || !begin || items_cap < static_cast<int64_t>(it.size())) return MUON_ERR_INVALID;
  for (size_t i = 0; i < it.size(); ++i) {
    items[4 * i] = it[i].x;
    items[4 * i + 1] = it[i].y;
    items[4 * i + 2] = it[i].z;
    items[4 * i + 3] = it[i].w;
  }
  for (size_t c = 0; c < bg.size(); ++c) begin[c] = bg[c];
  return MUON_OK;
}

muon_status muon_create(muon_handle* out, int device, const muon_config* cfg) {
  if (!out) return MUON_ERR_INVALID;
  *out = nullptr;
  if (cfg && (cfg->steps < 0 || cfg->steps > kMaxSteps || !(cfg->eps >= 0.0f) || !std::isfinite(cfg->a) ||
              !std::isfinite(cfg->b) || !std::isfinite(cfg->c) || !(cfg->weight_decay >= 0.0f) ||
              !std::isfinite(cfg->weight_decay) || (cfg->precise_carry < 0 || cfg->precise_carry > 2) ||
              (cfg->persistent < 0 || cfg->persistent > 2)))
    return MUON_ERR_INVALID;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) {
    cudaGetLastError();
    return MUON_ERR_CUDA;
  }
  if (device < 0 || device >= ndev) return MUON_ERR_INVALID;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MUON_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return MUON_ERR_UNSUPPORTED;
  DeviceGuard guard(device);
  auto h = std::make_unique<muon_ctx>();
  h->device = device;
  h->num_sms = prop.multiProcessorCount;

  muon_default_config(&h->cfg);
  if (cfg) h->cfg = *cfg;
  h->launch_mode = h->cfg.persistent;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return MUON_ERR_CUDA;
  h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  if (cudaMalloc(&h->err_dev, 256) != cudaSuccess) {
    cudaGetLastError();
    return MUON_ERR_NOMEM;
  }
  if (cudaMemset(h->err_dev, 0, 256) != cudaSuccess) {
    cudaFree(h->err_dev);
    return MUON_ERR_CUDA;
  }
  h->clk_dev = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(h->err_dev) + 64);
  auto kgram = ns_gemm_kernel<true, kGramBN, kGramStages, false>;
  auto kcomb = ns_gemm_kernel<false, kCombBN, kCombStages, false>;
  auto kfinal = ns_gemm_kernel<false, kCombBN, kCombStages, true>;
  auto kfused = ns_fused_kernel<kFusedStages>;
  cudaError_t e1 = cudaFuncSetAttribute(kgram, cudaFuncAttributeMaxDynamicSharedMemorySize, GramShape::SMEM_BYTES);
  cudaError_t e2 = cudaFuncSetAttribute(kcomb, cudaFuncAttributeMaxDynamicSharedMemorySize, CombShape::SMEM_BYTES);
  cudaError_t e3 = cudaFuncSetAttribute(kfinal, cudaFuncAttributeMaxDynamicSharedMemorySize, CombShape::SMEM_BYTES);
  cudaError_t e4 = cudaFuncSetAttribute(kfused, cudaFuncAttributeMaxDynamicSharedMemorySize, FusedShape::SMEM_BYTES);
  if (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess || e4 != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->err_dev);
    return MUON_ERR_CUDA;
  }
  // Persistent grids: as many tile lists as clusters that can be resident at once.
  h->max_lists = h->num_sms / kCluster;
  {
    cudaLaunchAttribute attr[2];
    int n1 = 0, n2 = 0, n3 = 0;
    cudaLaunchConfig_t c1 = gemm_config<true, kGramBN, kGramStages>(1, nullptr, attr);
    e1 = cudaOccupancyMaxActiveClusters(&n1, kgram, &c1);
    cudaLaunchConfig_t c2 = gemm_config<false, kCombBN, kCombStages>(1, nullptr, attr);
    e2 = cudaOccupancyMaxActiveClusters(&n2, kcomb, &c2);
    e3 = cudaOccupancyMaxActiveClusters(&n3, kfinal, &c2);
    int n4 = 0;
    cudaLaunchConfig_t c4 = fused_config(1, nullptr, attr);
    e4 = cudaOccupancyMaxActiveClusters(&n4, kfused, &c4);
    if (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess || e4 != cudaSuccess || n1 < 1 || n2 < 1 ||
        n3 < 1 || n4 < 1) {
      cudaGetLastError();
      cudaFree(h->err_dev);
      return MUON_ERR_UNSUPPORTED;
    }
    h->max_lists = std::min(std::min(n1, n4), std::min(n2, n3));
  }
  *out = h.release();
  return MUON_OK;
}

muon_status muon_destroy(muon_handle h) {
  if (!h) return MUON_OK;
  {
    DeviceGuard guard(h->device);
    cudaDeviceSynchronize();
    for (auto& kv : h->plans) free_plan(h, kv.second.get());
    if (h->err_dev) cudaFree(h->err_dev);
    for (auto& r : h->recs) {
      cudaEventDestroy(r.a);
      cudaEventDestroy(r.b);
    }
    for (cudaEvent_t e : h->event_pool) cudaEventDestroy(e);
  }
  delete h;
  return MUON_OK;
}

muon_status muon_orthogonalize(muon_handle h, const muon_matrix* in, const muon_matrix* out, int count, int steps,
                               float a, float b, float c, void* stream) {
  if (!h) return MUON_ERR_INVALID;
  char msg[256] = {0};
  muon_status st = muon_check_orthogonalize(in, out, count, steps, msg, sizeof(msg));
  if (st != MUON_OK) return fail(h, st, "%s", msg);
  if (!std::isfinite(a) || !std::isfinite(b) || !std::isfinite(c))
    return fail(h, MUON_ERR_INVALID, "non-finite coefficient");
  if (count == 0 || all_skipped(in, count)) return MUON_OK;
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Plan* P = nullptr;
  if ((st = get_plan(h, shape_key(in, count), uses_carry(h->cfg, c), &P)) != MUON_OK) return st;
  if ((st = launch_momentum<false>(h, *P, in, nullptr, 0.f, 0, 0, s)) != MUON_OK) return st;
  if ((st = launch_map<kScale>(h, *P, in, 0, 0.f, s, K_SCALE)) != MUON_OK) return st;
  int xk = 0;
  if (per_phase_launches(P->groups, h->launch_mode, c != 0.0f, h->max_lists)) {
    const bool direct = steps >= 1 && prepare_final(h, *P, out, false, 0.f);
    if ((st = run_iterations(h, *P, steps, a, b, c, s, &xk, direct)) != MUON_OK) return st;
    if (direct) return MUON_OK;
    return launch_map<kCopy>(h, *P, out, xk, 0.f, s, K_COPY);
  }
  const bool direct = steps >= 1 && prepare_final_slots(h, *P, out, false, 0.f);
  if ((st = run_iterations_fused(h, *P, steps, a, b, c, s, &xk, direct, false)) != MUON_OK) return st;
  if (direct) return MUON_OK;
  return launch_map<kCopy>(h, *P, out, xk, 0.f, s, K_COPY);
}

muon_status muon_step(muon_handle h, const muon_matrix* params, const muon_matrix* grads, const muon_matrix* momentum,
                      int count, float lr, float beta, int nesterov, void* stream) {
  if (!h) return MUON_ERR_INVALID;
  char msg[256] = {0};
  muon_status st = muon_check_step(params, grads, momentum, count, msg, sizeof(msg));
  if (st != MUON_OK) return fail(h, st, "%s", msg);
  if (!std::isfinite(lr) || !std::isfinite(beta)) return fail(h, MUON_ERR_INVALID, "non-finite lr or beta");
  if (count == 0 || all_skipped(params, count)) return MUON_OK;
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Plan* P = nullptr;
  if ((st = get_plan(h, shape_key(params, count), uses_carry(h->cfg, h->cfg.c), &P)) != MUON_OK) return st;
  // u goes into the first X buffer unscaled; its 1/(||u||_F + eps) is folded into the first
  // iteration's Gram and combine, except for norms outside the safe range, where the momentum
  // kernel scales u in place (and always with zero iterations).
  const int steps = h->cfg.steps;
  if ((st = launch_momentum<true>(h, *P, grads, momentum, beta, nesterov, steps == 0 ? 1 : 0, s)) != MUON_OK)
    return st;
  int xk = 0;
  // The update happens in the last combine's epilogue when the parameters allow it.
  if (per_phase_launches(P->groups, h->launch_mode, h->cfg.c != 0.0f, h->max_lists)) {
    const bool direct = steps >= 1 && prepare_final(h, *P, params, true, lr);
    if ((st = run_iterations(h, *P, steps, h->cfg.a, h->cfg.b, h->cfg.c, s, &xk, direct, true)) != MUON_OK)
      return st;
    if (direct) return MUON_OK;
    return launch_map<kUpdate>(h, *P, params, xk, lr, s, K_UPDATE);
  }
  const bool direct = steps >= 1 && prepare_final_slots(h, *P, params, true, lr);
  if ((st = run_iterations_fused(h, *P, steps, h->cfg.a, h->cfg.b, h->cfg.c, s, &xk, direct, true)) != MUON_OK)
    return st;
  if (direct) return MUON_OK;
  return launch_map<kUpdate>(h, *P, params, xk, lr, s, K_UPDATE);
}

muon_status muon_get_error(muon_handle h, void* stream) {
  if (!h) return MUON_ERR_INVALID;
  DeviceGuard guard(h->device);
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "stream synchronize");
  int v = 0;
  e = cudaMemcpy(&v, h->err_dev, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e, "error flag read");
  if (v != 0) {
    const int zero = 0;
    cudaMemcpy(h->err_dev, &zero, sizeof(int), cudaMemcpyHostToDevice);
    return fail(h, MUON_ERR_TIMEOUT, "a device-side wait expired");
  }
  return MUON_OK;
}

muon_status muon_selftest_wait(muon_handle h, int64_t limit_ns, void* stream) {
  if (!h) return MUON_ERR_INVALID;
  if (limit_ns < 1000000 || limit_ns > 2000000000) return fail(h, MUON_ERR_INVALID, "limit_ns out of [1e6, 2e9]");
  DeviceGuard guard(h->device);
  wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(h->err_dev, static_cast<uint64_t>(limit_ns));
  return launch_checked(h, cudaPeekAtLastError(), "wait self-test kernel");
}

muon_status muon_selftest_persistent(muon_handle h, int64_t limit_ns, void* stream) {
  if (!h) return MUON_ERR_INVALID;
  if (limit_ns < 1000000 || limit_ns > 2000000000) return fail(h, MUON_ERR_INVALID, "limit_ns out of [1e6, 2e9]");
  DeviceGuard guard(h->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // One 256 x 256 matrix, one iteration, with the first item of the first list waiting for a stage
  // count its matrix never reaches.
  Plan* P = nullptr;
  muon_status st = get_plan(h, {{256, 256}}, false, &P);
  if (st != MUON_OK) return st;
  std::vector<int4> items;
  std::vector<int> begin;
  fused_schedule(*P, false, 1, false, h->max_lists, items, begin);
  if (items.empty()) return fail(h, MUON_ERR_CUDA, "empty self-test schedule");
  items[begin[0]].w = 1 << 30;
  const size_t ib = items.size() * sizeof(int4), bb = begin.size() * sizeof(int);
  void* buf = nullptr;
  cudaError_t e = cudaMalloc(&buf, ib + bb);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(h, MUON_ERR_NOMEM, "self-test schedule: %s", cudaGetErrorString(e));
  }
  e = cudaMemcpy(buf, items.data(), ib, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(static_cast<uint8_t*>(buf) + ib, begin.data(), bb, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) {
    FusedArgs fa;
    memset(&fa, 0, sizeof(fa));
    fa.maps = P->maps_dev;
    fa.groups = P->groups_dev;
    fa.items = static_cast<int4*>(buf);
    fa.begin = reinterpret_cast<int*>(static_cast<uint8_t*>(buf) + ib);
    fa.counters = P->counters;
    fa.done = P->done;
    fa.num_slots = 1;
    fa.num_groups = static_cast<int>(P->groups.size());
    fa.a = 1.5f;
    fa.b = -0.5f;
    fa.err = h->err_dev;
    fa.wait_ns = static_cast<uint64_t>(limit_ns);
    static const FinalArgs<kMaxFinal> kNone = {};
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = fused_config(static_cast<int>(begin.size()) - 1, s, attr);
    e = cudaLaunchKernelEx(&cfg, ns_fused_kernel<kFusedStages>, fa, kNone);
    // The schedule buffer must outlive the launch; this call waits for it.
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  cudaFree(buf);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(h, e, "persistent self-test");
  }
  return MUON_OK;
}

muon_status muon_set_workspace_limit(muon_handle h, int64_t bytes) {
  if (!h || bytes < 0) return MUON_ERR_INVALID;
  h->plan_limit = static_cast<size_t>(bytes);
  return MUON_OK;
}

muon_status muon_workspace_bytes(muon_handle h, int64_t* bytes) {
  if (!h || !bytes) return MUON_ERR_INVALID;
  *bytes = static_cast<int64_t>(h->plan_bytes);
  return MUON_OK;
}

muon_status muon_profile_enable(muon_handle h, int enable) {
  if (!h) return MUON_ERR_INVALID;
  if (enable && !h->profiling) {
    DeviceGuard guard(h->device);
    if (cudaMemset(h->clk_dev, 0, 2 * sizeof(unsigned long long)) != cudaSuccess) {
      cudaGetLastError();
      return MUON_ERR_CUDA;
    }
  }
  h->profiling = enable != 0;
  return MUON_OK;
}

muon_status muon_profile_clock(muon_handle h, double* sm_mhz) {
  if (!h || !sm_mhz) return MUON_ERR_INVALID;
  DeviceGuard guard(h->device);
  unsigned long long v[2] = {0, 0};
  if (cudaMemcpy(v, h->clk_dev, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return MUON_ERR_CUDA;
  }
  *sm_mhz = v[1] ? 1e3 * static_cast<double>(v[0]) / static_cast<double>(v[1]) : 0.0;
  return MUON_OK;
}

muon_status muon_profile_read(muon_handle h, double* ms, int64_t* launches) {
  if (!h) return MUON_ERR_INVALID;
  DeviceGuard guard(h->device);
  double acc[MUON_KERNEL_KINDS] = {0};
  int64_t cnt[MUON_KERNEL_KINDS] = {0};
  muon_status st = MUON_OK;
  for (auto& r : h->recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) st = MUON_ERR_CUDA;
    float t = 0.f;
    if (st == MUON_OK && cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess) {
      acc[r.kind] += t;
      cnt[r.kind] += 1;
    }
    h->event_pool.push_back(r.a);
    h->event_pool.push_back(r.b);
  }
  h->recs.clear();
  for (int k = 0; k < MUON_KERNEL_KINDS; ++k) {
    if (ms) ms[k] = acc[k];
    if (launches) launches[k] = cnt[k];
  }
  if (st != MUON_OK) cudaGetLastError();
  return st;
}

}  // extern "C"
