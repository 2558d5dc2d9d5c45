// C-ABI entry points: argument checks, row grouping, slicing, TMA
// descriptors and launches.  No allocation, no stream synchronisation.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <new>
#include <cmath>
#include <cstring>
#include <unordered_map>
#include <vector>

#include "params.h"
#include "tfpa.h"

using namespace tfpa;

namespace {

// ------------------------------------------------------------ launch hook
// Set from one thread while no other call runs (a test facility); read by
// every call without a lock.
std::atomic<tfpa_launch_hook> g_hook_fn{nullptr};
std::atomic<void*> g_hook_user{nullptr};
std::atomic<int> g_hook_dry{0};

bool dry_run() {
  return g_hook_dry.load(std::memory_order_relaxed) != 0 &&
         g_hook_fn.load(std::memory_order_relaxed) != nullptr;
}

void record(int kind, int row0, int rows, int runs, int items, int grid, int64_t qoff,
            int64_t ooff) {
  const tfpa_launch_hook fn = g_hook_fn.load(std::memory_order_acquire);
  if (!fn) return;
  tfpa_launch_record r;
  r.kind = kind;
  r.row0 = row0;
  r.rows = rows;
  r.runs = runs;
  r.items = items;
  r.grid = grid;
  r.q_offset = qoff;
  r.out_offset = ooff;
  fn(&r, g_hook_user.load(std::memory_order_relaxed));
}

// ------------------------------------------------------------ device info
// SM count and compute capability of each device, read once per device.
struct DeviceInfo {
  std::atomic<int> ready{0};
  int sm_count = 0;
  int major = 0;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];

// The current device's info, or nullptr if a CUDA call fails.
const DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceInfo& d = g_dev[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    int n = 0, major = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
      return nullptr;
    d.sm_count = n;     // two threads may both get here: they store the same values
    d.major = major;
    d.ready.store(1, std::memory_order_release);
  }
  return &d;
}

int sm_count() {
  if (dry_run()) return 152;
  const DeviceInfo* d = device_info();
  return d ? d->sm_count : 0;
}

int check_device() {
  if (dry_run()) return TFPA_OK;
  const DeviceInfo* d = device_info();
  if (!d) return TFPA_ECUDA;
  return d->major == 10 ? TFPA_OK : TFPA_EDEVICE;
}

// ------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

struct MapKey {
  const void* ptr;
  uint64_t rows;
  int fp8, box_inner, box_rows;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && rows == o.rows && fp8 == o.fp8 && box_inner == o.box_inner &&
           box_rows == o.box_rows;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    size_t h = std::hash<const void*>()(k.ptr);
    h ^= std::hash<uint64_t>()(k.rows) + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
    h ^= (size_t)(k.fp8 * 131 + k.box_inner * 7 + k.box_rows);
    return h;
  }
};
// Each host thread keeps its own cache of encoded maps, so calls from
// several threads share no lock.  A map only describes an address range and
// a box, so it stays valid for any buffer later placed at the same address
// with the same extent.
thread_local std::unordered_map<MapKey, CUtensorMap, MapKeyHash> t_maps;

// A 2D view [rows][128] of a K or V buffer, 128B swizzle, box
// [box_inner elements][box_rows rows].
int get_map(const void* ptr, uint64_t rows, bool fp8, int box_inner, int box_rows,
            CUtensorMap* out) {
  if (dry_run()) {
    std::memset(out, 0, sizeof(*out));
    return TFPA_OK;
  }
  MapKey key{ptr, rows, fp8 ? 1 : 0, box_inner, box_rows};
  auto it = t_maps.find(key);
  if (it != t_maps.end()) {
    *out = it->second;
    return TFPA_OK;
  }
  auto fn = encode_fn();
  if (!fn) return TFPA_ECUDA;
  const uint64_t esz = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(kHeadDim * esz)};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  CUresult r = fn(&m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return TFPA_ECUDA;
  if (t_maps.size() > 4096) t_maps.clear();
  t_maps.emplace(key, m);
  *out = m;
  return TFPA_OK;
}

// q of one launch as a 3D tensor [rows][hq][128] bf16, 128B swizzle; box
// 64 x 1 x 128 (prefill: one head's 128-row tile, half the head dim) or
// 64 x G x 128 / G (verify: a kv head's query vectors of 128 / G rows).
int get_qmap(const void* q, int hq, int rows, int box_heads, int box_rows, CUtensorMap* out) {
  if (dry_run()) {
    std::memset(out, 0, sizeof(*out));
    return TFPA_OK;
  }
  auto fn = encode_fn();
  if (!fn) return TFPA_ECUDA;
  cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)hq, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)hq * kHeadDim * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TFPA_OK : TFPA_ECUDA;
}

// ------------------------------------------------------------ validation
// Q tiles of the prompt and verify paths are loaded by TMA, from device (or
// managed) memory only: pinned host memory, which the decode path takes for
// q, is refused for them before anything is enqueued.
int check_tma_source(const void* q) {
  if (dry_run()) return TFPA_OK;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
    cudaGetLastError();   // the failed query's error stays with this call
    return TFPA_EINVAL;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged ? TFPA_OK
                                                                              : TFPA_EINVAL;
}

int32_t pages_of(int32_t L) { return (L + kPage - 1) / kPage; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_cache(const tfpa_cache* c) {
  if (!c) return TFPA_EINVAL;
  if (c->dtype != TFPA_BF16 && c->dtype != TFPA_FP8_E4M3) return TFPA_EINVAL;
  if (c->head_dim != kHeadDim || c->hkv < 1 || c->hq < 1 || c->hq % c->hkv) return TFPA_EINVAL;
  if (c->dtype == TFPA_FP8_E4M3 && (!c->k_scale || !c->v_scale)) return TFPA_EINVAL;
  if ((c->k_pool && !aligned(c->k_pool, 16)) || (c->v_pool && !aligned(c->v_pool, 16)))
    return TFPA_EINVAL;
  return TFPA_OK;
}

int check_segs(const tfpa_cache* c, const tfpa_seg* segs, int32_t nseg) {
  if (nseg < 0 || (nseg > 0 && !segs)) return TFPA_EINVAL;
  for (int32_t s = 0; s < nseg; ++s) {
    const tfpa_seg& g = segs[s];
    if (g.seq_len < 1) return TFPA_EINVAL;
    if (g.page_table) {
      if (!c->k_pool || !c->v_pool || c->num_pages < 1) return TFPA_EINVAL;
      if ((int64_t)c->num_pages * c->hkv * kPage > INT32_MAX) return TFPA_EINVAL;
      if (g.page_table_host) {
        const int32_t n = pages_of(g.seq_len);
        for (int32_t i = 0; i < n; ++i)
          if (g.page_table_host[i] < 0 || g.page_table_host[i] >= c->num_pages)
            return TFPA_ERANGE;
      }
    } else {
      if (!g.k_slab || !g.v_slab) return TFPA_EINVAL;
      if (!aligned(g.k_slab, 16) || !aligned(g.v_slab, 16)) return TFPA_EINVAL;
      if (g.slab_cap % kPage || g.slab_cap < pages_of(g.seq_len) * kPage) return TFPA_EINVAL;
      if ((int64_t)c->hkv * g.slab_cap > INT32_MAX) return TFPA_EINVAL;
    }
  }
  return TFPA_OK;
}

// A run: consecutive rows of one segment at consecutive positions.
struct Run {
  int32_t seg, row0, nrows, pos0;
};

int build_runs(const tfpa_seg* segs, int32_t nseg, const int32_t* row_seg,
               const int32_t* row_pos, int32_t rows, std::vector<Run>& out) {
  out.clear();
  if (rows < 0 || (rows > 0 && (!row_seg || !row_pos))) return TFPA_EINVAL;
  for (int32_t r = 0; r < rows; ++r) {
    const int32_t s = row_seg[r], p = row_pos[r];
    if (s < 0 || s >= nseg) return TFPA_ERANGE;
    if (p < 0 || p >= segs[s].seq_len) return TFPA_ERANGE;
    if (!out.empty()) {
      Run& b = out.back();
      if (b.seg == s && b.pos0 + b.nrows == p) {
        ++b.nrows;
        continue;
      }
    }
    out.push_back(Run{s, r, 1, p});
  }
  return TFPA_OK;
}

// Runs of four or more m-tiles (16 query vectors each, so at least 49
// vectors per kv head) are dense enough for the tensor cores: they take the
// prefill kernel in verify mode, when a tile holds the group's heads.
bool on_verify_path(const Run& r, int G) {
  return G <= kVerifyVectors && (r.nrows * G + 15) / 16 >= 4;
}

int to_err(cudaError_t e) { return e == cudaSuccess ? TFPA_OK : TFPA_ECUDA; }

}  // namespace

// A call's launches, planned and kept by value for a later tfpa_plan_launch.
// In device mode (dyn_base set) each decode, merge and write launch owns a
// 16-byte aligned slot of the caller's device buffer at dyn_base, from which
// it reads its dynamic data; the plan keeps the host image in the launch's
// parameters (`d`) for tfpa_plan_dyn_pack.
struct tfpa_plan {
  enum Kind : int { kDecode, kVerify, kMerge, kWrite };
  struct Entry {
    Kind kind;
    bool fp8;
    int grid;
    size_t index;   // into the vector of its kind
  };
  std::vector<Entry> entries;
  std::vector<DecodeParams> decode;
  std::vector<PrefillParams> verify;
  std::vector<MergeParams> merge;
  std::vector<WriteParams> write;
  uint8_t* dyn_base = nullptr;   // DEVICE, or nullptr: parameter mode
  size_t dyn_cap = 0;
  size_t dyn_used = 0;           // bytes of dyn_base handed out
  cudaGraphExec_t exec = nullptr;   // tfpa_plan_capture's graph
  uint64_t exec_shape = 0;          // the plan's shape when it was captured
  uint64_t shape = 0;               // the shape of the launches held now
  bool captured = false;
  ~tfpa_plan() {
    if (exec) cudaGraphExecDestroy(exec);
  }
};

namespace {

// Where a call's launches go: enqueued on a stream now, or appended to a
// plan.  A planning call that fails takes back what it appended (Mark).
struct Sink {
  cudaStream_t stream = nullptr;
  tfpa_plan* plan = nullptr;
  struct Mark {
    size_t e, d, v, m, w, dyn;
  };
  // Device mode: launch shapes must not depend on the streams' lengths.
  bool device() const { return plan && plan->dyn_base; }
  Mark mark() const {
    return plan ? Mark{plan->entries.size(), plan->decode.size(), plan->verify.size(),
                       plan->merge.size(), plan->write.size(), plan->dyn_used}
                : Mark{0, 0, 0, 0, 0, 0};
  }
  void rollback(const Mark& k) const {
    if (!plan) return;
    plan->entries.resize(k.e);
    plan->decode.resize(k.d);
    plan->verify.resize(k.v);
    plan->merge.resize(k.m);
    plan->write.resize(k.w);
    plan->dyn_used = k.dyn;
  }
  template <typename P>
  int keep(tfpa_plan::Kind kind, std::vector<P>& v, const P& p, bool fp8, int grid) const {
    v.push_back(p);
    plan->entries.push_back(tfpa_plan::Entry{kind, fp8, grid, v.size() - 1});
    return TFPA_OK;
  }
  // keep() for a launch with dynamic data: in device mode the launch takes
  // the next slot of the plan's device buffer.
  template <typename P>
  int keep_dyn(tfpa_plan::Kind kind, std::vector<P>& v, const P& p, bool fp8, int grid) const {
    const size_t off = plan->dyn_used;
    if (plan->dyn_base) {
      const size_t end = (off + sizeof(p.d) + 15) & ~size_t(15);
      if (end > plan->dyn_cap) return TFPA_ECAPACITY;
      plan->dyn_used = end;
    }
    keep(kind, v, p, fp8, grid);
    v.back().dyn = plan->dyn_base
                       ? reinterpret_cast<decltype(p.dyn)>(plan->dyn_base + off)
                       : nullptr;
    return TFPA_OK;
  }
  int decode(const DecodeParams& p, bool fp8, int grid) const {
    if (plan) return keep_dyn(tfpa_plan::kDecode, plan->decode, p, fp8, grid);
    return dry_run() ? TFPA_OK : to_err(launch_decode_partial(p, fp8, grid, stream));
  }
  int verify(const PrefillParams& p, bool fp8, int tiles) const {
    // the tensor-core verify launch's grid follows the streams' lengths
    if (device()) return TFPA_EINVAL;
    if (plan) return keep(tfpa_plan::kVerify, plan->verify, p, fp8, tiles);
    return dry_run() ? TFPA_OK : to_err(launch_verify(p, fp8, tiles, stream));
  }
  int merge(const MergeParams& p) const {
    if (plan) return keep_dyn(tfpa_plan::kMerge, plan->merge, p, false, 0);
    return dry_run() ? TFPA_OK : to_err(launch_merge(p, stream));
  }
  int write(const WriteParams& p) const {
    if (plan) return keep_dyn(tfpa_plan::kWrite, plan->write, p, false, 0);
    return dry_run() ? TFPA_OK : to_err(launch_write_kv(p, stream));
  }
};

}  // namespace

// One page per split up to 16 pages (a short stream's keys spread over as
// many CTAs as it has pages), then at least two.
extern "C" int32_t tfpa_pages_per_split(int32_t seq_len) {
  const int32_t np = pages_of(std::max(seq_len, 1));
  if (np <= 16) return 1;
  return std::max<int32_t>(2, (np + kMaxSplits - 1) / kMaxSplits);
}

extern "C" int32_t tfpa_num_splits(int32_t seq_len) {
  const int32_t np = pages_of(std::max(seq_len, 1));
  const int32_t pps = tfpa_pages_per_split(seq_len);
  return (np + pps - 1) / pps;
}

namespace {

// Splits of a run on the tensor-core verify path: at least 24 pages and at
// most 7 a stream.  A verify tile carries a fixed cost (set-up, its first
// loads, a cold first softmax step and the epilogue: about a quarter of a
// 24-page tile), so a long stream takes a few long tiles.  A function of the
// stream's length only, like the decode splits, so a stream's bytes do not
// depend on its batch.  On 65,536-key streams (7 splits of 37 pages), 8
// streams x 8 kv heads make 448 tiles, 2.95 waves of 152 SMs; 16-node trees
// took 294 / 345 us (e4m3 / bf16 cache) with 11 splits of 24 pages, 279 /
// 331 with 9 of 29, 263 / 325 with 7 of 37 and 295 / 348 with 6 of 43.
// Other batches fill the waves differently.  Never more splits than the
// decode path's, so a scratch sized for decode holds them.
int32_t verify_pages_per_split(int32_t seq_len) {
  const int32_t np = pages_of(std::max(seq_len, 1));
  return std::max<int32_t>(24, (np + 6) / 7);
}
int32_t verify_num_splits(int32_t seq_len) {
  const int32_t np = pages_of(std::max(seq_len, 1));
  const int32_t pps = verify_pages_per_split(seq_len);
  return (np + pps - 1) / pps;
}

// K/V sources of one launch: source 0 is the pool, 1.. are slab streams.
struct SourceSet {
  int slab_seg[kMaxSlabs];
  int nslab = 0;
  bool pool = false;
  // Source index for segment `s`, or -1 if the set is full.
  int add(const tfpa_seg* segs, int s) {
    if (segs[s].page_table) {
      pool = true;
      return 0;
    }
    for (int i = 0; i < nslab; ++i)
      if (slab_seg[i] == s) return i + 1;
    if (nslab == kMaxSlabs) return -1;
    slab_seg[nslab] = s;
    return ++nslab;
  }
};

int fill_maps(const tfpa_cache* c, const tfpa_seg* segs, const SourceSet& ss, bool fp8,
              int box_inner, int box_rows, KVMaps* maps, int32_t& nsrc) {
  int e;
  if (ss.pool) {
    const uint64_t rows = (uint64_t)c->num_pages * c->hkv * kPage;
    if ((e = get_map(c->k_pool, rows, fp8, box_inner, box_rows, &maps[0].k))) return e;
    if ((e = get_map(c->v_pool, rows, fp8, box_inner, box_rows, &maps[0].v))) return e;
  }
  for (int i = 0; i < ss.nslab; ++i) {
    const tfpa_seg& g = segs[ss.slab_seg[i]];
    const uint64_t rows = (uint64_t)c->hkv * g.slab_cap;
    if ((e = get_map(g.k_slab, rows, fp8, box_inner, box_rows, &maps[i + 1].k))) return e;
    if ((e = get_map(g.v_slab, rows, fp8, box_inner, box_rows, &maps[i + 1].v))) return e;
  }
  nsrc = 1 + ss.nslab;
  return TFPA_OK;
}

void fill_run(RunInfo& ri, const tfpa_seg& g, int src, int row0, int nrows, int pos0) {
  ri.page_table = g.page_table;
  ri.src = src;
  ri.seq_len = g.seq_len;
  ri.row0 = row0;
  ri.nrows = nrows;
  ri.pos0 = pos0;
  ri.nsplit = tfpa_num_splits(g.seq_len);
  ri.pps = tfpa_pages_per_split(g.seq_len);
  ri.item0 = 0;
  ri.slab_cap = g.page_table ? 0 : g.slab_cap;
  ri.pad_ = 0;
}

// Key stages of decode work item (m-tile mt, split sigma) of a run: its
// split's keys, cut at the stream's end and at the last position of the
// item's rows (the kernel's item key range, in units of the kernel's chunk).
int item_stages(const RunInfo& ri, int G, int mt, int sigma, int chunk) {
  const int nq = ri.nrows * G;
  const int last_qv = std::min(16 * mt + 15, nq - 1);
  const int maxpos = ri.pos0 + last_qv / G;
  const int klo = sigma * ri.pps * kPage;
  const int khi = std::min(std::min(klo + ri.pps * kPage, ri.seq_len), maxpos + 1);
  return khi > klo ? (khi - klo + chunk - 1) / chunk : 0;
}

// Per-CTA item ranges of a decode partial launch, balanced by work: an item
// weighs its key stages plus a fixed cost (its query load and combine), and
// CTA b starts at the first item whose prefix weight reaches b / grid of the
// total.  Items are walked in the kernel's order: run, kv head, m-tile,
// split.  An item's weight does not depend on its kv head, so each run's
// (m-tile, split) prefix weights are computed once, and each CTA boundary is
// found by a binary search in the block of the kv head that holds it.
void plan_cta_ranges(DecodeParams& p, int nr, int G, bool fp8, int grid) {
  const int chunk = fp8 ? 256 : 128;
  // The fixed cost, in key stages, was measured on the overcommitted pool
  // (17 streams of 1k-262k keys, e4m3): 0 -> 380 us, 1 -> 341 us, 2 -> 348 us,
  // 4 -> 377 us, 8 -> 444 us; uniform batches do not depend on it.
  constexpr int64_t kItemCost = 1;
  thread_local std::vector<int64_t> cum;     // per run: 0, w0, w0 + w1, ...
  int32_t blk[kMaxRuns + 1];                 // run r's prefix weights: cum[blk[r] .. blk[r + 1]]
  cum.clear();
  int64_t total = 0;
  for (int r = 0; r < nr; ++r) {
    const RunInfo& ri = p.d.runs[r];
    const int mtiles = (ri.nrows * G + 15) / 16;
    blk[r] = (int32_t)cum.size();
    int64_t sum = 0;
    cum.push_back(0);
    for (int mt = 0; mt < mtiles; ++mt)
      for (int sg = 0; sg < ri.nsplit; ++sg) {
        sum += item_stages(ri, G, mt, sg, chunk) + kItemCost;
        cum.push_back(sum);
      }
    total += sum * p.hkv;
  }
  blk[nr] = (int32_t)cum.size();
  int b = 1, item = 0;
  int64_t prefix = 0;   // weight of the items before the current block
  p.d.cta_item0[0] = 0;
  for (int r = 0; r < nr && b < grid; ++r) {
    const int64_t* c = cum.data() + blk[r];
    const int32_t n = blk[r + 1] - blk[r] - 1;   // items of one kv head's block
    for (int g = 0; g < p.hkv && b < grid; ++g) {
      // CTA b starts at the first item whose prefix weight P satisfies
      // P * grid >= total * b, i.e. P >= ceil(total * b / grid)
      while (b < grid) {
        const int64_t need = (total * b + grid - 1) / grid - prefix;
        const int32_t i = (int32_t)(std::lower_bound(c, c + n, need) - c);
        if (i >= n) break;
        p.d.cta_item0[b++] = item + i;
      }
      prefix += c[n];
      item += n;
    }
  }
  // CTAs past the last boundary get empty ranges at the end
  int n_items = 0;
  for (int r = 0; r < nr; ++r) n_items += (blk[r + 1] - blk[r] - 1) * p.hkv;
  while (b <= grid) p.d.cta_item0[b++] = n_items;
}

// Streams of at most this many splits (1,024 positions) are merged inside
// the partial kernel when the scratch has arrival counters.
constexpr int kFusedMergeMaxSplits = 4;

struct RopeArgs {
  const int32_t* pos;   // DEVICE [rows] or nullptr (the storage positions)
  const float* cos;     // DEVICE [n][64] or nullptr (plain store)
  const float* sin;
  int32_t n;
};
int write_impl(const tfpa_cache* c, const tfpa_seg* segs, int32_t nseg, const void* k_rows,
               const void* v_rows, const int32_t* row_seg, const int32_t* row_pos, int32_t rows,
               const RopeArgs& rope, const Sink& sink);

// Partial (and optionally merge) launches over the call's rows.  With
// `sliced`, each launch's partials start at scratch row 0 and are merged
// before the next launch; otherwise partials land at the call's own row and
// no merge runs.
// With k_rows / v_rows (append), the rows' K and V are stored as well: by
// the decode partial kernel itself when every run takes it and no segment
// has two runs (a run's CTAs store the new rows they read before reading
// them), else by a KV write launch ahead of the decode launches.
int decode_impl(const tfpa_cache* c, const tfpa_seg* segs, int32_t nseg, const void* q,
                const int32_t* row_seg, const int32_t* row_pos, const uint64_t* anc,
                int32_t rows, float scale, const tfpa_scratch* sc, void* out, float* lse,
                const Sink& sink, bool sliced, const void* k_rows = nullptr,
                const void* v_rows = nullptr) {
  int e;
  if ((e = check_cache(c)) || (e = check_segs(c, segs, nseg))) return e;
  if (!sc || !sc->part_o || !sc->part_ml || sc->cap_rows < 1 || sc->max_splits < 1)
    return TFPA_EINVAL;
  if (rows > 0 && (!q || !aligned(q, 16))) return TFPA_EINVAL;
  if (sliced && rows > 0 && (!out || !aligned(out, 8))) return TFPA_EINVAL;
  if (anc && !aligned(anc, 8)) return TFPA_EINVAL;
  if (!std::isfinite(scale) || !(scale > 0.f)) return TFPA_EINVAL;
  if (!sliced && rows > sc->cap_rows) return TFPA_ECAPACITY;
  thread_local std::vector<Run> runs;   // reused by every call of this thread
  if ((e = build_runs(segs, nseg, row_seg, row_pos, rows, runs))) return e;
  for (const Run& r : runs)
    if (tfpa_num_splits(segs[r.seg].seq_len) > sc->max_splits) return TFPA_ECAPACITY;
  if (rows == 0) return TFPA_OK;
  if ((e = check_device())) return e;
  const bool fp8 = c->dtype == TFPA_FP8_E4M3;
  const int G = c->hq / c->hkv;
  for (const Run& r : runs)
    if (on_verify_path(r, G)) {
      if ((e = check_tma_source(q))) return e;
      break;
    }
  if (k_rows || v_rows) {
    if (!k_rows || !v_rows || !aligned(k_rows, 16) || !aligned(v_rows, 16)) return TFPA_EINVAL;
    bool fuse = true;
    for (size_t i = 0; fuse && i < runs.size(); ++i) {
      fuse = !on_verify_path(runs[i], G);   // the decode partial path
      for (size_t j = 0; fuse && j < i; ++j) fuse = runs[j].seg != runs[i].seg;
    }
    if (!fuse) {
      if ((e = write_impl(c, segs, nseg, k_rows, v_rows, row_seg, row_pos, rows,
                          RopeArgs{nullptr, nullptr, nullptr, 0}, sink)))
        return e;
      k_rows = v_rows = nullptr;
    }
  }
  const int nsm = sm_count();
  if (nsm < 1) return TFPA_ECUDA;
  const size_t hd = (size_t)c->hq * kHeadDim;

  size_t ri = 0;
  int32_t taken = 0;  // rows of runs[ri] already launched
  // Launch parameters are large (kernel arguments by value): each host
  // thread builds them in its own buffers.
  thread_local DecodeParams p;
  thread_local PrefillParams pv;   // the tensor-core verify launch of the same rows
  thread_local MergeParams mp;
  // Runs of four or more m-tiles (16 query vectors each, so at least 49
  // vectors per kv head) are dense enough for the tensor cores: they go to
  // the prefill kernel in verify mode (128 / G rows x the group's G heads
  // per tile), the rest to the decode partial kernel.  Decided on the
  // call's whole run, so every slice of it computes its rows with the same
  // arithmetic (slices give the same bytes as one launch).  A group wider
  // than a tile (more than 128 query heads per kv head) stays on the decode
  // kernel (on_verify_path).
  const int vrows = G <= kVerifyVectors ? kVerifyVectors / G : 1;   // rows of a verify tile
  while (ri < runs.size()) {
    SourceSet ss;
    const int32_t base = runs[ri].row0 + taken;  // first call row of this launch
    int32_t nrows = 0, items = 0, tiles = 0;
    int nr = 0, nd = 0, nv = 0;  // runs of the slice: all, decode, verify
    while (ri < runs.size() && nr < kMaxRuns && nrows < sc->cap_rows) {
      const Run& r = runs[ri];
      const int src = ss.add(segs, r.seg);
      if (src < 0) break;
      const int32_t take = std::min(r.nrows - taken, sc->cap_rows - nrows);
      const tfpa_seg& g = segs[r.seg];
      if (on_verify_path(r, G)) {
        if (nv == 0) std::memset(&pv, 0, sizeof(pv));   // only launches that run are built
        RunInfo& info = pv.runs[nv++];
        fill_run(info, g, src, nrows, take, r.pos0 + taken);
        info.pps = verify_pages_per_split(g.seq_len);
        info.nsplit = verify_num_splits(g.seq_len);
        info.item0 = tiles;
        tiles += c->hkv * ((take + vrows - 1) / vrows) * info.nsplit;
        mp.d.runs[nr] = MergeRun{nrows, take, info.nsplit, 0};
      } else {
        if (nd == 0) std::memset(&p, 0, sizeof(p));
        RunInfo& info = p.d.runs[nd++];
        fill_run(info, g, src, nrows, take, r.pos0 + taken);
        info.item0 = items;
        items += c->hkv * ((take * G + 15) / 16) * info.nsplit;
        mp.d.runs[nr] = MergeRun{nrows, take, info.nsplit, 0};
      }
      ++nr;
      nrows += take;
      taken += take;
      if (taken == r.nrows) {
        ++ri;
        taken = 0;
      }
    }
    const int32_t srow = sliced ? 0 : base;  // scratch row of this launch's first row
    const size_t srow_elems = (size_t)srow * c->hq * sc->max_splits;
    float* part_o = sc->part_o + srow_elems * kHeadDim;
    float* part_ml = sc->part_ml + srow_elems * 2;
    // With arrival counters, plain causal rows in parameter mode, no rows on
    // the verify path and few splits per stream, the partial kernel merges
    // the slice itself.  A group's merge runs on the one SM that finished
    // its last split, reading every split's partial: cheap for a few splits,
    // slower than a separate grid-wide merge for many.
    bool fused = sliced && nv == 0 && sc->arrive && !anc && !sink.device();
    for (int r = 0; fused && r < nd; ++r) fused = p.d.runs[r].nsplit <= kFusedMergeMaxSplits;
    if (nd > 0) {
      if ((e = fill_maps(c, segs, ss, fp8, fp8 ? 128 : 64, 128, p.maps, p.nsrc)))
        return e;
      p.q = static_cast<const __nv_bfloat16*>(q) + (size_t)base * hd;
      p.anc = anc ? anc + base : nullptr;   // the ancestor table shifts with the rows
      p.part_o = part_o;
      p.part_ml = part_ml;
      p.k_scale = c->k_scale;
      p.v_scale = c->v_scale;
      p.err_flag = c->err_flag;
      const size_t rd = (size_t)c->hkv * kHeadDim;
      p.k_rows = k_rows ? static_cast<const __nv_bfloat16*>(k_rows) + (size_t)base * rd : nullptr;
      p.v_rows = v_rows ? static_cast<const __nv_bfloat16*>(v_rows) + (size_t)base * rd : nullptr;
      if (k_rows) {
        // where each source's rows go: the pool, then the slabs in source order
        p.k_base[0] = c->k_pool;
        p.v_base[0] = c->v_pool;
        for (int i = 0; i < ss.nslab; ++i) {
          p.k_base[i + 1] = segs[ss.slab_seg[i]].k_slab;
          p.v_base[i + 1] = segs[ss.slab_seg[i]].v_slab;
        }
      }
      p.arrive = fused ? sc->arrive + (size_t)srow * c->hq : nullptr;
      p.out = fused ? static_cast<__nv_bfloat16*>(out) + (size_t)base * hd : nullptr;
      p.lse = fused && lse ? lse + (size_t)base * c->hq : nullptr;
      p.d.nruns = nd;
      p.d.n_items = items;
      p.hq = c->hq;
      p.hkv = c->hkv;
      p.group = G;
      p.max_splits = sc->max_splits;
      p.num_pages = c->num_pages;
      p.rows = nrows;
      p.scale_log2 = scale * 1.4426950408889634f;
      // In device mode the grid is one CTA per SM whatever the work, so
      // that the launch can be replayed as the streams grow.
      const int grid = std::min(sink.device() ? nsm : std::min(items, nsm), kMaxDecodeGrid);
      plan_cta_ranges(p, nd, G, fp8, grid);
      record(1, base, nrows, nd, items, grid, (int64_t)base * hd, 0);
      if ((e = sink.decode(p, fp8, grid))) return e;
    }
    if (nv > 0) {
      if ((e = fill_maps(c, segs, ss, fp8, fp8 ? 128 : 64, 128, pv.maps, pv.nsrc))) return e;
      // The kernel loads a verify tile's Q as two boxes of 64 query vectors
      // when G divides 64 (so that a tile of at most 64 vectors can hold
      // them twice, one copy per MMA slot), else as one box.
      const int qbox = 64 % G == 0 ? 64 / G : vrows;
      if ((e = get_qmap(static_cast<const __nv_bfloat16*>(q) + (size_t)base * hd, c->hq, nrows,
                        G, qbox, &pv.qmap)))
        return e;
      pv.q = static_cast<const __nv_bfloat16*>(q) + (size_t)base * hd;
      pv.anc = anc ? anc + base : nullptr;
      pv.part_o = part_o;
      pv.part_ml = part_ml;
      pv.k_scale = c->k_scale;
      pv.v_scale = c->v_scale;
      pv.err_flag = c->err_flag;
      pv.nruns = nv;
      pv.n_tiles = tiles;
      pv.hq = c->hq;
      pv.hkv = c->hkv;
      pv.group = G;
      pv.num_pages = c->num_pages;
      pv.rows = nrows;
      pv.max_splits = sc->max_splits;
      pv.scale_log2 = scale * 1.4426950408889634f;
      record(8, base, nrows, nv, tiles, tiles, (int64_t)base * hd, 0);
      if ((e = sink.verify(pv, fp8, tiles))) return e;
    }
    if (sliced && !fused) {
      mp.part_o = part_o;
      mp.part_ml = part_ml;
      mp.out = static_cast<__nv_bfloat16*>(out) + (size_t)base * hd;
      mp.lse = lse ? lse + (size_t)base * c->hq : nullptr;
      mp.d.nruns = nr;
      mp.d.rows = nrows;
      mp.hq = c->hq;
      mp.max_splits = sc->max_splits;
      record(2, base, nrows, nr, nrows * c->hq, (nrows * c->hq + 7) / 8, 0, (int64_t)base * hd);
      if ((e = sink.merge(mp))) return e;
    }
  }
  return TFPA_OK;
}

}  // namespace

extern "C" int tfpa_decode_partial(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                                   const void* q, const int32_t* row_seg, const int32_t* row_pos,
                                   int32_t rows, float softmax_scale, const tfpa_scratch* scratch,
                                   cudaStream_t stream) {
  return decode_impl(cache, segs, nseg, q, row_seg, row_pos, nullptr, rows, softmax_scale,
                     scratch, nullptr, nullptr, Sink{stream, nullptr}, false);
}

extern "C" int tfpa_decode(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                           const void* q, const int32_t* row_seg, const int32_t* row_pos,
                           int32_t rows, float softmax_scale, const tfpa_scratch* scratch,
                           void* out, float* lse, cudaStream_t stream) {
  return decode_impl(cache, segs, nseg, q, row_seg, row_pos, nullptr, rows, softmax_scale,
                     scratch, out, lse, Sink{stream, nullptr}, true);
}

extern "C" int tfpa_row_splits(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                               const int32_t* row_seg, const int32_t* row_pos, int32_t rows,
                               int32_t* nsplit) {
  int e;
  if ((e = check_cache(cache)) || (e = check_segs(cache, segs, nseg))) return e;
  if (rows > 0 && !nsplit) return TFPA_EINVAL;
  thread_local std::vector<Run> runs;
  if ((e = build_runs(segs, nseg, row_seg, row_pos, rows, runs))) return e;
  // the same choice of kernel as decode_impl: runs of four or more m-tiles
  // take the tensor-core verify path and its splits
  const int G = cache->hq / cache->hkv;
  for (const Run& r : runs) {
    const int32_t L = segs[r.seg].seq_len;
    const int32_t n = on_verify_path(r, G) ? verify_num_splits(L) : tfpa_num_splits(L);
    for (int32_t i = 0; i < r.nrows; ++i) nsplit[r.row0 + i] = n;
  }
  return TFPA_OK;
}

extern "C" int tfpa_decode_tree(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                                const void* q, const int32_t* row_seg, const int32_t* row_pos,
                                const uint64_t* row_anc, int32_t rows, float softmax_scale,
                                const tfpa_scratch* scratch, void* out, float* lse,
                                cudaStream_t stream) {
  if (rows > 0 && !row_anc) return TFPA_EINVAL;
  return decode_impl(cache, segs, nseg, q, row_seg, row_pos, row_anc, rows, softmax_scale,
                     scratch, out, lse, Sink{stream, nullptr}, true);
}

extern "C" int tfpa_decode_append(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                                  const void* k_rows, const void* v_rows, const void* q,
                                  const int32_t* row_seg, const int32_t* row_pos, int32_t rows,
                                  float softmax_scale, const tfpa_scratch* scratch, void* out,
                                  float* lse, cudaStream_t stream) {
  if (rows > 0 && (!k_rows || !v_rows)) return TFPA_EINVAL;
  return decode_impl(cache, segs, nseg, q, row_seg, row_pos, nullptr, rows, softmax_scale,
                     scratch, out, lse, Sink{stream, nullptr}, true, k_rows, v_rows);
}

extern "C" int tfpa_merge(const tfpa_scratch* sc, int32_t hq, int32_t rows,
                          const int32_t* nsplit, void* out, float* lse, cudaStream_t stream) {
  if (!sc || !sc->part_o || !sc->part_ml || hq < 1 || rows < 0) return TFPA_EINVAL;
  if (rows > sc->cap_rows) return TFPA_ECAPACITY;
  if (rows == 0) return TFPA_OK;
  if (!nsplit || !out || !aligned(out, 8)) return TFPA_EINVAL;
  for (int32_t r = 0; r < rows; ++r)
    if (nsplit[r] < 1 || nsplit[r] > std::min(sc->max_splits, kMaxSplits)) return TFPA_ECAPACITY;
  int e;
  if ((e = check_device())) return e;
  thread_local MergeParams mp;
  int32_t r = 0;
  while (r < rows) {
    std::memset(&mp, 0, sizeof(mp));
    const int32_t base = r;
    int nr = 0;
    while (r < rows && nr < (int)(sizeof(mp.d.runs) / sizeof(mp.d.runs[0]))) {
      int32_t n = 1;
      while (r + n < rows && nsplit[r + n] == nsplit[r]) ++n;
      mp.d.runs[nr++] = MergeRun{r - base, n, nsplit[r], 0};
      r += n;
    }
    const size_t srow = (size_t)base * hq * sc->max_splits;
    mp.part_o = sc->part_o + srow * kHeadDim;
    mp.part_ml = sc->part_ml + srow * 2;
    mp.out = static_cast<__nv_bfloat16*>(out) + (size_t)base * hq * kHeadDim;
    mp.lse = lse ? lse + (size_t)base * hq : nullptr;
    mp.d.nruns = nr;
    mp.d.rows = r - base;
    mp.hq = hq;
    mp.max_splits = sc->max_splits;
    record(2, base, r - base, nr, (r - base) * hq, ((r - base) * hq + 7) / 8, 0,
           (int64_t)base * hq * kHeadDim);
    if (!dry_run())
      if ((e = to_err(launch_merge(mp, stream)))) return e;
  }
  return TFPA_OK;
}

namespace {

int write_impl(const tfpa_cache* c, const tfpa_seg* segs, int32_t nseg, const void* k_rows,
               const void* v_rows, const int32_t* row_seg, const int32_t* row_pos, int32_t rows,
               const RopeArgs& rope, const Sink& sink) {
  int e;
  if ((e = check_cache(c)) || (e = check_segs(c, segs, nseg))) return e;
  if (rows > 0 && (!k_rows || !v_rows || !aligned(k_rows, 16) || !aligned(v_rows, 16)))
    return TFPA_EINVAL;
  if (rope.cos) {
    if (!rope.sin || rope.n < 1 || !aligned(rope.cos, 16) || !aligned(rope.sin, 16) ||
        (rope.pos && !aligned(rope.pos, 4)))
      return TFPA_EINVAL;
    if (!rope.pos)
      for (int32_t r = 0; r < rows; ++r)
        if (row_pos && row_pos[r] >= rope.n) return TFPA_ERANGE;
  }
  thread_local std::vector<Run> runs;   // reused by every call of this thread
  if ((e = build_runs(segs, nseg, row_seg, row_pos, rows, runs))) return e;
  if (rows == 0) return TFPA_OK;
  if ((e = check_device())) return e;
  const size_t rd = (size_t)c->hkv * kHeadDim;
  thread_local WriteParams p;
  size_t ri = 0;
  while (ri < runs.size()) {
    std::memset(&p, 0, sizeof(p));
    const int32_t base = runs[ri].row0;
    int nr = 0;
    int32_t nrows = 0;
    while (ri < runs.size() && nr < kMaxRuns) {
      const Run& r = runs[ri++];
      const tfpa_seg& g = segs[r.seg];
      WriteRun& w = p.d.runs[nr++];
      w.page_table = g.page_table;
      w.k_dst = g.page_table ? c->k_pool : g.k_slab;
      w.v_dst = g.page_table ? c->v_pool : g.v_slab;
      w.row0 = r.row0 - base;
      w.nrows = r.nrows;
      w.pos0 = r.pos0;
      w.slab_cap = g.slab_cap;
      w.seq_len = g.seq_len;
      nrows = r.row0 + r.nrows - base;
    }
    p.k_rows = static_cast<const __nv_bfloat16*>(k_rows) + (size_t)base * rd;
    p.v_rows = static_cast<const __nv_bfloat16*>(v_rows) + (size_t)base * rd;
    p.k_scale = c->k_scale;
    p.v_scale = c->v_scale;
    p.err_flag = c->err_flag;
    p.rope_cos = rope.cos;
    p.rope_sin = rope.sin;
    p.rope_pos = rope.pos ? rope.pos + base : nullptr;   // shifts with the rows
    p.rope_n = rope.n;
    p.d.nruns = nr;
    p.d.rows = nrows;
    p.hkv = c->hkv;
    p.num_pages = c->num_pages;
    p.fp8 = c->dtype == TFPA_FP8_E4M3;
    record(0, base, nrows, nr, nrows * c->hkv, (nrows * c->hkv + 15) / 16, 0, 0);
    if ((e = sink.write(p))) return e;
  }
  return TFPA_OK;
}

}  // namespace

extern "C" int tfpa_write_kv(const tfpa_cache* c, const tfpa_seg* segs, int32_t nseg,
                             const void* k_rows, const void* v_rows, const int32_t* row_seg,
                             const int32_t* row_pos, int32_t rows, cudaStream_t stream) {
  return write_impl(c, segs, nseg, k_rows, v_rows, row_seg, row_pos, rows,
                    RopeArgs{nullptr, nullptr, nullptr, 0}, Sink{stream, nullptr});
}

extern "C" int tfpa_write_kv_rope(const tfpa_cache* c, const tfpa_seg* segs, int32_t nseg,
                                  const void* k_rows, const void* v_rows,
                                  const int32_t* row_seg, const int32_t* row_pos,
                                  const int32_t* rope_pos, const float* rope_cos,
                                  const float* rope_sin, int32_t rope_n, int32_t rows,
                                  cudaStream_t stream) {
  if (!rope_cos) return TFPA_EINVAL;
  return write_impl(c, segs, nseg, k_rows, v_rows, row_seg, row_pos, rows,
                    RopeArgs{rope_pos, rope_cos, rope_sin, rope_n}, Sink{stream, nullptr});
}

// ------------------------------------------------------------ plans
namespace {
uint64_t compute_shape(const tfpa_plan* plan);
}  // namespace

extern "C" tfpa_plan* tfpa_plan_create(void) {
  tfpa_plan* plan = new (std::nothrow) tfpa_plan();
  if (plan) plan->shape = compute_shape(plan);
  return plan;
}

extern "C" void tfpa_plan_destroy(tfpa_plan* plan) { delete plan; }

extern "C" void tfpa_plan_clear(tfpa_plan* plan) {
  if (!plan) return;
  plan->entries.clear();
  plan->decode.clear();
  plan->verify.clear();
  plan->merge.clear();
  plan->write.clear();
  plan->dyn_used = 0;
  plan->shape = compute_shape(plan);
}

extern "C" int32_t tfpa_plan_launches(const tfpa_plan* plan) {
  return plan ? (int32_t)plan->entries.size() : 0;
}

extern "C" int tfpa_plan_set_device(tfpa_plan* plan, void* dyn, size_t bytes) {
  if (!plan || !plan->entries.empty()) return TFPA_EINVAL;
  if (dyn && (!aligned(dyn, 16) || bytes < 16)) return TFPA_EINVAL;
  plan->dyn_base = static_cast<uint8_t*>(dyn);
  plan->dyn_cap = dyn ? bytes : 0;
  plan->dyn_used = 0;
  plan->shape = compute_shape(plan);
  return TFPA_OK;
}

extern "C" size_t tfpa_plan_dyn_bytes(const tfpa_plan* plan) {
  return plan ? plan->dyn_used : 0;
}

extern "C" int tfpa_plan_dyn_pack(const tfpa_plan* plan, void* host, size_t bytes) {
  if (!plan || !plan->dyn_base) return TFPA_EINVAL;
  if (plan->dyn_used == 0) return TFPA_OK;
  if (!host) return TFPA_EINVAL;
  if (bytes < plan->dyn_used) return TFPA_ECAPACITY;
  uint8_t* dst = static_cast<uint8_t*>(host);
  auto put = [&](const void* slot, const void* d, size_t n) {
    std::memcpy(dst + (static_cast<const uint8_t*>(slot) - plan->dyn_base), d, n);
  };
  for (const DecodeParams& p : plan->decode) put(p.dyn, &p.d, sizeof(p.d));
  for (const MergeParams& p : plan->merge) put(p.dyn, &p.d, sizeof(p.d));
  for (const WriteParams& p : plan->write) put(p.dyn, &p.d, sizeof(p.d));
  return TFPA_OK;
}

namespace {
// A 64-bit hash of a byte range, eight bytes a step (multiply and
// xor-shift; FNV-1a for the tail).
uint64_t fnv1a(uint64_t h, const void* data, size_t n) {
  const uint8_t* b = static_cast<const uint8_t*>(data);
  size_t i = 0;
  for (; i + 8 <= n; i += 8) {
    uint64_t w;
    std::memcpy(&w, b + i, 8);
    h = (h ^ w) * 0x9E3779B97F4A7C15ull;
    h ^= h >> 29;
  }
  for (; i < n; ++i) h = (h ^ b[i]) * 1099511628211ull;
  return h;
}
// A launch's parameters without its dynamic data.
template <typename P>
uint64_t hash_static(uint64_t h, const P& p) {
  const uint8_t* b = reinterpret_cast<const uint8_t*>(&p);
  const size_t d0 = reinterpret_cast<const uint8_t*>(&p.d) - b;
  h = fnv1a(h, b, d0);
  return fnv1a(h, b + d0 + sizeof(p.d), sizeof(P) - d0 - sizeof(p.d));
}
}  // namespace

namespace {
uint64_t compute_shape(const tfpa_plan* plan) {
  uint64_t h = 14695981039346656037ull;
  for (const tfpa_plan::Entry& en : plan->entries) {
    const int32_t head[3] = {(int32_t)en.kind, (int32_t)en.fp8, en.grid};
    h = fnv1a(h, head, sizeof(head));
    switch (en.kind) {
      case tfpa_plan::kDecode: h = hash_static(h, plan->decode[en.index]); break;
      case tfpa_plan::kVerify: h = fnv1a(h, &plan->verify[en.index], sizeof(PrefillParams)); break;
      case tfpa_plan::kMerge: h = hash_static(h, plan->merge[en.index]); break;
      case tfpa_plan::kWrite: h = hash_static(h, plan->write[en.index]); break;
    }
  }
  return h;
}
}  // namespace

// The shape is recomputed after each planning call (while the GPU is busy
// with the previous step), so that a replay only compares two numbers.
extern "C" uint64_t tfpa_plan_shape(const tfpa_plan* plan) { return plan ? plan->shape : 0; }

extern "C" int tfpa_plan_capture(tfpa_plan* plan, const tfpa_copy* before, int32_t nbefore,
                                 const tfpa_copy* after, int32_t nafter, cudaStream_t stream) {
  if (!plan || plan->entries.empty() || nbefore < 0 || nafter < 0 ||
      (nbefore > 0 && !before) || (nafter > 0 && !after))
    return TFPA_EINVAL;
  for (int32_t i = 0; i < nbefore; ++i)
    if (before[i].bytes && (!before[i].dst || !before[i].src)) return TFPA_EINVAL;
  for (int32_t i = 0; i < nafter; ++i)
    if (after[i].bytes && (!after[i].dst || !after[i].src)) return TFPA_EINVAL;
  const uint64_t shape = tfpa_plan_shape(plan);
  if (dry_run()) {
    plan->exec_shape = shape;
    plan->captured = true;
    return TFPA_OK;
  }
  int e;
  if ((e = check_device())) return e;
  if (stream == nullptr || stream == cudaStreamLegacy) return TFPA_EINVAL;   // not capturable
  if (cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
    return TFPA_ECUDA;
  bool ok = true;
  for (int32_t i = 0; ok && i < nbefore; ++i)
    if (before[i].bytes)
      ok = cudaMemcpyAsync(before[i].dst, before[i].src, before[i].bytes, cudaMemcpyDefault,
                           stream) == cudaSuccess;
  if (ok) ok = tfpa_plan_launch(plan, stream) == TFPA_OK;
  for (int32_t i = 0; ok && i < nafter; ++i)
    if (after[i].bytes)
      ok = cudaMemcpyAsync(after[i].dst, after[i].src, after[i].bytes, cudaMemcpyDefault,
                           stream) == cudaSuccess;
  cudaGraph_t graph = nullptr;
  const bool ended = cudaStreamEndCapture(stream, &graph) == cudaSuccess;
  cudaGraphExec_t exec = nullptr;
  ok = ok && ended && graph && cudaGraphInstantiate(&exec, graph, 0ull) == cudaSuccess;
  if (graph) cudaGraphDestroy(graph);
  if (!ok) {
    cudaGetLastError();   // the failed call's error stays with this call
    return TFPA_ECUDA;
  }
  if (plan->exec) cudaGraphExecDestroy(plan->exec);
  plan->exec = exec;
  plan->exec_shape = shape;
  plan->captured = true;
  return TFPA_OK;
}

extern "C" int tfpa_plan_replay(const tfpa_plan* plan, cudaStream_t stream) {
  if (!plan || !plan->captured) return TFPA_EINVAL;
  if (tfpa_plan_shape(plan) != plan->exec_shape) return TFPA_EINVAL;
  if (dry_run()) return TFPA_OK;
  return to_err(cudaGraphLaunch(plan->exec, stream));
}

namespace {
// Runs a planning call into `plan`; on failure the plan is left as it was.
template <typename F>
int plan_call(tfpa_plan* plan, F&& fn) {
  if (!plan) return TFPA_EINVAL;
  const Sink sink{nullptr, plan};
  const Sink::Mark m = sink.mark();
  int e;
  try {
    e = fn(sink);
  } catch (const std::bad_alloc&) {
    e = TFPA_EINVAL;
  }
  if (e != TFPA_OK)
    sink.rollback(m);   // the plan, and so its shape, as before the call
  else
    plan->shape = compute_shape(plan);
  return e;
}
}  // namespace

extern "C" int tfpa_plan_write_kv(tfpa_plan* plan, const tfpa_cache* c, const tfpa_seg* segs,
                                  int32_t nseg, const void* k_rows, const void* v_rows,
                                  const int32_t* row_seg, const int32_t* row_pos,
                                  int32_t rows) {
  return plan_call(plan, [&](const Sink& sink) {
    return write_impl(c, segs, nseg, k_rows, v_rows, row_seg, row_pos, rows,
                      RopeArgs{nullptr, nullptr, nullptr, 0}, sink);
  });
}

extern "C" int tfpa_plan_decode(tfpa_plan* plan, const tfpa_cache* cache, const tfpa_seg* segs,
                                int32_t nseg, const void* q, const int32_t* row_seg,
                                const int32_t* row_pos, int32_t rows, float softmax_scale,
                                const tfpa_scratch* scratch, void* out, float* lse) {
  return plan_call(plan, [&](const Sink& sink) {
    return decode_impl(cache, segs, nseg, q, row_seg, row_pos, nullptr, rows, softmax_scale,
                       scratch, out, lse, sink, true);
  });
}

extern "C" int tfpa_plan_decode_append(tfpa_plan* plan, const tfpa_cache* cache,
                                       const tfpa_seg* segs, int32_t nseg, const void* k_rows,
                                       const void* v_rows, const void* q, const int32_t* row_seg,
                                       const int32_t* row_pos, int32_t rows, float softmax_scale,
                                       const tfpa_scratch* scratch, void* out, float* lse) {
  if (rows > 0 && (!k_rows || !v_rows)) return TFPA_EINVAL;
  return plan_call(plan, [&](const Sink& sink) {
    return decode_impl(cache, segs, nseg, q, row_seg, row_pos, nullptr, rows, softmax_scale,
                       scratch, out, lse, sink, true, k_rows, v_rows);
  });
}

extern "C" int tfpa_plan_launch(const tfpa_plan* plan, cudaStream_t stream) {
  if (!plan) return TFPA_EINVAL;
  if (dry_run()) return TFPA_OK;
  for (const tfpa_plan::Entry& en : plan->entries) {
    cudaError_t r = cudaSuccess;
    switch (en.kind) {
      case tfpa_plan::kDecode:
        r = launch_decode_partial(plan->decode[en.index], en.fp8, en.grid, stream);
        break;
      case tfpa_plan::kVerify:
        r = launch_verify(plan->verify[en.index], en.fp8, en.grid, stream);
        break;
      case tfpa_plan::kMerge:
        r = launch_merge(plan->merge[en.index], stream);
        break;
      case tfpa_plan::kWrite:
        r = launch_write_kv(plan->write[en.index], stream);
        break;
    }
    if (r != cudaSuccess) return TFPA_ECUDA;
  }
  return TFPA_OK;
}

extern "C" int tfpa_keep_kv(const tfpa_cache* c, const tfpa_seg* segs, int32_t nseg,
                            const int32_t* keep_seg, const int32_t* keep_src,
                            const int32_t* keep_dst, int32_t n, cudaStream_t stream) {
  int e;
  if ((e = check_cache(c)) || (e = check_segs(c, segs, nseg))) return e;
  if (n < 0 || (n > 0 && (!keep_seg || !keep_src || !keep_dst))) return TFPA_EINVAL;
  if (n > kMaxKeep) return TFPA_ECAPACITY;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t sg = keep_seg[i];
    if (sg < 0 || sg >= nseg) return TFPA_ERANGE;
    const tfpa_seg& g = segs[sg];
    if (keep_src[i] < 0 || keep_src[i] >= g.seq_len || keep_dst[i] < 0 ||
        keep_dst[i] >= g.seq_len)
      return TFPA_ERANGE;
    for (int32_t j = 0; j < i; ++j)          // one writer per destination row
      if (keep_seg[j] == sg && keep_dst[j] == keep_dst[i]) return TFPA_EINVAL;
  }
  if (n == 0) return TFPA_OK;
  if ((e = check_device())) return e;
  thread_local KeepParams p;
  std::memset(&p, 0, sizeof(p));
  for (int32_t i = 0; i < n; ++i) {
    const tfpa_seg& g = segs[keep_seg[i]];
    KeepPair& kp = p.pairs[i];
    kp.page_table = g.page_table;
    kp.k_slab = g.page_table ? nullptr : g.k_slab;
    kp.v_slab = g.page_table ? nullptr : g.v_slab;
    kp.slab_cap = g.page_table ? 0 : g.slab_cap;
    kp.src = keep_src[i];
    kp.dst = keep_dst[i];
  }
  p.k_pool = c->k_pool;
  p.v_pool = c->v_pool;
  p.err_flag = c->err_flag;
  p.n = n;
  p.hkv = c->hkv;
  p.num_pages = c->num_pages;
  p.row_bytes = c->dtype == TFPA_FP8_E4M3 ? kHeadDim : 2 * kHeadDim;
  record(4, 0, n, 0, n * c->hkv, c->hkv, 0, 0);
  if (!dry_run())
    if ((e = to_err(launch_keep(p, stream)))) return e;
  return TFPA_OK;
}

extern "C" int tfpa_stage_pages(int32_t* page_table, int32_t first, const int32_t* pages,
                                int32_t n, cudaStream_t stream) {
  if (!page_table || first < 0 || n < 0 || (n > 0 && !pages)) return TFPA_EINVAL;
  if (n == 0) return TFPA_OK;
  int e;
  if (!dry_run() && (e = check_device())) return e;
  thread_local StageParams p;
  for (int32_t done = 0; done < n; done += kMaxStage) {
    const int32_t m = std::min<int32_t>(kMaxStage, n - done);
    p.table = page_table;
    p.first = first + done;
    p.n = m;
    std::memcpy(p.ids, pages + done, sizeof(int32_t) * m);
    record(5, done, m, 0, m, 1, 0, 0);
    if (!dry_run())
      if ((e = to_err(launch_stage(p, stream)))) return e;
  }
  return TFPA_OK;
}

namespace {

int copy_impl(const tfpa_cache* c, const tfpa_seg* seg, int32_t p0, int32_t p1, const void* image,
              bool restore, cudaStream_t stream) {
  int e;
  if ((e = check_cache(c)) || (e = check_segs(c, seg, 1))) return e;
  if (!image || !aligned(image, 16)) return TFPA_EINVAL;
  if (p0 < 0 || p0 > p1 || p1 > seg->seq_len) return TFPA_ERANGE;
  if (p0 == p1) return TFPA_OK;
  if (!dry_run() && (e = check_device())) return e;
  CopyParams p{};
  p.page_table = seg->page_table;
  p.k_base = seg->page_table ? c->k_pool : seg->k_slab;
  p.v_base = seg->page_table ? c->v_pool : seg->v_slab;
  p.image = static_cast<uint8_t*>(const_cast<void*>(image));
  p.err_flag = c->err_flag;
  p.slab_cap = seg->page_table ? 0 : seg->slab_cap;
  p.p0 = p0;
  p.p1 = p1;
  p.page0 = p0 / kPage;
  p.hkv = c->hkv;
  p.num_pages = c->num_pages;
  p.row_bytes = c->dtype == TFPA_FP8_E4M3 ? kHeadDim : 2 * kHeadDim;
  p.restore = restore ? 1 : 0;
  const int npages = (p1 - 1) / kPage - p0 / kPage + 1;
  record(restore ? 7 : 6, p0, p1 - p0, 0, npages * c->hkv * 2, npages * c->hkv * 2, 0, 0);
  if (!dry_run())
    if ((e = to_err(launch_copy(p, npages, stream)))) return e;
  return TFPA_OK;
}

}  // namespace

extern "C" int tfpa_save_kv(const tfpa_cache* cache, const tfpa_seg* seg, int32_t p0, int32_t p1,
                            void* image, cudaStream_t stream) {
  return copy_impl(cache, seg, p0, p1, image, false, stream);
}

extern "C" int tfpa_restore_kv(const tfpa_cache* cache, const tfpa_seg* seg, int32_t p0,
                               int32_t p1, const void* image, cudaStream_t stream) {
  return copy_impl(cache, seg, p0, p1, image, true, stream);
}

extern "C" void tfpa_set_launch_hook(tfpa_launch_hook hook, void* user, int dry_run_flag) {
  g_hook_user.store(user, std::memory_order_relaxed);
  g_hook_dry.store(hook ? dry_run_flag : 0, std::memory_order_relaxed);
  g_hook_fn.store(hook, std::memory_order_release);
}

extern "C" const char* tfpa_strerror(int code) {
  switch (code) {
    case TFPA_OK: return "ok";
    case TFPA_EINVAL: return "invalid argument (dims, dtype, null pointer or alignment)";
    case TFPA_ERANGE: return "segment, position or page id out of range";
    case TFPA_ECAPACITY: return "scratch capacity exceeded (rows or splits)";
    case TFPA_ECUDA: return "CUDA call or launch failed";
    case TFPA_EDEVICE: return "current device is not sm_100-family";
    case TFPA_ELANEMEM: return "the page pool cannot hold the claim now (wait for releases)";
    default: return "unknown error";
  }
}

extern "C" const char* tfpa_version(void) { return "tfpa 0.1 (sm_103a)"; }

// ------------------------------------------------------------ prefill
namespace {
constexpr int kPrefillTileRows = 128;
}

extern "C" int tfpa_prefill(const tfpa_cache* c, const tfpa_seg* segs, int32_t nseg,
                            const void* q, const int32_t* row_seg, const int32_t* row_pos,
                            int32_t rows, float scale, int32_t max_rows_per_launch, void* out,
                            float* lse, cudaStream_t stream) {
  int e;
  if ((e = check_cache(c)) || (e = check_segs(c, segs, nseg))) return e;
  if (rows > 0 && (!q || !aligned(q, 16) || !out || !aligned(out, 16))) return TFPA_EINVAL;
  if (max_rows_per_launch < 0 || !std::isfinite(scale) || !(scale > 0.f)) return TFPA_EINVAL;
  thread_local std::vector<Run> runs;   // reused by every call of this thread
  if ((e = build_runs(segs, nseg, row_seg, row_pos, rows, runs))) return e;
  if (rows == 0) return TFPA_OK;
  if ((e = check_device()) || (e = check_tma_source(q))) return e;
  const bool fp8 = c->dtype == TFPA_FP8_E4M3;
  const int G = c->hq / c->hkv;
  const int npairs = (G + 1) / 2;
  const int32_t cap = max_rows_per_launch > 0 ? max_rows_per_launch : INT32_MAX;
  const int nsm = sm_count();
  if (nsm < 1) return TFPA_ECUDA;
  const size_t hd = (size_t)c->hq * kHeadDim;
  thread_local PrefillParams p;
  size_t ri = 0;
  int32_t taken = 0;
  while (ri < runs.size()) {
    std::memset(&p, 0, sizeof(p));
    SourceSet ss;
    const int32_t base = runs[ri].row0 + taken;
    int32_t nrows = 0, tiles = 0;
    int nr = 0;
    while (ri < runs.size() && nr < kMaxRuns && nrows < cap) {
      const Run& r = runs[ri];
      const int src = ss.add(segs, r.seg);
      if (src < 0) break;
      const int32_t take = std::min(r.nrows - taken, cap - nrows);
      RunInfo& info = p.runs[nr++];
      fill_run(info, segs[r.seg], src, nrows, take, r.pos0 + taken);
      info.item0 = tiles;
      tiles += c->hkv * npairs * ((take + kPrefillTileRows - 1) / kPrefillTileRows);
      nrows += take;
      taken += take;
      if (taken == r.nrows) {
        ++ri;
        taken = 0;
      }
    }
    if ((e = fill_maps(c, segs, ss, fp8, fp8 ? 128 : 64, 128, p.maps, p.nsrc))) return e;
    if ((e = get_qmap(static_cast<const __nv_bfloat16*>(q) + (size_t)base * hd, c->hq, nrows, 1,
                      kPrefillTileRows,
                      &p.qmap)))
      return e;
    p.q = static_cast<const __nv_bfloat16*>(q) + (size_t)base * hd;
    p.out = static_cast<__nv_bfloat16*>(out) + (size_t)base * hd;
    p.lse = lse ? lse + (size_t)base * c->hq : nullptr;
    p.k_scale = c->k_scale;
    p.v_scale = c->v_scale;
    p.err_flag = c->err_flag;
    p.nruns = nr;
    p.n_tiles = tiles;
    p.hq = c->hq;
    p.hkv = c->hkv;
    p.group = G;
    p.num_pages = c->num_pages;
    p.rows = nrows;
    p.scale_log2 = scale * 1.4426950408889634f;
    // A cluster of two CTAs per tile (each takes half of the tile's key
    // tiles), heaviest tiles first.
    record(3, base, nrows, nr, tiles, 2 * tiles, (int64_t)base * hd, (int64_t)base * hd);
    if (!dry_run())
      if ((e = to_err(launch_prefill(p, fp8, tiles, stream)))) return e;
  }
  return TFPA_OK;
}
