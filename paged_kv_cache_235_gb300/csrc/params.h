// Kernel launch parameters shared by the host planner and the kernels.
//
// A call's rows are grouped into runs: consecutive rows of one segment at
// consecutive positions.  Everything a kernel needs about a run travels in
// the launch parameters (passed by value, so a launch captured in a graph
// keeps them); only the bulk data (pages, tables, q, out, scratch) is in
// device memory.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace tfpa {

constexpr int kPage = 256;          // positions per page
constexpr int kHeadDim = 128;       // head size
constexpr int kMaxSplits = 32;      // split-K partials per (row, head), at most
constexpr int kMaxRuns = 64;        // runs per launch
constexpr int kMaxSlabs = 15;       // slab streams per launch (+1 source for the pool)
constexpr int kMaxSources = kMaxSlabs + 1;
constexpr int kMaxDecodeGrid = 256;  // CTAs of one decode partial launch, at most

// TMA descriptors of one K/V source: the page pool (source 0) or a slab.
struct KVMaps {
  CUtensorMap k;
  CUtensorMap v;
};

struct RunInfo {
  const int32_t* page_table;  // device; nullptr => slab source
  int32_t src;                // index into maps[]
  int32_t seq_len;
  int32_t row0;               // first row, relative to this launch
  int32_t nrows;
  int32_t pos0;               // position of the first row
  int32_t nsplit;             // decode and verify: splits of this stream
  int32_t pps;                // decode and verify: pages per split
  int32_t item0;              // first work item of this run
  int32_t slab_cap;           // slab capacity in positions (slab runs)
  int32_t pad_;
};

// The parts of a launch that change as streams grow (lengths, positions,
// split counts, item and CTA ranges).  A launch reads them from its own
// parameters, or, for a plan in device mode, from a device copy (`dyn`),
// which lets a captured launch be replayed step after step with new data.
struct DecodeDyn {
  RunInfo runs[kMaxRuns];
  int32_t nruns;
  int32_t n_items;
  int32_t pad_[2];
  // CTA b takes the work items [cta_item0[b], cta_item0[b + 1]), ranges the
  // host balances by the items' key stages.
  int32_t cta_item0[kMaxDecodeGrid + 1];
};

struct DecodeParams {
  KVMaps maps[kMaxSources];
  DecodeDyn d;
  const DecodeDyn* dyn;       // device copy of d to read instead, or nullptr
  const __nv_bfloat16* q;     // rows of this launch: [rows][hq][128]
  const uint64_t* anc;        // rows of this launch: ancestor masks, or nullptr (causal)
  float* part_o;              // [cap_rows][hq][max_splits][128]
  float* part_ml;             // [cap_rows][hq][max_splits][2]
  const float* k_scale;       // fp8: [hkv]
  const float* v_scale;
  int32_t* err_flag;
  // Append (k_rows != nullptr): the rows' new K and V ([rows][hkv][128]
  // bf16, rows of this launch) are stored by the CTAs whose keys include
  // them, before they read them; a source's K / V base is where its rows
  // go (pool: [num_pages][hkv][256][128], slab: [hkv][slab_cap][128]).
  const __nv_bfloat16* k_rows;
  const __nv_bfloat16* v_rows;
  void* k_base[kMaxSources];
  void* v_base[kMaxSources];
  // Merge in the partial kernel (arrive != nullptr): per (row, head) of a
  // group's first query vector, the splits finished so far; the last CTA
  // to finish one merges the group into out / lse (rows of this launch).
  uint32_t* arrive;           // [cap_rows][hq], scratch rows of this launch
  __nv_bfloat16* out;         // [rows][hq][128]
  float* lse;                 // [rows][hq] or nullptr
  int32_t nsrc;
  int32_t hq, hkv, group;     // group = hq / hkv
  int32_t max_splits;
  int32_t num_pages;
  int32_t rows;
  float scale_log2;           // softmax_scale * log2(e)
};

struct MergeRun {
  int32_t row0;
  int32_t nrows;
  int32_t nsplit;
  int32_t pad_;
};

struct MergeDyn {
  MergeRun runs[kMaxRuns * 2];
  int32_t nruns;
  int32_t rows;
  int32_t pad_[2];
};

struct MergeParams {
  MergeDyn d;
  const MergeDyn* dyn;        // device copy of d to read instead, or nullptr
  const float* part_o;
  const float* part_ml;
  __nv_bfloat16* out;         // rows of this launch: [rows][hq][128]
  float* lse;                 // [rows][hq] or nullptr
  int32_t hq;
  int32_t max_splits;
};

struct WriteRun {
  const int32_t* page_table;  // nullptr => slab
  void* k_dst;                // pool base or slab base
  void* v_dst;
  int32_t row0;               // first row of the run, relative to this launch
  int32_t nrows;
  int32_t pos0;
  int32_t slab_cap;
  int32_t seq_len;
  int32_t pad_;
};

struct WriteDyn {
  WriteRun runs[kMaxRuns];
  int32_t nruns;
  int32_t rows;
  int32_t pad_[2];
};

struct WriteParams {
  WriteDyn d;
  const WriteDyn* dyn;        // device copy of d to read instead, or nullptr
  const __nv_bfloat16* k_rows;  // [rows][hkv][128], rows of this launch
  const __nv_bfloat16* v_rows;
  const float* k_scale;
  const float* v_scale;
  int32_t* err_flag;
  // Rotary store (nullptr rope_cos: plain store): K is rotated by rope_pos[row]
  // (nullptr: the storage position) with the caller's cos/sin [rope_n][64].
  const float* rope_cos;
  const float* rope_sin;
  const int32_t* rope_pos;    // rows of this launch
  int32_t rope_n;
  int32_t hkv;
  int32_t num_pages;
  int32_t fp8;
};

// Keep: stored rows copied between positions of a stream (all kv heads).
constexpr int kMaxKeep = 256;
struct KeepPair {
  const int32_t* page_table;  // nullptr => slab
  void* k_slab;
  void* v_slab;
  int32_t slab_cap;
  int32_t src;
  int32_t dst;
  int32_t pad_;
};

struct KeepParams {
  KeepPair pairs[kMaxKeep];
  void* k_pool;
  void* v_pool;
  int32_t* err_flag;
  int32_t n;
  int32_t hkv;
  int32_t num_pages;
  int32_t row_bytes;          // 256 (bf16) or 128 (e4m3)
};

// Prefill: one work tile = (run, kv head g, query-head pair, 128 rows).
// The same kernel in verify mode (decode runs of many query vectors, on
// tensor cores): one work tile = (run, kv head g, 128 / G rows, key split);
// its query vectors (rows x the group's G heads, at most 128) form one Q
// tile that both MMA slots read, slot A taking the split's even key tiles
// and slot B the odd ones, each leaving its own split partial.
constexpr int kVerifyVectors = 128;
struct PrefillParams {
  KVMaps maps[kMaxSources];
  CUtensorMap qmap;           // q as 3D [rows][hq][128], 128B swizzle; box 64 x 1 x 128
                              // (prefill) or 64 x G x (128 / G) (verify)
  RunInfo runs[kMaxRuns];     // item0 = first tile of the run
  const __nv_bfloat16* q;     // [rows][hq][128]
  __nv_bfloat16* out;         // prefill
  float* lse;                 // prefill, or nullptr
  const uint64_t* anc;        // verify: the rows' ancestor masks, or nullptr (causal)
  float* part_o;              // verify: [rows][hq][max_splits][128]
  float* part_ml;             // verify: [rows][hq][max_splits][2]
  const float* k_scale;
  const float* v_scale;
  int32_t* err_flag;
  int32_t nruns;
  int32_t nsrc;
  int32_t n_tiles;
  int32_t hq, hkv, group;
  int32_t num_pages;
  int32_t rows;
  int32_t max_splits;         // verify
  float scale_log2;
};

// Page-table staging: ids written into a device page table on the stream.
constexpr int kMaxStage = 2048;
struct StageParams {
  int32_t* table;
  int32_t first;
  int32_t n;
  int32_t ids[kMaxStage];
};

// Save / restore of a stream's stored rows [p0, p1) to / from an image laid
// out [K, V][hkv][p1 - p0][row].
struct CopyParams {
  const int32_t* page_table;  // nullptr => slab
  void* k_base;               // pool or slab
  void* v_base;
  uint8_t* image;
  int32_t* err_flag;
  int32_t slab_cap;
  int32_t p0, p1;
  int32_t page0;              // first page of the range
  int32_t hkv;
  int32_t num_pages;
  int32_t row_bytes;          // 256 (bf16) or 128 (e4m3)
  int32_t restore;            // 0: cache -> image, 1: image -> cache
};

// Launchers (defined next to their kernels).
cudaError_t launch_write_kv(const WriteParams& p, cudaStream_t s);
cudaError_t launch_keep(const KeepParams& p, cudaStream_t s);
cudaError_t launch_stage(const StageParams& p, cudaStream_t s);
cudaError_t launch_copy(const CopyParams& p, int npages, cudaStream_t s);
cudaError_t launch_decode_partial(const DecodeParams& p, bool fp8, int grid, cudaStream_t s);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t s);
// Prefill launches a cluster of two CTAs per tile; verify one CTA per tile.
cudaError_t launch_prefill(const PrefillParams& p, bool fp8, int tiles, cudaStream_t s);
cudaError_t launch_verify(const PrefillParams& p, bool fp8, int tiles, cudaStream_t s);

}  // namespace tfpa
