// Causal prompt-chunk attention over a paged prefix on tcgen05/TMEM tiles
// (TensorFold PR #2011, "hpattn_p256_kernel": the page size a compile-time
// 256, a key tile's page looked up once; PR #1373, "What changes": the
// prompt tiles read pages through the page table, else the slab).
//
// One cluster of two CTAs per work tile = (run, kv head g, pair of query
// heads of g, 128 rows).  The tile's key tiles (128 keys, aligned to
// absolute positions) are cut at the midpoint: CTA 0 of the cluster takes
// the first half, CTA 1 the second (which holds the diagonal).  Each runs
// one online-softmax pass over its half.  Once CTA 0's MMAs are done with its
// K and V rings it tells CTA 1, which stores its (m, l, O) there through
// distributed shared memory; CTA 0 merges it with its own.  The cut depends
// only on the tile's key
// count, so a row's result never depends on how the rows are sliced into
// launches or tiles.  Two CTAs per tile halve the unit of work, so that the
// tiles of a prompt chunk fill the SMs' last wave (1,024 half tiles make
// 6.7 waves on 152 SMs where 512 whole tiles made 3.4).
//   warp 0      TMA producer: Q of both heads once, then K and V tiles into
//               2-stage rings (128B swizzle).  Each 128-key tile lies inside
//               one 256-position page: one page lookup per key tile.
//   warp 1      TMEM owner and MMA issuer: S_h = Q_h K^T (SS MMA, M=N=128,
//               K=16 x 8) into TMEM; O_h += P_h V (TS MMA, P read from TMEM,
//               V MN-major from shared memory).  The two heads ping-pong:
//               S_A(j+1) is issued right after PV_A(j), so head A's softmax
//               overlaps head B's MMAs and the other way round.
//   warps 4-7   softmax of head A, warps 8-11 of head B: one thread per row
//               (TMEM lane), causal mask on the diagonal tiles, online
//               max/sum, P written back over S as bf16 (f16 for e4m3
//               caches), O rescaled in TMEM only when the running max grows
//               by more than 2^8.
//   warps 12-15 (e4m3 caches only) converters: TMA lands e4m3 K/V tiles in
//               a staging buffer; these warps write the exact f16 operand
//               tiles (and zero V rows past the stream's end).
// With an e4m3 cache the MMAs run in f16: each softmax thread first turns its
// Q row into f16 scaled by a power of two (exact for every element within
// 2^28 of the row's largest), and the K and V scales are applied to the
// scores and to the output.  Verify tiles on an e4m3 cache instead split Q
// into two e4m3 tiles (hi + lo) and take S from 8-bit MMAs straight off the
// e4m3 K tiles, so only V passes through the converters.
// Verify mode (launch_verify): one CTA per tile (run, kv head, 128 / G rows,
// key split), no cluster.  One Q tile holds the group's query vectors (row x
// head) and both slots read it: slot A takes the split's even key tiles,
// slot B the odd ones, and the CTA merges the two into the split's partial.
// A verify tile of at most 64 query vectors holds them twice (M rows 0-63
// and 64-127) and each slot's softmax takes one copy, so the two slots run
// on different SM sub-partitions ("half mode").
// bf16: rings of three K and V stages over the slots' common tile order.
// e4m3: two e4m3 K stages per slot (8-bit S MMAs), two V staging tiles per
// slot, one f16 V stage per slot.
// TMEM (512 columns): S_A [0,128) O_A [128,256) S_B [256,384) O_B [384,512).
// CTA 1's partial lands in CTA 0's shared memory once CTA 0's MMAs are done:
// O (float32 [2 heads][128 rows][128], 16-byte chunks permuted by row against
// bank conflicts) over the K and V rings, (m, l) over the Q tiles.
#include <cuda_fp8.h>

#include "cluster.cuh"
#include "common.cuh"
#include "params.h"
#include "tcgen05.cuh"

namespace tfpa {
namespace {

constexpr int kTileRows = 128;
constexpr int kTileKeys = 128;
// bf16: warps 0-11.  e4m3: warps 0-15, warps 12-15 converting the staged
// e4m3 tiles (one warp per SM sub-partition, beside the softmax warps).
template <bool FP8>
constexpr int threads_of() { return FP8 ? 512 : 384; }
constexpr int kConvWarp0 = 12;
constexpr int kConvWarps = 4;
constexpr int kOffQ = 0;                 // 2 heads x [128 rows][128] 16-bit = 64 KB
constexpr int kOffK = 65536;             // 2 stages x 32 KB (16-bit operand tiles)
constexpr int kOffV = 131072;            // 2 stages x 32 KB
constexpr int kOffK8 = 196608;           // prefill, e4m3: the K staging tile, 16 KB
constexpr int kOffV8 = 212992;           // prefill, e4m3: the V staging tile, 16 KB
// Verify mode holds Q in the first Q tile (32 KB) only.  bf16: the second
// is K stage 2 of the rings of three.  e4m3: the Q tile becomes two e4m3
// tiles (hi and lo, 16 KB each) that feed 8-bit MMAs with K straight from
// its e4m3 stages, four of 16 KB over the 16-bit K region, two per slot; V
// still goes through the converters, from four e4m3 staging tiles (two per
// slot): the prefill staging pair and the second Q tile.
constexpr int kOffQ2 = 32768;
__device__ __forceinline__ int stage8_off(bool is_v) { return is_v ? kOffV8 : kOffK8; }
// Verify, e4m3: V staging tile i (2 x slot + step parity) and K stage i.
__device__ __forceinline__ int vstage8_off(int i) {
  return i < 2 ? kOffK8 + i * 16384 : kOffQ2 + (i - 2) * 16384;
}
__device__ __forceinline__ int kstage8_off(int i) { return kOffK + i * 16384; }
// Verify, bf16: a ring of three 16-bit stages each for K and V over the
// CTA's key tiles in the slots' common order (tile n = 2 step + slot in
// stage n mod 3): K stage 2 is the unused second Q tile, V stage 2 follows
// the prefill V ring.
__device__ __forceinline__ int kstage16_off(int t) { return t < 2 ? kOffK + t * 32768 : kOffQ2; }
template <bool FP8>
struct Layout {
  static constexpr int kOffBar = 229376;
  // Verify: the Q rows' scale factors (e4m3 caches; 128 floats) and slot
  // B's (m, l) per row for the merge of the two slots (128 float2).
  static constexpr int kOffDown = kOffBar + 256;
  static constexpr int kOffMl = kOffDown + 512;
  static constexpr int kSmemBytes = kOffMl + 1024 + 1024;
};
static_assert(Layout<true>::kSmemBytes <= 232448, "shared memory");
constexpr uint32_t kTmemCols = 512;
// Register split per warpgroup (setmaxnreg): warps 0-3 (TMA producer, MMA
// issuer) and the converters need few registers, the softmax warps (a
// row's 128 scores each) many.  A split hands out no more than the block
// launches with (e4m3: 512 x 128, bf16: 384 x 168), and no SM sub-partition
// (one warp of each warpgroup) more than its 16,384.  The bf16 split was
// picked by measurement: 64 / 216 ran 2.7 % faster than no split, where
// 56 / 224 and 72 / 216 (the latter without any spill) ran slower.  The
// e4m3 split 56 / 184 / 184 / 88 lets the converters issue all eight of a
// thread's staging loads at once (1.7 % on prompt chunks, 1 % on verify
// tiles, against 56 / 200 / 200 / 56 with four at a time); it uses each
// sub-partition's 16,384 registers exactly.
template <bool FP8>
struct Regs;
template <>
struct Regs<true> {
  static constexpr int kLow = 56, kHigh = 184, kConv = 88, kLaunch = 128;
};
template <>
struct Regs<false> {
  static constexpr int kLow = 64, kHigh = 216, kConv = 0, kLaunch = 168;
};
template <bool FP8>
constexpr int regs_split() {
  return 128 * (Regs<FP8>::kLow + 2 * Regs<FP8>::kHigh + Regs<FP8>::kConv);
}
static_assert(regs_split<true>() <= 512 * Regs<true>::kLaunch, "register split");
static_assert(regs_split<false>() <= 384 * Regs<false>::kLaunch, "register split");
static_assert(32 * (Regs<true>::kLow + 2 * Regs<true>::kHigh + Regs<true>::kConv) <= 16384,
              "sub-partition registers");
static_assert(32 * (Regs<false>::kLow + 2 * Regs<false>::kHigh) <= 16384,
              "sub-partition registers");
constexpr float kRescaleThreshold = 8.0f;   // log2 units
__device__ __forceinline__ uint32_t col_s(int hh) { return hh ? 256u : 0u; }
__device__ __forceinline__ uint32_t col_o(int hh) { return hh ? 384u : 128u; }

struct Bars {
  uint64_t* q_full;      // Q tiles landed (TMA)
  uint64_t* q_ready;     // Q operand ready for the MMA (e4m3 caches: after conversion)
  uint64_t* k_full;      // [2] K operand stage ready (verify: bf16 [3], e4m3 [4])
  uint64_t* k_empty;     // [2] (verify: bf16 [3], e4m3 [4])
  uint64_t* v_full;      // [2] (verify, bf16: [3])
  uint64_t* v_empty;     // [2] (verify, bf16: [3])
  uint64_t* k8_full;     // prefill, e4m3: the staging tile landed / free
  uint64_t* k8_empty;
  uint64_t* v8_full;     // (verify, e4m3: [4])
  uint64_t* v8_empty;    // (verify, e4m3: [4])
  uint64_t* s_full;      // [2] per head: S in TMEM
  uint64_t* p_ready;     // [2] per head: P in TMEM, O corrected
  uint64_t* o_final;
  uint64_t* drain;
  uint64_t* peer_ready;  // CTA 0: CTA 1's softmax threads stored their partial here
  uint64_t* dst_free;    // CTA 1: CTA 0's MMAs are done with its rings
  uint32_t* tmem_slot;
  volatile int* abort;
};

struct Tile {
  int run, g, hp, t, sigma;
};

// Prefill tiles are numbered heaviest first: the row-tile index is the
// slowest digit and runs from the last (longest causal range) to the first.
// Verify tiles: split, kv head, row tile (slowest first).
template <bool VERIFY>
__device__ __forceinline__ Tile tile_of(const PrefillParams& p, int i) {
  int r = 0;
  while (r + 1 < p.nruns && p.runs[r + 1].item0 <= i) ++r;
  const RunInfo& ru = p.runs[r];
  int local = i - ru.item0;
  const int npairs = (p.group + 1) >> 1;
  Tile x;
  x.run = r;
  if (VERIFY) {
    const int rt = kVerifyVectors / p.group;           // rows of a tile
    const int nrt = (ru.nrows + rt - 1) / rt;
    x.t = local % nrt;
    local /= nrt;
    x.g = local % p.hkv;
    x.sigma = local / p.hkv;
    x.hp = 0;
    return x;
  }
  const int pairs_total = p.hkv * npairs;
  const int ntr = (ru.nrows + kTileRows - 1) / kTileRows;
  const int t_rev = local / pairs_total;
  const int gp = local - t_rev * pairs_total;
  x.g = gp / npairs;
  x.hp = gp - x.g * npairs;
  x.t = ntr - 1 - t_rev;
  x.sigma = 0;
  return x;
}

// Verify tiles load Q as two boxes of 64 query vectors (M rows 0-63 and
// 64-127) when G divides 64.  A tile of at most 64 vectors then loads them
// into both halves ("half mode"): slot A's softmax takes TMEM lanes 0-63 and
// slot B's lanes 64-127, so the two slots' softmax threads sit on different
// SM sub-partitions (a warp reaches only its own quarter of the lanes).
__device__ __forceinline__ bool q_two_boxes(int group) { return 64 % group == 0; }

struct TileGeom {
  int row_lo;      // first row of the tile, relative to the run
  int nrows;       // valid rows in the tile
  int kend;        // the tile's rows see keys [0, kend)
  int kt0, nkt;    // this CTA's key tiles: kt0 .. kt0 + nkt - 1
};

// Key tiles of MMA slot hh and their order.  Prefill: both slots (two query
// heads) take every tile.  Verify: slot A the tiles kt0, kt0 + 2, ..., slot
// B kt0 + 1, kt0 + 3, ... (one Q tile, two independent online softmaxes).
template <bool VERIFY>
__device__ __forceinline__ int slot_tiles(const TileGeom& gm, int hh) {
  return VERIFY ? (gm.nkt + 1 - hh) >> 1 : gm.nkt;
}
template <bool VERIFY>
__device__ __forceinline__ int slot_tile(const TileGeom& gm, int jj, int hh) {
  return VERIFY ? gm.kt0 + 2 * jj + hh : gm.kt0 + jj;
}

// Prefill: key tiles [0, n / 2) go to CTA 0 of the cluster, [n / 2, n) to
// CTA 1 (CTA 0 has none when n = 1).  Verify: the key tiles of split sigma
// (pps pages of the stream each), cut at the tile's last position; a split
// past it has none.
template <bool VERIFY>
__device__ __forceinline__ TileGeom geom_of(const PrefillParams& p, const RunInfo& ru,
                                            const Tile& x, uint32_t rank) {
  TileGeom gm;
  const int rows = VERIFY ? kVerifyVectors / p.group : kTileRows;
  gm.row_lo = x.t * rows;
  gm.nrows = min(rows, ru.nrows - gm.row_lo);
  const int maxpos = ru.pos0 + gm.row_lo + gm.nrows - 1;
  gm.kend = min(ru.seq_len, maxpos + 1);
  const int n = (gm.kend + kTileKeys - 1) / kTileKeys;
  if (VERIFY) {
    const int per = ru.pps * (kPage / kTileKeys);
    gm.kt0 = x.sigma * per;
    gm.nkt = max(0, min(n, gm.kt0 + per) - gm.kt0);
    return gm;
  }
  const int mid = n >> 1;
  gm.kt0 = rank ? mid : 0;
  gm.nkt = rank ? n - mid : mid;
  return gm;
}

// Validity of the page under key tile j, read one page ahead so the table
// load is off the critical path (two key tiles share a page).
struct PageCheck {
  const int32_t* pt;
  int npages, num_pages, next_pid, stride;
  bool cur_bad, first;
  // Tiles j0, j0 + stride, ... (stride 1 or 2), n of them.
  __device__ __forceinline__ PageCheck(const PrefillParams& p, const RunInfo& ru,
                                       const TileGeom& gm, int j0, int n, int stride_)
      : pt(ru.page_table), npages((gm.kend + kPage - 1) / kPage), num_pages(p.num_pages),
        next_pid(0), stride(stride_), cur_bad(false), first(true) {
    if (pt && n > 0) next_pid = __ldg(pt + (j0 >> 1));
  }
  // Call for the tiles in order; true if tile j's page is bad.
  __device__ __forceinline__ bool bad(int j) {
    if (!pt) return false;
    if ((j & 1) == 0 || first || stride == 2) {
      first = false;
      const int page = j >> 1;
      cur_bad = (unsigned)next_pid >= (unsigned)num_pages;
      if (page + 1 < npages) next_pid = __ldg(pt + page + 1);
    }
    return cur_bad;
  }
};

// First V row of key tile j that must read as zero: keys past the stream's
// end, or every row of a tile whose page id is bad.
__device__ __forceinline__ int v_zero_from(const RunInfo& ru, int j, bool page_bad) {
  if (page_bad) return 0;
  const int kt = j * kTileKeys;
  return kt + kTileKeys > ru.seq_len ? ru.seq_len - kt : kTileKeys;
}


template <bool FP8, bool VERIFY>
__device__ void producer(const PrefillParams& p, const RunInfo& ru, const Tile& x,
                         const TileGeom& gm, uint8_t* smem, const Bars& b) {
  const CUtensorMap* mk = &p.maps[ru.src].k;
  const CUtensorMap* mv = &p.maps[ru.src].v;
  if (gm.nkt == 0) return;
  if (VERIFY) {
    // One Q tile, both slots: 128 / G rows x the group's G heads (box 64 x G
    // x rows, landing as M row G (row) + head).  Rows past the run hold the
    // next rows or zeros, which no output reads.
    const int rt = kVerifyVectors / p.group;
    mbar_arrive_expect_tx(b.q_full, 2u * 128u * (uint32_t)(p.group * rt));
    if (q_two_boxes(p.group)) {
      const bool half = gm.nrows * p.group <= 64;
      for (int rg = 0; rg < 2; ++rg)
        for (int hb = 0; hb < 2; ++hb)
          tma_load_3d(smem + kOffQ + rg * 16384 + hb * 8192, &p.qmap, rg * 64, x.g * p.group,
                      ru.row0 + gm.row_lo + (half ? 0 : hb * (64 / p.group)), b.q_full);
    } else {
      for (int rg = 0; rg < 2; ++rg)
        tma_load_3d(smem + kOffQ + rg * 16384, &p.qmap, rg * 64, x.g * p.group,
                    ru.row0 + gm.row_lo, b.q_full);
    }
  } else {
    // Slot hh is query head h0 + hh, 128 rows (box 64 x 1 x 128).
    mbar_arrive_expect_tx(b.q_full, 65536);
    for (int hh = 0; hh < 2; ++hh)
      for (int rg = 0; rg < 2; ++rg)
        tma_load_3d(smem + kOffQ + hh * 32768 + rg * 16384, &p.qmap, rg * 64,
                    x.g * p.group + 2 * x.hp + hh, ru.row0 + gm.row_lo, b.q_full);
  }
  // Row coordinate of key tile j in its source; one page lookup per page.  A
  // bad page id is flagged and a valid page read in its place (its keys are
  // masked).
  int cached_page = -1, cached_pid = 0;
  auto row_of = [&](int j) {
    const int kt = j * kTileKeys;
    if (!ru.page_table) return x.g * ru.slab_cap + kt;
    const int page = kt >> 8;
    if (page != cached_page) {
      cached_pid = __ldg(ru.page_table + page);
      cached_page = page;
      if ((unsigned)cached_pid >= (unsigned)p.num_pages) {
        flag_error(p.err_flag, kErrBadPage);
        cached_pid = 0;
      }
    }
    return (cached_pid * p.hkv + x.g) * kPage + (kt & (kPage - 1));
  };
  // Loads into a 16-bit operand stage (bf16), or (prefill, e4m3) into the
  // staging tile that the converters move on, K and V in their order.
  int staged_k = 0, staged_v = 0;       // e4m3: staging loads issued
  auto load = [&](bool is_v, int stage, uint32_t parity, int y) {
    if (FP8) {
      int& n = is_v ? staged_v : staged_k;
      uint64_t* empty = is_v ? b.v8_empty : b.k8_empty;
      uint64_t* full = is_v ? b.v8_full : b.k8_full;
      if (!mbar_wait_or_abort(empty, (n & 1) ^ 1, p.err_flag, b.abort)) return false;
      mbar_arrive_expect_tx(full, 16384);
      tma_load_2d(smem + stage8_off(is_v), is_v ? mv : mk, 0, y, full);
      ++n;
      return true;
    }
    uint64_t* empty = is_v ? &b.v_empty[stage] : &b.k_empty[stage];
    uint64_t* full = is_v ? &b.v_full[stage] : &b.k_full[stage];
    if (!mbar_wait_or_abort(empty, parity ^ 1, p.err_flag, b.abort)) return false;
    uint8_t* dst = smem + (is_v ? kOffV + stage * 32768
                                : (VERIFY ? kstage16_off(stage) : kOffK + stage * 32768));
    mbar_arrive_expect_tx(full, 32768);
    tma_load_2d(dst, is_v ? mv : mk, 0, y, full);
    tma_load_2d(dst + 16384, is_v ? mv : mk, 64, y, full);
    return true;
  };
  // Last load issued into each 16-bit stage (phase parity, or -1): an
  // aborting CTA waits for these before it exits.
  int last_k0 = -1, last_k1 = -1, last_k2 = -1, last_v0 = -1, last_v1 = -1, last_v2 = -1;
  auto issued = [&](bool is_v, int stage, uint32_t ph) {
    int& w = is_v ? (stage == 2 ? last_v2 : stage ? last_v1 : last_v0)
                  : (stage == 2 ? last_k2 : stage ? last_k1 : last_k0);
    w = (int)ph;
  };
  if (VERIFY && FP8) {
    // Step jj, slot hh: K into e4m3 stage 2 hh + (jj & 1), V into staging
    // tile 2 hh + (jj & 1), each at phase (jj >> 1) & 1; K of both slots,
    // then V of both.  last_k*, last_v*: each slot's last step loaded.
    bool ok = true;
    for (int jj = 0; ok && jj < slot_tiles<true>(gm, 0); ++jj) {
      const uint32_t ph = (jj >> 1) & 1;
      for (int kv = 0; ok && kv < 2; ++kv)
        for (int hh = 0; ok && hh < 2; ++hh) {
          if (jj >= slot_tiles<true>(gm, hh)) continue;
          const int i = 2 * hh + (jj & 1);
          uint64_t* empty = kv ? b.v8_empty + i : b.k_empty + i;
          uint64_t* full = kv ? b.v8_full + i : b.k_full + i;
          const int y = row_of(slot_tile<true>(gm, jj, hh));
          if (!(ok = mbar_wait_or_abort(empty, ph ^ 1, p.err_flag, b.abort))) break;
          mbar_arrive_expect_tx(full, 16384);
          tma_load_2d(smem + (kv ? vstage8_off(i) : kstage8_off(i)), kv ? mv : mk, 0, y, full);
          if (kv) {
            (hh ? last_v1 : last_v0) = jj;
          } else {
            (hh ? last_k1 : last_k0) = jj;
          }
        }
    }
  } else if (VERIFY) {
    // Step jj, slot hh: tile n = 2 jj + hh (kt0 + n) into stage n mod 3 at
    // phase (n / 3) & 1; K of both slots, then V of both.
    bool ok = true;
    for (int jj = 0; ok && jj < slot_tiles<true>(gm, 0); ++jj) {
      for (int kv = 0; ok && kv < 2; ++kv)
        for (int hh = 0; ok && hh < 2; ++hh) {
          if (jj >= slot_tiles<true>(gm, hh)) continue;
          const int n = 2 * jj + hh;
          const uint32_t ph = (uint32_t)((n / 3) & 1);
          ok = load(kv == 1, n % 3, ph, row_of(slot_tile<true>(gm, jj, hh)));
          if (ok) issued(kv == 1, n % 3, ph);
        }
    }
  } else {
    for (int jj = 0; jj < gm.nkt; ++jj) {   // jj counts this CTA's tiles
      const int s = jj & 1;
      const uint32_t ph = (jj >> 1) & 1;
      const int y = row_of(gm.kt0 + jj);
      if (!load(false, s, ph, y)) break;
      issued(false, s, ph);
      if (!load(true, s, ph, y)) break;
      issued(true, s, ph);
    }
  }
  if (*b.abort) {
    // Let this CTA's loads in flight land before it exits.
    mbar_wait(b.q_full, 0, p.err_flag);
    if (VERIFY && FP8) {
      // each slot's last two steps loaded (buffers alternate by step)
      const int lasts[4] = {last_k0, last_k1, last_v0, last_v1};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int hh = u & 1;
        uint64_t* full = u < 2 ? b.k_full : b.v8_full;
#pragma unroll
        for (int d = 0; d < 2; ++d) {
          const int jj = lasts[u] - d;
          if (jj >= 0) mbar_wait(full + 2 * hh + (jj & 1), (uint32_t)((jj >> 1) & 1), p.err_flag);
        }
      }
    } else if (FP8) {
      if (staged_k > 0) mbar_wait(b.k8_full, (uint32_t)((staged_k - 1) & 1), p.err_flag);
      if (staged_v > 0) mbar_wait(b.v8_full, (uint32_t)((staged_v - 1) & 1), p.err_flag);
    } else {
      if (last_k0 >= 0) mbar_wait(&b.k_full[0], (uint32_t)last_k0, p.err_flag);
      if (last_k1 >= 0) mbar_wait(&b.k_full[1], (uint32_t)last_k1, p.err_flag);
      if (last_k2 >= 0) mbar_wait(&b.k_full[2], (uint32_t)last_k2, p.err_flag);
      if (last_v0 >= 0) mbar_wait(&b.v_full[0], (uint32_t)last_v0, p.err_flag);
      if (last_v1 >= 0) mbar_wait(&b.v_full[1], (uint32_t)last_v1, p.err_flag);
      if (last_v2 >= 0) mbar_wait(&b.v_full[2], (uint32_t)last_v2, p.err_flag);
    }
  }
}


// Zero rows [z0, 128) of a 16-bit V operand tile (both 64-column halves):
// keys past the stream's end, or a tile whose page id was bad, must add
// exactly nothing to O even if the bytes there are not finite.
__device__ __forceinline__ void zero_v_rows(uint8_t* vtile, int z0, int lane) {
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int i = z0 * 16 + lane; i < kTileKeys * 16; i += 32) {
    const int row = i >> 4, c = i & 15;     // 16 chunks of 16 B per row (2 halves)
    *reinterpret_cast<uint4*>(vtile + (c >> 3) * 16384 + row * 128 + (c & 7) * 16) = z;
  }
  fence_proxy_async_smem();
  __syncwarp();
}

// e4m3 staging tile [128 rows][128 B] (128B swizzle) -> f16 operand tile
// [128 rows][2 halves of 64] (128B swizzle), 64 threads; rows >= z0 become 0.
__device__ __forceinline__ void convert_tile(const uint8_t* src, uint8_t* dst, int z0, int t) {
  const uint32_t sb = smem_u32(src), db = smem_u32(dst);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = t + 128 * k;             // (row, 16-byte source chunk)
    const int row = i >> 3, c8 = i & 7;    // source chunk c8 = head dims 16*c8 .. +15
    uint4 w = lds128(swz128(sb, row, c8));
    if (row >= z0) w = make_uint4(0, 0, 0, 0);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    uint32_t h[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      h[2 * q] = e4m3x2_to_f16x2((uint16_t)(ws[q] & 0xFFFF));
      h[2 * q + 1] = e4m3x2_to_f16x2((uint16_t)(ws[q] >> 16));
    }
    const uint32_t half = db + (uint32_t)(c8 >> 2) * 16384u;
    const int c16 = 2 * (c8 & 3);
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(swz128(half, row, c16)),
                 "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3]) : "memory");
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(swz128(half, row, c16 + 1)),
                 "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7]) : "memory");
  }
}

// Warps 12-15 for e4m3 caches: staging -> f16 operand stages, in the order
// the producer fills the staging tiles.  Prefill: K and V of each key tile
// through one staging tile each.  Verify: V only (K feeds 8-bit MMAs), slot
// hh's step jj from staging tile 2 hh + (jj & 1).
template <bool VERIFY>
__device__ void converter(const PrefillParams& p, const RunInfo& ru, const TileGeom& gm,
                          uint8_t* smem, const Bars& b) {
  const int t = threadIdx.x - kConvWarp0 * 32;   // 0..127
  const int lane = threadIdx.x & 31;
  // Staging tile `src` (K, or V with rows from z0 on zeroed: past the
  // stream's end, or all rows of a bad page) into 16-bit stage s.
  auto convert = [&](bool is_v, int s, uint32_t ph, int z0, int src, uint32_t ph8,
                     uint64_t* full8, uint64_t* empty8) {
    uint64_t* empty = is_v ? &b.v_empty[s] : &b.k_empty[s];
    uint64_t* full = is_v ? &b.v_full[s] : &b.k_full[s];
    if (!mbar_wait_or_abort(full8, ph8, p.err_flag, b.abort)) return false;
    if (!mbar_wait_or_abort(empty, ph ^ 1, p.err_flag, b.abort)) return false;
    convert_tile(smem + src, smem + (is_v ? kOffV : kOffK) + s * 32768, is_v ? z0 : kTileKeys, t);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(empty8);
      mbar_arrive(full);
    }
    return true;
  };
  if (VERIFY) {
    PageCheck pc0(p, ru, gm, gm.kt0, slot_tiles<true>(gm, 0), 2);
    PageCheck pc1(p, ru, gm, gm.kt0 + 1, slot_tiles<true>(gm, 1), 2);
    bool ok = true;
    for (int jj = 0; ok && jj < slot_tiles<true>(gm, 0); ++jj) {
      for (int hh = 0; ok && hh < 2; ++hh) {
        if (jj >= slot_tiles<true>(gm, hh)) continue;
        const int j = slot_tile<true>(gm, jj, hh);
        const int z0 = v_zero_from(ru, j, hh ? pc1.bad(j) : pc0.bad(j));
        const int i = 2 * hh + (jj & 1);
        ok = convert(true, hh, jj & 1, z0, vstage8_off(i), (uint32_t)((jj >> 1) & 1),
                     b.v8_full + i, b.v8_empty + i);
      }
    }
    return;
  }
  PageCheck pc(p, ru, gm, gm.kt0, gm.nkt, 1);
  for (int jj = 0; jj < gm.nkt; ++jj) {
    const int j = gm.kt0 + jj;
    const int z0 = v_zero_from(ru, j, pc.bad(j));
    const int s = jj & 1;
    const uint32_t ph = (jj >> 1) & 1;
    // one staging tile each for K and V: its jj-th fill is phase jj & 1
    const uint32_t ph8 = (uint32_t)(jj & 1);
    if (!convert(false, s, ph, z0, stage8_off(false), ph8, b.k8_full, b.k8_empty)) return;
    if (!convert(true, s, ph, z0, stage8_off(true), ph8, b.v8_full, b.v8_empty)) return;
  }
}

template <bool FP8, bool VERIFY>
__device__ void mma_issuer(const PrefillParams& p, const RunInfo& ru, const TileGeom& gm,
                           uint8_t* smem, uint32_t tmem, const Bars& b) {
  const int lane = threadIdx.x & 31;
  const bool leader = lane == 0;
  constexpr uint32_t kIdescQK = umma::idesc_f16(128, 128, !FP8, false);
  constexpr uint32_t kIdescPV = umma::idesc_f16(128, 128, !FP8, true);
  const uint32_t qb = smem_u32(smem + kOffQ);
  const uint32_t kb = smem_u32(smem + kOffK);
  const uint32_t vb = smem_u32(smem + kOffV);

  constexpr uint32_t kIdescQK8 = umma::idesc_e4m3(128, 128);
  auto issue_s = [&](int hh, int s) {     // S_hh = Q_hh K_s^T (verify: one Q tile)
    if constexpr (VERIFY && FP8) {
      // S_hh = Q_hi K^T + Q_lo K^T over e4m3 K stage s (K = 32 per MMA)
      const uint32_t k8 = smem_u32(smem + kstage8_off(s));
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t a = umma::smem_desc_sw128(qb + q * 16384 + ks * 32, 16, 1024);
          const uint64_t bd = umma::smem_desc_sw128(k8 + ks * 32, 16, 1024);
          umma::mma_ss_f8(tmem + col_s(hh), a, bd, kIdescQK8, (q | ks) ? 1u : 0u);
        }
    } else {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
        const uint64_t a = umma::smem_desc_sw128(qb + (VERIFY ? 0 : hh * 32768) + off, 16, 1024);
        const uint32_t k16 = VERIFY ? smem_u32(smem + kstage16_off(s)) : kb + s * 32768;
        const uint64_t bd = umma::smem_desc_sw128(k16 + off, 16, 1024);
        umma::mma_ss(tmem + col_s(hh), a, bd, kIdescQK, ks > 0 ? 1u : 0u);
      }
    }
  };
  auto issue_pv = [&](int hh, int s, bool acc) {   // O_hh (+)= P_hh V_s
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t bd = umma::smem_desc_sw128(vb + s * 32768 + kk * 2048, 16384, 1024);
      umma::mma_ts(tmem + col_o(hh), tmem + col_s(hh) + kk * 8, bd, kIdescPV,
                   (acc || kk > 0) ? 1u : 0u);
    }
  };

  if (gm.nkt == 0) {                  // no keys in this half: nothing to wait for
    if (leader) mbar_arrive(b.o_final);
    __syncwarp();
    return;
  }
  if (VERIFY) {
    // Slot hh, step jj.  bf16: K and V of tile n = 2 jj + hh in stage n mod
    // 3 at phase (n / 3) & 1.  e4m3: K in e4m3 stage 2 hh + (jj & 1) at phase
    // (jj >> 1) & 1, V in 16-bit stage hh at phase jj & 1.
    auto kst = [&](int hh, int jj) { return FP8 ? 2 * hh + (jj & 1) : (2 * jj + hh) % 3; };
    auto kph = [&](int hh, int jj) {
      return (uint32_t)(FP8 ? (jj >> 1) & 1 : ((2 * jj + hh) / 3) & 1);
    };
    auto vst = [&](int hh, int jj) { return FP8 ? hh : (2 * jj + hh) % 3; };
    auto vph = [&](int hh, int jj) { return (uint32_t)(FP8 ? jj & 1 : ((2 * jj + hh) / 3) & 1); };
    bool ok = mbar_wait_or_abort(b.q_ready, 0, p.err_flag, b.abort);
    for (int hh = 0; ok && hh < 2; ++hh) {
      if (slot_tiles<true>(gm, hh) == 0) continue;
      if (!(ok = mbar_wait_or_abort(&b.k_full[kst(hh, 0)], 0, p.err_flag, b.abort))) break;
      umma::fence_after_sync();
      if (leader) {
        issue_s(hh, kst(hh, 0));
        umma::commit(&b.s_full[hh]);
        umma::commit(&b.k_empty[kst(hh, 0)]);
      }
      __syncwarp();
    }
    PageCheck pc0(p, ru, gm, gm.kt0, slot_tiles<true>(gm, 0), 2);
    PageCheck pc1(p, ru, gm, gm.kt0 + 1, slot_tiles<true>(gm, 1), 2);
    for (int jj = 0; ok && jj < slot_tiles<true>(gm, 0); ++jj) {
      for (int hh = 0; ok && hh < 2; ++hh) {
        const int n = slot_tiles<true>(gm, hh);
        if (jj >= n) continue;
        const int j = slot_tile<true>(gm, jj, hh);
        const bool page_bad = hh ? pc1.bad(j) : pc0.bad(j);
        const int vs = vst(hh, jj);
        if (!(ok = mbar_wait_or_abort(&b.v_full[vs], vph(hh, jj), p.err_flag, b.abort))) break;
        if (!FP8) {
          const int z0 = v_zero_from(ru, j, page_bad);
          if (z0 < kTileKeys) zero_v_rows(smem + kOffV + vs * 32768, z0, lane);
        }
        if (!(ok = mbar_wait_or_abort(&b.p_ready[hh], jj & 1, p.err_flag, b.abort))) break;
        umma::fence_after_sync();
        if (leader) {
          issue_pv(hh, vs, jj > 0);
          umma::commit(&b.v_empty[vs]);
        }
        __syncwarp();
        if (jj + 1 < n) {
          const int ks = kst(hh, jj + 1);
          if (!(ok = mbar_wait_or_abort(&b.k_full[ks], kph(hh, jj + 1), p.err_flag, b.abort)))
            break;
          umma::fence_after_sync();
          if (leader) {
            issue_s(hh, ks);
            umma::commit(&b.s_full[hh]);
            umma::commit(&b.k_empty[ks]);
          }
          __syncwarp();
        }
      }
    }
    if (leader) {
      if (ok) {
        umma::commit(b.o_final);
      } else {
        umma::commit(b.drain);        // let issued MMAs finish before TMEM is freed
        mbar_wait(b.drain, 0, p.err_flag);
      }
    }
    __syncwarp();
    return;
  }
  bool ok = mbar_wait_or_abort(b.q_ready, 0, p.err_flag, b.abort) &&
            mbar_wait_or_abort(&b.k_full[0], 0, p.err_flag, b.abort);
  if (ok) {
    umma::fence_after_sync();
    if (leader) {
      issue_s(0, 0);
      umma::commit(&b.s_full[0]);
      issue_s(1, 0);
      umma::commit(&b.s_full[1]);
      umma::commit(&b.k_empty[0]);
    }
    __syncwarp();
  }
  PageCheck pc(p, ru, gm, gm.kt0, gm.nkt, 1);
  for (int jj = 0; ok && jj < gm.nkt; ++jj) {
    const int j = gm.kt0 + jj;
    const bool page_bad = pc.bad(j);
    const int s = jj & 1;
    const uint32_t ph = (jj >> 1) & 1;
    const int s1 = (jj + 1) & 1;
    const uint32_t ph1 = ((jj + 1) >> 1) & 1;
    const bool more = jj + 1 < gm.nkt;
    if (!(ok = mbar_wait_or_abort(&b.v_full[s], ph, p.err_flag, b.abort))) break;
    if (!FP8) {   // the e4m3 converters zero these rows themselves
      const int z0 = v_zero_from(ru, j, page_bad);
      if (z0 < kTileKeys) zero_v_rows(smem + kOffV + s * 32768, z0, lane);
    }
    // head A
    if (!(ok = mbar_wait_or_abort(&b.p_ready[0], jj & 1, p.err_flag, b.abort))) break;
    umma::fence_after_sync();
    if (leader) issue_pv(0, s, jj > 0);
    if (more) {
      if (!(ok = mbar_wait_or_abort(&b.k_full[s1], ph1, p.err_flag, b.abort))) break;
      umma::fence_after_sync();
      if (leader) {
        issue_s(0, s1);
        umma::commit(&b.s_full[0]);
      }
    }
    // head B
    if (!(ok = mbar_wait_or_abort(&b.p_ready[1], jj & 1, p.err_flag, b.abort))) break;
    umma::fence_after_sync();
    if (leader) {
      issue_pv(1, s, jj > 0);
      if (more) {
        issue_s(1, s1);
        umma::commit(&b.s_full[1]);
        umma::commit(&b.k_empty[s1]);
      }
      umma::commit(&b.v_empty[s]);
    }
    __syncwarp();
  }
  if (leader) {
    if (ok) {
      umma::commit(b.o_final);
    } else {
      umma::commit(b.drain);          // let issued MMAs finish before TMEM is freed
      mbar_wait(b.drain, 0, p.err_flag);
    }
  }
  __syncwarp();
}

// e4m3 caches: turn this thread's Q row (bf16, in the operand tile) into f16
// in place, scaled by 2^e so its largest element lies in [2^13, 2^14).
// Returns 2^-e, the factor that undoes the scaling.
__device__ __forceinline__ float q_row_to_f16(uint8_t* qtile, int r) {
  const uint32_t base = smem_u32(qtile);
  uint32_t v[64];
#pragma unroll
  for (int ch = 0; ch < 16; ++ch) {
    const uint4 w = lds128(swz128(base + (ch >> 3) * 16384u, r, ch & 7));
    v[4 * ch + 0] = w.x;
    v[4 * ch + 1] = w.y;
    v[4 * ch + 2] = w.z;
    v[4 * ch + 3] = w.w;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    amax = fmaxf(amax, fabsf(__uint_as_float(v[i] << 16)));
    amax = fmaxf(amax, fabsf(__uint_as_float(v[i] & 0xFFFF0000u)));
  }
  int ex;
  frexpf(amax, &ex);
  ex = max(min(ex, 120), -100);
  const float up = __int_as_float((127 + 14 - ex) << 23);
#pragma unroll
  for (int i = 0; i < 64; ++i)
    v[i] = pack_f16x2(__uint_as_float(v[i] << 16) * up, __uint_as_float(v[i] & 0xFFFF0000u) * up);
#pragma unroll
  for (int ch = 0; ch < 16; ++ch)
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};"
                 ::"r"(swz128(base + (ch >> 3) * 16384u, r, ch & 7)), "r"(v[4 * ch]),
                   "r"(v[4 * ch + 1]), "r"(v[4 * ch + 2]), "r"(v[4 * ch + 3])
                 : "memory");
  return __int_as_float((127 - 14 + ex) << 23);
}

// Verify with an e4m3 cache: this thread's Q row (bf16, in the operand
// tile) becomes two e4m3 rows for the 8-bit MMAs, hi = e4m3(q 2^e) and
// lo = e4m3(q 2^e - hi), both rounded to nearest, with e putting the row's
// largest magnitude in [2^7, 2^8).  q 2^e - hi is exact in float32 and has
// at most four significant bits, so hi + lo = q 2^e exactly for every
// element of magnitude 2^-2 or more after scaling (within 2^9 of the row's
// largest), and to within one e4m3 rounding of the remainder below that.
// hi lands over the first 64-column half (a [128 rows][128 B] tile, 128B
// swizzle, as TMA lays out an e4m3 K tile), lo over the second; each thread
// reads its whole row before it writes.  Returns 2^-e.
__device__ __forceinline__ float q_row_to_e4m3_pair(uint8_t* qtile, int r) {
  const uint32_t base = smem_u32(qtile);
  uint32_t v[64];
#pragma unroll
  for (int ch = 0; ch < 16; ++ch) {
    const uint4 w = lds128(swz128(base + (ch >> 3) * 16384u, r, ch & 7));
    v[4 * ch + 0] = w.x;
    v[4 * ch + 1] = w.y;
    v[4 * ch + 2] = w.z;
    v[4 * ch + 3] = w.w;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    amax = fmaxf(amax, fabsf(__uint_as_float(v[i] << 16)));
    amax = fmaxf(amax, fabsf(__uint_as_float(v[i] & 0xFFFF0000u)));
  }
  int ex;
  frexpf(amax, &ex);
  ex = max(min(ex, 120), -100);
  const float up = __int_as_float((127 + 8 - ex) << 23);
  // Word i of a row: dims 4i .. 4i + 3, dim 4i in the low byte.
  auto e4m3x2 = [](float a, float b) -> uint32_t {   // a in the low byte
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  };
  auto rest2 = [](float a, float b, uint32_t h2) -> float2 {   // (a, b) - their e4m3 pair
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
    return make_float2(a - f.x, b - f.y);
  };
  uint32_t hi[32], lo[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float x0 = __uint_as_float(v[2 * i] << 16) * up;
    const float x1 = __uint_as_float(v[2 * i] & 0xFFFF0000u) * up;
    const float x2 = __uint_as_float(v[2 * i + 1] << 16) * up;
    const float x3 = __uint_as_float(v[2 * i + 1] & 0xFFFF0000u) * up;
    const uint32_t h01 = e4m3x2(x0, x1), h23 = e4m3x2(x2, x3);
    const float2 r01 = rest2(x0, x1, e4m3x2_to_f16x2((uint16_t)h01));
    const float2 r23 = rest2(x2, x3, e4m3x2_to_f16x2((uint16_t)h23));
    hi[i] = h01 | (h23 << 16);
    lo[i] = e4m3x2(r01.x, r01.y) | (e4m3x2(r23.x, r23.y) << 16);
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};"
                 ::"r"(swz128(base, r, c)), "r"(hi[4 * c]), "r"(hi[4 * c + 1]),
                   "r"(hi[4 * c + 2]), "r"(hi[4 * c + 3])
                 : "memory");
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};"
                 ::"r"(swz128(base + 16384u, r, c)), "r"(lo[4 * c]), "r"(lo[4 * c + 1]),
                   "r"(lo[4 * c + 2]), "r"(lo[4 * c + 3])
                 : "memory");
  }
  return __int_as_float((127 - 8 + ex) << 23);
}

// Offsets of CTA 1's partial for (head hh, row r) in CTA 0's shared memory:
// O over the K/V rings, (m, l) over the Q tiles.
__device__ __forceinline__ uint32_t part_o_row(uint32_t smem_base, int hh, int r) {
  return smem_base + kOffK + hh * 65536 + r * 512;
}
__device__ __forceinline__ uint32_t part_o_chunk(int r, int c) {   // c: 16-byte chunk 0..31
  return (uint32_t)((c ^ (r & 7)) * 16);
}
__device__ __forceinline__ uint32_t part_ml(uint32_t smem_base, int hh, int r) {
  return smem_base + kOffQ + (hh * kTileRows + r) * 8;
}

template <bool FP8, bool VERIFY>
__device__ void softmax_role(const PrefillParams& p, const RunInfo& ru, const Tile& x,
                             const TileGeom& gm, uint32_t rank, int hh, uint8_t* smem,
                             uint32_t tmem, const Bars& b) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = 32 * (warp & 3) + lane;                 // row of the tile = TMEM lane
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  const uint32_t tS = tmem + lane_off + col_s(hh);
  const uint32_t tO = tmem + lane_off + col_o(hh);
  // Verify: TMEM lane r holds query vector v = r (row v / G, head v % G of
  // the group) in both slots, or in half mode v = r - 64 hh for the lanes of
  // slot hh's half; the slots see alternate key tiles.
  const bool half = VERIFY && q_two_boxes(p.group) && gm.nrows * p.group <= 64;
  const bool mine = !half || (r >> 6) == hh;            // half mode: this slot's lanes
  const int v = half ? (r & 63) : r;                    // query vector of this lane
  const int rho = VERIFY ? v / p.group : r;             // row within the tile
  const int hig = VERIFY ? v - rho * p.group : 0;       // verify: head within the group
  const bool valid =
      mine && rho < gm.nrows && (!VERIFY || v < p.group * (kVerifyVectors / p.group));
  const int pos = ru.pos0 + gm.row_lo + (valid ? rho : 0);
  const int nt = slot_tiles<VERIFY>(gm, hh);             // this slot's key tiles
  // Verify with ancestor masks: key pos - d (d < 64) is visible iff bit d of
  // the row's mask is set; keys further back always are.  Bit-reversed, the
  // mask lines up with key order: key lim - d of a tile is bit 63 - d.
  const bool tree = VERIFY && p.anc != nullptr;
  const uint64_t anc_rev =
      __brevll(tree && valid ? __ldg(p.anc + ru.row0 + gm.row_lo + rho) : ~0ull);
  float sl2 = p.scale_log2;
  bool ok = true;
  if (FP8 && gm.nkt > 0) {
    // Prefill: each slot's warps turn their head's Q rows into f16.  Verify:
    // slot A's warps turn the one Q tile, publish each row's factor, and
    // slot B's take it once they see the tile ready.
    float* down_s = reinterpret_cast<float*>(smem + Layout<FP8>::kOffDown);
    if (!VERIFY || hh == 0) {
      ok = mbar_wait_or_abort(b.q_full, 0, p.err_flag, b.abort);
      if (ok) {
        const float down = VERIFY ? q_row_to_e4m3_pair(smem + kOffQ, r)
                                  : q_row_to_f16(smem + kOffQ + hh * 32768, r);
        sl2 = p.scale_log2 * down * __ldg(p.k_scale + x.g);
        if (VERIFY) down_s[r] = down;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(b.q_ready);
      }
    } else {
      ok = mbar_wait_or_abort(b.q_ready, 0, p.err_flag, b.abort);
      if (ok) sl2 = p.scale_log2 * down_s[r] * __ldg(p.k_scale + x.g);
    }
  }
  float m_run = -INFINITY, l = 0.f;
  PageCheck pc(p, ru, gm, VERIFY ? gm.kt0 + hh : gm.kt0, nt, VERIFY ? 2 : 1);
  // A warp whose 32 rows all lie past the tile's last row (a short run or
  // a small draft tree) has nothing to compute: its rows' P and O are never
  // read into any output.  It still waits for each S and arrives on p_ready,
  // which keeps it in step with the MMA issuer.
  const bool idle = !__any_sync(0xffffffffu, valid);

  for (int jj = 0; ok && jj < nt; ++jj) {
    const int j = slot_tile<VERIFY>(gm, jj, hh);
    const bool page_bad = pc.bad(j);
    if (!(ok = mbar_wait_or_abort(&b.s_full[hh], jj & 1, p.err_flag, b.abort))) break;
    if (idle) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&b.p_ready[hh]);
      continue;
    }
    umma::fence_after_sync();
    const int kt = j * kTileKeys;
    const int lim = page_bad ? -1 : pos - kt;            // key kt+i visible iff i <= lim
    const bool full_tile = lim >= kTileKeys - 1 + (tree ? 64 : 0);
    uint32_t sv[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) umma::tmem_ld32(tS + 32 * c, sv[c]);
    umma::tmem_ld_wait();
    if (!full_tile) {
      // Masked keys' scores become -inf: they take no part in the max, and
      // with a positive scale their exponentials are exactly 0.  Bit b of
      // word w: key kt + 32 w + b is visible (causal bound, then the
      // ancestor bits over the 64 keys up to the row's position).
      uint32_t vis[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int n = lim - 32 * w + 1;                  // causal keys in this word
        vis[w] = n >= 32 ? ~0u : (n <= 0 ? 0u : (1u << n) - 1u);
        if (tree) {
          const int o = 32 * w - lim + 63;               // reversed-mask bit of key 32 w
          uint32_t win = 0u, bits = 0u;
          if (o >= 0 && o < 64) {
            win = (uint32_t)(~0ull >> o);
            bits = (uint32_t)(anc_rev >> o);
          } else if (o < 0 && o > -32) {
            win = (uint32_t)(~0ull << -o);
            bits = (uint32_t)(anc_rev << -o);
          }
          vis[w] = (vis[w] & ~win) | (bits & win);
        }
      }
#pragma unroll
      for (int i = 0; i < 128; ++i)
        if (!((vis[i >> 5] >> (i & 31)) & 1u)) sv[i >> 5][i & 31] = 0xff800000u;   // -inf
    }
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < 64; ++k)
      mx = fmax3(mx, __uint_as_float(sv[(2 * k) >> 5][(2 * k) & 31]),
                 __uint_as_float(sv[(2 * k + 1) >> 5][(2 * k + 1) & 31]));
    mx = mx * sl2;
    const float m_new = fmaxf(m_run, mx);
    const bool resc = m_new > m_run + kRescaleThreshold;
    float alpha = 1.f;
    if (resc) {
      alpha = fast_exp2(m_run - m_new);
      l *= alpha;
      m_run = m_new;
    }
    const float nbase = m_run == -INFINITY ? 0.f : -m_run;
    // p = 2^(s*scale - m) on pairs of columns (packed f32x2 FMA and add),
    // packed to 16-bit pairs in place (pair k lands in slot k <= 2k, after
    // both of its inputs are read), then written over the first 64 columns
    // of S.  The row sum is kept as two interleaved partial sums.
    f2 acc = {0.f, 0.f};
    const f2 sc2 = {sl2, sl2}, nb2 = {nbase, nbase};
#pragma unroll
    for (int k = 0; k < 64; ++k) {
      const int i0 = 2 * k;
      f2 t = ffma2({__uint_as_float(sv[i0 >> 5][i0 & 31]),
                    __uint_as_float(sv[(i0 + 1) >> 5][(i0 + 1) & 31])}, sc2, nb2);
      const f2 e = {fast_exp2(t.x), fast_exp2(t.y)};
      acc = fadd2(acc, e);
      sv[k >> 5][k & 31] = FP8 ? pack_f16x2(e.x, e.y) : pack_bf16x2(e.x, e.y);
    }
    const float rs = acc.x + acc.y;
    umma::tmem_st32(tS, sv[0]);
    umma::tmem_st32(tS + 32, sv[1]);
    if (jj > 0 && __any_sync(0xffffffffu, resc)) {     // O *= alpha in TMEM
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        umma::tmem_ld32(tO + 32 * c, o);
        umma::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        umma::tmem_st32(tO + 32 * c, o);
      }
    }
    l += rs;
    umma::tmem_st_wait();
    umma::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&b.p_ready[hh]);
  }
  if (ok) ok = mbar_wait_or_abort(b.o_final, 0, p.err_flag, b.abort);
  if (ok) umma::fence_after_sync();

  if (VERIFY) {
    // Merge the two slots (the same query vectors over alternate key tiles)
    // into split sigma's partial, as the decode partial kernel leaves it: m
    // in log2 units, l, and O (unnormalised, V scale applied).  Slot B's
    // threads leave their (m, l) in shared memory; after one barrier of all
    // eight softmax warps (which every one of them reaches), slot A's read
    // both slots' O from TMEM (the same lane quarter) and write.  A slot
    // without tiles counts as m = -inf, l = 0, O = 0.
    // In half mode slot B's lanes are not slot A's: slot B's threads also
    // leave their O rows in shared memory (over the V stages, free once the
    // MMAs are done; 16-byte chunks permuted by vector against conflicts).
    float2* ml_s = reinterpret_cast<float2*>(smem + Layout<FP8>::kOffMl);
    const uint32_t obuf = smem_u32(smem + kOffV) + (uint32_t)v * 512u;
    if (hh == 1) {
      if (mine) ml_s[v] = make_float2(m_run, l);
      // tcgen05.ld is warp-wide: the condition is the same for every lane
      // (mine and nt are per warp), and only the stores follow `valid`
      const bool wok = __all_sync(0xffffffffu, ok);
      if (half && mine && nt > 0 && wok) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          umma::tmem_ld32(tO + 32 * c, o);
          umma::tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                               obuf + part_o_chunk(v, 8 * c + q)),
                           "r"(o[4 * q]), "r"(o[4 * q + 1]), "r"(o[4 * q + 2]),
                           "r"(o[4 * q + 3])
                           : "memory");
          }
        }
      }
    }
    __syncwarp();
    named_bar_sync(1, 256);
    if (hh == 1 || !__all_sync(0xffffffffu, ok)) return;
    const float2 mlb = ml_s[v];
    const float mx = fmaxf(m_run, mlb.x);
    const float a0 = m_run == -INFINITY ? 0.f : fast_exp2(m_run - mx);
    const float a1 = mlb.x == -INFINITY ? 0.f : fast_exp2(mlb.x - mx);
    const float vs = FP8 ? __ldg(p.v_scale + x.g) : 1.f;
    const float c0 = a0 * vs, c1 = a1 * vs;
    const int nb = slot_tiles<true>(gm, 1);
    const size_t slot =
        ((size_t)(ru.row0 + gm.row_lo + rho) * p.hq + x.g * p.group + hig) * p.max_splits +
        x.sigma;
    float4* po = reinterpret_cast<float4*>(p.part_o + slot * kHeadDim);
    const uint32_t tOb = tmem + lane_off + col_o(1);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t oa[32], ob[32];
      if (nt > 0) {
        umma::tmem_ld32(tO + 32 * c, oa);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) oa[i] = 0u;
      }
      if (nb > 0 && half) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 w = lds128(obuf + part_o_chunk(v, 8 * c + q));
          ob[4 * q] = w.x;
          ob[4 * q + 1] = w.y;
          ob[4 * q + 2] = w.z;
          ob[4 * q + 3] = w.w;
        }
      } else if (nb > 0) {
        umma::tmem_ld32(tOb + 32 * c, ob);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) ob[i] = 0u;
      }
      umma::tmem_ld_wait();
      if (valid) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            v[e] = __fmaf_rn(__uint_as_float(oa[4 * q + e]), c0,
                             __fmul_rn(__uint_as_float(ob[4 * q + e]), c1));
          po[8 * c + q] = make_float4(v[0], v[1], v[2], v[3]);
        }
      }
    }
    if (valid)
      *reinterpret_cast<float2*>(p.part_ml + slot * 2) =
          make_float2(mx, __fmaf_rn(l, a0, __fmul_rn(mlb.y, a1)));
    return;
  }

  const uint32_t sbase = smem_u32(smem);

  if (rank == 1) {
    // Store (m, l, O) into CTA 0 once its rings are free; arrive on its
    // barrier whatever happened, so that it never waits out the time limit
    // on this CTA's account.
    const bool free = mbar_wait_cluster(b.dst_free, 0, p.err_flag);
    if (ok && free) {
      const uint32_t orow = mapa_shared(part_o_row(sbase, hh, r), 0);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        umma::tmem_ld32(tO + 32 * c, o);
        umma::tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 8; ++q)
          st_cluster128(orow + part_o_chunk(r, 8 * c + q), o[4 * q], o[4 * q + 1], o[4 * q + 2],
                        o[4 * q + 3]);
      }
      st_cluster_f2(mapa_shared(part_ml(sbase, hh, r), 0), m_run, l);
    }
    mbar_arrive_remote(mapa_shared(smem_u32(b.peer_ready), 0));
    return;
  }

  // CTA 0: its MMAs are done (or it gave up), so CTA 1 may store into the
  // rings.  Then merge CTA 1's half into this one, normalise, write.
  if (threadIdx.x == 128) mbar_arrive_remote(mapa_shared(smem_u32(b.dst_free), 1));
  const bool peer = mbar_wait_cluster(b.peer_ready, 0, p.err_flag);
  if (!ok || !peer) return;
  float2 ml1;
  asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(ml1.x), "=f"(ml1.y)
               : "r"(part_ml(sbase, hh, r)) : "memory");
  const float m_all = fmaxf(m_run, ml1.x);
  const float a0 = m_run == -INFINITY ? 0.f : fast_exp2(m_run - m_all);
  const float a1 = ml1.x == -INFINITY ? 0.f : fast_exp2(ml1.x - m_all);
  const float l_all = __fmaf_rn(l, a0, __fmul_rn(ml1.y, a1));
  const float inv = (l_all > 0.f ? 1.f / l_all : 0.f) * (FP8 ? __ldg(p.v_scale + x.g) : 1.f);
  const float c0 = a0 * inv, c1 = a1 * inv;
  const int h = x.g * p.group + 2 * x.hp + hh;
  const bool write = valid && (2 * x.hp + hh) < p.group;
  uint4* dst = reinterpret_cast<uint4*>(
      p.out + ((size_t)(ru.row0 + gm.row_lo + r) * p.hq + h) * kHeadDim);
  const uint32_t prow = part_o_row(sbase, hh, r);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t o[32];
    if (gm.nkt > 0) {
      umma::tmem_ld32(tO + 32 * c, o);
      umma::tmem_ld_wait();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = 0u;
    }
    float f[32];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint4 w = lds128(prow + part_o_chunk(r, 8 * c + q));
      f[4 * q + 0] = __fmaf_rn(__uint_as_float(o[4 * q + 0]), c0, __fmul_rn(__uint_as_float(w.x), c1));
      f[4 * q + 1] = __fmaf_rn(__uint_as_float(o[4 * q + 1]), c0, __fmul_rn(__uint_as_float(w.y), c1));
      f[4 * q + 2] = __fmaf_rn(__uint_as_float(o[4 * q + 2]), c0, __fmul_rn(__uint_as_float(w.z), c1));
      f[4 * q + 3] = __fmaf_rn(__uint_as_float(o[4 * q + 3]), c0, __fmul_rn(__uint_as_float(w.w), c1));
    }
    if (write) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 v;
        v.x = pack_bf16x2(f[8 * q + 0], f[8 * q + 1]);
        v.y = pack_bf16x2(f[8 * q + 2], f[8 * q + 3]);
        v.z = pack_bf16x2(f[8 * q + 4], f[8 * q + 5]);
        v.w = pack_bf16x2(f[8 * q + 6], f[8 * q + 7]);
        dst[4 * c + q] = v;
      }
    }
  }
  if (write && p.lse)
    p.lse[(size_t)(ru.row0 + gm.row_lo + r) * p.hq + h] =
        l_all > 0.f ? (m_all + log2f(l_all)) * 0.6931471805599453f : -INFINITY;
}

template <bool FP8, bool VERIFY>
__global__ void __launch_bounds__(threads_of<FP8>(), 1)
    prefill_kernel(const __grid_constant__ PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Layout<FP8>::kOffBar);
  Bars b;
  b.q_full = bars + 0;
  b.q_ready = FP8 ? bars + 1 : bars + 0;
  // Verify with an e4m3 cache: four K stages (bars 2-5 full, 10-13 empty)
  // and four V staging tiles (24-27 full, 28-31 empty); no K staging.
  // Verify with a bf16 cache: rings of three, K full 24-26 and empty 27-29,
  // V full 2-4 and empty 5-7.
  constexpr bool kDirectK = VERIFY && FP8;
  constexpr bool kRing3 = VERIFY && !FP8;
  b.k_full = kRing3 ? bars + 24 : bars + 2;
  b.k_empty = kDirectK ? bars + 10 : kRing3 ? bars + 27 : bars + 4;
  b.v_full = kRing3 ? bars + 2 : bars + 6;
  b.v_empty = kRing3 ? bars + 5 : bars + 8;
  b.k8_full = bars + 10;
  b.k8_empty = bars + 11;
  b.v8_full = kDirectK ? bars + 24 : bars + 12;
  b.v8_empty = kDirectK ? bars + 28 : bars + 13;
  b.s_full = bars + 14;
  b.p_ready = bars + 16;
  b.o_final = bars + 18;
  b.drain = bars + 19;
  b.tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  b.abort = reinterpret_cast<volatile int*>(bars + 21);
  b.peer_ready = bars + 22;
  b.dst_free = bars + 23;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    const uint32_t stage_arrivals = FP8 ? kConvWarps : 1;   // the converters, or the producer
    mbar_init(b.q_full, 1);
    mbar_init(bars + 1, VERIFY ? 4 : 8);           // q_ready: the (slot A) softmax warps
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b.s_full[i], 1);
      mbar_init(&b.p_ready[i], 4);
    }
    for (int i = 0; i < (kRing3 ? 3 : 2); ++i) {
      mbar_init(&b.v_full[i], stage_arrivals);
      mbar_init(&b.v_empty[i], 1);
    }
    if (kDirectK) {
      for (int i = 0; i < 4; ++i) {
        mbar_init(&b.k_full[i], 1);                // the producer's TMA
        mbar_init(&b.k_empty[i], 1);
        mbar_init(&b.v8_full[i], 1);
        mbar_init(&b.v8_empty[i], kConvWarps);
      }
    } else {
      for (int i = 0; i < (kRing3 ? 3 : 2); ++i) {
        mbar_init(&b.k_full[i], stage_arrivals);
        mbar_init(&b.k_empty[i], 1);
      }
      if (FP8) {
        mbar_init(b.k8_full, 1);
        mbar_init(b.k8_empty, kConvWarps);
        mbar_init(b.v8_full, 1);
        mbar_init(b.v8_empty, kConvWarps);
      }
    }
    mbar_init(b.o_final, 1);
    mbar_init(b.drain, 1);
    mbar_init(b.peer_ready, 256);                  // every softmax thread of CTA 1
    mbar_init(b.dst_free, 1);
    *b.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.qmap);
    for (int i = 0; i < p.nsrc; ++i) {
      tma_prefetch_desc(&p.maps[i].k);
      tma_prefetch_desc(&p.maps[i].v);
    }
  }
  if (warp == 1) umma::tmem_alloc(b.tmem_slot, kTmemCols);
  umma::fence_before_sync();
  __syncthreads();
  if (!VERIFY) cluster_sync();   // both CTAs' barriers initialised before any remote arrival
  umma::fence_after_sync();
  const uint32_t tmem = *b.tmem_slot;
  allow_next_grid();
  wait_prior_grid();

  // Prefill: two CTAs (a cluster) per tile; verify: one CTA per tile.
  const uint32_t rank = VERIFY ? 0 : cluster_ctarank();
  const Tile x = tile_of<VERIFY>(p, VERIFY ? blockIdx.x : blockIdx.x >> 1);
  const RunInfo& ru = p.runs[x.run];
  const TileGeom gm = geom_of<VERIFY>(p, ru, x, rank);

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Regs<FP8>::kLow));
    if (warp == 0) {
      if (lane == 0) producer<FP8, VERIFY>(p, ru, x, gm, smem, b);
    } else if (warp == 1) {
      mma_issuer<FP8, VERIFY>(p, ru, gm, smem, tmem, b);
    }
  } else if (warp < kConvWarp0) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Regs<FP8>::kHigh));
    softmax_role<FP8, VERIFY>(p, ru, x, gm, rank, (warp - 4) >> 2, smem, tmem, b);
  } else if (FP8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Regs<FP8>::kConv));
    converter<VERIFY>(p, ru, gm, smem, b);
  }
  umma::fence_before_sync();
  __syncthreads();
  if (!VERIFY) cluster_sync();   // CTA 1's shared memory stays until CTA 0 has read it
  if (warp == 1) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool FP8, bool VERIFY>
cudaError_t launch(const PrefillParams& p, int tiles, cudaStream_t s) {
  static PerDeviceOnce configured;
  const cudaError_t e = configured.run([] {
    // The register split only works if the block launches with at least the
    // registers it hands out; otherwise setmaxnreg.inc would wait forever.
    cudaFuncAttributes attr;
    cudaError_t r = cudaFuncGetAttributes(&attr, prefill_kernel<FP8, VERIFY>);
    if (r != cudaSuccess) return r;
    if (attr.numRegs * threads_of<FP8>() < regs_split<FP8>()) return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(prefill_kernel<FP8, VERIFY>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Layout<FP8>::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  if (VERIFY)
    return launch_pdl(prefill_kernel<FP8, VERIFY>, dim3(tiles), dim3(threads_of<FP8>()),
                      Layout<FP8>::kSmemBytes, s, p);
  return launch_pdl_cluster(prefill_kernel<FP8, VERIFY>, dim3(2 * tiles),
                            dim3(threads_of<FP8>()), Layout<FP8>::kSmemBytes, s, p, 2);
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, bool fp8, int tiles, cudaStream_t s) {
  if (tiles <= 0) return cudaSuccess;
  return fp8 ? launch<true, false>(p, tiles, s) : launch<false, false>(p, tiles, s);
}

cudaError_t launch_verify(const PrefillParams& p, bool fp8, int tiles, cudaStream_t s) {
  if (tiles <= 0) return cudaSuccess;
  return fp8 ? launch<true, true>(p, tiles, s) : launch<false, true>(p, tiles, s);
}

}  // namespace tfpa
