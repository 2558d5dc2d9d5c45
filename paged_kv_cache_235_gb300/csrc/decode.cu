// Decode/verify attention as split-K partials plus a log-sum-exp merge
// (TensorFold Issue #1344, "Mechanism": partial kernels write running max,
// sum and unnormalised output per split, then attn_merge combines them).
//
// Partial kernel: persistent CTAs, each taking a contiguous range of work
// items (run, kv head g, m-tile of 16 query vectors, split).  A split is a
// fixed number of whole pages chosen from the stream's own length, so a
// row's partials never depend on its batch or on how rows are sliced.
// Per CTA (four warpgroups):
//   warp 12     producer: looks each page up once (PR #2011, "the decode
//               tiles ... look a page up once"), stages K and V chunks into
//               shared memory with TMA tiled loads (128B swizzle), a ring
//               of three 64 KB key chunks (bf16: a chunk is one stage;
//               e4m3: two stages, read by consumer warps 0-3 and 4-7);
//   warps 0..7  consumers: each takes an eighth of every chunk's keys, runs
//               QK^T and PV on mma.sync m16n8k16 (bf16, or f16 for e4m3
//               caches, whose bytes convert to f16 exactly) and an online
//               softmax reduced with warp shuffles; at the end of an item
//               each warp stores its state (O, m, l) into tensor memory and
//               goes straight on to the next item;
//   warps 8..11 combiners: warp 8+q reads the states of consumer warps q and
//               q+4 (the two warps that share its TMEM lane quarter and its
//               fragment layout), folds them, and the four combiners add
//               their folds in a fixed order and write the partial.
// TMEM holds two items' states, so the combine of one item overlaps the
// next item's loads and math.
// Paged and slab streams differ only in the TMA row coordinate, so they
// produce the same bytes (PR #1373, "What changes").
#include <climits>

#include "common.cuh"
#include "kvstore.cuh"
#include "params.h"
#include "tcgen05.cuh"

namespace tfpa {
namespace {

// The ring holds three key chunks (64 KB of K and V each); a chunk arrives
// as Cfg::kSub stages (see Cfg), at most kMaxStages in the ring.
constexpr int kRingBytes = 3 * 65536;
constexpr int kMaxStages = 6;
constexpr int kConsumerWarps = 8;
constexpr int kCombineWarp0 = 8;      // warps 8..11
constexpr int kCombineWarps = 4;
constexpr int kProducerWarp = 12;     // warps 13..15 only take part in the register split
constexpr int kThreads = 16 * 32;
// Registers after the split: the block launches with 512 x 128 = 65,536 and
// 128 x (2 x kRegsConsumer + kRegsCombine + kRegsProducer) must not exceed it.
constexpr int kRegsConsumer = 184;
constexpr int kRegsCombine = 112;
constexpr int kRegsProducer = 32;
static_assert(128 * (2 * kRegsConsumer + kRegsCombine + kRegsProducer) <= 65536, "register split");
// TMEM: two buffers (item parity) x two halves (consumer warps q, q+4) of
// 64 O columns + (m0, l0, m1, l1); lane quarter q belongs to warps q, q+4, 8+q.
constexpr int kTmemCols = 512;
constexpr int kBufCols = 256;
constexpr int kHalfCols = 128;
// Fold buffer: [slot q][PV n-tile][lane] float4, the C-fragment order of the
// consumer warps (conflict-free float4 stores and loads).
constexpr int kCombBytes = kCombineWarps * 16 * 32 * 16;
constexpr int kMlBytes = kConsumerWarps * 16 * 2 * 4;
constexpr int kNumBars = 2 * kMaxStages + 7;
constexpr int kSmemBytes =
    kRingBytes + kCombBytes + kMlBytes + kMaxStages * 4 + 8 + kNumBars * 8 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory");
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <bool FP8>
struct Cfg {
  static constexpr int kChunk = FP8 ? 256 : 128;      // keys per chunk
  // e4m3: a chunk in two stages of 128 keys (K 16 KB + V 16 KB), the first
  // read by consumer warps 0-3, the second by 4-7, so a stage is released
  // after half the warps' work (fp8 verify partial 174.2 -> 172.5 us);
  // bf16: one stage of 128 keys (two stages measured 0.7 % slower).
  static constexpr int kSub = FP8 ? 2 : 1;
  static constexpr int kStages = 3 * kSub;
  static constexpr int kStageBytes = 65536 / kSub;
  static constexpr int kStageKeys = kChunk / kSub;     // 128 either way
  static constexpr int kSubWarps = kConsumerWarps / kSub;   // warps reading a stage
  static constexpr int kKeysPerWarp = kChunk / kConsumerWarps;
  static constexpr int kNT = kKeysPerWarp / 8;         // score n-tiles per warp
  static constexpr int kKS = kKeysPerWarp / 16;        // PV k-steps per warp
};

// A work item: (run, kv head g, m-tile mt of 16 query vectors, split sigma).
struct Item {
  int run, g, mt, sigma;
};

__device__ __forceinline__ int mtiles_of(const RunInfo& ru, int group) {
  return (ru.nrows * group + 15) >> 4;
}

// The run holding item `it`, by binary search over the runs' first items
// (a few dependent loads when the runs sit in device memory).
__device__ __forceinline__ int run_of(const DecodeDyn& D, int it) {
  int lo = 0, hi = D.nruns - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (D.runs[mid].item0 <= it) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Work item `it`; r is the run of an earlier item of this CTA (or of `it`)
// and becomes `it`'s: a CTA walks its items in order, so the run only moves
// forward.
__device__ __forceinline__ Item item_of(const DecodeParams& p, const DecodeDyn& D, int it,
                                        int& r) {
  while (r + 1 < D.nruns && D.runs[r + 1].item0 <= it) ++r;
  const RunInfo& ru = D.runs[r];
  int local = it - ru.item0;
  const int mgroups = mtiles_of(ru, p.group);
  Item x;
  x.run = r;
  x.sigma = local % ru.nsplit;
  local /= ru.nsplit;
  x.mt = local % mgroups;
  x.g = local / mgroups;
  return x;
}

// Items [begin, end) of this CTA: a contiguous share balanced by work on the
// host, so consecutive items are mostly consecutive splits of one (stream,
// kv head, m-tile).
__device__ __forceinline__ void cta_items(const DecodeDyn& D, int& begin, int& end) {
  begin = D.cta_item0[blockIdx.x];
  end = D.cta_item0[blockIdx.x + 1];
}

// Key range [klo, khi) an item must read: its split's pages, cut at the
// stream length and at the last position among the item's rows.
__device__ __forceinline__ void item_keys(const DecodeParams& p, const DecodeDyn& D, const Item& x,
                                          int& klo, int& khi) {
  const RunInfo& ru = D.runs[x.run];
  const int nq = ru.nrows * p.group;
  const int last_qv = min(16 * x.mt + 15, nq - 1);
  const int maxpos = ru.pos0 + last_qv / p.group;
  klo = x.sigma * ru.pps * kPage;
  khi = min(min(klo + ru.pps * kPage, ru.seq_len), maxpos + 1);
}

// Append: the producer warp stores the new K and V of kv head g at
// positions [k0, k1) of run ru (rows of this launch from ru.row0), as the
// KV write kernel stores them: lanes 0-15 a K row's 8-element slices, lanes
// 16-31 a V row's.  Each lane then fences its stores against the TMA
// loads that follow (async proxy), and the warp meets.
template <bool FP8>
__device__ void store_new_rows(const DecodeParams& p, const RunInfo& ru, int g, int k0, int k1,
                               int lane) {
  const bool is_v = lane >= 16;
  const int t = lane & 15;
  const __nv_bfloat16* src_rows = is_v ? p.v_rows : p.k_rows;
  void* base = is_v ? p.v_base[ru.src] : p.k_base[ru.src];
  for (int key = k0; key < k1; ++key) {
    size_t dst_row;
    if (ru.page_table) {
      const int pid = __ldg(ru.page_table + (key >> 8));
      if ((unsigned)pid >= (unsigned)p.num_pages) {   // flagged by the loads of that page
        continue;
      }
      dst_row = ((size_t)pid * p.hkv + g) * kPage + (key & (kPage - 1));
    } else {
      dst_row = (size_t)g * ru.slab_cap + key;
    }
    const int row = ru.row0 + (key - ru.pos0);
    const uint4 in =
        *reinterpret_cast<const uint4*>(src_rows + ((size_t)row * p.hkv + g) * kHeadDim + t * 8);
    if (FP8) {
      float f[8];
      unpack8(in, f);
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(base) + dst_row * kHeadDim + t * 8) =
          quant8(f, __ldg((is_v ? p.v_scale : p.k_scale) + g));
    } else {
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + dst_row * kHeadDim + t * 8) =
          in;
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncwarp();
}

template <bool FP8>
__device__ __forceinline__ bool load_item(const DecodeParams& p, const RunInfo& ru, const Item& x,
                                          int klo, int khi, uint8_t* stage_mem, uint64_t* full,
                                          uint64_t* empty, int* stage_bad, uint32_t& stage);

// Producer warp: lane 0 looks pages up and issues the TMA loads; with
// append (APPEND), the whole warp first stores the new rows an item reads.
template <bool FP8, bool APPEND>
__device__ void producer(const DecodeParams& p, const DecodeDyn& D, uint8_t* stage_mem,
                         uint64_t* full, uint64_t* empty, int* stage_bad) {
  const int lane = threadIdx.x & 31;
  if (!APPEND && lane != 0) return;
  int ib, ie;
  cta_items(D, ib, ie);
  int rh = ib < ie ? run_of(D, ib) : 0;   // run of the current item
  uint32_t stage = 0;
  bool ok = true;
  for (int it = ib; ok && it < ie; ++it) {
    const Item x = item_of(p, D, it, rh);
    const RunInfo& ru = D.runs[x.run];
    int klo, khi;
    item_keys(p, D, x, klo, khi);
    if constexpr (APPEND) {
      const int k0 = max(klo, ru.pos0), k1 = min(khi, ru.pos0 + ru.nrows);
      if (k0 < k1) store_new_rows<FP8>(p, ru, x.g, k0, k1, lane);
      // the warp moves on item by item with lane 0, and leaves with it
      ok = __shfl_sync(0xffffffffu, lane == 0 ? load_item<FP8>(p, ru, x, klo, khi, stage_mem,
                                                                full, empty, stage_bad, stage)
                                              : true,
                       0);
    } else {
      ok = load_item<FP8>(p, ru, x, klo, khi, stage_mem, full, empty, stage_bad, stage);
    }
  }
}

// Lane 0 of the producer warp: the TMA loads of one item's key chunks into
// the ring, one page lookup per page.  False if a wait gave up.
template <bool FP8>
__device__ __forceinline__ bool load_item(const DecodeParams& p, const RunInfo& ru, const Item& x,
                                          int klo, int khi, uint8_t* stage_mem, uint64_t* full,
                                          uint64_t* empty, int* stage_bad, uint32_t& stage) {
  using C = Cfg<FP8>;
  {
    const CUtensorMap* mk = &p.maps[ru.src].k;
    const CUtensorMap* mv = &p.maps[ru.src].v;
    int cached_page = -1, cached_pid = 0;
    // a chunk (and so each of its stages) lies within one page
    for (int k0 = klo; k0 < khi; k0 += C::kChunk) {
      const int page = k0 >> 8;
      int y, bad = 0;
      if (ru.page_table) {
        if (page != cached_page) {  // one lookup per page
          cached_pid = __ldg(ru.page_table + page);
          cached_page = page;
        }
        int pid = cached_pid;
        if ((unsigned)pid >= (unsigned)p.num_pages) {
          flag_error(p.err_flag, kErrBadPage);
          bad = 1;
          pid = 0;
        }
        y = (pid * p.hkv + x.g) * kPage + (k0 & (kPage - 1));
      } else {
        y = x.g * ru.slab_cap + k0;
      }
      for (int h = 0; h < C::kSub; ++h, ++stage, y += C::kStageKeys) {
        const int buf = stage % C::kStages;
        const uint32_t ph = (stage / C::kStages) & 1;
        if (!mbar_wait(&empty[buf], ph ^ 1, p.err_flag)) return false;
        stage_bad[buf] = bad;
        uint64_t* fb = &full[buf];
        uint8_t* sb = stage_mem + (size_t)buf * C::kStageBytes;
        mbar_arrive_expect_tx(fb, C::kStageBytes);
        if (FP8) {
          tma_load_2d(sb, mk, 0, y, fb);
          tma_load_2d(sb + C::kStageBytes / 2, mv, 0, y, fb);
        } else {
          tma_load_2d(sb, mk, 0, y, fb);
          tma_load_2d(sb + C::kStageBytes / 4, mk, 64, y, fb);
          tma_load_2d(sb + C::kStageBytes / 2, mv, 0, y, fb);
          tma_load_2d(sb + 3 * C::kStageBytes / 4, mv, 64, y, fb);
        }
      }
    }
  }
  return true;
}

// Real head-dim index of C-fragment column n of PV n-tile nt (the V fragments
// are loaded so a thread's sixteen n-tiles cover contiguous 16-byte chunks).
template <bool FP8>
__device__ __forceinline__ int out_col(int nt, int n) {
  if (FP8) return 16 * n + nt;
  return nt < 8 ? 8 * n + nt : 64 + 8 * n + (nt - 8);
}

// Query fragments of rows gq and gq+8 of an m-tile, the rows' causal limits,
// their ancestor masks (all ones for causal rows) and their score multipliers
// (f16 operands for e4m3 caches: each row is scaled by a power of two into
// f16 range, exact for every element within 2^28 of the row's largest).
template <bool FP8, bool GEN>
__device__ __forceinline__ void load_q(const DecodeParams& p, const RunInfo& ru, const Item& x,
                                       int gq, int c, uint32_t (&qr)[2][16], int (&lim)[2],
                                       uint64_t (&anc)[2], float (&sc)[2]) {
  const int nq = ru.nrows * p.group;
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int qv = x.mt * 16 + gq + 8 * hr;
    uint4 v[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                  make_uint4(0, 0, 0, 0)};
    lim[hr] = -1;
    anc[hr] = ~0ull;
    if (qv < nq) {
      const int r = qv / p.group;
      const int h = x.g * p.group + (qv - r * p.group);
      lim[hr] = ru.pos0 + r;
      if (GEN && p.anc) anc[hr] = __ldg(p.anc + ru.row0 + r);
      const uint4* qp =
          reinterpret_cast<const uint4*>(p.q + ((size_t)(ru.row0 + r) * p.hq + h) * kHeadDim);
      if (FP8) {
#pragma unroll
        for (int m = 0; m < 4; ++m) v[m] = __ldg(qp + 4 * c + m);
      } else {
        v[0] = __ldg(qp + 2 * c);
        v[1] = __ldg(qp + 2 * c + 1);
        v[2] = __ldg(qp + 8 + 2 * c);
        v[3] = __ldg(qp + 8 + 2 * c + 1);
      }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      qr[hr][4 * m + 0] = v[m].x;
      qr[hr][4 * m + 1] = v[m].y;
      qr[hr][4 * m + 2] = v[m].z;
      qr[hr][4 * m + 3] = v[m].w;
    }
    sc[hr] = p.scale_log2;
    if (FP8) {
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        amax = fmaxf(amax, fabsf(__uint_as_float(qr[hr][j] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(qr[hr][j] & 0xFFFF0000u)));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      int ex;
      frexpf(amax, &ex);
      ex = max(min(ex, 120), -100);
      const float up = __int_as_float((127 + 14 - ex) << 23);
      const float down = __int_as_float((127 - 14 + ex) << 23);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float lo = __uint_as_float(qr[hr][j] << 16) * up;
        const float hi = __uint_as_float(qr[hr][j] & 0xFFFF0000u) * up;
        qr[hr][j] = pack_f16x2(lo, hi);
      }
      sc[hr] = p.scale_log2 * down * __ldg(p.k_scale + x.g);
    }
  }
}

struct CombBars {
  uint64_t* posted;      // [2] by item parity: the 8 consumer warps stored their state
  uint64_t* tmem_free;   // [2] by item parity: the combiners read that TMEM buffer
  uint64_t* pub;         // the combiners published their pairs' (m, l)
  uint64_t* folded;      // the combiners wrote their folds
  uint64_t* done;        // the combiners finished the item (fold buffer free)
};

// This warp's kKeysPerWarp keys, keys key_base.. at rows r0.. of the stage
// at sb: scores, the causal or ancestor mask, the online softmax, and
// O += P V.
template <bool FP8, bool GEN>
__device__ __forceinline__ void attend_block(uint32_t sb, int r0, int key_base, int seq_len,
                                             const uint32_t (&qr)[2][16], const int (&lim)[2],
                                             const float (&sc)[2], const uint64_t (&anc)[2],
                                             int tree_low, int gq, int c, float (&m_run)[2],
                                             float (&l_run)[2], float (&o)[16][4]) {
  using C = Cfg<FP8>;
  constexpr int kNT = C::kNT;             // score n-tiles
  constexpr int kKS = C::kKS;             // PV k-steps
  constexpr int kKeys = C::kKeysPerWarp;
  // ---- S = Q K^T over this warp's keys
  float s[kNT][4];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    const int kr = r0 + nt * 8 + gq;
    uint32_t kb[16];
    if (FP8) {
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const uint4 w = lds128(swz128(sb, kr, 2 * c + ch));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          kb[8 * ch + 2 * i] = e4m3x2_to_f16x2((uint16_t)(ws[i] & 0xFFFF));
          kb[8 * ch + 2 * i + 1] = e4m3x2_to_f16x2((uint16_t)(ws[i] >> 16));
        }
      }
    } else {
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const uint32_t base = sb + (ch >> 1) * (uint32_t)(C::kStageBytes / 4);
        const uint4 w = lds128(swz128(base, kr, 2 * c + (ch & 1)));
        kb[4 * ch + 0] = w.x;
        kb[4 * ch + 1] = w.y;
        kb[4 * ch + 2] = w.z;
        kb[4 * ch + 3] = w.w;
      }
    }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t a[4] = {qr[0][2 * ks], qr[1][2 * ks], qr[0][2 * ks + 1],
                             qr[1][2 * ks + 1]};
      if (FP8)
        mma_f16(s[nt], a, kb[2 * ks], kb[2 * ks + 1]);
      else
        mma_bf16(s[nt], a, kb[2 * ks], kb[2 * ks + 1]);
    }
  }
  // ---- scale, causal (or ancestor) mask, online softmax (rows gq,
  // gq+8; a row's keys are spread over the 4 threads of a quad).  The
  // running max is only moved when it grows by more than 2^8, so O is
  // rarely rescaled.  Ancestor masks are only consulted where a key
  // lies within 63 positions of some row of the warp.
  const bool tree_zone = GEN && key_base + kKeys > tree_low;
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int hr = j >> 1;
      const int key = key_base + nt * 8 + 2 * c + (j & 1);
      bool vis = key <= lim[hr];
      if (tree_zone) {
        const int dd = lim[hr] - key;
        vis = vis && (dd > 63 || ((anc[hr] >> dd) & 1ull));
      }
      const float v = vis ? s[nt][j] * sc[hr] : -INFINITY;
      s[nt][j] = v;
      mx[hr] = fmaxf(mx[hr], v);
    }
  }
  float alpha[2];
  bool resc = false;
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
    mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
    alpha[hr] = 1.f;
    if (mx[hr] > m_run[hr] + kRescaleThreshold) {
      alpha[hr] = fast_exp2(m_run[hr] - mx[hr]);
      l_run[hr] *= alpha[hr];
      m_run[hr] = mx[hr];
      resc = true;
    }
  }
  if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      o[nt][0] *= alpha[0];
      o[nt][1] *= alpha[0];
      o[nt][2] *= alpha[1];
      o[nt][3] *= alpha[1];
    }
  }
  const float base0 = m_run[0] == -INFINITY ? 0.f : m_run[0];
  const float base1 = m_run[1] == -INFINITY ? 0.f : m_run[1];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float e = fast_exp2(s[nt][j] - ((j >> 1) ? base1 : base0));
      s[nt][j] = e;
      l_run[j >> 1] += e;
    }
  }
  // ---- O += P V
  const uint32_t vb = sb + (uint32_t)(C::kStageBytes / 2);
#pragma unroll
  for (int kk = 0; kk < kKS; ++kk) {
    uint32_t a[4];
    if (FP8) {
      a[0] = pack_f16x2(s[2 * kk][0], s[2 * kk][1]);
      a[1] = pack_f16x2(s[2 * kk][2], s[2 * kk][3]);
      a[2] = pack_f16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      a[3] = pack_f16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
    } else {
      a[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
      a[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
      a[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      a[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
    }
    const int kv0 = r0 + 16 * kk + 2 * c;    // rows kv0, kv0+1, kv0+8, kv0+9
    const int krow[4] = {kv0, kv0 + 1, kv0 + 8, kv0 + 9};
    if (FP8) {
      uint32_t w[4][4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint4 t = lds128(swz128(vb, krow[q4], gq));
        if (key_base - r0 + krow[q4] >= seq_len) t = make_uint4(0, 0, 0, 0);
        w[q4][0] = t.x; w[q4][1] = t.y; w[q4][2] = t.z; w[q4][3] = t.w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t x01 = prmt(w[0][i], w[1][i], 0x5140);
        const uint32_t y01 = prmt(w[0][i], w[1][i], 0x7362);
        const uint32_t x23 = prmt(w[2][i], w[3][i], 0x5140);
        const uint32_t y23 = prmt(w[2][i], w[3][i], 0x7362);
        mma_f16(o[4 * i + 0], a, e4m3x2_to_f16x2((uint16_t)(x01 & 0xFFFF)),
                e4m3x2_to_f16x2((uint16_t)(x23 & 0xFFFF)));
        mma_f16(o[4 * i + 1], a, e4m3x2_to_f16x2((uint16_t)(x01 >> 16)),
                e4m3x2_to_f16x2((uint16_t)(x23 >> 16)));
        mma_f16(o[4 * i + 2], a, e4m3x2_to_f16x2((uint16_t)(y01 & 0xFFFF)),
                e4m3x2_to_f16x2((uint16_t)(y23 & 0xFFFF)));
        mma_f16(o[4 * i + 3], a, e4m3x2_to_f16x2((uint16_t)(y01 >> 16)),
                e4m3x2_to_f16x2((uint16_t)(y23 >> 16)));
      }
    } else {
      uint32_t r[4][8];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint4 t0 = lds128(swz128(vb, krow[q4], gq));
        uint4 t1 = lds128(swz128(vb + (uint32_t)(C::kStageBytes / 4), krow[q4], gq));
        if (key_base - r0 + krow[q4] >= seq_len) {
          t0 = make_uint4(0, 0, 0, 0);
          t1 = t0;
        }
        r[q4][0] = t0.x; r[q4][1] = t0.y; r[q4][2] = t0.z; r[q4][3] = t0.w;
        r[q4][4] = t1.x; r[q4][5] = t1.y; r[q4][6] = t1.z; r[q4][7] = t1.w;
      }
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const uint32_t sel = (nt & 1) ? 0x7632u : 0x5410u;
        const uint32_t b0 = prmt(r[0][nt >> 1], r[1][nt >> 1], sel);
        const uint32_t b1 = prmt(r[2][nt >> 1], r[3][nt >> 1], sel);
        mma_bf16(o[nt], a, b0, b1);
      }
    }
  }
}

template <bool FP8, bool GEN>
__device__ void consumer(const DecodeParams& p, const DecodeDyn& D, uint8_t* stage_mem,
                         uint64_t* full, uint64_t* empty, const int* stage_bad, uint32_t tmem,
                         CombBars bars) {
  using C = Cfg<FP8>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2, c = lane & 3;
  const uint32_t sbase = smem_u32(stage_mem);
  uint32_t chunk = 0;                       // key chunks read so far
  int ib, ie;
  cta_items(D, ib, ie);
  int rh = ib < ie ? run_of(D, ib) : 0;   // run of the current item
  int q_run = -1, q_g = -1, q_mt = -1;     // the m-tile whose query is loaded
  int lim[2] = {-1, -1};
  uint64_t anc[2] = {~0ull, ~0ull};
  float sc[2] = {0.f, 0.f};
  uint32_t qr[2][16];
  int maxlim = -1;
  int tree_low = INT_MAX;     // keys from here on may be hidden by an ancestor mask

  for (int it = ib; it < ie; ++it) {
    const Item x = item_of(p, D, it, rh);
    const RunInfo& ru = D.runs[x.run];
    int klo, khi;
    item_keys(p, D, x, klo, khi);
    // The chunk's 8 sub-blocks of kKeysPerWarp keys go to the 8 warps.
    const int sub0 = warp;
    if (x.run != q_run || x.g != q_g || x.mt != q_mt) {
      load_q<FP8, GEN>(p, ru, x, gq, c, qr, lim, anc, sc);
      maxlim = __reduce_max_sync(0xffffffffu, max(lim[0], lim[1]));
      if (GEN && p.anc) {
        const int mn = min(lim[0] >= 0 ? lim[0] : INT_MAX, lim[1] >= 0 ? lim[1] : INT_MAX);
        tree_low = (int)__reduce_min_sync(0xffffffffu, (unsigned)mn) - 63;
      }
      q_run = x.run;
      q_g = x.g;
      q_mt = x.mt;
    }

    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    float o[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

    // Chunk n's stage n * kSub + h holds the keys of warps h * kSubWarps ..
    // (h + 1) * kSubWarps - 1; this warp reads its stage only.
    for (int k0 = klo; k0 < khi; k0 += C::kChunk, ++chunk) {
      const uint32_t st = chunk * C::kSub + sub0 / C::kSubWarps;
      const int buf = st % C::kStages;
      const uint32_t ph = (st / C::kStages) & 1;
      if (!mbar_wait(&full[buf], ph, p.err_flag)) return;
      const uint32_t sb = sbase + (uint32_t)buf * C::kStageBytes;
      const int wk0 = sub0 * C::kKeysPerWarp;
      const int r0 = wk0 - (sub0 / C::kSubWarps) * C::kStageKeys;
      if (!stage_bad[buf] && k0 + wk0 <= maxlim)
        attend_block<FP8, GEN>(sb, r0, k0 + wk0, ru.seq_len, qr, lim, sc, anc, tree_low, gq, c,
                               m_run, l_run, o);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[buf]);
    }

    // ---- hand the state to the combiners: O and (m, l) into this warp's
    // lanes of TMEM buffer (item & 1), once the combine of item - 2 has
    // read that buffer.
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
      l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
    }
    const int rel = it - ib;
    const int b = rel & 1;
    if (rel >= 2 &&
        !mbar_wait(&bars.tmem_free[b], (uint32_t)((rel >> 1) - 1) & 1u, p.err_flag))
      return;
    umma::fence_after_sync();
    const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16) +
                        (uint32_t)(b * kBufCols + (warp >> 2) * kHalfCols);
    {
      uint32_t ov[64];
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
        for (int j = 0; j < 4; ++j) ov[4 * nt + j] = __float_as_uint(o[nt][j]);
      }
      umma::tmem_st64(ta, ov);
      const uint32_t ml[4] = {__float_as_uint(m_run[0]), __float_as_uint(l_run[0]),
                              __float_as_uint(m_run[1]), __float_as_uint(l_run[1])};
      umma::tmem_st4(ta + 64, ml);
    }
    umma::tmem_st_wait();
    umma::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.posted[b]);
  }
}

// The log-sum-exp merge of one (row, head) by one warp: lane s holds split
// s's (m, l), lane t owns head-dim elements 4t..4t+3.  M is the lanes' max,
// L the butterfly sum of l_s 2^(m_s - M), o = sum_s 2^(m_s - M) o_s taken in
// split order, out = o / L in bf16 and lse = ln2 (M + log2 L).  The o_s are
// loaded B splits at a time (every split at once in the merge kernel, fewer
// where registers are short); the arithmetic and its order do not depend on
// B, so every caller writes the same bytes.  CG: load through L2 only (the
// partials of other CTAs of a running grid).
template <int B, bool CG>
__device__ __forceinline__ void merge_vector(const float* part_o, const float* part_ml, int nsplit,
                                             __nv_bfloat16* out, float* lse) {
  const int lane = threadIdx.x & 31;
  const float4* po = reinterpret_cast<const float4*>(part_o) + lane;
  auto ld4 = [](const float4* a) { return CG ? __ldcg(a) : *a; };
  float4 v0[B];
#pragma unroll
  for (int u = 0; u < B; ++u)
    if (u < nsplit) v0[u] = ld4(po + u * (kHeadDim / 4));
  float m = -INFINITY, l = 0.f;
  if (lane < nsplit) {
    const float2* a = reinterpret_cast<const float2*>(part_ml) + lane;
    const float2 ml = CG ? __ldcg(a) : *a;
    m = ml.x;
    l = ml.y;
  }
  float M = m;
#pragma unroll
  for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float a = (m == -INFINITY) ? 0.f : fast_exp2(m - M);
  float L = a * l;
#pragma unroll
  for (int off = 16; off; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [&](int sp, const float4& v) {
    const float as = __shfl_sync(0xffffffffu, a, sp);
    acc.x = __fmaf_rn(as, v.x, acc.x);
    acc.y = __fmaf_rn(as, v.y, acc.y);
    acc.z = __fmaf_rn(as, v.z, acc.z);
    acc.w = __fmaf_rn(as, v.w, acc.w);
  };
  for (int u0 = 0; u0 < nsplit; u0 += B) {
    if (u0 > 0) {
#pragma unroll
      for (int u = 0; u < B; ++u)
        if (u0 + u < nsplit) v0[u] = ld4(po + (u0 + u) * (kHeadDim / 4));
    }
#pragma unroll
    for (int u = 0; u < B; ++u)
      if (u0 + u < nsplit) add(u0 + u, v0[u]);
  }
  const float inv = 1.f / L;
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(out + lane * 4) = packed;
  if (lse && lane == 0) *lse = (M + log2f(L)) * 0.6931471805599453f;
}

// Merge in the partial kernel, run by the four combiner warps after they
// wrote an item's partial: the item's group (run, kv head, m-tile) counts
// its finished splits in p.arrive, at the (row, head) of its first query
// vector; the CTA that finishes the last split resets the counter and
// merges the group's query vectors, warp 8+q taking vectors q, q+4, ...
// Every thread fences its partial stores before the count, and the merging
// threads fence after it and load the partials through L2.
__device__ __forceinline__ void merge_if_last(const DecodeParams& p, const RunInfo& ru,
                                              const Item& x, int nq, int* merge_flag) {
  const int q = (threadIdx.x >> 5) - kCombineWarp0;
  __threadfence();
  named_bar_sync(1, 32 * kCombineWarps);
  if (threadIdx.x == 32 * kCombineWarp0) {
    const int qv0 = x.mt * 16;
    const int r0 = qv0 / p.group;
    uint32_t* ctr = p.arrive + (size_t)(ru.row0 + r0) * p.hq + x.g * p.group + (qv0 - r0 * p.group);
    const uint32_t old = atomicAdd(ctr, 1u);
    const int last = old + 1u == (uint32_t)ru.nsplit;
    if (last) atomicExch(ctr, 0u);
    *merge_flag = last;
  }
  named_bar_sync(1, 32 * kCombineWarps);
  if (!*merge_flag) return;
  __threadfence();
  for (int j = q; j < 16; j += kCombineWarps) {
    const int qv = x.mt * 16 + j;
    if (qv >= nq) break;
    const int r = qv / p.group;
    const size_t rh = (size_t)(ru.row0 + r) * p.hq + x.g * p.group + (qv - r * p.group);
    const size_t slot0 = rh * p.max_splits;
    merge_vector<4, true>(p.part_o + slot0 * kHeadDim, p.part_ml + slot0 * 2, ru.nsplit,
                          p.out + rh * kHeadDim, p.lse ? p.lse + rh : nullptr);
  }
}

// Combiner warp 8+q: for every item of the CTA, reads the states of consumer
// warps q and q+4 from TMEM, and
// (1) publishes their (m, l) so that each combiner knows the eight-warp max;
// (2) folds the two O's, each rescaled to that max, into fold slot q;
// (3) adds the four slots in order for PV n-tiles 4q..4q+3 and writes that
//     part of the partial o (warp 8 also writes m and l).  The sums are
//     taken in a fixed order, so a partial's bits depend only on its keys.
// Each of pub, folded and done completes once per item (parity = item & 1);
// a combiner waits for done of the previous item before publishing, so the
// fold and (m, l) buffers are never overwritten while still being read.
template <bool FP8, bool GEN, bool MERGE>
__device__ void combiner(const DecodeParams& p, const DecodeDyn& D, uint32_t tmem, float4* fold,
                         float* ml_buf, int* merge_flag, CombBars bars) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q = warp - kCombineWarp0;
  const int gq = lane >> 2, c = lane & 3;
  int ib, ie;
  cta_items(D, ib, ie);
  int rh = ib < ie ? run_of(D, ib) : 0;   // run of the current item
  const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
  for (int it = ib; it < ie; ++it) {
    const Item x = item_of(p, D, it, rh);
    const RunInfo& ru = D.runs[x.run];
    const int nq = ru.nrows * p.group;
    const int rel = it - ib;
    const int b = rel & 1;
    const uint32_t par = (uint32_t)rel & 1u;
    if (!mbar_wait(&bars.posted[b], (uint32_t)(rel >> 1) & 1u, p.err_flag)) return;
    umma::fence_after_sync();
    const uint32_t tA = tl + (uint32_t)(b * kBufCols);          // consumer warp q
    const uint32_t tB = tA + kHalfCols;                          // consumer warp q + 4
    uint32_t mlA[4], mlB[4];
    umma::tmem_ld4(tA + 64, mlA);
    umma::tmem_ld4(tB + 64, mlB);
    umma::tmem_ld_wait();
    if (rel > 0 && !mbar_wait(bars.done, par ^ 1u, p.err_flag)) return;
    if (c == 0) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int row = gq + 8 * hr;
        ml_buf[(q * 16 + row) * 2 + 0] = __uint_as_float(mlA[2 * hr]);
        ml_buf[(q * 16 + row) * 2 + 1] = __uint_as_float(mlA[2 * hr + 1]);
        ml_buf[((q + 4) * 16 + row) * 2 + 0] = __uint_as_float(mlB[2 * hr]);
        ml_buf[((q + 4) * 16 + row) * 2 + 1] = __uint_as_float(mlB[2 * hr + 1]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.pub);
    if (!mbar_wait(bars.pub, par, p.err_flag)) return;
    float M[2], aA[2], aB[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int row = gq + 8 * hr;
      M[hr] = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M[hr] = fmaxf(M[hr], ml_buf[(w * 16 + row) * 2]);
      const float mA = __uint_as_float(mlA[2 * hr]), mB = __uint_as_float(mlB[2 * hr]);
      aA[hr] = mA == -INFINITY ? 0.f : fast_exp2(mA - M[hr]);
      aB[hr] = mB == -INFINITY ? 0.f : fast_exp2(mB - M[hr]);
    }
    // fold: TMEM column f of a consumer lane holds o[f / 4][f % 4]
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t xa[16], xb[16];
      umma::tmem_ld16(tA + 16 * k, xa);
      umma::tmem_ld16(tB + 16 * k, xb);
      umma::tmem_ld_wait();
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = 4 * u + j, hr = j >> 1;
          v[j] = __fmaf_rn(aB[hr], __uint_as_float(xb[i]), __fmul_rn(aA[hr], __uint_as_float(xa[i])));
        }
        fold[(q * 16 + 4 * k + u) * 32 + lane] = make_float4(v[0], v[1], v[2], v[3]);
      }
    }
    umma::fence_before_sync();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&bars.tmem_free[b]);
      mbar_arrive(bars.folded);
    }
    if (!mbar_wait(bars.folded, par, p.err_flag)) return;
    // final: n-tiles 4q..4q+3 of this lane's fragment, summed over the slots
    {
      float4 acc[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int nt = 4 * q + u;
        float4 a = fold[nt * 32 + lane];
#pragma unroll
        for (int sl = 1; sl < kCombineWarps; ++sl) {
          const float4 t = fold[(sl * 16 + nt) * 32 + lane];
          a.x += t.x;
          a.y += t.y;
          a.z += t.z;
          a.w += t.w;
        }
        acc[u] = a;
      }
      const float vs = FP8 ? __ldg(p.v_scale + x.g) : 1.f;
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int qv = x.mt * 16 + gq + 8 * hr;
        if (qv >= nq) continue;
        const int r = qv / p.group;
        const int h = x.g * p.group + (qv - r * p.group);
        const size_t pslot = ((size_t)(ru.row0 + r) * p.hq + h) * p.max_splits + x.sigma;
        float* orow = p.part_o + pslot * kHeadDim;
        // fragment element j = 2 hr + e sits at column out_col(nt, 2c + e);
        // over nt = 4q..4q+3 those are four consecutive columns
        const float4 o0 = hr ? make_float4(acc[0].z, acc[1].z, acc[2].z, acc[3].z)
                             : make_float4(acc[0].x, acc[1].x, acc[2].x, acc[3].x);
        const float4 o1 = hr ? make_float4(acc[0].w, acc[1].w, acc[2].w, acc[3].w)
                             : make_float4(acc[0].y, acc[1].y, acc[2].y, acc[3].y);
        *reinterpret_cast<float4*>(orow + out_col<FP8>(4 * q, 2 * c)) =
            make_float4(o0.x * vs, o0.y * vs, o0.z * vs, o0.w * vs);
        *reinterpret_cast<float4*>(orow + out_col<FP8>(4 * q, 2 * c + 1)) =
            make_float4(o1.x * vs, o1.y * vs, o1.z * vs, o1.w * vs);
        if (q == 0 && c == 0) {
          const int row = gq + 8 * hr;
          float L = 0.f;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = ml_buf[(w * 16 + row) * 2];
            const float lw = ml_buf[(w * 16 + row) * 2 + 1];
            L += (mw == -INFINITY ? 0.f : fast_exp2(mw - M[hr])) * lw;
          }
          p.part_ml[pslot * 2 + 0] = M[hr];
          p.part_ml[pslot * 2 + 1] = L;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.done);
    if constexpr (MERGE) merge_if_last(p, ru, x, nq, merge_flag);
  }
}

// DEV: the runs and CTA ranges are read from p.dyn (a plan in device mode).
// MERGE: the combiners merge each finished group (p.arrive).
// APPEND: the producer warp stores the rows' new K and V (p.k_rows).
template <bool FP8, bool GEN, bool DEV, bool MERGE, bool APPEND>
__global__ void __launch_bounds__(kThreads, 1) decode_partial_kernel(
    const __grid_constant__ DecodeParams p) {
  const DecodeDyn& D = DEV ? *p.dyn : p.d;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stage_mem = smem;
  float4* fold = reinterpret_cast<float4*>(smem + kRingBytes);
  float* ml_buf = reinterpret_cast<float*>(smem + kRingBytes + kCombBytes);
  int* stage_bad = reinterpret_cast<int*>(ml_buf + kConsumerWarps * 16 * 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stage_bad + kMaxStages);
  int* merge_flag = reinterpret_cast<int*>(tmem_slot + 1);
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(merge_flag + 1) + 7) & ~uintptr_t(7));
  uint64_t* full = bars;
  uint64_t* empty = bars + kMaxStages;
  uint64_t* cbar = bars + 2 * kMaxStages;
  CombBars cb{cbar, cbar + 2, cbar + 4, cbar + 5, cbar + 6};

  const int warp = threadIdx.x >> 5;
  // With the launch data in the parameters, the producer's first page id is
  // brought into L2 while the block sets up: a prefetch reads no value, so
  // it may come before the wait for the previous grid (which can write the
  // table).  Batched decode partial 46.6 -> 45.9 us; not with append, whose
  // producer stores the new rows first (the step measured 0.4 us slower).
  if (!DEV && !APPEND && warp == kProducerWarp && (threadIdx.x & 31) == 0) {
    int ib, ie;
    cta_items(D, ib, ie);
    if (ib < ie) {
      int r = run_of(D, ib);
      const Item x = item_of(p, D, ib, r);
      if (D.runs[x.run].page_table) {
        int klo, khi;
        item_keys(p, D, x, klo, khi);
        prefetch_l2(D.runs[x.run].page_table + (klo >> 8));
      }
    }
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg<FP8>::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], Cfg<FP8>::kSubWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&cb.posted[i], kConsumerWarps);
      mbar_init(&cb.tmem_free[i], kCombineWarps);
    }
    mbar_init(cb.pub, kCombineWarps);
    mbar_init(cb.folded, kCombineWarps);
    mbar_init(cb.done, kCombineWarps);
    fence_mbar_init();
  }
  if (warp == kProducerWarp && (threadIdx.x & 31) == 0) {
    for (int i = 0; i < p.nsrc; ++i) {
      tma_prefetch_desc(&p.maps[i].k);
      tma_prefetch_desc(&p.maps[i].v);
    }
  }
  if (warp == kCombineWarp0) umma::tmem_alloc(tmem_slot, kTmemCols);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  allow_next_grid();
  wait_prior_grid();
  if (warp < kCombineWarp0) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsConsumer));
    consumer<FP8, GEN>(p, D, stage_mem, full, empty, stage_bad, tmem, cb);
  } else if (warp < kProducerWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCombine));
    combiner<FP8, GEN, MERGE>(p, D, tmem, fold, ml_buf, merge_flag, cb);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsProducer));
    if (warp == kProducerWarp) producer<FP8, APPEND>(p, D, stage_mem, full, empty, stage_bad);
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == kCombineWarp0) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- merge
// One warp per (row, head): lane s holds split s's (m, l); lanes own 4
// consecutive head-dim elements of the output.  Fixed summation order.
// DEV: the runs are read from p.dyn (a plan in device mode).
template <bool DEV>
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ MergeParams p) {
  allow_next_grid();
  wait_prior_grid();
  const MergeDyn& D = DEV ? *p.dyn : p.d;
  const int wid = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= D.rows * p.hq) return;
  const int row = wid / p.hq;
  const int h = wid - row * p.hq;
  int ri = 0;
  if (DEV) {
    // runs in device memory: 32 runs' first rows per round of loads; the
    // row's run is the last whose first row is at or before it
    for (int base = 0; base < D.nruns; base += 32) {
      const int i = base + lane;
      const unsigned m = __ballot_sync(0xffffffffu, i < D.nruns && D.runs[i].row0 <= row);
      if (m) ri = base + 31 - __clz(m);
      if (m != 0xffffffffu) break;
    }
  } else {
    while (ri + 1 < D.nruns && D.runs[ri + 1].row0 <= row) ++ri;
  }
  const int nsplit = D.runs[ri].nsplit;
  const size_t slot0 = ((size_t)row * p.hq + h) * p.max_splits;
  // Every slot below nsplit was written by the partial kernel (an empty split
  // holds o = 0 with weight 0).  Every split's o chunk is loaded together
  // with the (m, l) pairs, before the reductions that need them, so a merge
  // waits for one round of loads.
  static_assert(kMaxSplits == 32, "one load per split");
  merge_vector<kMaxSplits, false>(p.part_o + slot0 * kHeadDim, p.part_ml + slot0 * 2, nsplit,
                                  p.out + ((size_t)row * p.hq + h) * kHeadDim,
                                  p.lse ? p.lse + (size_t)row * p.hq + h : nullptr);
}

template <bool FP8, bool GEN, bool DEV, bool MERGE, bool APPEND>
cudaError_t launch_partial(const DecodeParams& p, int grid, cudaStream_t s) {
  static PerDeviceOnce configured;
  cudaError_t e = configured.run([] {
    // The register split only works if the block launches with at least the
    // registers it hands out; otherwise setmaxnreg.inc would wait forever.
    cudaFuncAttributes attr;
    cudaError_t r = cudaFuncGetAttributes(&attr, decode_partial_kernel<FP8, GEN, DEV, MERGE, APPEND>);
    if (r != cudaSuccess) return r;
    if (attr.numRegs * kThreads < 128 * (2 * kRegsConsumer + kRegsCombine + kRegsProducer))
      return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(decode_partial_kernel<FP8, GEN, DEV, MERGE, APPEND>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  e =
      launch_pdl(decode_partial_kernel<FP8, GEN, DEV, MERGE, APPEND>, dim3(grid), dim3(kThreads), kSmemBytes, s, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool DEV>
cudaError_t launch_partial_dev(const DecodeParams& p, bool fp8, int grid, cudaStream_t s) {
  // Rows with ancestor masks take the general instantiation, so the plain
  // causal calls keep their own kernel's code.
  if (p.anc)
    return fp8 ? launch_partial<true, true, DEV, false, false>(p, grid, s)
               : launch_partial<false, true, DEV, false, false>(p, grid, s);
  if (p.k_rows)
    return fp8 ? launch_partial<true, false, DEV, false, true>(p, grid, s)
               : launch_partial<false, false, DEV, false, true>(p, grid, s);
  return fp8 ? launch_partial<true, false, DEV, false, false>(p, grid, s)
             : launch_partial<false, false, DEV, false, false>(p, grid, s);
}

}  // namespace

// The launch shape comes from the parameters' own copy of the dynamic data
// (p.d), which a device-mode plan keeps fixed from step to step.
cudaError_t launch_decode_partial(const DecodeParams& p, bool fp8, int grid, cudaStream_t s) {
  if (grid <= 0 || p.d.n_items == 0) return cudaSuccess;
  // The merge in the kernel is built for plain causal rows in parameter mode.
  if (p.k_rows && p.anc) return cudaErrorInvalidValue;   // append has no tree rows
  if (p.arrive) {
    if (p.anc || p.dyn || !p.out) return cudaErrorInvalidValue;
    if (p.k_rows)
      return fp8 ? launch_partial<true, false, false, true, true>(p, grid, s)
                 : launch_partial<false, false, false, true, true>(p, grid, s);
    return fp8 ? launch_partial<true, false, false, true, false>(p, grid, s)
               : launch_partial<false, false, false, true, false>(p, grid, s);
  }
  return p.dyn ? launch_partial_dev<true>(p, fp8, grid, s)
               : launch_partial_dev<false>(p, fp8, grid, s);
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t s) {
  const int warps = p.d.rows * p.hq;
  if (warps == 0) return cudaSuccess;
  return p.dyn ? launch_pdl(merge_kernel<true>, dim3((warps + 7) / 8), dim3(256), 0, s, p)
               : launch_pdl(merge_kernel<false>, dim3((warps + 7) / 8), dim3(256), 0, s, p);
}

}  // namespace tfpa
