// Causal prompt-chunk attention over a paged prefix on tcgen05/TMEM tiles
// (TensorFold PR #2011, "hpattn_p256_kernel": the page size a compile-time
// 256, a key tile's page looked up once; PR #1373, "What changes": the
// prompt tiles read pages through the page table, else the slab).
//
// One CTA per work tile = (run, kv head g, pair of query heads of g, 128
// rows).  One online-softmax pass over key tiles of 128 keys aligned to
// absolute positions, so a row's result never depends on how the rows are
// sliced into launches or tiles.
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
//               max/sum, P written back over S as bf16, O rescaled in TMEM
//               only when the running max grows by more than 2^8.
// TMEM (512 columns): S_A [0,128) O_A [128,256) S_B [256,384) O_B [384,512).
#include "common.cuh"
#include "params.h"
#include "tcgen05.cuh"

namespace tfpa {
namespace {

constexpr int kTileRows = 128;
constexpr int kTileKeys = 128;
constexpr int kThreads = 384;
constexpr int kOffQ = 0;                 // 2 heads x [128 rows][128] bf16 = 64 KB
constexpr int kOffK = 65536;             // 2 stages x 32 KB
constexpr int kOffV = 131072;            // 2 stages x 32 KB
constexpr int kOffBar = 196608;
constexpr int kSmemBytes = kOffBar + 256 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

__device__ __forceinline__ uint32_t col_s(int hh) { return hh ? 256u : 0u; }
__device__ __forceinline__ uint32_t col_o(int hh) { return hh ? 384u : 128u; }

struct Tile {
  int run, g, hp, t;
};

// Tiles are numbered heaviest first: the row-tile index is the slowest digit
// and runs from the last (longest causal range) to the first.
__device__ __forceinline__ Tile tile_of(const PrefillParams& p, int i) {
  int r = 0;
  while (r + 1 < p.nruns && p.runs[r + 1].item0 <= i) ++r;
  const RunInfo& ru = p.runs[r];
  const int local = i - ru.item0;
  const int npairs = (p.group + 1) >> 1;
  const int pairs_total = p.hkv * npairs;
  const int ntr = (ru.nrows + kTileRows - 1) / kTileRows;
  const int t_rev = local / pairs_total;
  const int gp = local - t_rev * pairs_total;
  Tile x;
  x.run = r;
  x.g = gp / npairs;
  x.hp = gp - x.g * npairs;
  x.t = ntr - 1 - t_rev;
  return x;
}

struct TileGeom {
  int row_lo;      // first row of the tile, relative to the run
  int nrows;       // valid rows in the tile
  int kend;        // keys [0, kend) are read
  int nkt;         // key tiles
};

__device__ __forceinline__ TileGeom geom_of(const RunInfo& ru, const Tile& x) {
  TileGeom gm;
  gm.row_lo = x.t * kTileRows;
  gm.nrows = min(kTileRows, ru.nrows - gm.row_lo);
  const int maxpos = ru.pos0 + gm.row_lo + gm.nrows - 1;
  gm.kend = min(ru.seq_len, maxpos + 1);
  gm.nkt = (gm.kend + kTileKeys - 1) / kTileKeys;
  return gm;
}

// Page id of key tile j (paged runs), or -1 if it is outside the pool.
__device__ __forceinline__ int tile_page(const PrefillParams& p, const RunInfo& ru, int j) {
  const int pid = __ldg(ru.page_table + ((j * kTileKeys) >> 8));
  return (unsigned)pid < (unsigned)p.num_pages ? pid : -1;
}

__device__ void producer(const PrefillParams& p, const RunInfo& ru, const Tile& x,
                         const TileGeom& gm, uint8_t* smem, uint64_t* q_full, uint64_t* k_full,
                         uint64_t* k_empty, uint64_t* v_full, uint64_t* v_empty,
                         volatile int* abort) {
  const CUtensorMap* mk = &p.maps[ru.src].k;
  const CUtensorMap* mv = &p.maps[ru.src].v;
  const int h0 = x.g * p.group + 2 * x.hp;
  mbar_arrive_expect_tx(q_full, 65536);
  for (int hh = 0; hh < 2; ++hh)
    for (int rg = 0; rg < 2; ++rg)
      tma_load_3d(smem + kOffQ + hh * 32768 + rg * 16384, &p.qmap, rg * 64, h0 + hh,
                  ru.row0 + gm.row_lo, q_full);
  int cached_page = -1, cached_pid = 0;
  int issued_k = 0, issued_v = 0;
  for (int j = 0; j < gm.nkt; ++j) {
    const int s = j & 1;
    const uint32_t ph = (j >> 1) & 1;
    const int kt = j * kTileKeys;
    int y;
    if (ru.page_table) {
      const int page = kt >> 8;
      if (page != cached_page) {          // one lookup per page
        cached_pid = __ldg(ru.page_table + page);
        cached_page = page;
        if ((unsigned)cached_pid >= (unsigned)p.num_pages) {
          flag_error(p.err_flag, kErrBadPage);
          cached_pid = 0;                  // read a valid page; its keys are masked
        }
      }
      y = (cached_pid * p.hkv + x.g) * kPage + (kt & (kPage - 1));
    } else {
      y = x.g * ru.slab_cap + kt;
    }
    if (!mbar_wait_or_abort(&k_empty[s], ph ^ 1, p.err_flag, abort)) break;
    mbar_arrive_expect_tx(&k_full[s], 32768);
    tma_load_2d(smem + kOffK + s * 32768, mk, 0, y, &k_full[s]);
    tma_load_2d(smem + kOffK + s * 32768 + 16384, mk, 64, y, &k_full[s]);
    issued_k = j + 1;
    if (!mbar_wait_or_abort(&v_empty[s], ph ^ 1, p.err_flag, abort)) break;
    mbar_arrive_expect_tx(&v_full[s], 32768);
    tma_load_2d(smem + kOffV + s * 32768, mv, 0, y, &v_full[s]);
    tma_load_2d(smem + kOffV + s * 32768 + 16384, mv, 64, y, &v_full[s]);
    issued_v = j + 1;
  }
  if (*abort) {
    // Let this CTA's loads in flight land before it exits.
    for (int j = max(0, issued_k - 2); j < issued_k; ++j)
      mbar_wait(&k_full[j & 1], (j >> 1) & 1, p.err_flag);
    for (int j = max(0, issued_v - 2); j < issued_v; ++j)
      mbar_wait(&v_full[j & 1], (j >> 1) & 1, p.err_flag);
  }
}

// Zero rows [z0, 128) of a V tile (both 64-column halves) in shared memory:
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

__device__ void mma_issuer(const PrefillParams& p, const RunInfo& ru, const TileGeom& gm,
                           uint8_t* smem, uint32_t tmem, uint64_t* q_full, uint64_t* k_full,
                           uint64_t* k_empty, uint64_t* v_full, uint64_t* v_empty,
                           uint64_t* s_full, uint64_t* p_ready, uint64_t* o_final,
                           uint64_t* drain, volatile int* abort) {
  const int lane = threadIdx.x & 31;
  const bool leader = lane == 0;
  constexpr uint32_t kIdescQK = umma::idesc_f16(128, 128, true, false);
  constexpr uint32_t kIdescPV = umma::idesc_f16(128, 128, true, true);
  const uint32_t qb = smem_u32(smem + kOffQ);
  const uint32_t kb = smem_u32(smem + kOffK);
  const uint32_t vb = smem_u32(smem + kOffV);

  auto issue_s = [&](int hh, int s) {     // S_hh = Q_hh K_s^T
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
      const uint64_t a = umma::smem_desc_sw128(qb + hh * 32768 + off, 16, 1024);
      const uint64_t b = umma::smem_desc_sw128(kb + s * 32768 + off, 16, 1024);
      umma::mma_ss(tmem + col_s(hh), a, b, kIdescQK, ks > 0 ? 1u : 0u);
    }
  };
  auto issue_pv = [&](int hh, int s, bool acc) {   // O_hh (+)= P_hh V_s
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t b = umma::smem_desc_sw128(vb + s * 32768 + kk * 2048, 16384, 1024);
      umma::mma_ts(tmem + col_o(hh), tmem + col_s(hh) + kk * 8, b, kIdescPV,
                   (acc || kk > 0) ? 1u : 0u);
    }
  };

  bool ok = mbar_wait_or_abort(q_full, 0, p.err_flag, abort) &&
            mbar_wait_or_abort(&k_full[0], 0, p.err_flag, abort);
  if (ok) {
    umma::fence_after_sync();
    if (leader) {
      issue_s(0, 0);
      umma::commit(&s_full[0]);
      issue_s(1, 0);
      umma::commit(&s_full[1]);
      umma::commit(&k_empty[0]);
    }
    __syncwarp();
  }
  for (int j = 0; ok && j < gm.nkt; ++j) {
    const int s = j & 1;
    const uint32_t ph = (j >> 1) & 1;
    const int s1 = (j + 1) & 1;
    const uint32_t ph1 = ((j + 1) >> 1) & 1;
    const bool more = j + 1 < gm.nkt;
    if (!(ok = mbar_wait_or_abort(&v_full[s], ph, p.err_flag, abort))) break;
    const int kt = j * kTileKeys;
    int z0 = kTileKeys;
    if (kt + kTileKeys > ru.seq_len) z0 = ru.seq_len - kt;
    if (ru.page_table && tile_page(p, ru, j) < 0) z0 = 0;
    if (z0 < kTileKeys) zero_v_rows(smem + kOffV + s * 32768, z0, lane);
    // head A
    if (!(ok = mbar_wait_or_abort(&p_ready[0], j & 1, p.err_flag, abort))) break;
    umma::fence_after_sync();
    if (leader) issue_pv(0, s, j > 0);
    if (more) {
      if (!(ok = mbar_wait_or_abort(&k_full[s1], ph1, p.err_flag, abort))) break;
      umma::fence_after_sync();
      if (leader) {
        issue_s(0, s1);
        umma::commit(&s_full[0]);
      }
    }
    // head B
    if (!(ok = mbar_wait_or_abort(&p_ready[1], j & 1, p.err_flag, abort))) break;
    umma::fence_after_sync();
    if (leader) {
      issue_pv(1, s, j > 0);
      if (more) {
        issue_s(1, s1);
        umma::commit(&s_full[1]);
        umma::commit(&k_empty[s1]);
      }
      umma::commit(&v_empty[s]);
    }
    __syncwarp();
  }
  if (leader) {
    if (ok) {
      umma::commit(o_final);
    } else {
      umma::commit(drain);          // let issued MMAs finish before TMEM is freed
      mbar_wait(drain, 0, p.err_flag);
    }
  }
  __syncwarp();
}

__device__ void softmax_role(const PrefillParams& p, const RunInfo& ru, const Tile& x,
                             const TileGeom& gm, int hh, uint32_t tmem, uint64_t* s_full,
                             uint64_t* p_ready, uint64_t* o_final, volatile int* abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = 32 * (warp & 3) + lane;                 // row of the tile = TMEM lane
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  const uint32_t tS = tmem + lane_off + col_s(hh);
  const uint32_t tO = tmem + lane_off + col_o(hh);
  const bool valid = r < gm.nrows;
  const int pos = ru.pos0 + gm.row_lo + (valid ? r : 0);
  const float sl2 = p.scale_log2;
  float m_run = -INFINITY, l = 0.f;
  int cached_page = -1;
  bool page_bad = false;

  for (int j = 0; j < gm.nkt; ++j) {
    if (!mbar_wait_or_abort(&s_full[hh], j & 1, p.err_flag, abort)) return;
    umma::fence_after_sync();
    const int kt = j * kTileKeys;
    if (ru.page_table && (kt >> 8) != cached_page) {
      cached_page = kt >> 8;
      page_bad = tile_page(p, ru, j) < 0;
    }
    const int lim = page_bad ? -1 : pos - kt;            // key kt+i visible iff i <= lim
    const bool full_tile = lim >= kTileKeys - 1;
    uint32_t sv[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) umma::tmem_ld32(tS + 32 * c, sv[c]);
    umma::tmem_ld_wait();
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 128; ++i) {
      const float v = __uint_as_float(sv[i >> 5][i & 31]);
      mx = (full_tile || i <= lim) ? fmaxf(mx, v) : mx;
    }
    mx = mx * sl2;
    const float m_new = fmaxf(m_run, mx);
    const bool resc = m_new > m_run + kRescaleThreshold;
    float alpha = 1.f;
    if (resc) {
      alpha = fast_exp2(m_run - m_new);
      l *= alpha;
      m_run = m_new;
    }
    const float base = m_run == -INFINITY ? 0.f : m_run;
    // p = 2^(s*scale - m), packed to bf16 pairs in place (pair k lands in
    // slot k <= 2k, after both of its inputs are read), then written over
    // the first 64 columns of S.
    float rs = 0.f;
#pragma unroll
    for (int k = 0; k < 64; ++k) {
      const int i0 = 2 * k;
      const float s0 =
          (full_tile || i0 <= lim) ? __uint_as_float(sv[i0 >> 5][i0 & 31]) * sl2 : -INFINITY;
      const float s1 = (full_tile || i0 + 1 <= lim)
                           ? __uint_as_float(sv[(i0 + 1) >> 5][(i0 + 1) & 31]) * sl2
                           : -INFINITY;
      const float p0 = fast_exp2(s0 - base);
      const float p1 = fast_exp2(s1 - base);
      rs += p0 + p1;
      sv[k >> 5][k & 31] = pack_bf16x2(p0, p1);
    }
    umma::tmem_st32(tS, sv[0]);
    umma::tmem_st32(tS + 32, sv[1]);
    if (j > 0 && __any_sync(0xffffffffu, resc)) {      // O *= alpha in TMEM
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
    if (lane == 0) mbar_arrive(&p_ready[hh]);
  }
  if (!mbar_wait_or_abort(o_final, 0, p.err_flag, abort)) return;
  umma::fence_after_sync();
  const int h = x.g * p.group + 2 * x.hp + hh;
  const bool write = valid && (2 * x.hp + hh) < p.group;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  uint4* dst = reinterpret_cast<uint4*>(
      p.out + ((size_t)(ru.row0 + gm.row_lo + r) * p.hq + h) * kHeadDim);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t o[32];
    umma::tmem_ld32(tO + 32 * c, o);
    umma::tmem_ld_wait();
    if (write) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 v;
        v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
        v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
        v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
        v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
        dst[4 * c + q] = v;
      }
    }
  }
  if (write && p.lse)
    p.lse[(size_t)(ru.row0 + gm.row_lo + r) * p.hq + h] =
        l > 0.f ? (m_run + log2f(l)) * 0.6931471805599453f : -INFINITY;
}

__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = bars + 3;
  uint64_t* v_full = bars + 5;
  uint64_t* v_empty = bars + 7;
  uint64_t* s_full = bars + 9;
  uint64_t* p_ready = bars + 11;
  uint64_t* o_final = bars + 13;
  uint64_t* drain = bars + 14;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort = reinterpret_cast<volatile int*>(bars + 17);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_ready[i], 4);
    }
    mbar_init(o_final, 1);
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.qmap);
    for (int i = 0; i < p.nsrc; ++i) {
      tma_prefetch_desc(&p.maps[i].k);
      tma_prefetch_desc(&p.maps[i].v);
    }
  }
  if (warp == 1) umma::tmem_alloc(tmem_slot, kTmemCols);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const Tile x = tile_of(p, blockIdx.x);
  const RunInfo& ru = p.runs[x.run];
  const TileGeom gm = geom_of(ru, x);

  if (warp == 0) {
    if (lane == 0) producer(p, ru, x, gm, smem, q_full, k_full, k_empty, v_full, v_empty, abort);
  } else if (warp == 1) {
    mma_issuer(p, ru, gm, smem, tmem, q_full, k_full, k_empty, v_full, v_empty, s_full, p_ready,
               o_final, drain, abort);
  } else if (warp >= 4) {
    softmax_role(p, ru, x, gm, (warp - 4) >> 2, tmem, s_full, p_ready, o_final, abort);
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, bool fp8, int grid, cudaStream_t s) {
  if (fp8) return cudaErrorNotSupported;
  if (grid <= 0) return cudaSuccess;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  prefill_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace tfpa
