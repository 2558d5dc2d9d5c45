// KV write: new rows' K and V into their pages or slab, bf16 copy or e4m3
// quantisation (TensorFold PR #1373, "What changes": the page-run layout the
// KV store kernels write), optionally with K rotated by its rotary position
// first; and keep: stored rows copied between positions of a stream (the
// PR #1373 review lists "rope stores and keep" among the paged store's
// checks).
//
// Write: one 16-thread group per (row, kv head); each thread moves 8
// elements (16 bytes of bf16 in; 16 bytes of bf16 or 8 bytes of e4m3 out).
// The page is looked up once per (row, head).  The rotation pairs element i
// with i + 64 (rotate-half), so a thread also reads its partner's 8
// elements; every product and sum is rounded on its own (no fused
// multiply-add), so the stored code is a function of the inputs alone.
#include <cuda_fp8.h>

#include "common.cuh"
#include "kvstore.cuh"
#include "params.h"

namespace tfpa {

namespace {

__device__ __forceinline__ uint4 pack8_bf16(const float (&x)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace

// DEV: the runs are read from p.dyn (a plan in device mode).
template <bool DEV>
__global__ void __launch_bounds__(256) write_kv_kernel(const __grid_constant__ WriteParams p) {
  allow_next_grid();
  wait_prior_grid();
  const WriteDyn& D = DEV ? *p.dyn : p.d;
  const int gid = blockIdx.x * 16 + (threadIdx.x >> 4);  // (row, head) pair
  const int t = threadIdx.x & 15;                          // 8-element slice
  const bool live = gid < D.rows * p.hkv;
  const int row = gid / p.hkv;
  const int g = gid - row * p.hkv;
  int ri = 0;
  if (DEV) {
    // runs in device memory: each 16-thread group reads 16 runs' first
    // rows per round (every lane of the warp takes part in the ballots);
    // the row's run is the last whose first row is at or before it
    const int sh = threadIdx.x & 16;
    for (int base = 0; base < D.nruns; base += 16) {
      const int i = base + t;
      const unsigned m =
          (__ballot_sync(0xffffffffu, i < D.nruns && D.runs[i].row0 <= row) >> sh) & 0xFFFFu;
      if (m) ri = base + 31 - __clz(m);
    }
  } else if (live) {
    while (ri + 1 < D.nruns && D.runs[ri + 1].row0 <= row) ++ri;
  }
  if (!live) return;
  const WriteRun& run = D.runs[ri];
  const int pos = run.pos0 + (row - run.row0);

  size_t dst_row;  // element index of the destination row
  if (run.page_table) {
    const int pid = __ldg(run.page_table + (pos >> 8));
    if ((unsigned)pid >= (unsigned)p.num_pages) {
      if (t == 0) flag_error(p.err_flag, kErrBadPage);
      return;
    }
    dst_row = ((size_t)pid * p.hkv + g) * kPage + (pos & (kPage - 1));
  } else {
    dst_row = (size_t)g * run.slab_cap + pos;
  }
  const size_t src_row = ((size_t)row * p.hkv + g) * kHeadDim;
  const size_t src = src_row + t * 8;
  const uint4 kv = *reinterpret_cast<const uint4*>(p.k_rows + src);
  const uint4 vv = *reinterpret_cast<const uint4*>(p.v_rows + src);

  float kf[8];
  unpack8(kv, kf);
  if (p.rope_cos) {
    const int rpos = p.rope_pos ? __ldg(p.rope_pos + row) : pos;
    if ((unsigned)rpos >= (unsigned)p.rope_n) {
      if (t == 0) flag_error(p.err_flag, kErrRopeRange);
      return;
    }
    const bool second = t >= 8;                // elements 64.. of the head
    const int i0 = (t & 7) * 8;                // index within the half
    float other[8];
    unpack8(*reinterpret_cast<const uint4*>(p.k_rows + src_row + (second ? i0 : 64 + i0)),
            other);
    const float4* cp = reinterpret_cast<const float4*>(p.rope_cos + (size_t)rpos * 64 + i0);
    const float4* sp = reinterpret_cast<const float4*>(p.rope_sin + (size_t)rpos * 64 + i0);
    const float4 c0 = __ldg(cp), c1 = __ldg(cp + 1), s0 = __ldg(sp), s1 = __ldg(sp + 1);
    const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float a = second ? other[e] : kf[e];   // element i
      const float b = second ? kf[e] : other[e];   // element i + 64
      kf[e] = second ? __fadd_rn(__fmul_rn(b, c[e]), __fmul_rn(a, s[e]))
                     : __fsub_rn(__fmul_rn(a, c[e]), __fmul_rn(b, s[e]));
    }
  }
  if (!p.fp8) {
    __nv_bfloat16* kd = static_cast<__nv_bfloat16*>(run.k_dst) + dst_row * kHeadDim + t * 8;
    __nv_bfloat16* vd = static_cast<__nv_bfloat16*>(run.v_dst) + dst_row * kHeadDim + t * 8;
    *reinterpret_cast<uint4*>(kd) = p.rope_cos ? pack8_bf16(kf) : kv;
    *reinterpret_cast<uint4*>(vd) = vv;
    return;
  }
  float vf[8];
  unpack8(vv, vf);
  uint8_t* kd = static_cast<uint8_t*>(run.k_dst) + dst_row * kHeadDim + t * 8;
  uint8_t* vd = static_cast<uint8_t*>(run.v_dst) + dst_row * kHeadDim + t * 8;
  *reinterpret_cast<uint2*>(kd) = quant8(kf, __ldg(p.k_scale + g));
  *reinterpret_cast<uint2*>(vd) = quant8(vf, __ldg(p.v_scale + g));
}

// Keep: CTA g handles kv head g of every pair.  The pairs' source and
// destination row addresses (K and V) are looked up once into shared memory;
// then every source row is read into shared memory before any destination is
// written, so chains of moves within a call (2 -> 1, 5 -> 2) copy the rows
// as they were.  A pair whose source or destination page id is out of range
// is skipped and flagged.
constexpr int kKeepThreads = 1024;
__global__ void __launch_bounds__(kKeepThreads)
    keep_kernel(const __grid_constant__ KeepParams p) {
  extern __shared__ uint4 stash[];                 // [n][K, V][row_bytes / 16]
  __shared__ uint4* src_row[kMaxKeep][2];
  __shared__ uint4* dst_row[kMaxKeep][2];
  allow_next_grid();
  wait_prior_grid();
  const int g = blockIdx.x;
  const int cpr = p.row_bytes / 16;               // 16-byte chunks per row
  auto row_ptr = [&](const KeepPair& kp, int which, int pos) -> uint4* {
    uint8_t* base;
    size_t idx;
    if (kp.page_table) {
      const int pid = __ldg(kp.page_table + (pos >> 8));
      if ((unsigned)pid >= (unsigned)p.num_pages) return nullptr;
      base = static_cast<uint8_t*>(which ? p.v_pool : p.k_pool);
      idx = ((size_t)pid * p.hkv + g) * kPage + (pos & (kPage - 1));
    } else {
      base = static_cast<uint8_t*>(which ? kp.v_slab : kp.k_slab);
      idx = (size_t)g * kp.slab_cap + pos;
    }
    return reinterpret_cast<uint4*>(base + idx * p.row_bytes);
  };
  for (int i = threadIdx.x; i < 2 * p.n; i += blockDim.x) {
    const KeepPair& kp = p.pairs[i >> 1];
    uint4* s = row_ptr(kp, i & 1, kp.src);
    uint4* d = row_ptr(kp, i & 1, kp.dst);
    if (!s || !d) {
      flag_error(p.err_flag, kErrBadPage);
      s = d = nullptr;
    }
    src_row[i >> 1][i & 1] = s;
    dst_row[i >> 1][i & 1] = d;
  }
  __syncthreads();
  // Each thread issues its (up to) kUnroll loads before any shared store, so
  // they are in flight together rather than one round trip each.
  constexpr int kUnroll = 8;
  const int total = p.n * 2 * cpr;
  for (int i0 = threadIdx.x; i0 < total; i0 += kUnroll * blockDim.x) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * blockDim.x;
      v[u] = make_uint4(0, 0, 0, 0);
      if (i < total) {
        const uint4* s = src_row[i / (2 * cpr)][(i / cpr) & 1];
        if (s) v[u] = s[i % cpr];
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < total) stash[i] = v[u];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    uint4* d = dst_row[i / (2 * cpr)][(i / cpr) & 1];
    if (d) d[i % cpr] = stash[i];
  }
}

cudaError_t launch_write_kv(const WriteParams& p, cudaStream_t s) {
  const int pairs = p.d.rows * p.hkv;
  const int grid = (pairs + 15) / 16;
  if (grid == 0) return cudaSuccess;
  return p.dyn ? launch_pdl(write_kv_kernel<true>, dim3(grid), dim3(256), 0, s, p)
               : launch_pdl(write_kv_kernel<false>, dim3(grid), dim3(256), 0, s, p);
}

cudaError_t launch_keep(const KeepParams& p, cudaStream_t s) {
  if (p.n == 0) return cudaSuccess;
  const int smem = p.n * 2 * p.row_bytes;
  static PerDeviceOnce configured;
  if (smem > 48 * 1024) {
    const cudaError_t e = configured.run([] {
      return cudaFuncSetAttribute(keep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kMaxKeep * 2 * 256);
    });
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(keep_kernel, dim3(p.hkv), dim3(kKeepThreads), smem, s, p);
}

}  // namespace tfpa
