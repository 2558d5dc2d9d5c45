// KV write: new rows' K and V into their pages or slab, bf16 copy or e4m3
// quantisation (TensorFold PR #1373, "What changes": the page-run layout the
// KV store kernels write).
//
// One 16-thread group per (row, kv head); each thread moves 8 elements
// (16 bytes of bf16 in; 16 bytes of bf16 or 8 bytes of e4m3 out).  The page
// is looked up once per (row, head).
#include <cuda_fp8.h>

#include "common.cuh"
#include "params.h"

namespace tfpa {

__global__ void __launch_bounds__(256) write_kv_kernel(const __grid_constant__ WriteParams p) {
  allow_next_grid();
  wait_prior_grid();
  const int gid = blockIdx.x * 16 + (threadIdx.x >> 4);  // (row, head) pair
  const int t = threadIdx.x & 15;                          // 8-element slice
  if (gid >= p.rows * p.hkv) return;
  const int row = gid / p.hkv;
  const int g = gid - row * p.hkv;
  int ri = 0;
  while (ri + 1 < p.nruns && p.runs[ri + 1].row0 <= row) ++ri;
  const WriteRun& run = p.runs[ri];
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
  const size_t src = ((size_t)row * p.hkv + g) * kHeadDim + t * 8;
  const uint4 kv = *reinterpret_cast<const uint4*>(p.k_rows + src);
  const uint4 vv = *reinterpret_cast<const uint4*>(p.v_rows + src);
  if (!p.fp8) {
    __nv_bfloat16* kd = static_cast<__nv_bfloat16*>(run.k_dst) + dst_row * kHeadDim + t * 8;
    __nv_bfloat16* vd = static_cast<__nv_bfloat16*>(run.v_dst) + dst_row * kHeadDim + t * 8;
    *reinterpret_cast<uint4*>(kd) = kv;
    *reinterpret_cast<uint4*>(vd) = vv;
    return;
  }
  const float ks = __ldg(p.k_scale + g);
  const float vs = __ldg(p.v_scale + g);
  auto quant8 = [](const uint4& in, float s) {
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t out[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = __uint_as_float(w[i] << 16);
      const float hi = __uint_as_float(w[i] & 0xFFFF0000u);
      // value / scale rounded to float32 (IEEE division), then e4m3 RNE, saturating
      const float2 f = make_float2(__fdiv_rn(lo, s), __fdiv_rn(hi, s));
      const __nv_fp8x2_storage_t b = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      if (i & 1)
        out[i >> 1] |= (uint32_t)b << 16;
      else
        out[i >> 1] = (uint32_t)b;
    }
    return make_uint2(out[0], out[1]);
  };
  uint8_t* kd = static_cast<uint8_t*>(run.k_dst) + dst_row * kHeadDim + t * 8;
  uint8_t* vd = static_cast<uint8_t*>(run.v_dst) + dst_row * kHeadDim + t * 8;
  *reinterpret_cast<uint2*>(kd) = quant8(kv, ks);
  *reinterpret_cast<uint2*>(vd) = quant8(vv, vs);
}

cudaError_t launch_write_kv(const WriteParams& p, cudaStream_t s) {
  const int pairs = p.rows * p.hkv;
  const int grid = (pairs + 15) / 16;
  if (grid == 0) return cudaSuccess;
  return launch_pdl(write_kv_kernel, dim3(grid), dim3(256), 0, s, p);
}

}  // namespace tfpa
