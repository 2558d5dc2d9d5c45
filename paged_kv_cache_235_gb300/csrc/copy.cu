// Bulk moves around the hot path: page ids staged into a device page table
// on the stream, and a stream's stored rows saved to or restored from an
// image in memory the GPU can reach (PR #2011 review: page-table staging
// between prompt chunks; save and restore copies, where a kernel writing
// mapped host memory measured faster than per-page copies).  On GB300 a
// pinned host image sits behind NVLink-C2C, so the save is one kernel that
// streams every (page, kv head) block straight to it.
#include "common.cuh"
#include "params.h"

namespace tfpa {

__global__ void __launch_bounds__(256) stage_kernel(const __grid_constant__ StageParams p) {
  allow_next_grid();
  wait_prior_grid();
  for (int i = threadIdx.x; i < p.n; i += blockDim.x) p.table[p.first + i] = p.ids[i];
}

// Block (page, kv head, K or V): the rows of the range inside that page are
// contiguous both in the page block and in the image, so the block moves one
// contiguous span of up to 64 KB in 16-byte pieces, four in flight a thread.
__global__ void __launch_bounds__(256) copy_kernel(const __grid_constant__ CopyParams p) {
  allow_next_grid();
  wait_prior_grid();
  const int which = blockIdx.x & 1;
  const int g = (blockIdx.x >> 1) % p.hkv;
  const int page = p.page0 + (blockIdx.x >> 1) / p.hkv;
  const int lo = max(p.p0, page * kPage), hi = min(p.p1, (page + 1) * kPage);
  if (lo >= hi) return;
  size_t row;
  if (p.page_table) {
    const int pid = __ldg(p.page_table + page);
    if ((unsigned)pid >= (unsigned)p.num_pages) {
      if (threadIdx.x == 0) flag_error(p.err_flag, kErrBadPage);
      return;
    }
    row = ((size_t)pid * p.hkv + g) * kPage + (lo & (kPage - 1));
  } else {
    row = (size_t)g * p.slab_cap + lo;
  }
  uint4* dev = reinterpret_cast<uint4*>(static_cast<uint8_t*>(which ? p.v_base : p.k_base) +
                                        row * p.row_bytes);
  uint4* img = reinterpret_cast<uint4*>(
      p.image + (((size_t)which * p.hkv + g) * (p.p1 - p.p0) + (lo - p.p0)) * p.row_bytes);
  const uint4* src = p.restore ? img : dev;
  uint4* dst = p.restore ? dev : img;
  const int n = (hi - lo) * p.row_bytes / 16;
  int i = threadIdx.x;
  for (; i + 3 * 256 < n; i += 4 * 256) {
    const uint4 a = src[i], b = src[i + 256], c = src[i + 512], d = src[i + 768];
    dst[i] = a;
    dst[i + 256] = b;
    dst[i + 512] = c;
    dst[i + 768] = d;
  }
  for (; i < n; i += 256) dst[i] = src[i];
}

cudaError_t launch_stage(const StageParams& p, cudaStream_t s) {
  if (p.n == 0) return cudaSuccess;
  return launch_pdl(stage_kernel, dim3(1), dim3(256), 0, s, p);
}

cudaError_t launch_copy(const CopyParams& p, int npages, cudaStream_t s) {
  if (npages == 0 || p.p1 <= p.p0) return cudaSuccess;
  return launch_pdl(copy_kernel, dim3(npages * p.hkv * 2), dim3(256), 0, s, p);
}

}  // namespace tfpa
