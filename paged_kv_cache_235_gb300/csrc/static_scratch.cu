// tfpa_decode_static: decode with the split-K scratch held in a file-scope
// device array, for callers that cannot allocate device memory themselves.
//
// The array is a fixed part of the library image: every device that loads
// the library keeps it until the process exits.  Its device address is looked
// up once per device (cudaGetSymbolAddress with that device current) on the
// first call made on that device; the host never passes the array's name to
// a kernel, since in host code that name is only a host-side stand-in.
#include <mutex>

#include "params.h"
#include "tfpa.h"

namespace {

constexpr int kStaticSlots = TFPA_STATIC_SCRATCH_SLOTS;   // (row, head, split) slots
constexpr size_t kStaticFloats = (size_t)kStaticSlots * (tfpa::kHeadDim + 2);

// o partials ([slots][128]) followed by (m, l) pairs ([slots][2]).
static __device__ __align__(256) float g_static_scratch[kStaticFloats];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
float* g_static_addr[kMaxDevices] = {};

// Device address of the array on the current device (set up on first use).
int static_scratch_address(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TFPA_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return TFPA_EDEVICE;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return TFPA_ECUDA;
    g_static_addr[dev] = static_cast<float*>(p);
  }
  *out = g_static_addr[dev];
  return TFPA_OK;
}

}  // namespace

extern "C" int tfpa_decode_static(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                                  const void* q, const int32_t* row_seg,
                                  const int32_t* row_pos, int32_t rows, float softmax_scale,
                                  void* out, float* lse, cudaStream_t stream) {
  if (!cache || cache->hq < 1) return TFPA_EINVAL;
  // One row needs hq * TFPA_MAX_SPLITS slots; larger head counts do not fit.
  const int32_t per_row = cache->hq * TFPA_MAX_SPLITS;
  if (per_row > kStaticSlots) return TFPA_ECAPACITY;
  float* base = nullptr;
  const int e = static_scratch_address(&base);
  if (e != TFPA_OK) return e;
  tfpa_scratch sc;
  sc.part_o = base;
  sc.part_ml = base + (size_t)kStaticSlots * tfpa::kHeadDim;
  sc.cap_rows = kStaticSlots / per_row;
  sc.max_splits = TFPA_MAX_SPLITS;
  return tfpa_decode(cache, segs, nseg, q, row_seg, row_pos, rows, softmax_scale, &sc, out, lse,
                     stream);
}
