// tfpa_decode_static: decode with the split-K scratch held in a file-scope
// device array, for callers that cannot allocate device memory themselves.
//
// The array is a fixed part of the library image: every device that loads
// the library keeps it until the process exits.  Its device address is looked
// up (cudaGetSymbolAddress, with the device current) on the first call made
// in a device's context, and again only if that context has been replaced
// (after a cudaDeviceReset the module is loaded anew and the array may move).
// The host never passes the array's name to a kernel: in host code that name
// is only a host-side stand-in.
#include <cudaTypedefs.h>

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
struct StaticAddr {
  unsigned long long ctx_id = 0;   // the context the address was taken in (0: none yet)
  float* addr = nullptr;
};
StaticAddr g_static_addr[kMaxDevices];

// Driver calls that identify the current context (cuCtxGetId gives an id
// unique within the process, so a replaced context never matches).
struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};
const CtxFns& ctx_fns() {
  static const CtxFns f = [] {
    CtxFns r;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      r.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      r.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    return r;
  }();
  return f;
}

// Id of the current context, 0 if there is none yet.
int current_ctx_id(unsigned long long* id) {
  const CtxFns& f = ctx_fns();
  if (!f.get_current || !f.get_id) return TFPA_ECUDA;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS) return TFPA_ECUDA;
  *id = 0;
  if (ctx && f.get_id(ctx, id) != CUDA_SUCCESS) return TFPA_ECUDA;
  return TFPA_OK;
}

// Device address of the array on the current device.
int static_scratch_address(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TFPA_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return TFPA_EDEVICE;
  std::lock_guard<std::mutex> lock(g_static_mu);
  unsigned long long id = 0;
  int e = current_ctx_id(&id);
  if (e != TFPA_OK) return e;
  StaticAddr& a = g_static_addr[dev];
  if (id == 0 || id != a.ctx_id || !a.addr) {
    // cudaGetSymbolAddress makes the device's primary context current if
    // no context is yet, so the id is read again after it.
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return TFPA_ECUDA;
    if ((e = current_ctx_id(&id)) != TFPA_OK) return e;
    a.ctx_id = id;
    a.addr = static_cast<float*>(p);
  }
  *out = a.addr;
  return TFPA_OK;
}

}  // namespace

extern "C" int tfpa_decode_static(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                                  const void* q, const int32_t* row_seg,
                                  const int32_t* row_pos, int32_t rows, float softmax_scale,
                                  void* out, float* lse, cudaStream_t stream) {
  if (!cache || cache->hq < 1) return TFPA_EINVAL;
  // One row needs hq * TFPA_MAX_SPLITS slots; larger head counts do not fit
  // (checked before the product is formed, so no head count overflows it).
  if (cache->hq > kStaticSlots / TFPA_MAX_SPLITS) return TFPA_ECAPACITY;
  const int32_t per_row = cache->hq * TFPA_MAX_SPLITS;
  float* base = nullptr;
  const int e = static_scratch_address(&base);
  if (e != TFPA_OK) return e;
  tfpa_scratch sc;
  sc.part_o = base;
  sc.part_ml = base + (size_t)kStaticSlots * tfpa::kHeadDim;
  sc.cap_rows = kStaticSlots / per_row;
  sc.max_splits = TFPA_MAX_SPLITS;
  sc.arrive = nullptr;   // the separate merge launch
  return tfpa_decode(cache, segs, nseg, q, row_seg, row_pos, rows, softmax_scale, &sc, out, lse,
                     stream);
}
