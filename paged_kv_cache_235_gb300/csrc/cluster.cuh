// Thread-block cluster helpers: a cluster launch, the cluster barrier, and
// distributed shared memory (addresses in another CTA of the cluster, stores
// there, and mbarrier arrivals there).
#pragma once

#include "common.cuh"

namespace tfpa {

// As launch_pdl, in clusters of `cluster` CTAs along x.
template <typename P>
cudaError_t launch_pdl_cluster(void (*kernel)(P), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t s, const P& p, int cluster) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster executes this the same number of
// times.  It orders each thread's earlier shared-memory writes (barrier
// initialisation, partial results) before the other CTAs' later accesses,
// and no CTA passes it, and so none exits, before all have arrived.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of the same offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                              uint32_t d) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b),
               "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void st_cluster_f2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1,%2};" ::"r"(addr), "f"(a), "f"(b)
               : "memory");
}

// Arrival, with release at cluster scope, on an mbarrier of another CTA of
// the cluster (`cluster_addr` from mapa_shared).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// As mbar_wait, acquiring at cluster scope: what other CTAs' threads wrote
// before their release arrivals is visible after it returns true.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, int32_t* err) {
  const uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((++n & 255u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
      flag_error(err, kErrTimeout);
      return false;
    }
  }
}

}  // namespace tfpa
