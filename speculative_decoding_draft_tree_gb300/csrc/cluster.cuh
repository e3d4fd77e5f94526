// Thread-block cluster primitives shared by the verification kernels: the CTA's rank, hardware
// cluster barriers and loads from another CTA's shared memory (distributed shared memory).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <map>
#include <mutex>
#include <tuple>

#include "tc_ptx.cuh"

namespace spec {

__device__ __forceinline__ int cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return int(r);
}
__device__ __forceinline__ int cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return int(n);
}
// every thread of every CTA of the cluster; release / acquire order the shared-memory
// accesses on either side
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_addr(const void* p, int rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(tc::smem_u32(p)), "r"(rank));
  return ra;
}
__device__ __forceinline__ float ld_cluster_f32(const void* p, int rank) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr(p, rank)) : "memory");
  return v;
}
__device__ __forceinline__ int ld_cluster_s32(const void* p, int rank) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(cluster_addr(p, rank)) : "memory");
  return v;
}
// the two halves of cluster_sync, for a barrier whose wait comes later
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- host side
// clusters of n CTAs of `threads` threads and `smem` bytes of dynamic shared memory each that
// device `dev` holds at once (0 when none fits), cached per kernel and shape
template <typename K>
inline int active_clusters(K kernel, int dev, int n, int threads, long long smem) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int, int, long long>, int> cache;
  const auto key = std::make_tuple(reinterpret_cast<const void*>(kernel), dev, n, threads, smem);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(n));
  cfg.blockDim = dim3(unsigned(threads));
  cfg.dynamicSmemBytes = size_t(smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(n);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int c = 0;
  if (cudaOccupancyMaxActiveClusters(&c, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    c = 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = c;
  return c;
}


}  // namespace spec
