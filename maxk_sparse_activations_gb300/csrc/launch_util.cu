// Grid sizing for the persistent kernels: one cache entry per (device, kernel).
#include <mutex>

#include "launch.h"

namespace rtopk {
namespace {

struct Entry {
  int device;
  const void* kernel;
  int threads;
  size_t smem;
  int cluster;  // 0: plain blocks; else CTAs per cluster (and `blocks` counts clusters)
  int blocks;
};
constexpr int kMaxEntries = 256;
Entry g_cache[kMaxEntries];
int g_used = 0;
std::mutex g_mu;

}  // namespace

int persistent_blocks(const void* kernel, int threads, size_t smem, int64_t blocks_needed) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  int per_gpu = 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < g_used; ++i) {
      if (g_cache[i].device == dev && g_cache[i].kernel == kernel && g_cache[i].threads == threads &&
          g_cache[i].smem == smem && g_cache[i].cluster == 0) {
        per_gpu = g_cache[i].blocks;
        break;
      }
    }
  }
  if (per_gpu == 0) {
    int sms = 0, occ = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem) != cudaSuccess)
      return 0;
    per_gpu = sms * (occ > 0 ? occ : 1);
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_used < kMaxEntries) g_cache[g_used++] = Entry{dev, kernel, threads, smem, 0, per_gpu};
  }
  if (blocks_needed < 1) blocks_needed = 1;
  return int(blocks_needed < per_gpu ? blocks_needed : per_gpu);
}

int persistent_clusters(const void* kernel, int threads, int cluster, int64_t clusters_needed) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  int per_gpu = 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < g_used; ++i) {
      if (g_cache[i].device == dev && g_cache[i].kernel == kernel && g_cache[i].threads == threads &&
          g_cache[i].cluster == cluster) {
        per_gpu = g_cache[i].blocks;
        break;
      }
    }
  }
  if (per_gpu == 0) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(unsigned(cluster));
    cfg.blockDim = dim3(unsigned(threads));
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) return 0;
    per_gpu = n > 0 ? n : 0;
    if (per_gpu == 0) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_used < kMaxEntries) g_cache[g_used++] = Entry{dev, kernel, threads, 0, cluster, per_gpu};
  }
  if (clusters_needed < 1) clusters_needed = 1;
  return int(clusters_needed < per_gpu ? clusters_needed : per_gpu);
}

}  // namespace rtopk
