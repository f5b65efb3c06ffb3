// Host-side helpers shared by the C-ABI entry points.
#pragma once
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "tv.h"

namespace tv {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch with or without programmatic dependent launch (the kernel may start
// while the previous kernel on the stream is finishing; it orders itself with
// griddepcontrol.wait).
template <typename... KArgs, typename... Args>
inline void launch_k(bool overlap, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (overlap) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_k with a thread-block cluster of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
inline void launch_k_cluster(bool overlap, int cluster_x, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                             size_t smem, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (overlap) {
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline bool tree_overlap(const tv_tree* t) { return t && (t->flags & TV_TREE_OVERLAP) != 0; }

// Status of the launches just enqueued.  Clears a sticky-free launch error
// so that the next call starts clean.
inline tv_status launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

// Streaming multiprocessors of the current device.
inline int num_sms() {
  static int cached = 0;
  if (cached > 0) return cached;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  cached = n > 0 ? n : 1;
  return cached;
}

inline bool tree_ok(const tv_tree* t) {
  return t && t->n_seq >= 1 && t->n_seq <= TV_MAX_SEQ && t->n_max >= 1 && t->n_max <= TV_MAX_NODES &&
         t->n_total >= t->n_seq && t->n_total <= t->n_seq * t->n_max && t->node_off && t->parent &&
         t->meta && t->status && aligned16(t->node_off) && aligned16(t->parent) && aligned16(t->meta) &&
         aligned16(t->status);
}

}  // namespace tv
