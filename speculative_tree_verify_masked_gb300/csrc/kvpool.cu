// KV pool ("Parallel requests", "The shared KV pool"): a cache tensor's whole
// window is reserved as virtual addresses, and physical pages are mapped only
// for the rows a sequence writes.  The tensor keeps the shape, dtype and
// strides of a static buffer, so the verify, commit and decode kernels, the
// tensor maps they build and any captured graph see the same addresses and
// produce the same bits.
//
// Host code only: the driver's virtual memory calls are reached through
// runtime driver entry points (no link against the driver library), and each
// call runs with the pool's device current, restoring the caller's device.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <vector>

#include "tv.h"

namespace {

struct Driver {
  PFN_cuMemCreate_v10020 create = nullptr;
  PFN_cuMemRelease_v10020 release = nullptr;
  PFN_cuMemMap_v10020 map = nullptr;
  PFN_cuMemUnmap_v10020 unmap = nullptr;
  PFN_cuMemSetAccess_v10020 set_access = nullptr;
  PFN_cuMemAddressReserve_v10020 reserve = nullptr;
  PFN_cuMemAddressFree_v10020 free_va = nullptr;
  PFN_cuMemGetAllocationGranularity_v10020 granularity = nullptr;
  bool ok = false;
};

template <typename F>
bool entry(const char* name, F& f) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || p == nullptr) {
    cudaGetLastError();
    return false;
  }
  f = reinterpret_cast<F>(p);
  return true;
}

const Driver& driver() {
  static const Driver d = [] {
    Driver x;
    x.ok = entry("cuMemCreate", x.create) && entry("cuMemRelease", x.release) && entry("cuMemMap", x.map) &&
           entry("cuMemUnmap", x.unmap) && entry("cuMemSetAccess", x.set_access) &&
           entry("cuMemAddressReserve", x.reserve) && entry("cuMemAddressFree", x.free_va) &&
           entry("cuMemGetAllocationGranularity", x.granularity);
    return x;
  }();
  return d;
}

CUmemAllocationProp device_prop(int device) {
  CUmemAllocationProp prop{};
  prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
  prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  prop.location.id = device;
  return prop;
}

size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

// The pool's device current for the duration of a call.
struct DeviceScope {
  int prev = -1;
  bool ok = false;
  explicit DeviceScope(int device) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    ok = cudaSetDevice(device) == cudaSuccess;
    if (!ok) cudaGetLastError();
  }
  ~DeviceScope() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

struct Reservation {
  size_t bytes = 0;
  std::vector<CUmemGenericAllocationHandle> page;  // 0: not mapped
};

}  // namespace

struct tv_kv_pool {
  int device = 0;
  size_t page = 0;
  std::mutex mu;
  std::map<uintptr_t, Reservation> res;  // by base address
  size_t committed = 0, reserved = 0;
};

namespace {

// Pages [p0, p1) of the reservation at `base` that some head's rows [0, rows) touch.
template <typename Fn>
void for_row_pages(size_t page, int32_t n_heads, size_t head_stride, size_t row_bytes, int64_t rows, Fn fn) {
  if (rows <= 0) return;
  for (int32_t h = 0; h < n_heads; h++) {
    const size_t lo = static_cast<size_t>(h) * head_stride;
    const size_t hi = lo + static_cast<size_t>(rows) * row_bytes;
    fn(lo / page, (hi + page - 1) / page);
  }
}

tv_status unmap_page(tv_kv_pool* p, uintptr_t base, Reservation& r, size_t i) {
  const Driver& d = driver();
  const CUdeviceptr va = static_cast<CUdeviceptr>(base + i * p->page);
  if (d.unmap(va, p->page) != CUDA_SUCCESS || d.release(r.page[i]) != CUDA_SUCCESS) return TV_ERR_CUDA;
  r.page[i] = 0;
  p->committed -= p->page;
  return TV_OK;
}

bool rows_fit(const Reservation& r, int32_t n_heads, size_t head_stride, size_t row_bytes, int64_t rows) {
  if (n_heads < 1 || head_stride == 0 || row_bytes == 0 || rows < 0) return false;
  if (static_cast<size_t>(rows) * row_bytes > head_stride) return false;
  return static_cast<size_t>(n_heads) * head_stride <= r.bytes;
}

}  // namespace

extern "C" size_t tv_kvpool_page_bytes(int32_t device, size_t page_bytes) {
  const Driver& d = driver();
  if (!d.ok || device < 0) return 0;
  CUmemAllocationProp prop = device_prop(device);
  size_t g = 0;
  if (d.granularity(&g, &prop, CU_MEM_ALLOC_GRANULARITY_MINIMUM) != CUDA_SUCCESS || g == 0) return 0;
  return round_up(page_bytes ? page_bytes : (static_cast<size_t>(2) << 20), g);
}

extern "C" tv_status tv_kvpool_create(int32_t device, size_t page_bytes, tv_kv_pool** pool) {
  if (pool == nullptr || device < 0) return TV_ERR_ARG;
  *pool = nullptr;
  const size_t page = tv_kvpool_page_bytes(device, page_bytes);
  if (page == 0) return TV_ERR_CUDA;
  tv_kv_pool* p = new tv_kv_pool;
  p->device = device;
  p->page = page;
  *pool = p;
  return TV_OK;
}

extern "C" tv_status tv_kvpool_reserve(tv_kv_pool* p, size_t bytes, void** base) {
  if (p == nullptr || base == nullptr || bytes == 0) return TV_ERR_ARG;
  *base = nullptr;
  const Driver& d = driver();
  std::lock_guard<std::mutex> lock(p->mu);
  DeviceScope dev(p->device);
  if (!dev.ok) return TV_ERR_CUDA;
  const size_t size = round_up(bytes, p->page);
  CUdeviceptr va = 0;
  if (d.reserve(&va, size, p->page, 0, 0) != CUDA_SUCCESS) return TV_ERR_CUDA;
  Reservation r;
  r.bytes = size;
  r.page.assign(size / p->page, 0);
  p->res.emplace(static_cast<uintptr_t>(va), std::move(r));
  p->reserved += size;
  *base = reinterpret_cast<void*>(va);
  return TV_OK;
}

extern "C" tv_status tv_kvpool_commit_rows(tv_kv_pool* p, void* base, int32_t n_heads, size_t head_stride,
                                           size_t row_bytes, int64_t rows, tv_stream stream) {
  if (p == nullptr || base == nullptr) return TV_ERR_ARG;
  const Driver& d = driver();
  std::lock_guard<std::mutex> lock(p->mu);
  auto it = p->res.find(reinterpret_cast<uintptr_t>(base));
  if (it == p->res.end() || !rows_fit(it->second, n_heads, head_stride, row_bytes, rows)) return TV_ERR_ARG;
  Reservation& r = it->second;
  DeviceScope dev(p->device);
  if (!dev.ok) return TV_ERR_CUDA;
  const CUmemAllocationProp prop = device_prop(p->device);
  CUmemAccessDesc access{};
  access.location = prop.location;
  access.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
  tv_status st = TV_OK;
  for_row_pages(p->page, n_heads, head_stride, row_bytes, rows, [&](size_t p0, size_t p1) {
    for (size_t i = p0; i < p1 && st == TV_OK; i++) {
      if (r.page[i] != 0) continue;
      CUmemGenericAllocationHandle h = 0;
      const CUresult cr = d.create(&h, p->page, &prop, 0);
      if (cr != CUDA_SUCCESS) {
        st = cr == CUDA_ERROR_OUT_OF_MEMORY ? TV_ERR_CAPACITY : TV_ERR_CUDA;
        break;
      }
      const CUdeviceptr va = static_cast<CUdeviceptr>(it->first + i * p->page);
      if (d.map(va, p->page, 0, h, 0) != CUDA_SUCCESS) {
        d.release(h);
        st = TV_ERR_CUDA;
        break;
      }
      r.page[i] = h;
      p->committed += p->page;
      if (d.set_access(va, p->page, &access, 1) != CUDA_SUCCESS) {
        unmap_page(p, it->first, r, i);
        st = TV_ERR_CUDA;
        break;
      }
      // a fresh page reads as zeros, as a zero-filled static buffer would
      if (cudaMemsetAsync(reinterpret_cast<void*>(va), 0, p->page, reinterpret_cast<cudaStream_t>(stream)) !=
          cudaSuccess) {
        cudaGetLastError();
        st = TV_ERR_CUDA;
        break;
      }
    }
  });
  return st;
}

extern "C" tv_status tv_kvpool_release_rows(tv_kv_pool* p, void* base, int32_t n_heads, size_t head_stride,
                                            size_t row_bytes, int64_t keep_rows) {
  if (p == nullptr || base == nullptr) return TV_ERR_ARG;
  std::lock_guard<std::mutex> lock(p->mu);
  auto it = p->res.find(reinterpret_cast<uintptr_t>(base));
  if (it == p->res.end() || !rows_fit(it->second, n_heads, head_stride, row_bytes, keep_rows)) return TV_ERR_ARG;
  Reservation& r = it->second;
  DeviceScope dev(p->device);
  if (!dev.ok) return TV_ERR_CUDA;
  std::vector<char> keep(r.page.size(), 0);
  for_row_pages(p->page, n_heads, head_stride, row_bytes, keep_rows, [&](size_t p0, size_t p1) {
    for (size_t i = p0; i < p1; i++) keep[i] = 1;
  });
  // work already queued may still read the pages being given back
  if (cudaDeviceSynchronize() != cudaSuccess) return TV_ERR_CUDA;
  for (size_t i = 0; i < r.page.size(); i++)
    if (r.page[i] != 0 && !keep[i] && unmap_page(p, it->first, r, i) != TV_OK) return TV_ERR_CUDA;
  return TV_OK;
}

extern "C" size_t tv_kvpool_committed_bytes(const tv_kv_pool* p) {
  if (p == nullptr) return 0;
  std::lock_guard<std::mutex> lock(const_cast<tv_kv_pool*>(p)->mu);
  return p->committed;
}

extern "C" size_t tv_kvpool_reserved_bytes(const tv_kv_pool* p) {
  if (p == nullptr) return 0;
  std::lock_guard<std::mutex> lock(const_cast<tv_kv_pool*>(p)->mu);
  return p->reserved;
}

extern "C" tv_status tv_kvpool_destroy(tv_kv_pool* p) {
  if (p == nullptr) return TV_ERR_ARG;
  const Driver& d = driver();
  tv_status st = TV_OK;
  {
    std::lock_guard<std::mutex> lock(p->mu);
    DeviceScope dev(p->device);
    if (!dev.ok || cudaDeviceSynchronize() != cudaSuccess) st = TV_ERR_CUDA;
    for (auto& kv : p->res) {
      for (size_t i = 0; i < kv.second.page.size(); i++)
        if (kv.second.page[i] != 0 && unmap_page(p, kv.first, kv.second, i) != TV_OK) st = TV_ERR_CUDA;
      if (d.free_va(static_cast<CUdeviceptr>(kv.first), kv.second.bytes) != CUDA_SUCCESS) st = TV_ERR_CUDA;
    }
    p->res.clear();
  }
  delete p;
  return st;
}
