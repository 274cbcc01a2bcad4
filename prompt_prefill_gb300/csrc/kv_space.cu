// K/V cache memory that grows with the positions written ("Single-pass
// prefill", "What it unlocked": prefill pairs with grow-on-demand KV so
// memory stays bounded). The whole cache [2 L regions][positions][row] is one
// reserved virtual address range, so every kernel indexes it as if it were
// fully allocated; physical memory is created and mapped at the start of
// every region only as far as the positions a call writes, in steps of the
// device's allocation granularity, and released again on reset.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "pp_internal.cuh"

namespace pp {
namespace {

struct Vmm {
  PFN_cuMemAddressReserve_v10020 reserve = nullptr;
  PFN_cuMemAddressFree_v10020 addr_free = nullptr;
  PFN_cuMemCreate_v10020 create = nullptr;
  PFN_cuMemRelease_v10020 release = nullptr;
  PFN_cuMemMap_v10020 map = nullptr;
  PFN_cuMemUnmap_v10020 unmap = nullptr;
  PFN_cuMemSetAccess_v10020 set_access = nullptr;
  PFN_cuMemGetAllocationGranularity_v10020 granularity = nullptr;
  bool ok = false;
};

template <class F>
bool entry(const char* name, F* fn) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, 10020, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !f)
    return false;
  *fn = reinterpret_cast<F>(f);
  return true;
}

const Vmm& vmm() {
  static Vmm v = [] {
    Vmm x;
    x.ok = entry("cuMemAddressReserve", &x.reserve) && entry("cuMemAddressFree", &x.addr_free) &&
           entry("cuMemCreate", &x.create) && entry("cuMemRelease", &x.release) && entry("cuMemMap", &x.map) &&
           entry("cuMemUnmap", &x.unmap) && entry("cuMemSetAccess", &x.set_access) &&
           entry("cuMemGetAllocationGranularity", &x.granularity);
    return x;
  }();
  return v;
}

CUmemAllocationProp prop_for(int device) {
  CUmemAllocationProp p = {};
  p.type = CU_MEM_ALLOCATION_TYPE_PINNED;
  p.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  p.location.id = device;
  return p;
}

}  // namespace

cudaError_t kv_space_reserve(KvSpace* s, int device, int n_regions, size_t region_min_bytes) {
  const Vmm& v = vmm();
  if (!v.ok) return cudaErrorNotSupported;
  *s = KvSpace{};
  s->device = device;
  const CUmemAllocationProp p = prop_for(device);
  size_t g = 0;
  if (v.granularity(&g, &p, CU_MEM_ALLOC_GRANULARITY_RECOMMENDED) != CUDA_SUCCESS || g == 0) return cudaErrorUnknown;
  s->gran = g;
  s->region_bytes = (region_min_bytes + g - 1) / g * g;
  s->n_regions = n_regions;
  CUdeviceptr base = 0;
  if (v.reserve(&base, s->region_bytes * n_regions, g, 0, 0) != CUDA_SUCCESS) return cudaErrorMemoryAllocation;
  s->base = base;
  return cudaSuccess;
}

cudaError_t kv_space_grow(KvSpace* s, size_t region_bytes_needed) {
  const Vmm& v = vmm();
  if (!v.ok || !s->base) return cudaErrorNotSupported;
  if (region_bytes_needed > s->region_bytes) return cudaErrorInvalidValue;
  const size_t want = (region_bytes_needed + s->gran - 1) / s->gran * s->gran;
  if (want <= s->mapped) return cudaSuccess;
  const size_t step = want - s->mapped;
  const CUmemAllocationProp p = prop_for(s->device);
  CUmemAccessDesc acc = {};
  acc.location = p.location;
  acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
  const size_t first_new = s->maps.size();
  auto undo = [&] {  // all-or-nothing: drop only what this call mapped; earlier positions stay intact
    for (size_t i = first_new; i < s->maps.size(); ++i) {
      v.unmap((CUdeviceptr)s->maps[i].ptr, s->maps[i].size);
      v.release((CUmemGenericAllocationHandle)s->maps[i].handle);
    }
    s->maps.resize(first_new);
    return cudaErrorMemoryAllocation;
  };
  for (int r = 0; r < s->n_regions; ++r) {
    const CUdeviceptr at = s->base + (CUdeviceptr)(r * s->region_bytes + s->mapped);
    CUmemGenericAllocationHandle h = 0;
    if (v.create(&h, step, &p, 0) != CUDA_SUCCESS) return undo();
    if (v.map(at, step, 0, h, 0) != CUDA_SUCCESS) {
      v.release(h);
      return undo();
    }
    s->maps.push_back({(unsigned long long)at, step, (unsigned long long)h});
    if (v.set_access(at, step, &acc, 1) != CUDA_SUCCESS) return undo();
  }
  s->mapped = want;
  return cudaSuccess;
}

void kv_space_release(KvSpace* s) {
  const Vmm& v = vmm();
  if (!v.ok) return;
  for (const auto& m : s->maps) {
    v.unmap((CUdeviceptr)m.ptr, m.size);
    v.release((CUmemGenericAllocationHandle)m.handle);
  }
  s->maps.clear();
  s->mapped = 0;
}

void kv_space_free(KvSpace* s) {
  kv_space_release(s);
  const Vmm& v = vmm();
  if (v.ok && s->base) v.addr_free((CUdeviceptr)s->base, s->region_bytes * s->n_regions);
  s->base = 0;
}

}  // namespace pp
