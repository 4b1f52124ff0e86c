// Page-locked host memory for the arena (mt_host_alloc / mt_host_free).
//
// The arena's blocks leave and enter host memory as large DMA bursts (chestersoft digest,
// Methodik, "Layer-Contiguous Tiling"), so what matters is that every page of it moves at the
// host link's full rate. Measured on GB300 (Grace host, 64 KB base pages): once other
// processes have used and released host memory, memory from cudaHostAlloc, or base pages
// registered with cudaHostRegister, has regions that copy at 8-40 GB/s instead of ~210 GB/s,
// and every such 512 MB region probed was made of scattered base pages; regions backed by
// transparent huge pages (512 MB on that kernel) copied at full rate in the same state. So the
// arena is an anonymous mapping aligned to the huge-page size and advised to use huge pages,
// faulted in one huge page at a time by one thread (faulting from all host threads at once
// left more of it in base pages: 3-6 of 162 regions of an 81 GB arena, against none), then
// registered. Spare huge pages are faulted in with it; a copy of every huge page is timed, and
// spares that copy at full rate are moved (mremap) over pages that copy below 0.6 x the median,
// in up to three rounds, before the unused spares are released. Where transparent huge pages
// are switched off, or the mapping or registration fails, cudaHostAlloc is used.
#include <cuda_runtime.h>
#include <sys/mman.h>
#include <unistd.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "kernels.h"

namespace mt {

namespace {

struct Mapping {
  uint64_t len;
  HostAllocInfo info;
};
std::mutex g_mu;
std::map<void*, Mapping> g_maps;  // registered huge-page mappings by base address

std::string read_file(const char* path) {
  std::string s;
  if (FILE* f = std::fopen(path, "r")) {
    char buf[256];
    size_t n = std::fread(buf, 1, sizeof buf - 1, f);
    buf[n] = 0;
    s = buf;
    std::fclose(f);
  }
  return s;
}

// Size of a transparent huge page, or 0 when they cannot be used.
uint64_t thp_size() {
  const std::string mode = read_file("/sys/kernel/mm/transparent_hugepage/enabled");
  if (mode.empty() || mode.find("[never]") != std::string::npos) return 0;
  const uint64_t hp = std::strtoull(read_file("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size").c_str(), nullptr, 10);
  const long page = sysconf(_SC_PAGESIZE);
  if (hp == 0 || page <= 0 || hp % static_cast<uint64_t>(page)) return 0;
  return hp;
}

// Times host-to-device copies of huge pages into one device buffer of a huge page, with events
// on a private stream. ok() is false if the buffer or the stream cannot be had (the caller then
// skips the check).
class Prober {
 public:
  explicit Prober(uint64_t chunk) : chunk_(chunk) {
    ok_ = cudaMalloc(&d_, chunk) == cudaSuccess && cudaStreamCreateWithFlags(&st_, cudaStreamNonBlocking) == cudaSuccess &&
          cudaEventCreate(&a_) == cudaSuccess && cudaEventCreate(&b_) == cudaSuccess;
    if (!ok_) cudaGetLastError();
  }
  ~Prober() {
    if (a_) cudaEventDestroy(a_);
    if (b_) cudaEventDestroy(b_);
    if (st_) cudaStreamDestroy(st_);
    if (d_) cudaFree(d_);
    cudaGetLastError();
  }
  bool ok() const { return ok_; }
  // GB/s of each of the n chunks from `base`; false (and gbs unusable) on any CUDA error.
  bool run(const uint8_t* base, uint64_t n, std::vector<double>& gbs) {
    gbs.assign(n, 0.0);
    for (uint64_t i = 0; ok_ && i < n; ++i) {
      float ms = 0.f;
      ok_ = cudaEventRecord(a_, st_) == cudaSuccess &&
            cudaMemcpyAsync(d_, base + i * chunk_, chunk_, cudaMemcpyHostToDevice, st_) == cudaSuccess &&
            cudaEventRecord(b_, st_) == cudaSuccess && cudaEventSynchronize(b_) == cudaSuccess &&
            cudaEventElapsedTime(&ms, a_, b_) == cudaSuccess;
      gbs[i] = ok_ && ms > 0.f ? chunk_ / (ms * 1e-3) / 1e9 : 0.0;
    }
    if (!ok_) cudaGetLastError();
    return ok_;
  }

 private:
  uint64_t chunk_;
  void* d_ = nullptr;
  cudaStream_t st_ = nullptr;
  cudaEvent_t a_ = nullptr, b_ = nullptr;
  bool ok_ = false;
};

double median_of(std::vector<double> v) {
  if (v.empty()) return 0.0;
  std::nth_element(v.begin(), v.begin() + v.size() / 2, v.end());
  return v[v.size() / 2];
}

void* huge_page_alloc(uint64_t bytes, HostAllocInfo* info) {
  const uint64_t hp = thp_size();
  if (hp == 0) return nullptr;
  const uint64_t len = (bytes + hp - 1) / hp * hp, n = len / hp;
  // spare huge pages to stand in for arena pages that copy slowly: 6 % of the arena, at least 8
  const uint64_t ns = std::max<uint64_t>(8, (6 * n + 99) / 100), total = len + ns * hp;
  void* raw = mmap(nullptr, total + hp, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (raw == MAP_FAILED) return nullptr;
  // keep exactly [base, base + total) with base on a huge-page boundary
  const uintptr_t r = reinterpret_cast<uintptr_t>(raw);
  const uintptr_t ub = (r + hp - 1) / hp * hp;
  if (ub > r) munmap(raw, ub - r);
  munmap(reinterpret_cast<void*>(ub + total), r + hp - ub);
  uint8_t* base = reinterpret_cast<uint8_t*>(ub);
  uint8_t* spare = base + len;
  if (madvise(base, total, MADV_HUGEPAGE) != 0) {
    munmap(base, total);
    return nullptr;
  }
  // fault the pages in, one huge page after the other (the kernel clears each on first touch)
  volatile uint8_t* b = base;
  for (uint64_t i = 0; i < n + ns; ++i) b[i * hp] = 0;
  if (cudaHostRegister(base, len, cudaHostRegisterDefault) != cudaSuccess) {
    cudaGetLastError();
    munmap(base, total);
    return nullptr;
  }
  // spares are registered one by one, so that each can be moved (or released) on its own
  std::vector<int> spare_state(ns, 0);  // 0 unregistered, 1 registered, 2 moved into the arena
  for (uint64_t j = 0; j < ns; ++j) {
    if (cudaHostRegister(spare + j * hp, hp, cudaHostRegisterDefault) == cudaSuccess)
      spare_state[j] = 1;
    else
      cudaGetLastError();
  }
  *info = HostAllocInfo{};
  info->chunk_bytes = hp;
  info->chunks = static_cast<int32_t>(n);
  info->spare = static_cast<int32_t>(ns);
  std::vector<double> gbs, sg;
  Prober prober(hp);
  bool probed = prober.ok() && prober.run(base, n, gbs);
  // up to three rounds: find arena pages that copy below 0.6 x the median, move good spare
  // pages over them, probe the arena again
  for (int round = 0; probed && round < 3; ++round) {
    const double med = median_of(gbs);
    std::vector<uint64_t> slow, good;
    for (uint64_t i = 0; i < n; ++i)
      if (gbs[i] < 0.6 * med) slow.push_back(i);
    if (round == 0) info->slow_found = static_cast<int32_t>(slow.size());
    if (slow.empty()) break;
    for (uint64_t j = 0; j < ns; ++j)
      if (spare_state[j] == 1 && prober.run(spare + j * hp, 1, sg) && sg[0] >= 0.6 * med) good.push_back(j);
    if (good.empty()) break;
    // neither range may be registered while pages move; a range that cannot be unregistered
    // stays where it is (the arena keeps its slow pages, a spare stays a spare)
    if (cudaHostUnregister(base) != cudaSuccess) {
      cudaGetLastError();
      break;
    }
    size_t k = 0;
    for (uint64_t i : slow) {
      if (k == good.size()) break;
      const uint64_t j = good[k++];
      if (cudaHostUnregister(spare + j * hp) != cudaSuccess) {
        cudaGetLastError();
        continue;
      }
      spare_state[j] = 0;
      if (mremap(spare + j * hp, hp, hp, MREMAP_MAYMOVE | MREMAP_FIXED, base + i * hp) != MAP_FAILED) {
        spare_state[j] = 2;
        ++info->replaced;
      }
    }
    if (cudaHostRegister(base, len, cudaHostRegisterDefault) != cudaSuccess) {
      cudaGetLastError();
      for (uint64_t j = 0; j < ns; ++j)
        if (spare_state[j] != 2) {
          if (spare_state[j] == 1) cudaHostUnregister(spare + j * hp);
          munmap(spare + j * hp, hp);
        }
      munmap(base, len);
      return nullptr;
    }
    probed = prober.run(base, n, gbs);
  }
  for (uint64_t j = 0; j < ns; ++j)
    if (spare_state[j] != 2) {
      if (spare_state[j] == 1) cudaHostUnregister(spare + j * hp);
      munmap(spare + j * hp, hp);
    }
  if (probed) {
    info->median_gbs = median_of(gbs);
    info->min_gbs = *std::min_element(gbs.begin(), gbs.end());
  }
  std::lock_guard<std::mutex> lk(g_mu);
  g_maps[base] = Mapping{len, *info};
  return base;
}

}  // namespace

cudaError_t host_alloc(uint64_t bytes, void** out) {
  HostAllocInfo info{};
  *out = huge_page_alloc(bytes, &info);
  if (*out) return cudaSuccess;
  return cudaHostAlloc(out, bytes, cudaHostAllocDefault);
}

bool host_alloc_info(const void* p, HostAllocInfo* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_maps.find(const_cast<void*>(p));
  if (it == g_maps.end()) return false;
  *out = it->second.info;
  return true;
}

cudaError_t host_free(void* p) {
  uint64_t len = 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_maps.find(p);
    if (it != g_maps.end()) {
      len = it->second.len;
      g_maps.erase(it);
    }
  }
  if (len == 0) return cudaFreeHost(p);
  const cudaError_t e = cudaHostUnregister(p);
  munmap(p, len);
  return e;
}

}  // namespace mt
