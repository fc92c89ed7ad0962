// Page-locked host memory on transparent huge pages, for the host-fed step.
//
// The gradients of zero_step_host cross the host link every step, so the
// link's rate bounds that step.  Memory pinned with cudaHostAlloc sits on
// base pages; on GB300 hosts its 1 GB copies measured anywhere from 38 to
// 212 GB/s, with more slow stretches in each later process on the same host,
// while memory mapped here (anonymous, advised for huge pages, populated,
// then registered) held 208-212 GB/s in the same processes.  The address
// translation of DMA over many small pages is the likely cost.

#include <sys/mman.h>
#include <unistd.h>

#include <cuda_runtime.h>

#include <algorithm>
#include <cerrno>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "zero_internal.h"
#include "zero_step.h"

namespace {

struct Mapping {
  void* base;      // what mmap returned
  size_t length;   // what was mapped
};

std::mutex g_mu;
std::map<void*, Mapping> g_maps;   // aligned address handed out -> its mapping

int fail(int code, const std::string& msg) { return zero::record_error(code, msg.c_str()); }

// Size of a transparent huge page (PMD size), 2 MiB if the kernel does not say.
size_t huge_page_bytes() {
  size_t bytes = 0;
  if (FILE* f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
    unsigned long long v = 0;
    if (std::fscanf(f, "%llu", &v) == 1) bytes = static_cast<size_t>(v);
    std::fclose(f);
  }
  return bytes ? bytes : (size_t(2) << 20);
}

// Write one byte in every base page so that all of it is backed now, in
// parallel over huge-page-sized pieces.
void populate(char* p, size_t len, size_t page, size_t piece) {
  const size_t pieces = (len + piece - 1) / piece;
  const unsigned hw = std::max(1u, std::thread::hardware_concurrency());
  const size_t nthreads = std::min<size_t>(std::min<size_t>(hw, 16), pieces);
  auto work = [&](size_t k0) {
    for (size_t k = k0; k < pieces; k += nthreads) {
      const size_t end = std::min(len, (k + 1) * piece);
      for (size_t off = k * piece; off < end; off += page) p[off] = 0;
    }
  };
  std::vector<std::thread> threads;
  for (size_t k = 1; k < nthreads; ++k) threads.emplace_back(work, k);
  work(0);
  for (auto& t : threads) t.join();
}

}  // namespace

extern "C" int zero_host_alloc(int64_t bytes, void** out) {
  if (out == nullptr) return fail(ZERO_E_ARG, "out is NULL");
  *out = nullptr;
  if (bytes <= 0) return fail(ZERO_E_ARG, "bytes must be > 0");
  const size_t huge = huge_page_bytes();
  const long page_l = sysconf(_SC_PAGESIZE);
  const size_t page = page_l > 0 ? static_cast<size_t>(page_l) : 4096;
  // Blocks of at least one huge page are whole huge pages, starting on a
  // huge-page boundary (the mapping has room for the shift), so that no part
  // of them is left on base pages; smaller blocks stay on base pages and
  // waste nothing.
  const bool use_huge = static_cast<size_t>(bytes) >= huge;
  const size_t unit = use_huge ? huge : page;
  const size_t len = (static_cast<size_t>(bytes) + unit - 1) / unit * unit;
  const size_t map_len = use_huge ? len + huge : len;
  void* base = mmap(nullptr, map_len, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (base == MAP_FAILED) return fail(ZERO_E_NOMEM, std::string("mmap failed: ") + std::strerror(errno));
  char* p = use_huge ? reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(base) + huge - 1) / huge * huge)
                     : static_cast<char*>(base);
#ifdef MADV_HUGEPAGE
  if (use_huge) madvise(p, len, MADV_HUGEPAGE);   // advice only: where huge pages are off, base pages serve
#endif
  populate(p, len, page, use_huge ? huge : (size_t(2) << 20));
#ifdef MADV_COLLAPSE
  // where the first touches got base pages (no free huge page at that
  // moment), ask the kernel to compact and collapse them now; advice only
  if (use_huge) madvise(p, len, MADV_COLLAPSE);
#endif
  const cudaError_t e = cudaHostRegister(p, len, cudaHostRegisterDefault);
  if (e != cudaSuccess) {
    munmap(base, map_len);
    return fail(ZERO_E_CUDA, std::string("cudaHostRegister: ") + cudaGetErrorString(e));
  }
  {
    std::lock_guard<std::mutex> lock(g_mu);
    g_maps[p] = {base, map_len};
  }
  *out = p;
  return ZERO_OK;
}

extern "C" int zero_host_free(void* p) {
  if (p == nullptr) return ZERO_OK;
  Mapping m;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_maps.find(p);
    if (it == g_maps.end()) return fail(ZERO_E_ARG, "not an address returned by zero_host_alloc");
    m = it->second;
    g_maps.erase(it);
  }
  const cudaError_t e = cudaHostUnregister(p);
  munmap(m.base, m.length);
  if (e != cudaSuccess) return fail(ZERO_E_CUDA, std::string("cudaHostUnregister: ") + cudaGetErrorString(e));
  return ZERO_OK;
}
