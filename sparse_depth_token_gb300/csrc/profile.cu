// Measurement support: a host-side count of kernel launches and optional
// per-kernel timing with CUDA events recorded on the launching stream.

#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"

namespace xmod {

namespace {
std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_enabled{0};
std::mutex g_mu;
struct Rec {
  const char* kind;
  cudaEvent_t start, stop;
};
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

ProfScope::ProfScope(const char* kind, cudaStream_t s) : kind_(kind), stream_(s) {
  if (!g_enabled.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  start_ = take_event();
  if (start_) cudaEventRecord(start_, stream_);
}

ProfScope::~ProfScope() {
  if (!start_) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t stop = take_event();
  if (!stop) return;
  cudaEventRecord(stop, stream_);
  g_recs.push_back({kind_, start_, stop});
}

}  // namespace xmod

using namespace xmod;

extern "C" {

uint64_t xmod_launch_count(void) { return g_launches.load(); }

int xmod_profile_enable(int enable) {
  g_enabled.store(enable ? 1 : 0);
  return XMOD_OK;
}

int xmod_profile_read(xmod_kernel_time* out, int max_kinds, int* n_kinds) {
  std::lock_guard<std::mutex> lk(g_mu);
  int n = 0;
  int st = XMOD_OK;
  for (const Rec& r : g_recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) {
      st = XMOD_ERR_CUDA;
      ms = 0.f;
    }
    int k = 0;
    for (; k < n; ++k)
      if (out && strncmp(out[k].name, r.kind, sizeof(out[k].name)) == 0) break;
    if (k == n) {
      if (!out || n >= max_kinds) {
        g_pool.push_back(r.start);
        g_pool.push_back(r.stop);
        continue;
      }
      memset(&out[k], 0, sizeof(out[k]));
      strncpy(out[k].name, r.kind, sizeof(out[k].name) - 1);
      ++n;
    }
    out[k].launches += 1;
    out[k].total_ms += ms;
    g_pool.push_back(r.start);
    g_pool.push_back(r.stop);
  }
  g_recs.clear();
  if (n_kinds) *n_kinds = n;
  return st;
}

}  // extern "C"
