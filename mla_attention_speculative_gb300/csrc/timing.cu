// Per-kernel timing for benchmarks (mla_kernel_timing_enable / _read).
//
// While enabled, each launch wrapped in a KernelTimer records a CUDA event on
// the launching stream before and after the kernel.  Events come from a pool
// owned here and are recycled when the totals are read; no device memory is
// involved.  Reading waits for the recorded events, so it synchronises with
// the streams that carry them.

#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "mla_internal.h"

namespace mla {
namespace {

struct Pending {
  int id;
  cudaEvent_t start, stop;
};

std::atomic<bool> g_enabled{false};
std::mutex g_mu;
std::vector<std::string> g_names;
std::vector<long long> g_launches;
std::vector<double> g_ms;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_free;

int kernel_id(const char* name) {
  for (size_t i = 0; i < g_names.size(); ++i)
    if (g_names[i] == name) return (int)i;
  g_names.emplace_back(name);
  g_launches.push_back(0);
  g_ms.push_back(0.0);
  return (int)g_names.size() - 1;
}

cudaEvent_t take_event() {
  if (!g_free.empty()) {
    cudaEvent_t e = g_free.back();
    g_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

bool timing_enabled() { return g_enabled.load(std::memory_order_relaxed); }

KernelTimer::KernelTimer(const char* name, cudaStream_t stream) : stream_(stream) {
  if (!timing_enabled()) return;
  std::lock_guard<std::mutex> lk(g_mu);
  start_ = take_event();
  if (start_ == nullptr) return;
  id_ = kernel_id(name);
  cudaEventRecord(start_, stream_);
}

KernelTimer::~KernelTimer() {
  if (id_ < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t stop = take_event();
  if (stop == nullptr) {
    g_free.push_back(start_);
    return;
  }
  cudaEventRecord(stop, stream_);
  g_pending.push_back({id_, start_, stop});
}

}  // namespace mla

using namespace mla;

extern "C" mla_status_t mla_kernel_timing_enable(int32_t on) {
  g_enabled.store(on != 0);
  return MLA_OK;
}

extern "C" mla_status_t mla_kernel_timing_read(char* names, size_t names_len, int32_t* launches,
                                               double* total_ms, int32_t max_kernels,
                                               int32_t* n_kernels, int32_t reset) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (const Pending& p : g_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.stop) != cudaSuccess ||
        cudaEventElapsedTime(&ms, p.start, p.stop) != cudaSuccess) {
      set_error("timing event failed: %s", cudaGetErrorString(cudaGetLastError()));
      return MLA_ERR_CUDA;
    }
    g_launches[p.id] += 1;
    g_ms[p.id] += ms;
    g_free.push_back(p.start);
    g_free.push_back(p.stop);
  }
  g_pending.clear();
  const int n = (int)g_names.size();
  if (n_kernels) *n_kernels = n;
  std::string joined;
  for (int i = 0; i < n; ++i) {
    if (i) joined += ';';
    joined += g_names[i];
    if (i < max_kernels) {
      if (launches) launches[i] = (int32_t)g_launches[i];
      if (total_ms) total_ms[i] = g_ms[i];
    }
  }
  if (names && names_len) {
    const size_t k = joined.size() < names_len - 1 ? joined.size() : names_len - 1;
    memcpy(names, joined.data(), k);
    names[k] = '\0';
  }
  if (reset) {
    for (int i = 0; i < n; ++i) {
      g_launches[i] = 0;
      g_ms[i] = 0.0;
    }
  }
  return MLA_OK;
}
