// gma_profile.cu -- launch counter and optional per-kernel CUDA-event timing.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "gma_internal.h"
#include "gma_profile.h"

namespace gma {
namespace {

std::atomic<unsigned long long> g_launches{0};
std::atomic<bool> g_recording{false};

struct Rec {
  const char* name;
  cudaEvent_t start, stop;
};

std::mutex g_mu;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_free;

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

void* prof_before(cudaStream_t st, const char* name) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_recording.load(std::memory_order_relaxed)) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  Rec r{name, take_event(), take_event()};
  if (!r.start || !r.stop) return nullptr;
  cudaEventRecord(r.start, st);
  g_recs.push_back(r);
  return (void*)(uintptr_t)g_recs.size();
}

void prof_after(cudaStream_t st, void* token) {
  if (!token) return;
  std::lock_guard<std::mutex> lock(g_mu);
  size_t i = (size_t)(uintptr_t)token - 1;
  if (i < g_recs.size()) cudaEventRecord(g_recs[i].stop, st);
}

}  // namespace gma

using namespace gma;

extern "C" {

unsigned long long gma_launch_count(void) { return g_launches.load(); }

void gma_debug_withhold_first_load(void) { gma::tc_set_fault_injection(1u); }

gma_status_t gma_profile_enable(int on) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (on) {
    for (auto& r : g_recs) {
      g_free.push_back(r.start);
      g_free.push_back(r.stop);
    }
    g_recs.clear();
  }
  g_recording.store(on != 0);
  return GMA_OK;
}

int gma_profile_read(char* buf, size_t len) {
  std::lock_guard<std::mutex> lock(g_mu);
  std::map<std::string, std::pair<int, double>> agg;
  for (auto& r : g_recs) {
    if (cudaEventSynchronize(r.stop) != cudaSuccess) return -1;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) return -1;
    auto& a = agg[r.name];
    a.first += 1;
    a.second += ms;
  }
  std::string out;
  for (auto& kv : agg) {
    char line[160];
    snprintf(line, sizeof line, "%s %d %.6f\n", kv.first.c_str(), kv.second.first, kv.second.second);
    out += line;
  }
  if (buf && len) {
    size_t n = out.size() < len - 1 ? out.size() : len - 1;
    memcpy(buf, out.data(), n);
    buf[n] = 0;
  }
  return (int)agg.size();
}

}  // extern "C"
