// profiler.cu -- optional per-launch timing inside libnsa.so.
//
// When enabled (nsa_profile_enable(1)), every kernel launch of the library is
// bracketed by two CUDA events recorded on the launching stream.
// nsa_profile_read() synchronises those events and returns, per kernel name,
// the number of launches and the summed device time.  Disabled (the default),
// it costs one branch per launch.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "nsa.h"
#include "profiler.hpp"

namespace nsa {
namespace prof {

namespace {
struct Rec {
  std::string name;
  cudaEvent_t a, b;
};
struct State {
  std::mutex mu;
  bool on = false;
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
} g_state;

cudaEvent_t take_event() {
  if (!g_state.pool.empty()) {
    cudaEvent_t e = g_state.pool.back();
    g_state.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
}  // namespace

bool enabled() { return g_state.on; }

void begin(const char* name, cudaStream_t s) {
  if (!g_state.on) return;
  std::lock_guard<std::mutex> lk(g_state.mu);
  Rec r;
  r.name = name;
  r.a = take_event();
  r.b = take_event();
  cudaEventRecord(r.a, s);
  g_state.recs.push_back(r);
}

void end(cudaStream_t s) {
  if (!g_state.on) return;
  std::lock_guard<std::mutex> lk(g_state.mu);
  if (!g_state.recs.empty()) cudaEventRecord(g_state.recs.back().b, s);
}

}  // namespace prof
}  // namespace nsa

using namespace nsa::prof;

extern "C" {

int nsa_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_state.mu);
  g_state.on = on != 0;
  return NSA_OK;
}

int nsa_profile_read(int max_kernels, char* names, size_t name_cap, int* launches, float* total_ms) {
  std::lock_guard<std::mutex> lk(g_state.mu);
  std::vector<std::string> keys;
  std::vector<int> cnt;
  std::vector<double> tot;
  for (Rec& r : g_state.recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return -NSA_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return -NSA_ERR_CUDA;
    size_t k = 0;
    while (k < keys.size() && keys[k] != r.name) ++k;
    if (k == keys.size()) {
      keys.push_back(r.name);
      cnt.push_back(0);
      tot.push_back(0.0);
    }
    cnt[k] += 1;
    tot[k] += ms;
    g_state.pool.push_back(r.a);
    g_state.pool.push_back(r.b);
  }
  g_state.recs.clear();
  std::string joined;
  const int n = (int)keys.size() < max_kernels ? (int)keys.size() : max_kernels;
  for (int k = 0; k < n; ++k) {
    if (k) joined += ",";
    joined += keys[k];
    if (launches) launches[k] = cnt[k];
    if (total_ms) total_ms[k] = (float)tot[k];
  }
  if (names && name_cap) {
    std::strncpy(names, joined.c_str(), name_cap - 1);
    names[name_cap - 1] = '\0';
  }
  return n;
}

}  // extern "C"
