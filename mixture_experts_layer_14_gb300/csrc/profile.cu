// Per-launch CUDA-event timing used by benchmarks (mok_timing_enable / mok_timing_collect).
#include <cstring>
#include <string>
#include <vector>

#include "mok_internal.h"

namespace mok {
namespace {
struct Rec {
  const char* name;
  cudaEvent_t a, b;
};
struct Prof {
  bool on = false;
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
};
thread_local Prof g_prof;
}  // namespace

void prof_begin(const char* name, cudaStream_t s) {
  if (!g_prof.on) return;
  Rec r{name, g_prof.get(), g_prof.get()};
  cudaEventRecord(r.a, s);
  g_prof.recs.push_back(r);
}

void prof_end(cudaStream_t s) {
  if (!g_prof.on || g_prof.recs.empty()) return;
  cudaEventRecord(g_prof.recs.back().b, s);
}

}  // namespace mok

extern "C" {

int mok_timing_enable(int enable) {
  mok::g_prof.on = enable != 0;
  return MOK_OK;
}

int mok_timing_collect(char* names, int* launches, double* ms, int max_kernels, int* n_out) {
  using namespace mok;
  if (!names || !launches || !ms || !n_out || max_kernels <= 0) return MOK_ERR_INVALID_ARG;
  std::vector<std::string> keys;
  std::vector<int> cnt;
  std::vector<double> tot;
  int rc = MOK_OK;
  for (auto& r : g_prof.recs) {
    float t = 0.0f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      rc = MOK_ERR_CUDA;
    size_t i = 0;
    while (i < keys.size() && keys[i] != r.name) ++i;
    if (i == keys.size()) {
      keys.emplace_back(r.name);
      cnt.push_back(0);
      tot.push_back(0.0);
    }
    cnt[i] += 1;
    tot[i] += t;
    g_prof.pool.push_back(r.a);
    g_prof.pool.push_back(r.b);
  }
  g_prof.recs.clear();
  const int n = (int)std::min<size_t>(keys.size(), (size_t)max_kernels);
  for (int i = 0; i < n; ++i) {
    std::strncpy(names + 32 * i, keys[i].c_str(), 31);
    names[32 * i + 31] = 0;
    launches[i] = cnt[i];
    ms[i] = tot[i];
  }
  *n_out = n;
  return rc;
}

}  // extern "C"
