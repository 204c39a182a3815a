// Per-launch CUDA-event timing used by benchmarks (mok_timing_enable / mok_timing_collect).
#include <cstring>
#include <string>
#include <vector>

#include "mok_device.cuh"

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

// Failure-detection self-test: one CTA waits, with a bounded wait of `budget_ns`, on an mbarrier
// that nothing ever arrives on.  The wait gives up, records MOK_ERR_TIMEOUT in the status word
// and the kernel returns normally, leaving the context usable.
__global__ void selftest_wait_kernel(int* status, uint64_t budget_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&bar)), "r"(1) : "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, status, &abort_flag, budget_ns);
  __syncthreads();
}

}  // namespace mok

extern "C" {

int mok_selftest_bounded_wait(void* ws, int64_t budget_ns, mok_stream_t stream) {
  if (!ws || budget_ns <= 0 || budget_ns > (int64_t)mok::kWaitNs) return MOK_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mok::selftest_wait_kernel<<<1, 32, 0, s>>>(static_cast<int*>(ws), (uint64_t)budget_ns);
  return cudaGetLastError() == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}

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
