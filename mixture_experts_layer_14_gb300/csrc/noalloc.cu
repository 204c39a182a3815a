// mok_dispatch_index_noalloc: the pull-schedule counting sort with its scratch in a fixed,
// library-owned device array instead of a caller-provided workspace.
//
// Who needs it: callers that are not allowed to allocate device memory at the point where they
// build the routing — for example a serving runtime that reserves all device memory up front and
// forbids cudaMalloc afterwards (a cudaMalloc/cudaFree can synchronise the device and stall
// every stream), or host code that runs on a thread without access to the framework's caching
// allocator.  They still own and pass every input and output buffer; only the scratch moves.
#include <mutex>

#include "mok_internal.h"

namespace mok {

// Scratch of the no-allocation dispatch: a 256-byte header (word 0 is the status word of the
// call) followed by a 1 MiB histogram of (expert, token block) counts, so that E * ceil(T / 64)
// counts fit when that product is at most 262144 (T = 65536 at E = 256).  Every device that
// loads the library keeps this array until the process exits.
constexpr int kNoAllocHeaderWords = 64;
constexpr size_t kNoAllocHistWords = size_t(1) << 18;
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocHeaderWords + kNoAllocHistWords];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
int32_t* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device.  Host code cannot use the
// symbol's name as a pointer (on the host it names a stand-in, not device memory), so the
// address is looked up once per device, with that device current, and cached.
int32_t* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_ptr[dev] = static_cast<int32_t*>(p);
  }
  return g_noalloc_ptr[dev];
}
}  // namespace

}  // namespace mok

extern "C" int mok_dispatch_index_noalloc(const mok_dims* dims, const int32_t* topk_idx,
                                          const float* topk_w, int32_t* counts, int32_t* offsets,
                                          int32_t* sorted_tok, float* sorted_w, int32_t* inv_pos,
                                          mok_stream_t stream) {
  using namespace mok;
  if (!dims) return MOK_ERR_INVALID_ARG;
  if (dims->T < 0 || dims->T > 0x7fffffffLL / 8 || dims->k < 1 || dims->k > kMaxK ||
      dims->E < dims->k || dims->E > kMaxE || dims->E % 8)
    return MOK_ERR_UNSUPPORTED;
  if (!counts || !offsets ||
      (dims->T > 0 && (!topk_idx || !topk_w || !sorted_tok || !sorted_w || !inv_pos)))
    return MOK_ERR_INVALID_ARG;
  const int64_t nblk = (dims->T + kDispatchChunk - 1) / kDispatchChunk;
  const int64_t hist_words = (int64_t)dims->E * (nblk > 0 ? nblk : 1);
  if ((size_t)hist_words > kNoAllocHistWords) return MOK_ERR_WORKSPACE;

  int32_t* scratch = scratch_on_current_device();
  if (!scratch) return MOK_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the status word must start at zero; the histogram is fully rewritten by the call
  if (cudaMemsetAsync(scratch, 0, sizeof(int32_t), s) != cudaSuccess) return MOK_ERR_CUDA;
  int n = 0;
  const cudaError_t e =
      launch_dispatch(dims->T, dims->E, dims->k, topk_idx, topk_w, counts, offsets, sorted_tok,
                      sorted_w, inv_pos, scratch + kNoAllocHeaderWords, scratch, s, &n);
  return e == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}
