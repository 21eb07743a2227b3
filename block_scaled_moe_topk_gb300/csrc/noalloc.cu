// noalloc.cu -- moe_sort_by_expert_noalloc: the stable expert sort for callers that cannot
// hand the library any device memory beyond the sort's own inputs and outputs.
//
// Its scratch (the per-chunk expert histograms and a status word) lives in one fixed
// array compiled into the library, so every GPU that loads the library keeps these
// 4 MiB for the life of the process.  In host code the array's name is only a host-side
// stand-in; the device address is looked up once per device (and again if that device's
// context is replaced) with cudaGetSymbolAddress, with that device current, and handed to the same histogram / scan / scatter kernels the
// workspace version uses.  Every call on a device shares the array: the status word is
// cleared on each call, the histograms are fully rewritten before they are read.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "moe_internal.h"
#include "moe_topk.h"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;  // the fixed maximum: 4 MiB per device
constexpr size_t kStatusBytes = 256;              // status word, padded to keep alignment
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_sort_scratch[kScratchBytes];

// The current context's process-unique id (cuCtxGetId), or 0 when none is current or the
// driver entry points are unavailable.  The driver is reached through the runtime's entry-point
// query, so the library still links against the CUDA runtime alone.
unsigned long long current_context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of g_sort_scratch on the current device (nullptr on failure).  The first
// call on a device performs the lookup (which also brings up the device's primary context);
// later calls reuse it as long as the same context is current.  The cache is keyed on the
// context's unique id, so after cudaDeviceReset (a new primary context, a new module load) the
// address is looked up again instead of pointing into the destroyed context.
void* scratch_on_current_device() {
  struct Entry {
    unsigned long long ctx_id = 0;
    void* addr = nullptr;
  };
  static Entry cache[kMaxDevices];
  static std::mutex mu;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  Entry& e = cache[dev];
  const unsigned long long id = current_context_id();
  if (e.addr == nullptr || id == 0 || id != e.ctx_id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sort_scratch) != cudaSuccess) return nullptr;
    e.addr = p;
    e.ctx_id = current_context_id();  // the lookup made the primary context current if none was
  }
  return e.addr;
}

bool is_aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace

extern "C" moe_status_t moe_sort_by_expert_noalloc(const int32_t* topk_ids, int64_t T, int E, int k,
                                                   int32_t* counts, int64_t* offsets, int32_t* sorted_pair,
                                                   int32_t* inv, void* stream) {
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_ids || !sorted_pair || !inv)) return MOE_ERR_INVALID_ARG;
  if (T < 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
  if (k > moe::kMaxTopK || E > moe::kMaxExperts || T > (int64_t(1) << 24)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!is_aligned(topk_ids, 4) || !is_aligned(counts, 4) || !is_aligned(offsets, 8) ||
      !is_aligned(sorted_pair, 4) || !is_aligned(inv, 4))
    return MOE_ERR_MISALIGNED;
  const int64_t nchunk = (T + moe::kTokensPerChunk - 1) / moe::kTokensPerChunk;
  if (kStatusBytes + (size_t)E * (size_t)nchunk * sizeof(int32_t) > kScratchBytes)
    return MOE_ERR_WORKSPACE_TOO_SMALL;  // T * E beyond what the fixed scratch holds

  int dev = -1, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED_DEVICE;
  uint8_t* scratch = static_cast<uint8_t*>(scratch_on_current_device());
  if (scratch == nullptr) return MOE_ERR_CUDA;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* status = reinterpret_cast<uint32_t*>(scratch);
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (T == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(offsets, 0, sizeof(int64_t) * (E + 1), s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  moe::SortArgs sa{topk_ids, T, E, k, reinterpret_cast<int32_t*>(scratch + kStatusBytes), nchunk, counts, offsets,
                   nullptr, nullptr, sorted_pair, inv, nullptr, status};
  if (moe::launch_histogram(sa, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_sort(sa, s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}
