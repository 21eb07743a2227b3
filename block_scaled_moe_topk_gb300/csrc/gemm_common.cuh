// gemm_common.cuh -- pieces shared by the grouped GEMM kernels (gemm.cu, gemm_swap.cu):
// tile decoding over the experts' M tiles, bounded mbarrier waits, SwiGLU, and the driver
// entry point that encodes TMA tensor maps.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

struct Tile {
  int e, mt, nt;
};

// Tiles of expert e occupy [mtile_base[e]*NT, mtile_base[e+1]*NT); inside an expert the
// M tile is the fastest index so CTAs running side by side share the weight tile in L2.
__device__ __forceinline__ Tile decode_tile(int64_t tile, const int32_t* mtile_base, int E, int NT) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)mtile_base[mid] * NT <= tile) lo = mid;
    else hi = mid - 1;
  }
  const int mt_e = mtile_base[lo + 1] - mtile_base[lo];
  const int64_t local = tile - (int64_t)mtile_base[lo] * NT;
  Tile t;
  t.e = lo;
  t.nt = (int)(local / mt_e);
  t.mt = (int)(local % mt_e);
  return t;
}

struct Sync {
  volatile int* abort_flag;
  uint32_t* status;  // status[0]: status bits; status[1..6]: first expired wait (see below)
  uint64_t timeout_ns;
  uint32_t bar0;
};

// Poll a phase of an mbarrier until it completes, the CTA aborts, or the time limit passes.
// The limit is counted in SM clock cycles (clock64 is cheap; %globaltimer is not), at 2
// cycles per nanosecond of limit_ns, so at any SM clock >= 1 GHz the wait ends within
// 2 x limit_ns.  No clock is read during the first 64 probes, which is where a phase that
// is merely a little late completes.
// With drain = true the abort flag is ignored: used at exit to let this CTA's own copies and
// MMAs land (bounded by limit_ns alone) before TMEM is freed.
__device__ __noinline__ bool bounded_wait(uint32_t bar, uint32_t parity, const Sync& s, uint64_t limit_ns,
                                          bool drain = false) {
  const uint64_t limit_cycles = 2 * limit_ns;
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (!drain && *s.abort_flag) return false;
      const uint64_t now = clock64();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit_cycles) {
        *s.abort_flag = 1;
        atomicOr(s.status, kStatusTimeout);
        // first expiry only: barrier index, parity, CTA, warp, microseconds waited (at 2 GHz)
        if (atomicCAS(s.status + 1, 0u, 1u) == 0u) {
          s.status[2] = (bar - s.bar0) / 8;
          s.status[3] = parity;
          s.status[4] = blockIdx.x;
          s.status[5] = threadIdx.x / 32;
          s.status[6] = (uint32_t)((now - t0) / 2000);
        }
        return false;
      }
    }
  }
}

// Warp-uniform form: every lane polls, and the warp proceeds only if all lanes saw the
// phase complete, so no lane can run ahead into a .sync.aligned tcgen05 instruction
// while another one is leaving on the abort path.
// The common case (the phase already completed) costs one probe and one vote; the timed
// polling loop only runs after a miss.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Sync& s, uint64_t limit_ns,
                                          bool drain = false) {
  bool ok = mbar_try_wait(bar, parity);
  if (__all_sync(0xffffffffu, ok)) return true;
  if (!ok) ok = bounded_wait(bar, parity, s, limit_ns, drain);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ float silu_mul(float g, float u) { return __fdiv_rn(g, 1.0f + expf(-g)) * u; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

}  // namespace
}  // namespace moe
