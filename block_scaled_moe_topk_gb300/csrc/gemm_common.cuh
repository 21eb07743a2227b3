// gemm_common.cuh -- pieces of the grouped GEMM kernels: operand-format traits and the
// instruction descriptor, tile decoding over the experts' M tiles, bounded mbarrier waits, the epilogue stores (SwiGLU +
// MX requant, or bf16 rows), and the driver entry point that encodes TMA tensor maps.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "moe_internal.h"
#include "mx_device.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

template <int ACT>
struct ActTraits;
template <>
struct ActTraits<0> {                  // E4M3 activations x E2M1 weights
  static constexpr int kKPerStage = 128;
  static constexpr int kMmaK = 32;
  // The weight tile lands with an 8-byte gap after every 8 bytes of codes (32 KiB of shared
  // memory) but its transaction count is the 16 KiB of packed codes read from global memory.
  static constexpr int kBTxBytes = kNTile * 64;
  static constexpr uint32_t kIdescFmt = (0u << 7) | (5u << 10);
};
template <>
struct ActTraits<1> {                  // E2M1 x E2M1, packed
  static constexpr int kKPerStage = 256;
  static constexpr int kMmaK = 64;
  static constexpr int kBTxBytes = kNTile * 128;
  static constexpr uint32_t kIdescFmt = (1u << 7) | (1u << 10);
};

// Block-scaled instruction descriptor: formats, N>>3 at [17,23), E8M0 scales (bit 23),
// M>>4 at [24,29) (M = 128, one CTA); K-major A and B; scale-factor
// byte ids at [29,31) (A) and [4,6) (B).
template <int ACT>
__device__ __forceinline__ uint32_t make_idesc(uint32_t sf_id, int M) {
  return ActTraits<ACT>::kIdescFmt | ((uint32_t)(kNTile >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24) |
         (sf_id << 29) | (sf_id << 4);
}

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

// Single-thread form for roles that run on one lane (TMA and MMA issue): no vote.
__device__ __forceinline__ bool lane_wait(uint32_t bar, uint32_t parity, const Sync& s, uint64_t limit_ns,
                                          bool drain = false) {
  return mbar_try_wait(bar, parity) || bounded_wait(bar, parity, s, limit_ns, drain);
}

// h = silu(g) * u = g / (1 + exp(-g)) * u in fp32 with the fast exponential and reciprocal
// (a few ulp; the 128 per-thread evaluations share the SM with the MMA-issuing thread).  Large
// negative g: exp(-g) = inf, g / inf = -0, the limit.
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

// Epilogue of one thread: `acc` holds accumulator columns [half*128, half*128 + 128) of N tile
// nt for routed row prow (nothing is stored unless `valid`).  Called by all 32 lanes of a warp.
//   EPI 0 (GEMM1): h_j = silu(gate_j) * up_j over the 64 interleaved (gate, up) column pairs,
//                  then MX requantisation of h: two 32-wide blocks, E4M3 (ACT 0) or E2M1
//                  (ACT 1) codes into out_codes [rows, N/2 or N/4] and one E8M0 byte per block
//                  into out_sf (128x4 tile layout over N/2 columns).
//   EPI 1 (GEMM2): the fp32 row rounded to bf16 (nearest even) into out_bf16 [rows, N].
//   EPI 2 (GEMM1, bf16-out form): h_j = silu(gate_j) * up_j rounded to bf16 into out_bf16
//                  [rows, N/2], for a separate requantisation kernel.
//   EPI 3 (GEMM2, FP8 transport): the row times its routing weight row_w[prow] (fp32), four
//                  32-wide blocks as E4M3 codes into out_codes [rows, N] and one E8M0 byte per
//                  block into out_sf [rows, N/32] (row-major, for the combine).
template <int ACT, int EPI>
__device__ __forceinline__ void store_acc_rows(float (&acc)[128], bool valid, int64_t prow, int nt, int half, int N,
                                               uint8_t* out_codes, uint8_t* out_sf, uint16_t* out_bf16,
                                               const float* row_w = nullptr) {
  if (EPI == 0) {
    const int I = N / 2;
    // Padding rows of an expert's segment hold whatever the workspace held before: their
    // accumulators can be huge or non-finite, which sent an IEEE division in SwiGLU down its
    // slow path for the whole warp (measured: A4W4 GEMM1 1.5 -> 2.2 ms with stale bytes).
    // Skip warps with no routed row; give padding lanes of the others zeros.
    if (!__any_sync(0xffffffffu, valid)) return;
    if (!valid) {
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = silu_mul(acc[2 * i], acc[2 * i + 1]);  // h in place
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const float* h = acc + 32 * blk;
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(h[i]));
      const MxScale sc = mx_scale<ACT>(amax);
      const int kb = nt * 4 + half * 2 + blk;  // 32-wide block of h
      if (valid) {
        if (ACT == 0) {
          uint4* dst = reinterpret_cast<uint4*>(out_codes + prow * I + kb * 32);
          const uint2 c0 = pack_e4m3x8(h, sc.mult), c1 = pack_e4m3x8(h + 8, sc.mult);
          const uint2 c2 = pack_e4m3x8(h + 16, sc.mult), c3 = pack_e4m3x8(h + 24, sc.mult);
          dst[0] = make_uint4(c0.x, c0.y, c1.x, c1.y);
          dst[1] = make_uint4(c2.x, c2.y, c3.x, c3.y);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(out_codes + prow * (I / 2) + kb * 16);
          *dst = make_uint4(pack_e2m1x8(h, sc.mult), pack_e2m1x8(h + 8, sc.mult), pack_e2m1x8(h + 16, sc.mult),
                            pack_e2m1x8(h + 24, sc.mult));
        }
        out_sf[sf_tile_offset(prow, kb, I)] = sc.byte;
      }
    }
  } else if (EPI == 2) {
    if (!valid) return;  // padding rows: nothing stored (and no SwiGLU on their stale values)
    const int I = N / 2;
    uint4* d4 = reinterpret_cast<uint4*>(out_bf16 + prow * I + nt * (kNTile / 2) + half * 64);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t w[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = 8 * i + 2 * c;  // h columns j, j + 1 of this thread's 64
        const __nv_bfloat162 hb = __floats2bfloat162_rn(silu_mul(acc[2 * j], acc[2 * j + 1]),
                                                        silu_mul(acc[2 * j + 2], acc[2 * j + 3]));
        w[c] = *reinterpret_cast<const uint32_t*>(&hb);
      }
      d4[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else if (EPI == 3) {
    if (!valid) return;  // padding rows: nothing stored
    // the weight w >= 0 folds into the block maximum and the power-of-two multiplier:
    // max |w * acc| = w * max |acc| and (w * mult) * acc = (w * acc) * mult in fp32 (exact while
    // w * acc is a normal fp32 number: rounding is monotone, mult a power of two)
    const float wgt = row_w[prow];
    const int c0 = nt * kNTile + half * 128;
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
      const float* v = acc + 32 * blk;
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
      const MxScale sc = mx_scale<0>(amax * wgt);
      const float m = sc.mult * wgt;
      uint4* dst = reinterpret_cast<uint4*>(out_codes + prow * N + c0 + 32 * blk);
      const uint2 q0 = pack_e4m3x8(v, m), q1 = pack_e4m3x8(v + 8, m);
      const uint2 q2 = pack_e4m3x8(v + 16, m), q3 = pack_e4m3x8(v + 24, m);
      dst[0] = make_uint4(q0.x, q0.y, q1.x, q1.y);
      dst[1] = make_uint4(q2.x, q2.y, q3.x, q3.y);
      out_sf[prow * (N / 32) + c0 / 32 + blk] = sc.byte;
    }
  } else if (valid) {
    uint4* d4 = reinterpret_cast<uint4*>(out_bf16 + prow * N + nt * kNTile + half * 128);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      uint32_t w[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[8 * i + 2 * c], acc[8 * i + 2 * c + 1]);
        w[c] = *reinterpret_cast<const uint32_t*>(&b);
      }
      d4[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

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

// Tensor map of the activation codes [rows_cap, K] (E4M3: one byte per element; E2M1: two
// per byte): box of 128 bytes x `arows` rows, 128-byte swizzle (the layout the MMA's shared
// memory descriptors expect).  False if the driver rejects it.
inline bool encode_act_map(CUtensorMap* m, const uint8_t* act, int64_t rows_cap, int K, int act_fmt, int arows) {
  EncodeTiledFn encode = get_encode_fn();
  if (!encode) return false;
  const uint64_t row_bytes = act_fmt == 0 ? (uint64_t)K : (uint64_t)K / 2;
  const cuuint64_t dims[2] = {row_bytes, (cuuint64_t)rows_cap};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {128, (cuuint32_t)arows};
  const cuuint32_t es[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(act), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of the MXFP4 weights [E, N, K/2], box 128 K-elements x 256 rows x 1 expert.  With
// E4M3 activations (kind::mxf8f6f4) the packed codes land with an 8-byte gap after every 8
// bytes (16U4_ALIGN16B); with E2M1 activations (kind::mxf4) they stay packed.  Rows past N
// (a 128-row last tile) read as zeros.
inline bool encode_weight_map(CUtensorMap* m, const uint8_t* w, int E, int N, int K, int act_fmt) {
  EncodeTiledFn encode = get_encode_fn();
  if (!encode) return false;
  const uint64_t row_bytes = (uint64_t)K / 2;
  const cuuint64_t strides[2] = {row_bytes, row_bytes * (uint64_t)N};
  const cuuint32_t box[3] = {128, (cuuint32_t)kNTile, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  if (act_fmt == 0) {
    const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)N, (cuuint64_t)E};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<uint8_t*>(w), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t dims[3] = {row_bytes, (cuuint64_t)N, (cuuint64_t)E};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(w), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace moe
