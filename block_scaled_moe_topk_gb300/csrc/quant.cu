// quant.cu -- BF16 -> MXFP8 (E4M3) / MXFP4 (E2M1) quantisation with one E8M0 scale
// per 1x32 block ("add A4W4 and FP8 P2P transport support to MegaMoE", Technical
// Details; OCP Microscaling v1.0 scale rule s = floor(log2 amax) - emax + 127).
//
// Each thread owns 16 consecutive elements (two 16-byte loads); two threads form a
// 32-element block and agree on its amax with one shuffle.  In the forward the
// codes of token t are written straight to its k padded expert rows
// inv_padded[t*k + j] (the permute is fused here), and the scales go to the
// 128x4 tile layout that the GEMM's tensor-memory scale copy reads.
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "mx_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kQuantThreads = 256;

// Thread i of the grid owns elements [16c, 16c + 16) of row r, (r, c) = (i / (K/16), i % (K/16));
// lanes 2m and 2m+1 hold one 32-element block (K % 32 == 0 keeps the pairs inside a row) and
// agree on its amax with one shuffle.  Every lane of a warp runs the same number of rounds.
// Idx: the flat index type (32 bits whenever rows * K / 16 fits: a 64-bit division per element
// group is slow).
template <int FMT, typename Idx>
__global__ void __launch_bounds__(kQuantThreads) quant_kernel(QuantArgs a) {
  const int K = a.K;
  const Idx chunks = (Idx)(K / 16);
  const Idx n = (Idx)a.rows * chunks;
  const int lane = threadIdx.x & 31;
  const Idx stride = (Idx)gridDim.x * blockDim.x;
  for (Idx base = (Idx)blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < n; base += stride) {
    const Idx i = base + lane;
    const bool active = i < n;
    const int64_t row = active ? (int64_t)(i / chunks) : 0;
    const int col0 = active ? (int)(i - (Idx)row * chunks) * 16 : 0;
    float v[16];
    if (active) {
      const uint4* src = reinterpret_cast<const uint4*>(a.x + row * K + col0);
      const uint4 r0 = src[0], r1 = src[1];
      const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        v[2 * q] = __uint_as_float(w[q] << 16);
        v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = 0.0f;
    }
    float amax = 0.0f;
#pragma unroll
    for (int q = 0; q < 16; ++q) amax = fmaxf(amax, fabsf(v[q]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    if (!active) continue;  // both lanes of a pair are active or not (n is even)
    const MxScale sc = mx_scale<FMT>(amax);
    const int kb = col0 / 32;
    const bool scale_writer = (col0 & 31) == 0;
    if (FMT == 0) {
      const uint2 c0 = pack_e4m3x8(v, sc.mult), c1 = pack_e4m3x8(v + 8, sc.mult);
      if (a.inv_padded == nullptr) {  // caller's buffers: 8-byte alignment is what the API asks
        uint2* dst = reinterpret_cast<uint2*>(a.codes + row * K + col0);
        dst[0] = c0;
        dst[1] = c1;
        if (scale_writer) a.scales[row * (K / 32) + kb] = sc.byte;
      } else {  // workspace rows (256-byte aligned, K % 32 == 0): one 16-byte store per row
        if (col0 == 0 && a.row_w != nullptr)  // FP8 transport: each padded row's routing weight
          for (int j = 0; j < a.k; ++j) a.row_w[a.inv_padded[row * a.k + j]] = a.topk_w[row * a.k + j];
        const uint4 c = make_uint4(c0.x, c0.y, c1.x, c1.y);
        for (int j = 0; j < a.k; ++j) {
          const int64_t prow = a.inv_padded[row * a.k + j];
          *reinterpret_cast<uint4*>(a.codes + prow * K + col0) = c;
          if (scale_writer) a.scales[sf_tile_offset(prow, kb, K)] = sc.byte;
        }
      }
    } else {
      const uint2 c = make_uint2(pack_e2m1x8(v, sc.mult), pack_e2m1x8(v + 8, sc.mult));
      if (a.inv_padded == nullptr) {
        *reinterpret_cast<uint2*>(a.codes + row * (K / 2) + col0 / 2) = c;
        if (scale_writer) a.scales[row * (K / 32) + kb] = sc.byte;
      } else {
        if (col0 == 0 && a.row_w != nullptr)
          for (int j = 0; j < a.k; ++j) a.row_w[a.inv_padded[row * a.k + j]] = a.topk_w[row * a.k + j];
        for (int j = 0; j < a.k; ++j) {
          const int64_t prow = a.inv_padded[row * a.k + j];
          *reinterpret_cast<uint2*>(a.codes + prow * (K / 2) + col0 / 2) = c;
          if (scale_writer) a.scales[sf_tile_offset(prow, kb, K)] = sc.byte;
        }
      }
    }
  }
}

// Forward form: one block per token row, thread i owns elements [16i, 16i + 16) (lanes 2m and
// 2m+1 share a 32-element block); the row's k destination rows are read once per thread.  No
// grid-stride loop: every row's loads are in flight at once.
template <int FMT>
__global__ void __launch_bounds__(1024) quant_rows_kernel(QuantArgs a) {
  const int K = a.K;
  const int64_t row = blockIdx.x;
  const int col0 = (int)threadIdx.x * 16;
  const bool active = col0 < K;
  float v[16];
  if (active) {
    const uint4* src = reinterpret_cast<const uint4*>(a.x + row * K + col0);
    const uint4 r0 = src[0], r1 = src[1];
    const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      v[2 * q] = __uint_as_float(w[q] << 16);
      v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 16; ++q) v[q] = 0.0f;
  }
  int prow[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j)
    if (j < a.k) prow[j] = a.inv_padded[row * a.k + j];
  if (a.row_w != nullptr && threadIdx.x < a.k)  // FP8 transport: each padded row's routing weight
    a.row_w[a.inv_padded[row * a.k + threadIdx.x]] = a.topk_w[row * a.k + threadIdx.x];
  float amax = 0.0f;
#pragma unroll
  for (int q = 0; q < 16; ++q) amax = fmaxf(amax, fabsf(v[q]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  if (!active) return;  // whole lane pairs are active or not (K % 32 == 0)
  const MxScale sc = mx_scale<FMT>(amax);
  const int kb = col0 / 32;
  const bool scale_writer = (col0 & 31) == 0;
  if (FMT == 0) {
    const uint2 c0 = pack_e4m3x8(v, sc.mult), c1 = pack_e4m3x8(v + 8, sc.mult);
    const uint4 c = make_uint4(c0.x, c0.y, c1.x, c1.y);
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < a.k) {
        *reinterpret_cast<uint4*>(a.codes + (int64_t)prow[j] * K + col0) = c;
        if (scale_writer) a.scales[sf_tile_offset(prow[j], kb, K)] = sc.byte;
      }
  } else {
    const uint2 c = make_uint2(pack_e2m1x8(v, sc.mult), pack_e2m1x8(v + 8, sc.mult));
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < a.k) {
        *reinterpret_cast<uint2*>(a.codes + (int64_t)prow[j] * (K / 2) + col0 / 2) = c;
        if (scale_writer) a.scales[sf_tile_offset(prow[j], kb, K)] = sc.byte;
      }
  }
}

// Requantisation of the bf16-out GEMM1 form: one block per routed pair q, thread i owns
// elements [16i, 16i + 16) of the row's h; the codes and scales go to the same padded row.
template <int FMT>
__global__ void __launch_bounds__(1024) requant_rows_kernel(RequantArgs a) {
  const int K = a.K;
  const int64_t prow = a.inv_padded[blockIdx.x];
  const int col0 = (int)threadIdx.x * 16;
  const bool active = col0 < K;
  float v[16];
  if (active) {
    const uint4* src = reinterpret_cast<const uint4*>(a.h + prow * K + col0);
    const uint4 r0 = src[0], r1 = src[1];
    const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      v[2 * q] = __uint_as_float(w[q] << 16);
      v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 16; ++q) v[q] = 0.0f;
  }
  float amax = 0.0f;
#pragma unroll
  for (int q = 0; q < 16; ++q) amax = fmaxf(amax, fabsf(v[q]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  if (!active) return;
  const MxScale sc = mx_scale<FMT>(amax);
  const int kb = col0 / 32;
  if (FMT == 0) {
    const uint2 c0 = pack_e4m3x8(v, sc.mult), c1 = pack_e4m3x8(v + 8, sc.mult);
    *reinterpret_cast<uint4*>(a.codes + prow * K + col0) = make_uint4(c0.x, c0.y, c1.x, c1.y);
  } else {
    *reinterpret_cast<uint2*>(a.codes + prow * (K / 2) + col0 / 2) =
        make_uint2(pack_e2m1x8(v, sc.mult), pack_e2m1x8(v + 8, sc.mult));
  }
  if ((col0 & 31) == 0) a.scales[sf_tile_offset(prow, kb, K)] = sc.byte;
}

// Canonical E8M0 scales [rows, K/32] -> the 128x4 tile layout the GEMM copies to TMEM:
// thread i moves the 4 scale bytes (one 128-wide k-atom) of one row.
__global__ void __launch_bounds__(256) prepack_scales_kernel(const uint8_t* src, int64_t rows, int K, uint8_t* dst) {
  const int groups = K / 128;
  const int64_t n = rows * groups;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / groups;
    const int g = (int)(i % groups);
    const uint32_t v = *reinterpret_cast<const uint32_t*>(src + r * (K / 32) + 4 * g);
    *reinterpret_cast<uint32_t*>(dst + ((r >> 7) * groups + g) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4) = v;
  }
}

// Prequantised input: token t's code row (and its scales) copied to its k padded expert rows,
// scales into the 128x4 tile layout -- the quantiser's scatter without its arithmetic.  Idx as
// for quant_kernel.
template <typename Idx>
__global__ void __launch_bounds__(256) permute_rows_kernel(PermuteArgs a) {
  const int64_t row_bytes = a.code_bytes;        // multiple of 16
  const Idx chunks = (Idx)(row_bytes / 16);
  const Idx n = (Idx)a.rows * chunks;
  for (Idx i = (Idx)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (Idx)gridDim.x * blockDim.x) {
    const int64_t t = (int64_t)(i / chunks);
    const int64_t c = (int64_t)(i - (Idx)t * chunks);
    const uint4 v = *reinterpret_cast<const uint4*>(a.codes_in + t * row_bytes + c * 16);
    for (int j = 0; j < a.k; ++j)
      *reinterpret_cast<uint4*>(a.codes_out + (int64_t)a.inv_padded[t * a.k + j] * row_bytes + c * 16) = v;
  }
  if (a.row_w != nullptr)  // FP8 transport: each padded row's routing weight
    for (Idx q = (Idx)blockIdx.x * blockDim.x + threadIdx.x; q < (Idx)a.rows * a.k; q += (Idx)gridDim.x * blockDim.x)
      a.row_w[a.inv_padded[q]] = a.topk_w[q];
  const Idx nb = (Idx)(a.K / 32);
  const Idx ns = (Idx)a.rows * nb;
  for (Idx i = (Idx)blockIdx.x * blockDim.x + threadIdx.x; i < ns; i += (Idx)gridDim.x * blockDim.x) {
    const int64_t t = (int64_t)(i / nb);
    const int kb = (int)(i - (Idx)t * nb);
    const uint8_t v = a.scales_in[t * nb + kb];
    for (int j = 0; j < a.k; ++j) a.scales_out[sf_tile_offset(a.inv_padded[t * a.k + j], kb, a.K)] = v;
  }
}

}  // namespace

cudaError_t launch_permute_rows(const PermuteArgs& a, cudaStream_t s) {
  const int64_t n = a.rows * (a.code_bytes / 16);
  if (n == 0) return cudaSuccess;
  const unsigned grid = (unsigned)std::min<int64_t>((n + 255) / 256, 152 * 32);
  if (n < ((int64_t)1 << 31))  // rows * K / 32 <= n as well
    permute_rows_kernel<uint32_t><<<grid, 256, 0, s>>>(a);
  else
    permute_rows_kernel<int64_t><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_requant(const RequantArgs& a, cudaStream_t s) {
  if (a.R == 0) return cudaSuccess;
  if (a.K > 16 * 1024 || a.R > 0x7fffffff) return cudaErrorInvalidValue;
  const unsigned threads = (unsigned)((a.K / 16 + 31) / 32 * 32);
  if (a.fmt == 0) requant_rows_kernel<0><<<(unsigned)a.R, threads, 0, s>>>(a);
  else requant_rows_kernel<1><<<(unsigned)a.R, threads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prepack_scales(const uint8_t* src, int64_t rows, int K, uint8_t* dst, cudaStream_t s) {
  const int64_t n = rows * (K / 128);
  if (n == 0) return cudaSuccess;
  const unsigned grid = (unsigned)std::min<int64_t>((n + 255) / 256, 152 * 32);
  prepack_scales_kernel<<<grid, 256, 0, s>>>(src, rows, K, dst);
  return cudaGetLastError();
}

cudaError_t launch_quant(const QuantArgs& a, cudaStream_t s) {
  const int64_t n = a.rows * (a.K / 16);
  if (n == 0) return cudaSuccess;
  if (a.inv_padded != nullptr && a.K <= 16 * 1024 && a.rows <= 0x7fffffff) {
    // forward: one block per token row (threads rounded up to whole warps)
    const unsigned threads = (unsigned)((a.K / 16 + 31) / 32 * 32);
    if (a.fmt == 0) quant_rows_kernel<0><<<(unsigned)a.rows, threads, 0, s>>>(a);
    else quant_rows_kernel<1><<<(unsigned)a.rows, threads, 0, s>>>(a);
    return cudaGetLastError();
  }
  const unsigned grid = (unsigned)std::min<int64_t>((n + kQuantThreads - 1) / kQuantThreads, 152 * 8);
  const bool narrow = n < ((int64_t)1 << 31);
  if (a.fmt == 0) {
    if (narrow) quant_kernel<0, uint32_t><<<grid, kQuantThreads, 0, s>>>(a);
    else quant_kernel<0, int64_t><<<grid, kQuantThreads, 0, s>>>(a);
  } else {
    if (narrow) quant_kernel<1, uint32_t><<<grid, kQuantThreads, 0, s>>>(a);
    else quant_kernel<1, int64_t><<<grid, kQuantThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace moe
