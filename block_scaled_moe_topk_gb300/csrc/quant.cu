// quant.cu -- BF16 -> MXFP8 (E4M3) / MXFP4 (E2M1) quantisation with one E8M0 scale
// per 1x32 block ("add A4W4 and FP8 P2P transport support to MegaMoE", Technical
// Details; OCP Microscaling v1.0 scale rule s = floor(log2 amax) - emax + 127).
//
// Each thread owns 8 consecutive elements (one 16-byte load); four threads form a
// 32-element block and agree on its amax with two shuffles.  In the forward the
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
constexpr int kColsPerBlock = kQuantThreads * 8;

template <int FMT>
__global__ void __launch_bounds__(kQuantThreads) quant_kernel(QuantArgs a) {
  const int K = a.K;
  const int col_blocks = (K + kColsPerBlock - 1) / kColsPerBlock;
  const int64_t work = a.rows * col_blocks;
  for (int64_t wi = blockIdx.x; wi < work; wi += gridDim.x) {
    const int64_t row = wi / col_blocks;
    const int col0 = (int)(wi % col_blocks) * kColsPerBlock + threadIdx.x * 8;
    const bool active = col0 < K;
    float v[8];
    if (active) {
      const uint4 raw = *reinterpret_cast<const uint4*>(a.x + row * K + col0);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    if (!active) continue;  // whole 4-lane groups are active or not (K % 32 == 0)
    const MxScale sc = mx_scale<FMT>(amax);
    const int kb = col0 / 32;
    const bool scale_writer = (threadIdx.x & 3) == 0;
    if (FMT == 0) {
      const uint2 codes = pack_e4m3x8(v, sc.mult);
      if (a.inv_padded == nullptr) {
        *reinterpret_cast<uint2*>(a.codes + row * K + col0) = codes;
        if (scale_writer) a.scales[row * (K / 32) + kb] = sc.byte;
      } else {
        for (int j = 0; j < a.k; ++j) {
          const int64_t prow = a.inv_padded[row * a.k + j];
          *reinterpret_cast<uint2*>(a.codes + prow * K + col0) = codes;
          if (scale_writer) a.scales[sf_tile_offset(prow, kb, K)] = sc.byte;
        }
      }
    } else {
      const uint32_t codes = pack_e2m1x8(v, sc.mult);
      if (a.inv_padded == nullptr) {
        *reinterpret_cast<uint32_t*>(a.codes + row * (K / 2) + col0 / 2) = codes;
        if (scale_writer) a.scales[row * (K / 32) + kb] = sc.byte;
      } else {
        for (int j = 0; j < a.k; ++j) {
          const int64_t prow = a.inv_padded[row * a.k + j];
          *reinterpret_cast<uint32_t*>(a.codes + prow * (K / 2) + col0 / 2) = codes;
          if (scale_writer) a.scales[sf_tile_offset(prow, kb, K)] = sc.byte;
        }
      }
    }
  }
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
// scales into the 128x4 tile layout -- the quantiser's scatter without its arithmetic.
__global__ void __launch_bounds__(256) permute_rows_kernel(PermuteArgs a) {
  const int64_t row_bytes = a.code_bytes;        // multiple of 16
  const int64_t chunks = row_bytes / 16;
  const int64_t n = a.rows * chunks;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / chunks, c = i % chunks;
    const uint4 v = *reinterpret_cast<const uint4*>(a.codes_in + t * row_bytes + c * 16);
    for (int j = 0; j < a.k; ++j)
      *reinterpret_cast<uint4*>(a.codes_out + (int64_t)a.inv_padded[t * a.k + j] * row_bytes + c * 16) = v;
  }
  const int nb = a.K / 32;
  const int64_t ns = a.rows * nb;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < ns; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / nb;
    const int kb = (int)(i % nb);
    const uint8_t v = a.scales_in[t * nb + kb];
    for (int j = 0; j < a.k; ++j) a.scales_out[sf_tile_offset(a.inv_padded[t * a.k + j], kb, a.K)] = v;
  }
}

}  // namespace

cudaError_t launch_permute_rows(const PermuteArgs& a, cudaStream_t s) {
  const int64_t n = a.rows * (a.code_bytes / 16);
  if (n == 0) return cudaSuccess;
  const unsigned grid = (unsigned)std::min<int64_t>((n + 255) / 256, 152 * 32);
  permute_rows_kernel<<<grid, 256, 0, s>>>(a);
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
  const int col_blocks = (a.K + kColsPerBlock - 1) / kColsPerBlock;
  const int64_t work = a.rows * col_blocks;
  if (work == 0) return cudaSuccess;
  const unsigned grid = (unsigned)std::min<int64_t>(work, 152 * 16);
  if (a.fmt == 0) quant_kernel<0><<<grid, kQuantThreads, 0, s>>>(a);
  else quant_kernel<1><<<grid, kQuantThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
