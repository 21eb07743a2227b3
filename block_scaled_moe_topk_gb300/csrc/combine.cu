// combine.cu -- top-k weighted combine back to token order.
//
// out[t, n] = bf16_rne( sum_{j<k} topk_w[t, j] * y2[inv_padded[t*k + j], n] ), accumulated in
// fp32 in slot order: the page "add A4W4 and FP8 P2P transport support to MegaMoE" (Technical
// Details) sums the top-k contributions of a token in single precision; y2 rows are bf16.  Each thread owns 8
// consecutive columns: one 16-byte load per slot, one 16-byte bf16 store.  The flat index runs in
// 32 bits whenever T * H / 8 fits (a 64-bit division per element group cost 11-17 % of the
// kernel at T = 8192-32768).  With the FP8 transport of the GEMM2 rows the weights are already
// applied and the rows arrive as E4M3 codes with E8M0 scales (combine_fp8_kernel).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kCombineThreads = 256;

template <typename Idx>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineArgs a) {
  const int H = a.H, k = a.k;
  const Idx groups = (Idx)(H / 8);  // 8 columns per thread
  const Idx work = (Idx)a.T * groups;
  for (Idx i = (Idx)blockIdx.x * blockDim.x + threadIdx.x; i < work; i += (Idx)gridDim.x * blockDim.x) {
    const int64_t t = (int64_t)(i / groups);
    const int c0 = (int)(i - (Idx)t * groups) * 8;
    // all k row loads in flight before the first FMA (k <= kMaxTopK)
    int rows[kMaxTopK];
    float w[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) {
        rows[j] = a.inv_padded[t * k + j];
        w[j] = a.w[t * k + j];
      }
    uint4 raw[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) raw[j] = *reinterpret_cast<const uint4*>(a.y2 + (int64_t)rows[j] * H + c0);
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k) {  // slot order
        const uint32_t u[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          acc[2 * c] = fmaf(w[j], __uint_as_float(u[c] << 16), acc[2 * c]);              // low half: column c0+2c
          acc[2 * c + 1] = fmaf(w[j], __uint_as_float(u[c] & 0xFFFF0000u), acc[2 * c + 1]);
        }
      }
    }
    uint32_t packed[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * c], acc[2 * c + 1]);  // .x = low half
      packed[c] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(a.out + t * H + c0) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
}

// FP8 transport: the k rows of a token arrive already weighted, as E4M3 codes with one E8M0
// scale per 32 columns; out = bf16_rne(sum over slots of code value * 2^(scale - 127)), fp32 in
// slot order.  Each thread owns 8 consecutive columns: one 8-byte code load and one scale byte
// per slot.  The decode decides the speed: the hardware pair conversion E4M3 -> f16, then one
// mixed-precision FMA per value into the fp32 sum (below); with f16 -> f32 conversions in between
// the kernel was slower than the bf16 combine despite half the bytes, and an integer decode (sign
// and bits placed into an fp32 and rescaled) slower still.  It then runs at ~60 % of DRAM
// bandwidth with the ALU pipe ~60 % busy.
template <typename Idx>
__global__ void __launch_bounds__(kCombineThreads) combine_fp8_kernel(CombineArgs a) {
  const int H = a.H, k = a.k;
  const Idx groups = (Idx)(H / 8);
  const Idx work = (Idx)a.T * groups;
  for (Idx i = (Idx)blockIdx.x * blockDim.x + threadIdx.x; i < work; i += (Idx)gridDim.x * blockDim.x) {
    const int64_t t = (int64_t)(i / groups);
    const int c0 = (int)(i - (Idx)t * groups) * 8;
    int rows[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) rows[j] = a.inv_padded[t * k + j];
    uint2 raw[kMaxTopK];
    uint32_t sb[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) {
        raw[j] = *reinterpret_cast<const uint2*>(a.y2q + (int64_t)rows[j] * H + c0);
        sb[j] = a.y2s[(int64_t)rows[j] * (H / 32) + c0 / 32];
      }
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k) {  // slot order
        const uint32_t u[2] = {raw[j].x, raw[j].y};
        if (sb[j] >= 113 && sb[j] <= 142) {
          // 2^(s - 127) is a normal f16: one mixed-precision FMA per value (the f16 x f16 product is
          // exact in fp32, so the result equals the fp32 path's: one rounding in the add)
          const uint16_t sh = (uint16_t)((sb[j] - 112u) << 10);  // f16 bits of 2^(s - 127)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int b = 0; b < 4; b += 2) {
              const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((u[h] >> (8 * b)) & 0xFFFFu);
              const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
              const uint16_t lo = hr.x, hi = hr.y;
              asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc[4 * h + b]) : "h"(lo), "h"(sh));
              asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc[4 * h + b + 1]) : "h"(hi), "h"(sh));
            }
        } else {
          // 2^(s - 127) as an fp32 bit pattern (s = 0: the subnormal 2^-127)
          const float scale = sb[j] == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(sb[j] << 23);
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int b = 0; b < 4; b += 2) {  // element 2i in the low byte of each pair
              const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((u[h] >> (8 * b)) & 0xFFFFu);
              const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3)));
              acc[4 * h + b] = fmaf(f.x, scale, acc[4 * h + b]);
              acc[4 * h + b + 1] = fmaf(f.y, scale, acc[4 * h + b + 1]);
            }
        }
      }
    }
    uint32_t packed[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * c], acc[2 * c + 1]);
      packed[c] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(a.out + t * H + c0) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  const int64_t work = a.T * (a.H / 8);
  if (work == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((work + kCombineThreads - 1) / kCombineThreads, 152 * 16);
  const bool narrow = work < ((int64_t)1 << 31);
  if (a.y2 == nullptr) {  // FP8 transport
    if (narrow) combine_fp8_kernel<uint32_t><<<(unsigned)blocks, kCombineThreads, 0, s>>>(a);
    else combine_fp8_kernel<int64_t><<<(unsigned)blocks, kCombineThreads, 0, s>>>(a);
  } else if (narrow) {
    combine_kernel<uint32_t><<<(unsigned)blocks, kCombineThreads, 0, s>>>(a);
  } else {
    combine_kernel<int64_t><<<(unsigned)blocks, kCombineThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace moe
