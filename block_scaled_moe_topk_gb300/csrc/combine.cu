// combine.cu -- top-k weighted combine back to token order.
//
// out[t, n] = bf16_rne( sum_{j<k} topk_w[t, j] * y2[inv_padded[t*k + j], n] ), accumulated in
// fp32 in slot order ("add A4W4 and FP8 P2P transport support to MegaMoE", Technical
// Details: "accumulate TopK contributions in FP32").  Each thread owns 8 consecutive
// columns: two 16-byte loads per slot, one 16-byte bf16 store.
#include <cuda_bf16.h>

#include <algorithm>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kCombineThreads = 256;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineArgs a) {
  const int H = a.H, k = a.k;
  const int groups = H / 8;  // 8 columns per thread
  const int64_t work = a.T * groups;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < work; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / groups;
    const int c0 = (int)(i % groups) * 8;
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.0f;
    for (int j = 0; j < k; ++j) {
      const float w = a.w[t * k + j];
      const float4* src = reinterpret_cast<const float4*>(a.y2 + (int64_t)a.inv_padded[t * k + j] * H + c0);
      const float4 v0 = src[0], v1 = src[1];
      acc[0] = fmaf(w, v0.x, acc[0]);
      acc[1] = fmaf(w, v0.y, acc[1]);
      acc[2] = fmaf(w, v0.z, acc[2]);
      acc[3] = fmaf(w, v0.w, acc[3]);
      acc[4] = fmaf(w, v1.x, acc[4]);
      acc[5] = fmaf(w, v1.y, acc[5]);
      acc[6] = fmaf(w, v1.z, acc[6]);
      acc[7] = fmaf(w, v1.w, acc[7]);
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

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  const int64_t work = a.T * (a.H / 8);
  if (work == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((work + kCombineThreads - 1) / kCombineThreads, 152 * 16);
  combine_kernel<<<(unsigned)blocks, kCombineThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
