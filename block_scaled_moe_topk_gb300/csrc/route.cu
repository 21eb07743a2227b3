// route.cu -- top-k softmax gating (eight lanes per token up to 512 experts, a warp per
// token beyond), with the per-chunk expert histogram of the routed pairs fused in.
//
// Gating as in "[HIP] gfx950 A8W4 fused_moe configs for DSv4.1 TP-sharded
// experts" (Changes: the top-k softmax kernel): experts ranked by fp32 logit,
// descending, ties to the lower index; the k selected softmax probabilities are
// renormalised to sum 1, which reduces to exp(l_j - l_max) / sum_i exp(l_i - l_max)
// over the selected experts because the full softmax denominator cancels.
#include "moe_internal.h"
#include "route_device.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;

// Block b routes tokens [b*kTokensPerChunk, (b+1)*kTokensPerChunk) and, if asked,
// writes the chunk's expert histogram to chunk_hist[e * nchunk + b].
template <int kPerLane>
__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(RouteArgs a) {
  __shared__ int hist[kMaxExperts];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int E = a.E, k = a.k;
  // status word and the expired-wait record after it (8 words) start clean on every forward
  if (a.reset_status && blockIdx.x == 0 && threadIdx.x < 8) a.status[threadIdx.x] = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();

  const int64_t t_begin = (int64_t)blockIdx.x * kTokensPerChunk;
  const int64_t t_end = (a.T < t_begin + kTokensPerChunk) ? a.T : t_begin + kTokensPerChunk;
  for (int64_t t = t_begin + warp; t < t_end; t += kRouteWarps) {
    int my_id;
    float my_w;
    route_token_fast<kPerLane>(a.logits + t * E, E, k, lane, my_id, my_w);
    if (lane < k) {
      a.ids[t * k + lane] = my_id;
      a.w[t * k + lane] = my_w;
      if (a.chunk_hist) atomicAdd(&hist[my_id], 1);
    }
  }
  if (a.chunk_hist) {
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) a.chunk_hist[(int64_t)e * a.nchunk + blockIdx.x] = hist[e];
  }
}

// E <= 512: eight lanes per token, the block's 32 tokens in one pass (8 warps x 4 tokens).
template <int kV>
__global__ void __launch_bounds__(kRouteWarps * 32) route8_kernel(RouteArgs a) {
  static_assert(kRouteWarps * 4 == kTokensPerChunk, "one pass per chunk");
  __shared__ int hist[kV * 8];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, g = lane & 7;
  const int E = a.E, k = a.k;
  if (a.reset_status && blockIdx.x == 0 && threadIdx.x < 8) a.status[threadIdx.x] = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t t = (int64_t)blockIdx.x * kTokensPerChunk + warp * 4 + (lane >> 3);
  const bool valid = t < a.T;
  int my_id;
  float my_w;
  route_token8<kV>(a.logits + (valid ? t : 0) * E, valid, E, k, g, my_id, my_w);
  if (valid && g < k) {
    a.ids[t * k + g] = my_id;
    a.w[t * k + g] = my_w;
    if (a.chunk_hist) atomicAdd(&hist[my_id], 1);
  }
  if (a.chunk_hist) {
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) a.chunk_hist[(int64_t)e * a.nchunk + blockIdx.x] = hist[e];
  }
}

// Histogram of caller-supplied ids (the standalone sort entry point).
__global__ void __launch_bounds__(256) histogram_kernel(SortArgs a) {
  __shared__ int hist[kMaxExperts];
  const int E = a.E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t q_begin = (int64_t)blockIdx.x * kTokensPerChunk * a.k;
  const int64_t q_lim = q_begin + (int64_t)kTokensPerChunk * a.k;
  const int64_t q_end = (a.T * a.k < q_lim) ? a.T * a.k : q_lim;
  for (int64_t q = q_begin + threadIdx.x; q < q_end; q += blockDim.x) {
    const int id = a.ids[q];
    if (id >= 0 && id < E) atomicAdd(&hist[id], 1);
    else atomicOr(a.status, kStatusInvalidArg);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) a.chunk_hist[(int64_t)e * a.nchunk + blockIdx.x] = hist[e];
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
  const int64_t blocks = (a.T + kTokensPerChunk - 1) / kTokensPerChunk;
  if (blocks == 0) return cudaSuccess;
  const unsigned nb = (unsigned)blocks, nt = kRouteWarps * 32;
  if (a.E <= 64) route8_kernel<8><<<nb, nt, 0, s>>>(a);
  else if (a.E <= 128) route8_kernel<16><<<nb, nt, 0, s>>>(a);
  else if (a.E <= 256) route8_kernel<32><<<nb, nt, 0, s>>>(a);
  else if (a.E <= 384) route8_kernel<48><<<nb, nt, 0, s>>>(a);
  else if (a.E <= 512) route8_kernel<64><<<nb, nt, 0, s>>>(a);
  else route_kernel<32><<<nb, nt, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_histogram(const SortArgs& a, cudaStream_t s) {
  const int64_t blocks = (a.T + kTokensPerChunk - 1) / kTokensPerChunk;
  if (blocks == 0) return cudaSuccess;
  histogram_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
