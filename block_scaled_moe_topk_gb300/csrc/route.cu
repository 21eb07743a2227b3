// route.cu -- top-k softmax gating, one warp per token, with the per-chunk expert
// histogram of the routed pairs fused in.
//
// Gating as in "[HIP] gfx950 A8W4 fused_moe configs for DSv4.1 TP-sharded
// experts" (Changes: the top-k softmax kernel): experts ranked by fp32 logit,
// descending, ties to the lower index; the k selected softmax probabilities are
// renormalised to sum 1, which reduces to exp(l_j - l_max) / sum_i exp(l_i - l_max)
// over the selected experts because the full softmax denominator cancels.
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;
constexpr int kMaxPerLane = kMaxExperts / 32;

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Block b routes tokens [b*kTokensPerChunk, (b+1)*kTokensPerChunk) and, if asked,
// writes the chunk's expert histogram to chunk_hist[e * nchunk + b].
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
  const int per_lane = (E + 31) / 32;
  for (int64_t t = t_begin + warp; t < t_end; t += kRouteWarps) {
    const float* l = a.logits + t * E;
    float v[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      v[i] = (i < per_lane && e < E) ? l[e] : 0.0f;
    }
    uint32_t taken = 0;
    int my_id = 0;
    float my_val = 0.0f, lmax = 0.0f;
    for (int j = 0; j < k; ++j) {
      // lane-local best among the experts not yet taken
      float bv = 0.0f;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        const int e = lane + 32 * i;
        if (i < per_lane && e < E && !((taken >> i) & 1u)) {
          if (bi == 0x7fffffff || better(v[i], e, bv, bi)) {
            bv = v[i];
            bi = e;
          }
        }
      }
      // warp arg-max (value desc, index asc)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (oi != 0x7fffffff && (bi == 0x7fffffff || better(ov, oi, bv, bi))) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi / 32);
      if (j == 0) lmax = bv;
      if (lane == j) {
        my_id = bi;
        my_val = bv;
      }
    }
    // p_j = exp(l_j - l_max) without fp64 (scarce on this GPU): the difference is split
    // exactly into s + e (two-sum), so its rounding is not amplified by exp, and
    // exp(s + e) = expf(s) * (1 + e) because |e| <= ulp(s) / 2.
    float p = 0.0f;
    if (lane < k) {
      const float sdiff = my_val - lmax;
      const float bb = sdiff - my_val;
      const float e = (my_val - (sdiff - bb)) + (-lmax - bb);
      p = expf(sdiff) * (1.0f + e);
    }
    // z = sum of the k values as a compensated (hi, lo) pair, so w = p / z loses <= 1 ulp
    float zh = p, zl = 0.0f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float oh = __shfl_xor_sync(0xffffffffu, zh, off);
      const float ol = __shfl_xor_sync(0xffffffffu, zl, off);
      const float sum = zh + oh;
      const float bv = sum - zh;
      zl += ol + ((zh - (sum - bv)) + (oh - bv));
      zh = sum;
    }
    if (lane < k) {
      a.ids[t * k + lane] = my_id;
      a.w[t * k + lane] = __fdiv_rn(p, zh) * (1.0f - __fdiv_rn(zl, zh));
      if (a.chunk_hist) atomicAdd(&hist[my_id], 1);
    }
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
  route_kernel<<<(unsigned)blocks, kRouteWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_histogram(const SortArgs& a, cudaStream_t s) {
  const int64_t blocks = (a.T + kTokensPerChunk - 1) / kTokensPerChunk;
  if (blocks == 0) return cudaSuccess;
  histogram_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
