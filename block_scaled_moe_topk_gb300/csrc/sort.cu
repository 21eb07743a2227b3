// sort.cu -- deterministic, stable sort of the routed (token, slot) pairs by expert.
//
// The local form of the dispatch step of "feat(moe): FlyDSL MegaMoE fused EP-MoE
// integration" (description: dispatch+gemm1+quant+gemm2+combine).  Offsets are
// 64-bit: the same page reports an int32 kernel argument overflowing above 8192
// batched tokens per rank.
//
// Three phases, no atomics on the output order:
//   1. per-chunk expert histograms (route.cu, fused into the routing kernel);
//   2. a warp per expert: exclusive prefix over chunks -> chunk bases, counts;
//   3. a warp per chunk: prefixes over experts -> offsets, 128-row padded offsets,
//      M-tile bases (written once), then it walks its pairs in order and places each
//      at offset[e] + chunk_base[e] + rank, so equal experts keep pair order.
#include "moe_internal.h"
#include "route_device.cuh"

namespace moe {
namespace {

constexpr int kScanThreads = 1024;

template <typename T>
__device__ __forceinline__ T warp_inclusive_scan(T v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const T o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  return v;
}

// Phase 2a: one warp per expert turns its row of per-chunk counts into exclusive per-chunk
// bases (in place) and writes the expert's total to counts[e].  Rows are independent, so
// the experts spread over E / 8 blocks.
constexpr int kColWarps = 8;

__global__ void __launch_bounds__(kColWarps * 32) scan_cols_kernel(SortArgs a) {
  const int lane = threadIdx.x % 32;
  const int e = blockIdx.x * kColWarps + threadIdx.x / 32;
  if (e >= a.E) return;
  const int64_t nchunk = a.nchunk;
  int32_t* col = a.chunk_hist + (int64_t)e * nchunk;
  int running = 0;
  // 8 runs of 32 chunks are loaded before any is scanned, so the loads overlap
  constexpr int kRounds = 8;
  for (int64_t b0 = 0; b0 < nchunk; b0 += 32 * kRounds) {
    int v[kRounds];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int64_t b = b0 + 32 * r + lane;
      v[r] = (b < nchunk) ? col[b] : 0;
    }
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int64_t b = b0 + 32 * r + lane;
      const int incl = warp_inclusive_scan<int>(v[r], lane);
      if (b < nchunk) col[b] = running + incl - v[r];
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (lane == 0) a.counts[e] = running;
}

// Phase 2b + 3, one warp per chunk.  The warp first forms the exclusive prefixes over experts
// of the routed rows and of the 128-row padded rows from counts[] (every chunk's warp does
// this for itself; chunk 0's also writes offsets, padded offsets and M-tile bases), then walks
// its pairs in order and places each at offset[e] + chunk_base[e] + rank, so equal experts
// keep pair order.  Every global load (the expert totals, this chunk's column of the per-chunk
// histogram, the chunk's expert ids) is issued before the first is used, so the warp pays one
// load latency instead of one per phase and per pass.  Dynamic shared memory: E x (int64 offset,
// int64 padded offset, int32 next).
__global__ void __launch_bounds__(32) scatter_kernel(SortArgs a) {
  static_assert(kTokensPerChunk == 32, "one pass of the warp per slot");
  extern __shared__ __align__(8) uint8_t sort_smem[];
  const int lane = threadIdx.x;
  const int E = a.E, k = a.k;
  int64_t* off_s = reinterpret_cast<int64_t*>(sort_smem);
  int64_t* poff_s = off_s + E;
  int* next = reinterpret_cast<int*>(poff_s + E);
  const int64_t b = blockIdx.x;
  constexpr int kPer = kMaxExperts / 32;
  int cnt[kPer], col[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    cnt[i] = e < E ? a.counts[e] : 0;
    col[i] = e < E ? a.chunk_hist[(int64_t)e * a.nchunk + b] : 0;
  }
  const int64_t q_begin = b * kTokensPerChunk * k;
  const int64_t q_lim = q_begin + (int64_t)kTokensPerChunk * k;
  const int64_t q_end = (a.T * k < q_lim) ? a.T * k : q_lim;
  int idv[kMaxTopK];  // pass j holds pairs q_begin + 32 j + lane
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    const int64_t q = q_begin + 32 * j + lane;
    idv[j] = (j < k && q < q_end) ? a.ids[q] : -1;
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    if (lane + 32 * i < E) next[lane + 32 * i] = cnt[i];
  __syncwarp();
  // lane L owns experts [L * per, L * per + per)
  const int per = (E + 31) / 32;
  const int e0 = min(lane * per, E), e1 = min(e0 + per, E);
  int64_t s = 0, sp = 0;
  for (int e = e0; e < e1; ++e) {
    const int64_t c = next[e];
    s += c;
    sp += (c + kRowTile - 1) / kRowTile * kRowTile;
  }
  int64_t xs = warp_inclusive_scan<int64_t>(s, lane) - s;
  int64_t xsp = warp_inclusive_scan<int64_t>(sp, lane) - sp;
  const bool head = b == 0;
  for (int e = e0; e < e1; ++e) {
    const int64_t c = next[e];
    off_s[e] = xs;
    poff_s[e] = xsp;
    if (head) {
      a.offsets[e] = xs;
      if (a.padded_offsets) a.padded_offsets[e] = xsp;
      if (a.mtile_base) a.mtile_base[e] = (int32_t)(xsp / kRowTile);
    }
    xs += c;
    xsp += (c + kRowTile - 1) / kRowTile * kRowTile;
  }
  if (head && lane == 31) {  // lane 31 ends at the totals
    a.offsets[E] = xs;
    if (a.padded_offsets) a.padded_offsets[E] = xsp;
    if (a.mtile_base) a.mtile_base[E] = (int32_t)(xsp / kRowTile);
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    if (lane + 32 * i < E) next[lane + 32 * i] = col[i];
  __syncwarp();
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j >= k) break;
    const int64_t q = q_begin + 32 * j + lane;
    int id = idv[j];
    const bool valid = q < q_end && id >= 0 && id < E;
    if (!valid) id = -1 - lane;  // a group of its own
    const uint32_t peers = __match_any_sync(0xffffffffu, id);
    const int rank = __popc(peers & lt_mask);
    const int leader = __ffs(peers) - 1;
    int base = valid ? next[id] : 0;
    __syncwarp();
    if (valid && lane == leader) next[id] = base + __popc(peers);
    __syncwarp();
    if (valid) {
      const int64_t local = (int64_t)base + rank;
      const int64_t r = off_s[id] + local;
      a.sorted_pair[r] = (int32_t)q;
      a.inv[q] = (int32_t)r;
      if (a.inv_padded) a.inv_padded[q] = (int32_t)(poff_s[id] + local);
    }
  }
}

// Small batches (T <= kSmallRouteTokens): routing, histogram, the prefix sums and the stable
// scatter in one block, so a decode step pays one launch instead of three.  Same results as
// the routing kernel + scan_cols_kernel + scatter_kernel.
constexpr int kSmallMaxRows = kSmallRouteTokens * kMaxTopK;

template <int kPerLane, int kV>
__global__ void __launch_bounds__(kScanThreads) route_sort_small_kernel(RouteArgs ra, SortArgs sa) {
  __shared__ int cnt[kMaxExperts];
  __shared__ int next[kMaxExperts];
  __shared__ int64_t off_s[kMaxExperts];
  __shared__ int64_t poff_s[kMaxExperts];
  __shared__ int ids_s[kSmallMaxRows];
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int E = ra.E, k = ra.k;
  const int64_t T = ra.T;
  if (ra.reset_status && threadIdx.x < 8) ra.status[threadIdx.x] = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    cnt[e] = 0;
    next[e] = 0;
  }
  __syncthreads();
  if (kV > 0) {
    // eight lanes per token, four tokens per warp: the whole batch in one round
    const int g = lane & 7;
    for (int64_t t0 = (int64_t)warp * 4; t0 < T; t0 += (kScanThreads / 32) * 4) {
      const int64_t t = t0 + (lane >> 3);
      const bool valid = t < T;
      int id;
      float w;
      route_token8<(kV > 0 ? kV : 8)>(ra.logits + (valid ? t : 0) * E, valid, E, k, g, id, w);
      if (valid && g < k) {
        ra.ids[t * k + g] = id;
        ra.w[t * k + g] = w;
        ids_s[t * k + g] = id;
        atomicAdd(&cnt[id], 1);
      }
    }
  } else {
    for (int64_t t = warp; t < T; t += kScanThreads / 32) {
      int id;
      float w;
      route_token_fast<kPerLane>(ra.logits + t * E, E, k, lane, id, w);
      if (lane < k) {
        ra.ids[t * k + lane] = id;
        ra.w[t * k + lane] = w;
        ids_s[t * k + lane] = id;
        atomicAdd(&cnt[id], 1);
      }
    }
  }
  __syncthreads();
  if (warp != 0) return;
  // Warp 0 alone from here: the prefixes over experts (lane L owns experts [L * per, L * per +
  // per)), then the stable scatter; no block-wide barrier on a decode step's critical path.
  {
    const int per = (E + 31) / 32;
    const int e0 = min(lane * per, E), e1 = min(e0 + per, E);
    int64_t sum = 0, psum = 0;
    for (int e = e0; e < e1; ++e) {
      const int64_t c = cnt[e];
      sum += c;
      psum += (c + kRowTile - 1) / kRowTile * kRowTile;
    }
    int64_t xs = warp_inclusive_scan<int64_t>(sum, lane) - sum;
    int64_t xps = warp_inclusive_scan<int64_t>(psum, lane) - psum;
    for (int e = e0; e < e1; ++e) {
      const int c = cnt[e];
      sa.counts[e] = c;
      sa.offsets[e] = xs;
      sa.padded_offsets[e] = xps;
      sa.mtile_base[e] = (int32_t)(xps / kRowTile);
      off_s[e] = xs;
      poff_s[e] = xps;
      xs += c;
      xps += ((int64_t)c + kRowTile - 1) / kRowTile * kRowTile;
    }
    if (lane == 31) {  // lane 31 ends at the totals
      sa.offsets[E] = xs;
      sa.padded_offsets[E] = xps;
      sa.mtile_base[E] = (int32_t)(xps / kRowTile);
    }
  }
  __syncwarp();
  {  // stable scatter, pairs in ascending order
    const int64_t R = T * k;
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int64_t q0 = 0; q0 < R; q0 += 32) {
      const int64_t q = q0 + lane;
      const bool valid = q < R;
      const int id = valid ? ids_s[q] : -1 - lane;
      const uint32_t peers = __match_any_sync(0xffffffffu, id);
      const int rank = __popc(peers & lt_mask);
      const int leader = __ffs(peers) - 1;
      const int base = valid ? next[id] : 0;
      __syncwarp();
      if (valid && lane == leader) next[id] = base + __popc(peers);
      __syncwarp();
      if (valid) {
        const int64_t local = (int64_t)base + rank;
        const int64_t r = off_s[id] + local;
        sa.sorted_pair[r] = (int32_t)q;
        sa.inv[q] = (int32_t)r;
        sa.inv_padded[q] = (int32_t)(poff_s[id] + local);
      }
    }
  }
}

}  // namespace

cudaError_t launch_route_sort_small(const RouteArgs& ra, const SortArgs& sa, cudaStream_t s) {
  if (ra.T == 0) return cudaSuccess;
  // E <= 128: eight lanes per token (16 logits a lane), the batch in one round; more experts
  // made each token's rounds too long (E = 384: 17-25 -> 35-42 us at T = 8-64), so 32 lanes a
  // token and the warps take the tokens in turn
  if (ra.E <= 64) route_sort_small_kernel<16, 8><<<1, kScanThreads, 0, s>>>(ra, sa);
  else if (ra.E <= 128) route_sort_small_kernel<16, 16><<<1, kScanThreads, 0, s>>>(ra, sa);
  else if (ra.E <= 512) route_sort_small_kernel<16, 0><<<1, kScanThreads, 0, s>>>(ra, sa);
  else route_sort_small_kernel<32, 0><<<1, kScanThreads, 0, s>>>(ra, sa);
  return cudaGetLastError();
}

cudaError_t launch_scan(const SortArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  scan_cols_kernel<<<(unsigned)((a.E + kColWarps - 1) / kColWarps), kColWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_scatter(const SortArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const size_t smem = (size_t)a.E * (2 * sizeof(int64_t) + sizeof(int));  // <= 20 KB
  scatter_kernel<<<(unsigned)a.nchunk, 32, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_sort(const SortArgs& a, cudaStream_t s) {
  const cudaError_t err = launch_scan(a, s);
  return err != cudaSuccess ? err : launch_scatter(a, s);
}

}  // namespace moe
