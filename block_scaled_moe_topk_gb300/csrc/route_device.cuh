// route_device.cuh -- top-k softmax gating of one token by one warp (shared by the routing
// kernel and the fused small-batch route + sort kernel).
//
// "[HIP] gfx950 A8W4 fused_moe configs for DSv4.1 TP-sharded experts" (Changes: the top-k
// softmax kernel): experts ranked by fp32 logit, descending, ties to the lower index; the k
// selected softmax probabilities renormalised to sum 1, i.e. w_j = exp(l_j - l_max) /
// sum_i exp(l_i - l_max) over the selected experts (the full softmax denominator cancels).
#pragma once
#include <cstdint>

#include "moe_internal.h"

namespace moe {

__device__ __forceinline__ bool route_better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Lane j < k of the calling warp receives slot j: expert id and renormalised weight.  NaN
// logits (outside what the method defines) rank as -inf, lowest index first among equals, so
// the ids are always k distinct experts.
// kMaxPerLane >= ceil(E / 32): logits held per lane (fewer registers for smaller E).
template <int kMaxPerLane = kMaxExperts / 32>
__device__ __forceinline__ void route_token(const float* l, int E, int k, int lane, int& id_out, float& w_out) {
  static_assert(kMaxPerLane <= 32, "taken-mask width");
  const int per_lane = (E + 31) / 32;
  float v[kMaxPerLane];
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    const float x = (i < per_lane && e < E) ? l[e] : 0.0f;
    v[i] = x != x ? -INFINITY : x;  // a NaN logit ranks as -inf (below every number)
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
        if (bi == 0x7fffffff || route_better(v[i], e, bv, bi)) {
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
      if (oi != 0x7fffffff && (bi == 0x7fffffff || route_better(ov, oi, bv, bi))) {
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
    // an expert infinitely far below the maximum weighs exactly 0 (the two-sum term is NaN there)
    p = sdiff == -INFINITY ? 0.0f : expf(sdiff) * (1.0f + e);
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
  id_out = my_id;
  w_out = __fdiv_rn(p, zh) * (1.0f - __fdiv_rn(zl, zh));
}

// Order-preserving 32-bit key of a non-NaN float (larger value, larger key); -0 and +0 share
// the key of +0, as they compare equal.
__device__ __forceinline__ uint32_t route_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float route_key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// The same ranking and weights as route_token with a shorter dependency chain: each lane keeps
// its best remaining expert, each of the k rounds takes the warp's maximum key and, among the
// lanes holding it, the lowest expert index with two redux.sync reductions, and only the
// winning lane rescans its values.  A selected -0 logit reports +0 (the same weight).
template <int kMaxPerLane = kMaxExperts / 32>
__device__ __forceinline__ void route_token_fast(const float* l, int E, int k, int lane, int& id_out, float& w_out) {
  static_assert(kMaxPerLane <= 32, "availability-mask width");
  const int per_lane = (E + 31) / 32;
  uint32_t key[kMaxPerLane];
  uint32_t avail = 0;
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    const bool in = i < per_lane && e < E;
    const float x = in ? l[e] : 0.0f;
    key[i] = route_key(x != x ? -INFINITY : x);  // a NaN logit ranks as -inf
    if (in) avail |= 1u << i;
  }
  // this lane's best remaining expert: largest key, lowest index among equal keys (the first i)
  uint32_t best = 0;
  int best_i = -1;
  auto rescan = [&]() {
    best = 0;
    best_i = -1;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
      if (((avail >> i) & 1u) && (best_i < 0 || key[i] > best)) {
        best = key[i];
        best_i = i;
      }
  };
  rescan();
  int my_id = 0;
  float my_val = 0.0f, lmax = 0.0f;
  for (int j = 0; j < k; ++j) {
    // every available key is > 0 (route_key(-inf) = 0x007fffff), so 0 stands for "none left"
    const uint32_t mk = __reduce_max_sync(0xffffffffu, best_i >= 0 ? best : 0u);
    const uint32_t mine = (best_i >= 0 && best == mk) ? (uint32_t)(lane + 32 * best_i) : 0xffffffffu;
    const uint32_t mi = __reduce_min_sync(0xffffffffu, mine);
    const float mv = route_key_value(mk);
    if (j == 0) lmax = mv;
    if (lane == j) {
      my_id = (int)mi;
      my_val = mv;
    }
    if ((int)(mi & 31u) == lane) {
      avail &= ~(1u << (mi >> 5));
      rescan();
    }
  }
  // p_j = exp(l_j - l_max) and the compensated sum, exactly as route_token
  float p = 0.0f;
  if (lane < k) {
    const float sdiff = my_val - lmax;
    const float bb = sdiff - my_val;
    const float e = (my_val - (sdiff - bb)) + (-lmax - bb);
    p = sdiff == -INFINITY ? 0.0f : expf(sdiff) * (1.0f + e);
  }
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
  id_out = my_id;
  w_out = __fdiv_rn(p, zh) * (1.0f - __fdiv_rn(zl, zh));
}

// Eight lanes per token (lane g = lane % 8 of its group holds experts g + 8 i, i < kV), so a
// warp routes four tokens at once with three butterfly levels per selection instead of five.
// Same ranking and weights as route_token; kV >= ceil(E / 8), kV <= 64.  The local scan runs
// as two interleaved chains (even and odd i) to halve its dependency length.  Experts past E
// and the tokens of an invalid group hold NaN, which no comparison selects.
template <int kV>
__device__ __forceinline__ void route_token8(const float* l, bool valid, int E, int k, int g, int& id_out,
                                             float& w_out) {
  static_assert(kV % 2 == 0 && kV <= 64, "values per lane");
  constexpr int kNone = 0x7fffffff;
  const float nan = __int_as_float(0x7fc00000);
  float v[kV];
#pragma unroll
  for (int i = 0; i < kV; ++i) {
    const int e = g + 8 * i;
    const float x = (valid && e < E) ? l[e] : nan;
    // a NaN logit ranks as -inf, so a valid token always finds k experts; only the padding
    // (experts past E, tokens past T) stays NaN and is never selected
    v[i] = (valid && e < E && x != x) ? -INFINITY : x;
  }
  uint64_t taken = 0;
  int my_id = 0;
  float my_val = 0.0f, lmax = 0.0f;
  for (int j = 0; j < k; ++j) {
    float b0 = -INFINITY, b1 = -INFINITY;
    int i0 = kNone, i1 = kNone;
#pragma unroll
    for (int i = 0; i < kV; i += 2) {
      if (!((taken >> i) & 1ull) && route_better(v[i], g + 8 * i, b0, i0)) {
        b0 = v[i];
        i0 = g + 8 * i;
      }
      if (!((taken >> (i + 1)) & 1ull) && route_better(v[i + 1], g + 8 * (i + 1), b1, i1)) {
        b1 = v[i + 1];
        i1 = g + 8 * (i + 1);
      }
    }
    float bv = b0;
    int bi = i0;
    if (route_better(b1, i1, bv, bi)) {
      bv = b1;
      bi = i1;
    }
    // arg-max over the group's eight lanes (value desc, index asc); (-inf, kNone) is "none"
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (route_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi != kNone && (bi & 7) == g) taken |= 1ull << (bi >> 3);
    if (j == 0) lmax = bv;
    if (g == j) {
      my_id = bi;
      my_val = bv;
    }
  }
  float p = 0.0f;  // exp(l_j - l_max) as in route_token
  if (g < k) {
    const float sdiff = my_val - lmax;
    const float bb = sdiff - my_val;
    const float e = (my_val - (sdiff - bb)) + (-lmax - bb);
    p = sdiff == -INFINITY ? 0.0f : expf(sdiff) * (1.0f + e);
  }
  float zh = p, zl = 0.0f;  // compensated sum over the group
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, zh, off);
    const float ol = __shfl_xor_sync(0xffffffffu, zl, off);
    const float sum = zh + oh;
    const float bv = sum - zh;
    zl += ol + ((zh - (sum - bv)) + (oh - bv));
    zh = sum;
  }
  id_out = my_id;
  w_out = __fdiv_rn(p, zh) * (1.0f - __fdiv_rn(zl, zh));
}

}  // namespace moe
