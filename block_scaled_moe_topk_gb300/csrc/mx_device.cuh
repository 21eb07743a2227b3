// mx_device.cuh -- device helpers for the OCP MX formats used by the quantiser and the
// GEMM1 epilogue: the E8M0 scale of a 32-block and packing of E4M3 / E2M1 codes.
#pragma once
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace moe {

struct MxScale {
  uint8_t byte;  // E8M0 scale byte s, value 2^(s-127)
  float mult;    // 2^(127-s): multiplying by it divides by the scale exactly; 0 for a
                 // zero / subnormal block, which turns every element into a signed zero
};

// s = floor(log2 amax) - emax + 127, clamped to [0, 254]; emax = 8 (E4M3) or 2 (E2M1).
// floor(log2 amax) is read from the exponent field, so no log2f is involved.
template <int FMT>
__device__ __forceinline__ MxScale mx_scale(float amax) {
  constexpr int kEmax = FMT == 0 ? 8 : 2;
  const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
  MxScale r;
  if (ef == 0) {
    r.byte = 0;
    r.mult = 0.0f;
  } else {
    const int s = min(max(ef - kEmax, 0), 254);
    r.byte = (uint8_t)s;
    r.mult = __uint_as_float((uint32_t)(254 - s) << 23);
  }
  return r;
}

// Eight values -> eight E4M3 bytes (round to nearest even, saturate to +-448),
// element 0 in the lowest byte.
__device__ __forceinline__ uint2 pack_e4m3x8(const float* v, float mult) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_fp8x2_storage_t c =
        __nv_cvt_float2_to_fp8x2(make_float2(v[2 * i] * mult, v[2 * i + 1] * mult), __NV_SATFINITE, __NV_E4M3);
    w[i] = (uint32_t)c;
  }
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// Eight values -> four bytes of E2M1 codes (nearest even, saturate to +-6),
// element 2i in the low nibble of byte i.
__device__ __forceinline__ uint32_t pack_e2m1x8(const float* v, float mult) {
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_fp4x2_storage_t c =
        __nv_cvt_float2_to_fp4x2(make_float2(v[2 * i] * mult, v[2 * i + 1] * mult), __NV_E2M1, cudaRoundNearest);
    r |= (uint32_t)c << (8 * i);
  }
  return r;
}

// Byte offset of the scale of (row, 32-block kb) in the 128x4 tile layout of a
// [rows, K] operand: tiles of 128 rows x 4 blocks (512 bytes), row-major over
// (row/128, kb/4); inside a tile byte (r%32)*16 + ((r%128)/32)*4 + kb%4.  This is
// the order in which tcgen05.cp (32x128b, warpx4) lands the scales of row r in
// TMEM lane r%32, column r/32 (mod 4), byte kb%4.
__device__ __forceinline__ int64_t sf_tile_offset(int64_t row, int kb, int K) {
  return ((row >> 7) * (K >> 7) + (kb >> 2)) * 512 + (row & 31) * 16 + ((row & 127) >> 5) * 4 + (kb & 3);
}

}  // namespace moe
