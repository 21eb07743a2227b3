// moe_internal.h -- launchers shared between the host API and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace moe {

// Routing chunk: tokens handled by one routing block (its expert histogram is one
// column of chunk_hist).
constexpr int kTokensPerChunk = 32;  // 8 warps x 4 tokens: enough warps to route T=8192 on 152 SMs
constexpr int kRowTile = 128;   // rows per GEMM M tile; expert segments are padded to it
constexpr int kNTile = 256;     // output columns per GEMM N tile
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 8;

// Device status word bits (the host maps them to moe_status_t).
constexpr uint32_t kStatusInvalidArg = 1u;  // an expert id outside [0, E)
constexpr uint32_t kStatusTimeout = 2u;     // a bounded in-kernel wait expired

struct RouteArgs {
  const float* logits;  // [T, E]
  int64_t T;
  int E, k;
  int32_t* ids;         // [T, k]
  float* w;             // [T, k]
  int32_t* chunk_hist;  // [E, nchunk] or null
  int64_t nchunk;
  uint32_t* status;     // reset to 0 by block 0 when reset_status
  int reset_status;
};

struct SortArgs {
  const int32_t* ids;  // [T*k]
  int64_t T;
  int E, k;
  int32_t* chunk_hist;       // [E, nchunk]: histogram in, exclusive per-expert chunk base out
  int64_t nchunk;
  int32_t* counts;           // [E]
  int64_t* offsets;          // [E+1]
  int64_t* padded_offsets;   // [E+1] or null
  int32_t* mtile_base;       // [E+1] or null
  int32_t* sorted_pair;      // [T*k]
  int32_t* inv;              // [T*k]
  int32_t* inv_padded;       // [T*k] or null
  uint32_t* status;
};

// route.cu
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s);
// Histogram of externally supplied ids (standalone sort entry point).
cudaError_t launch_histogram(const SortArgs& a, cudaStream_t s);
// sort.cu: per-expert chunk bases + offsets (scan), then the stable scatter.
cudaError_t launch_scan(const SortArgs& a, cudaStream_t s);
cudaError_t launch_scatter(const SortArgs& a, cudaStream_t s);
cudaError_t launch_sort(const SortArgs& a, cudaStream_t s);
// Batches of at most kSmallRouteTokens tokens: routing + sort (with padded outputs) in one
// single-block kernel.
constexpr int kSmallRouteTokens = 64;
cudaError_t launch_route_sort_small(const RouteArgs& ra, const SortArgs& sa, cudaStream_t s);

// quant.cu
struct QuantArgs {
  const uint16_t* x;      // bf16 [rows, K]
  int64_t rows;
  int K;
  int fmt;                // 0 = E4M3, 1 = E2M1
  uint8_t* codes;
  uint8_t* scales;
  // Permuted mode (forward): row t goes to rows inv_padded[t*k + j], j < k, and
  // its scales to the 128x4 tile layout.  Canonical mode when inv_padded == null.
  const int32_t* inv_padded;
  int k;
  // permuted mode, FP8 transport of the GEMM2 rows: row_w[inv_padded[t*k + j]] = topk_w[t*k + j]
  const float* topk_w;
  float* row_w;
};
cudaError_t launch_quant(const QuantArgs& a, cudaStream_t s);
// Prequantised activations [rows, code_bytes] + canonical scales [rows, K/32] -> padded expert
// rows inv_padded[t*k + j] and the 128x4 tile layout (code_bytes % 16 == 0).
struct PermuteArgs {
  const uint8_t* codes_in;
  const uint8_t* scales_in;
  int64_t rows;
  int K;
  int64_t code_bytes;
  const int32_t* inv_padded;
  int k;
  uint8_t* codes_out;
  uint8_t* scales_out;
  const float* topk_w;  // with row_w: row_w[inv_padded[q]] = topk_w[q] (as QuantArgs)
  float* row_w;
};
cudaError_t launch_permute_rows(const PermuteArgs& a, cudaStream_t s);
// bf16 rows h [rows_cap, K] at the padded rows inv_padded[q] of the R routed pairs -> MX codes
// of the same rows (E4M3 or E2M1) and their scales in the 128x4 tile layout (K % 128 == 0).
struct RequantArgs {
  const uint16_t* h;
  const int32_t* inv_padded;
  int64_t R;
  int K;
  int fmt;
  uint8_t* codes;
  uint8_t* scales;
};
cudaError_t launch_requant(const RequantArgs& a, cudaStream_t s);
// Canonical [rows, K/32] scales -> 128x4 tile layout (rows % 128 == 0, K % 128 == 0).
cudaError_t launch_prepack_scales(const uint8_t* src, int64_t rows, int K, uint8_t* dst, cudaStream_t s);

// gemm.cu
struct GemmArgs {
  int act_fmt;            // 0: E4M3 activations (kind::mxf8f6f4), 1: E2M1 (kind::mxf4)
  int epilogue;           // 0: SwiGLU + MX requant (GEMM1), 1: bf16 rows (GEMM2), 2: bf16 SwiGLU
                          // rows h [rows_cap, N/2] into out_bf16 (GEMM1, bf16-out form), 3: rows
                          // weighted by row_w as E4M3 codes [rows_cap, N] in out_codes and one E8M0
                          // byte per 1x32 block [rows_cap, N/32] in out_sf (GEMM2, FP8 transport)
  const uint8_t* act;     // activation codes [rows_cap, K or K/2]
  const uint8_t* act_sf;  // [rows_cap/128][K/128][512]
  int64_t rows_cap;
  const uint8_t* w;       // MXFP4 [E, N, K/2]
  const uint8_t* w_sf;    // E8M0 [E, N, K/32], or its 128x4 tile layout when w_sf_tiled
  int w_sf_tiled;
  int E, N, K;
  const int32_t* counts;
  const int32_t* mtile_base;  // [E+1]; expert e's padded rows start at 128 * mtile_base[e]
  int64_t max_tiles;      // host upper bound on tiles (grid sizing)
  uint8_t* out_codes;     // GEMM1: A2 codes [rows_cap, N/2 or N/4]
  uint8_t* out_sf;        // GEMM1: A2 scales, 128x4 tile layout over N/2 columns
  uint16_t* out_bf16;     // GEMM2: y2 bf16 [rows_cap, N]
  uint32_t* status;
  uint64_t timeout_ns;
  int num_sms;
  int test_stall;         // test hook: the producer issues nothing, so the MMA warp's wait expires
  int a_rows;             // single-CTA tiles: activation rows staged per K stage (16, 64 or 128;
                          // 16 requires every tile to hold at most 16 routed rows)
  int tail_only;          // single-CTA tiles, A8W4, 128 rows: only each expert's odd last M tile
                          // (after launch_gemm_pair took the whole pairs)
  uint8_t* act_sf_rot;    // split GEMMs with the wide tail pass: launch_gemm_pair writes the A-scale
                          // atoms of each expert's odd last M tile here, halves swapped, for
                          // launch_gemm_tail_wide (same layout as act_sf); null otherwise
  const float* row_w;     // epilogue 3: the routing weight of each padded row [rows_cap]
};
// Single-CTA GEMMs stage 16 activation rows when T <= 16, and 64 rows (in 64-row work units)
// when the batch routes at most this many rows per expert on average (T * k <= 16 * E) and the
// GEMM's K spans at least kUnit64MinStages stages: with skewed routing or a short K, experts
// split into two units or the per-unit overhead cost more than the deeper ring gained.
constexpr int kUnit64MaxRowsPerExpert = 16;
constexpr int kUnit64MinStages = 16;
// gemm.cu: one CTA per 128-row x 256-column tile (any weight-scale layout).
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s);
// gemm_pair.cu: the whole pairs of each expert's M tiles on CTA pairs (prepacked weight scales,
// N a multiple of 256); gemm.cu's tail pass (tail_only) then takes each odd last M tile.
cudaError_t launch_gemm_pair(const GemmArgs& a, cudaStream_t s);
// gemm_pair.cu: the tail pass of a split GEMM on CTA pairs (cta_group::2, M = 128), each pair
// tile an expert's odd last M tile by 512 output columns (N a multiple of 512), reading the
// rotated A-scale atoms launch_gemm_pair wrote to act_sf_rot.  Five 43 KiB stages keep 80 KiB of
// weight bytes in flight per SM, against 64 KiB for the single-CTA tail tiles.
constexpr int kTailWideN = 2 * kNTile;
cudaError_t launch_gemm_tail_wide(const GemmArgs& a, cudaStream_t s);
// The wide tail pass serves GEMMs with N a multiple of 512 and at least kTailWideMinStages K
// stages: with short K (V4.1-Flash and draft GEMM2, 5-9 stages a tile) the accumulator hand-off
// between tiles and the pair kernel's fixed cost outweighed the deeper ring (+6 to +20 % for
// those layers at T = 1024-8192).
constexpr int kTailWideMinStages = 16;
inline bool gemm_tail_wide(int N, int K) { return N % kTailWideN == 0 && K / 128 >= kTailWideMinStages; }
// The kernel chain splits a GEMM into the pair kernel and a tail pass when its tiles are the
// 128-row A8W4 ones, the weight scales are prepacked and N is a multiple of 256, and
//   * its tail pass is the wide one and the batch routes more than kUnit64MaxRowsPerExpert rows
//     per expert on average: measured on V4-Pro A8W4 against single-CTA tiles throughout, -7 to
//     -9 % for the layer at T = 1025-6144, and at T = 8192 GEMM1 / GEMM2 tails 860 / 460 ->
//     779 / 440 us; or
//   * the batch routes at least kPairMinRowsPerExpert rows per expert on average (then about
//     half the experts or more have a second M tile): with the single-CTA tail pass, GEMM1
//     -8.7 % and GEMM2 -6.8 % at T = 8192, -4.7 % / -3 % at T = 16384, equal at T = 32768.
constexpr int kPairMinRowsPerExpert = 128;
inline bool gemm_pair_split(int64_t T, int E, int k, int act_fmt, bool prepacked, int N, int K, int a_rows) {
  if (act_fmt != 0 || !prepacked || N % kNTile != 0 || a_rows != kRowTile) return false;
  const int64_t rows = T * (int64_t)k;
  return rows >= (int64_t)kPairMinRowsPerExpert * E ||
         (gemm_tail_wide(N, K) && rows > (int64_t)kUnit64MaxRowsPerExpert * E);
}
// Whether a batch may split a GEMM with the wide tail pass (the workspace then holds sf_rot).
inline bool gemm_split_rows(int64_t T, int E, int k, int act_fmt) {
  return act_fmt == 0 && T * (int64_t)k > (int64_t)kUnit64MaxRowsPerExpert * E;
}


// decode.cu: the whole layer for a small batch in one persistent kernel (T <= kDecodeMaxTokens).
// Every CTA routes and sorts the batch itself; CTA b quantises token b; GEMM1 and GEMM2 are
// each spread over all CTAs by K stages; GEMM2 stages of an expert wait for its A2 rows; the
// combine runs as each output column block completes.  Counters live in the workspace's
// sync region, which the host zeroes before the launch.
constexpr int kDecodeMaxTokens = kSmallRouteTokens;
// MOE_SCHEDULE_AUTO takes the fused kernel for T <= 2 on every shape, and up to 16 tokens when
// the intermediate size I is at least 1024 (measured on the GB300 over the configs' shapes:
// with I = 640 the items of GEMM2 are five K stages long and the kernel chain wins from 4-8
// tokens on)
constexpr int kDecodeAutoMaxTokens = 16;
constexpr int kDecodeAutoAlwaysTokens = 2;
constexpr int kDecodeAutoMinI = 1024;

constexpr int kDecodeMaxPairs = kDecodeMaxTokens * kMaxTopK;  // routed rows, also active experts
constexpr int kDecodeMaxCtas = 160;                           // grid = min(SMs, this)
constexpr int kDecodeMaxHidden = 16384;                       // H of the fused schedule (staged row)
inline bool decode_auto(int64_t T, int H, int I) {
  if (H > kDecodeMaxHidden) return false;
  return T <= kDecodeAutoAlwaysTokens || (T <= kDecodeAutoMaxTokens && I >= kDecodeAutoMinI);
}
// sync region (uint32 words)
constexpr int kSyncQuant = 0;                                     // tokens quantised
constexpr int kSyncDone2 = 1;                                     // GEMM2 parts final
constexpr int kSyncRouted = 2;                                    // tokens routed (above 11 tokens)
constexpr int kSyncReady = 16;                                    // [active expert] GEMM1 parts final
constexpr int kSyncTicket = kSyncReady + kDecodeMaxPairs;         // [phase][first CTA][warp] tickets
constexpr int kSyncWords = kSyncTicket + 2 * kDecodeMaxCtas * 8;
// activation rows staged per K stage: every expert of a batch of T tokens has at most T rows
inline int decode_arows(int64_t T) { return T <= 16 ? 16 : 64; }
// partial-accumulator slots: per CTA, per GEMM, its first and last item
inline size_t decode_part_bytes(int64_t T) {
  return (size_t)kDecodeMaxCtas * 4 * (size_t)decode_arows(T) * kNTile * sizeof(float);
}

struct DecodeArgs {
  int act_fmt;
  const uint16_t* x;          // bf16 [T, H], or null when the input is prequantised:
  const uint8_t* xq_in;       //   codes [T, H or H/2]
  const uint8_t* xs_in;       //   canonical E8M0 scales [T, H/32]
  const float* logits;        // [T, E]
  const uint8_t* w1;
  const uint8_t* w1_sf;
  const uint8_t* w2;
  const uint8_t* w2_sf;
  int w_sf_tiled;
  int64_t rows_cap;
  uint8_t* xq;                // padded expert rows + 128x4 tile scales (as the kernel chain)
  uint8_t* xs;
  uint8_t* a2;
  uint8_t* a2s;
  float* part;                // decode_part_bytes(T)
  float* y2f;                 // fp32 GEMM2 rows [T*k, H], unpadded row order
  uint16_t* out;              // bf16 [T, H]
  int32_t* ids;               // routing / sort results, as the kernel chain writes them
  float* tw;
  int32_t* counts;
  int64_t* offsets;
  int64_t* padded_offsets;
  int32_t* mtile_base;
  int32_t* sorted_pair;
  int32_t* inv;
  int32_t* inv_padded;
  uint32_t* sync;             // kSyncWords, zero at launch
  uint32_t* status;
  uint64_t timeout_ns;
  int num_sms;
  int test_stall;
  int64_t T;
  int H, I, E, k;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);

// combine.cu
struct CombineArgs {
  const uint16_t* y2;       // bf16 [rows_cap, H]
  const float* w;           // [T, k]
  const int32_t* inv_padded;
  int64_t T;
  int H, k;
  uint16_t* out;            // bf16 [T, H]
  // FP8 transport (y2 null): the rows already weighted, as E4M3 codes y2q [rows_cap, H] and one
  // E8M0 byte per 1x32 block y2s [rows_cap, H/32]; out = bf16(sum over slots of their values)
  const uint8_t* y2q;
  const uint8_t* y2s;
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);

}  // namespace moe
