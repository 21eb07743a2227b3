// moe_api.cu -- the exported C ABI: argument validation, workspace layout and the launch
// sequence of the expert layer.  Nothing here allocates device memory or synchronises,
// except moe_read_device_status, whose job is to read the status word back.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "moe_internal.h"
#include "moe_topk.h"

namespace {

using moe::kMaxExperts;
using moe::kMaxTopK;
using moe::kRowTile;
using moe::kTokensPerChunk;

constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;  // bound of every in-kernel wait

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

moe_status_t check_sizes(int64_t T, int H, int I, int E, int k, moe_act_fmt_t fmt) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
  if (fmt != MOE_ACT_MXFP8 && fmt != MOE_ACT_MXFP4) return MOE_ERR_INVALID_ARG;
  if (k > E) return MOE_ERR_INVALID_ARG;
  if (k > kMaxTopK || E > kMaxExperts) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (H % 128 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (H > 65536 || I > 65536) return MOE_ERR_UNSUPPORTED_SHAPE;
  // row indices are int32 on the device: keep the padded row space below 2^31
  const int64_t R = T * (int64_t)k;
  if (T > (int64_t(1) << 24) || R + (int64_t)127 * std::min<int64_t>(E, R) > (int64_t(1) << 30))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

struct DeviceInfo {
  int ok = -1;  // -1 unknown, 0 unsupported, 1 sm_103
  int num_sms = 0;
};

moe_status_t device_info(DeviceInfo* out) {
  static DeviceInfo cache[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& d = cache[dev];
  if (d.ok < 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    d.ok = (major == 10 && minor == 3) ? 1 : 0;
    d.num_sms = sms;
  }
  *out = d;
  return d.ok == 1 ? MOE_OK : MOE_ERR_UNSUPPORTED_DEVICE;
}

moe_status_t layout(int64_t T, int H, int I, int E, int k, moe_act_fmt_t fmt, moe_workspace_layout_t* L) {
  const moe_status_t st = check_sizes(T, H, I, E, k, fmt);
  if (st != MOE_OK) return st;
  memset(L, 0, sizeof(*L));
  const int64_t R = T * (int64_t)k;
  const int64_t rows_cap =
      R == 0 ? 0 : (R + (int64_t)(kRowTile - 1) * std::min<int64_t>(E, R) + kRowTile - 1) / kRowTile * kRowTile;
  const int64_t nchunk = (T + kTokensPerChunk - 1) / kTokensPerChunk;
  const size_t hb = fmt == MOE_ACT_MXFP8 ? (size_t)H : (size_t)H / 2;
  const size_t ib = fmt == MOE_ACT_MXFP8 ? (size_t)I : (size_t)I / 2;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L->status = take(sizeof(uint32_t) * 8);
  L->sync = take(sizeof(uint32_t) * moe::kSyncWords);  // right after the status words: one memset clears both
  L->topk_ids = take(sizeof(int32_t) * R);
  L->topk_w = take(sizeof(float) * R);
  L->counts = take(sizeof(int32_t) * E);
  L->offsets = take(sizeof(int64_t) * (E + 1));
  L->padded_offsets = take(sizeof(int64_t) * (E + 1));
  L->mtile_base = take(sizeof(int32_t) * (E + 1));
  L->chunk_hist = take(sizeof(int32_t) * (size_t)E * nchunk);
  L->sorted_pair = take(sizeof(int32_t) * R);
  L->inv = take(sizeof(int32_t) * R);
  L->inv_padded = take(sizeof(int32_t) * R);
  L->xq = take(hb * rows_cap);
  L->xs = take((size_t)H / 32 * rows_cap);
  L->a2 = take(ib * rows_cap);
  L->a2s = take((size_t)I / 32 * rows_cap);
  L->y2 = take(sizeof(uint16_t) * (size_t)H * rows_cap);
  // the split GEMMs' rotated A-scale atoms (only a batch the chain may split needs them)
  const bool split_rows = moe::gemm_split_rows(T, E, k, fmt == MOE_ACT_MXFP8 ? 0 : 1);
  L->sf_rot = take(split_rows ? (size_t)std::max(H, I) / 32 * rows_cap : 0);
  // the single-kernel decode schedule (T <= 64): partial accumulators and fp32 GEMM2 rows
  const bool decode = T <= moe::kDecodeMaxTokens;
  L->part = take(decode ? moe::decode_part_bytes(T) : 0);
  L->y2f = take(decode ? sizeof(float) * (size_t)R * H : 0);
  L->total = off;
  L->rows_cap = rows_cap;
  L->nchunk = nchunk;
  return MOE_OK;
}

uint64_t wait_timeout_ns() {
  static uint64_t v = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    v = kDefaultTimeoutNs;
    if (const char* s = getenv("MOE_WAIT_TIMEOUT_NS")) {
      const unsigned long long x = strtoull(s, nullptr, 10);
      if (x > 0) v = x;
    }
  });
  return v;
}

// Test hook for the failure path: MOE_TEST_STALL_PRODUCER=1 makes the GEMM producers issue
// nothing, so the first wait of the MMA warp expires after MOE_WAIT_TIMEOUT_NS and the kernel
// reports MOE_ERR_DEVICE_TIMEOUT through the workspace status words (no fault, no hang).
int test_stall_producer() {
  static int v = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    if (const char* s = getenv("MOE_TEST_STALL_PRODUCER")) v = atoi(s) != 0;
  });
  return v;
}

#define MOE_CUDA_TRY(expr)                          \
  do {                                              \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

// The forward's launch sequence.  With `ev` (kForwardKernels + 1 events) an event is
// recorded before the first kernel and after every kernel, for per-kernel timing.
// Kernel chain, T > 64: route, scan, scatter, quant, gemm1, gemm2, combine; T <= 64:
// route_sort, quant, gemm1, gemm2, combine.  Fused schedule (T <= 64): one decode kernel.
constexpr int kForwardKernels = 7;
constexpr int kMaxForwardKernels = 9;  // the chain with both GEMMs split (pair kernel + tail pass)
bool valid_schedule(int schedule) {
  return schedule == MOE_SCHEDULE_AUTO || schedule == MOE_SCHEDULE_CHAIN || schedule == MOE_SCHEDULE_FUSED ||
         schedule == MOE_SCHEDULE_CHAIN_BF16_H || schedule == MOE_SCHEDULE_CHAIN_SINGLE_CTA ||
         schedule == MOE_SCHEDULE_CHAIN_FP8_Y2;
}
bool use_fused(int64_t T, int schedule, int H, int I) {
  return schedule == MOE_SCHEDULE_FUSED || (schedule == MOE_SCHEDULE_AUTO && moe::decode_auto(T, H, I));
}
int launch_count(int64_t T, int H, int I, int schedule = MOE_SCHEDULE_AUTO) {
  if (T <= 0) return 0;
  if (use_fused(T, schedule, H, I)) return 1;
  const int requant = schedule == MOE_SCHEDULE_CHAIN_BF16_H ? 1 : 0;  // the separate requant kernel
  return (T <= moe::kSmallRouteTokens ? 5 : kForwardKernels) + requant;
}
// Activation rows a single-CTA GEMM of reduction length K stages per K stage (GemmArgs::a_rows).
int gemm_a_rows(int64_t T, int E, int k, int K) {
  if (T <= 16) return 16;
  const bool few_rows = T * (int64_t)k <= (int64_t)moe::kUnit64MaxRowsPerExpert * E;
  return few_rows && K / 128 >= moe::kUnit64MinStages ? 64 : kRowTile;
}
// Whether the chain runs a GEMM of N output columns and reduction length K as the pair kernel
// plus the tail pass (moe::gemm_pair_split).
bool split_gemm(int64_t T, int E, int k, int afmt, bool prepacked, int schedule, int N, int K) {
  if (schedule == MOE_SCHEDULE_CHAIN_SINGLE_CTA || schedule == MOE_SCHEDULE_CHAIN_BF16_H) return false;
  return moe::gemm_pair_split(T, E, k, afmt, prepacked, N, K, gemm_a_rows(T, E, k, K));
}
int launch_count_cfg(int64_t T, int H, int I, int E, int k, int afmt, int schedule, bool prepacked) {
  const int n = launch_count(T, H, I, schedule);
  if (n <= 1) return n;
  return n + (split_gemm(T, E, k, afmt, prepacked, schedule, 2 * I, H) ? 1 : 0) +
         (split_gemm(T, E, k, afmt, prepacked, schedule, H, I) ? 1 : 0);
}

// x is bf16 [T, H] when x_scale is null, else prequantised codes [T, H or H/2] with canonical
// E8M0 scales x_scale [T, H/32] (the quantiser is then replaced by a permuting copy).
moe_status_t forward(const void* x, const uint8_t* x_scale, const float* logits, const uint8_t* w1,
                     const uint8_t* w1s, const uint8_t* w2, const uint8_t* w2s, void* out, int64_t T, int H,
                     int I, int E, int k, void* ws, size_t ws_bytes, void* stream, moe_act_fmt_t fmt,
                     bool tiled_scales, cudaEvent_t* ev = nullptr, int schedule = MOE_SCHEDULE_AUTO) {
  // with T == 0 nothing is read or written, so empty x / logits / out may be null
  if ((T > 0 && (!x || !logits || !out)) || !w1 || !w1s || !w2 || !w2s || !ws) return MOE_ERR_INVALID_ARG;
  moe_workspace_layout_t L;
  moe_status_t st = layout(T, H, I, E, k, fmt, &L);
  if (st != MOE_OK) return st;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(logits, 4) || !aligned(w1, 32) || !aligned(w2, 32) ||
      !aligned(w1s, tiled_scales ? 16 : 4) || !aligned(w2s, tiled_scales ? 16 : 4) || !aligned(ws, 256))
    return MOE_ERR_MISALIGNED;
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!valid_schedule(schedule)) return MOE_ERR_INVALID_ARG;
  // the bf16-out GEMM1 keeps h in the y2 region (rows_cap x H bf16), requantised by a kernel of
  // at most 1024 threads of 16 elements
  if (schedule == MOE_SCHEDULE_CHAIN_BF16_H && (I > H || I > 16384)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (schedule == MOE_SCHEDULE_FUSED && (T > moe::kDecodeMaxTokens || H > moe::kDecodeMaxHidden))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T == 0) return MOE_OK;
  DeviceInfo dev;
  st = device_info(&dev);
  if (st != MOE_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* W = static_cast<uint8_t*>(ws);
  auto at = [&](size_t o) { return W + o; };
  uint32_t* status = reinterpret_cast<uint32_t*>(at(L.status));
  int32_t* ids = reinterpret_cast<int32_t*>(at(L.topk_ids));
  float* tw = reinterpret_cast<float*>(at(L.topk_w));
  int32_t* counts = reinterpret_cast<int32_t*>(at(L.counts));
  int64_t* offsets = reinterpret_cast<int64_t*>(at(L.offsets));
  int64_t* poff = reinterpret_cast<int64_t*>(at(L.padded_offsets));
  int32_t* mtb = reinterpret_cast<int32_t*>(at(L.mtile_base));
  int32_t* chunk_hist = reinterpret_cast<int32_t*>(at(L.chunk_hist));
  int32_t* inv_padded = reinterpret_cast<int32_t*>(at(L.inv_padded));

  int evi = 0;
  auto mark = [&]() { return ev ? cudaEventRecord(ev[evi++], s) : cudaSuccess; };
  const int afmt = fmt == MOE_ACT_MXFP8 ? 0 : 1;
  if (use_fused(T, schedule, H, I) && dev.num_sms >= moe::kDecodeMaxTokens) {
    // the status words and the decode kernel's counters start at zero on every call
    MOE_CUDA_TRY(cudaMemsetAsync(W + L.status, 0, L.sync + sizeof(uint32_t) * moe::kSyncWords - L.status, s));
    MOE_CUDA_TRY(mark());
    moe::DecodeArgs da{};
    da.act_fmt = afmt;
    da.x = x_scale == nullptr ? static_cast<const uint16_t*>(x) : nullptr;
    da.xq_in = x_scale == nullptr ? nullptr : static_cast<const uint8_t*>(x);
    da.xs_in = x_scale;
    da.logits = logits;
    da.w1 = w1;
    da.w1_sf = w1s;
    da.w2 = w2;
    da.w2_sf = w2s;
    da.w_sf_tiled = tiled_scales ? 1 : 0;
    da.rows_cap = L.rows_cap;
    da.xq = at(L.xq);
    da.xs = at(L.xs);
    da.a2 = at(L.a2);
    da.a2s = at(L.a2s);
    da.part = reinterpret_cast<float*>(at(L.part));
    da.y2f = reinterpret_cast<float*>(at(L.y2f));
    da.out = static_cast<uint16_t*>(out);
    da.ids = ids;
    da.tw = tw;
    da.counts = counts;
    da.offsets = offsets;
    da.padded_offsets = poff;
    da.mtile_base = mtb;
    da.sorted_pair = reinterpret_cast<int32_t*>(at(L.sorted_pair));
    da.inv = reinterpret_cast<int32_t*>(at(L.inv));
    da.inv_padded = inv_padded;
    da.sync = reinterpret_cast<uint32_t*>(at(L.sync));
    da.status = status;
    da.timeout_ns = wait_timeout_ns();
    da.num_sms = dev.num_sms;
    da.test_stall = test_stall_producer();
    da.T = T;
    da.H = H;
    da.I = I;
    da.E = E;
    da.k = k;
    MOE_CUDA_TRY(moe::launch_decode(da, s));
    MOE_CUDA_TRY(mark());
    return MOE_OK;
  }
  // FP8 transport of the GEMM2 rows: their E4M3 codes [rows_cap, H], E8M0 scales [rows_cap, H/32]
  // and each padded row's routing weight [rows_cap] share the y2 region (2 H bytes a row)
  const bool fp8_y2 = schedule == MOE_SCHEDULE_CHAIN_FP8_Y2;
  uint8_t* y2q = fp8_y2 ? at(L.y2) : nullptr;
  uint8_t* y2s = fp8_y2 ? y2q + (size_t)L.rows_cap * H : nullptr;
  float* row_w = fp8_y2 ? reinterpret_cast<float*>(y2s + align256((size_t)L.rows_cap * (H / 32))) : nullptr;
  MOE_CUDA_TRY(mark());
  moe::RouteArgs ra{logits, T, E, k, ids, tw, chunk_hist, L.nchunk, status, 1};
  moe::SortArgs sa{ids, T, E, k, chunk_hist, L.nchunk, counts, offsets, poff, mtb,
                   reinterpret_cast<int32_t*>(at(L.sorted_pair)), reinterpret_cast<int32_t*>(at(L.inv)),
                   inv_padded, status};
  if (T <= moe::kSmallRouteTokens) {
    MOE_CUDA_TRY(moe::launch_route_sort_small(ra, sa, s));  // one launch for a decode step
    MOE_CUDA_TRY(mark());
  } else {
    MOE_CUDA_TRY(moe::launch_route(ra, s));
    MOE_CUDA_TRY(mark());
    MOE_CUDA_TRY(moe::launch_scan(sa, s));
    MOE_CUDA_TRY(mark());
    MOE_CUDA_TRY(moe::launch_scatter(sa, s));
    MOE_CUDA_TRY(mark());
  }
  if (x_scale == nullptr) {
    moe::QuantArgs qa{static_cast<const uint16_t*>(x), T, H, afmt, at(L.xq), at(L.xs), inv_padded, k, tw, row_w};
    MOE_CUDA_TRY(moe::launch_quant(qa, s));
  } else {
    moe::PermuteArgs pa{static_cast<const uint8_t*>(x), x_scale, T, H, afmt == 0 ? (int64_t)H : (int64_t)H / 2,
                        inv_padded, k, at(L.xq), at(L.xs), tw, row_w};
    MOE_CUDA_TRY(moe::launch_permute_rows(pa, s));
  }
  MOE_CUDA_TRY(mark());

  const int64_t mtiles_cap = L.rows_cap / kRowTile;
  moe::GemmArgs g1{};
  g1.act_fmt = afmt;
  g1.epilogue = 0;
  g1.act = at(L.xq);
  g1.act_sf = at(L.xs);
  g1.rows_cap = L.rows_cap;
  g1.w = w1;
  g1.w_sf = w1s;
  g1.w_sf_tiled = tiled_scales ? 1 : 0;
  g1.E = E;
  g1.N = 2 * I;
  g1.K = H;
  g1.counts = counts;
  g1.mtile_base = mtb;
  g1.max_tiles = mtiles_cap * (2 * I / moe::kNTile);
  g1.out_codes = at(L.a2);
  g1.out_sf = at(L.a2s);
  g1.status = status;
  g1.timeout_ns = wait_timeout_ns();
  g1.num_sms = dev.num_sms;
  g1.test_stall = test_stall_producer();
  // T <= 16: no expert receives more than T rows (a token routes to an expert at most once);
  // few rows per expert on average and a long K: 64-row work units
  auto a_rows_for = [&](int K) { return gemm_a_rows(T, E, k, K); };
  g1.a_rows = a_rows_for(H);
  // a GEMM, split into the pair kernel and the tail pass where that pays (split_gemm)
  // (the tail pass on CTA pairs, 512 columns a pair tile, when N allows: its odd CTAs read the
  // rotated A-scale atoms the pair kernel writes to sf_rot)
  auto run_gemm = [&](const moe::GemmArgs& g) -> cudaError_t {
    if (g.epilogue != 2 && split_gemm(T, E, k, afmt, tiled_scales, schedule, g.N, g.K)) {
      moe::GemmArgs t = g;
      const bool wide = moe::gemm_tail_wide(g.N, g.K);
      t.act_sf_rot = wide ? at(L.sf_rot) : nullptr;
      cudaError_t e = moe::launch_gemm_pair(t, s);
      if (e != cudaSuccess) return e;
      e = mark();
      if (e != cudaSuccess) return e;
      if (wide) return moe::launch_gemm_tail_wide(t, s);
      t.tail_only = 1;
      return moe::launch_gemm(t, s);
    }
    return moe::launch_gemm(g, s);
  };
  const bool bf16_h = schedule == MOE_SCHEDULE_CHAIN_BF16_H;
  if (bf16_h) {
    // GEMM1 leaves h = SwiGLU(acc) as bf16 rows in the y2 region; a separate kernel requantises
    // the routed rows into A2 (GEMM2 overwrites the region with y2 afterwards)
    g1.epilogue = 2;
    g1.out_codes = nullptr;
    g1.out_sf = nullptr;
    g1.out_bf16 = reinterpret_cast<uint16_t*>(at(L.y2));
  }
  MOE_CUDA_TRY(run_gemm(g1));
  MOE_CUDA_TRY(mark());
  if (bf16_h) {
    moe::RequantArgs rq{reinterpret_cast<const uint16_t*>(at(L.y2)), inv_padded, T * (int64_t)k, I, afmt, at(L.a2),
                        at(L.a2s)};
    MOE_CUDA_TRY(moe::launch_requant(rq, s));
    MOE_CUDA_TRY(mark());
  }

  moe::GemmArgs g2 = g1;
  g2.epilogue = 1;
  g2.act = at(L.a2);
  g2.act_sf = at(L.a2s);
  g2.w = w2;
  g2.w_sf = w2s;
  g2.N = H;
  g2.K = I;
  g2.max_tiles = mtiles_cap * ((H + moe::kNTile - 1) / moe::kNTile);  // last N tile may be 128 wide
  g2.a_rows = a_rows_for(I);
  g2.out_codes = nullptr;
  g2.out_sf = nullptr;
  g2.out_bf16 = reinterpret_cast<uint16_t*>(at(L.y2));
  if (fp8_y2) {
    g2.epilogue = 3;
    g2.out_codes = y2q;
    g2.out_sf = y2s;
    g2.out_bf16 = nullptr;
    g2.row_w = row_w;
  }
  MOE_CUDA_TRY(run_gemm(g2));
  MOE_CUDA_TRY(mark());

  moe::CombineArgs ca{fp8_y2 ? nullptr : reinterpret_cast<const uint16_t*>(at(L.y2)), tw, inv_padded, T, H, k,
                      static_cast<uint16_t*>(out), y2q, y2s};
  MOE_CUDA_TRY(moe::launch_combine(ca, s));
  MOE_CUDA_TRY(mark());
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "MOE_ERR_UNSUPPORTED_DEVICE";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
  }
  return "MOE_UNKNOWN_STATUS";
}

moe_status_t moe_get_workspace_layout(int64_t T, int H, int I, int E, int k, moe_act_fmt_t fmt,
                                      moe_workspace_layout_t* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  return layout(T, H, I, E, k, fmt, out);
}

size_t moe_workspace_bytes(int64_t T, int H, int I, int E, int k, moe_act_fmt_t fmt) {
  moe_workspace_layout_t L;
  return layout(T, H, I, E, k, fmt, &L) == MOE_OK ? L.total : 0;
}

moe_status_t moe_topk_route(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w, void* stream) {
  if (!logits || !ids || !w) return MOE_ERR_INVALID_ARG;
  if (T < 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
  if (k > kMaxTopK || E > kMaxExperts) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(logits, 4) || !aligned(ids, 4) || !aligned(w, 4)) return MOE_ERR_MISALIGNED;
  if (T == 0) return MOE_OK;
  DeviceInfo dev;
  const moe_status_t st = device_info(&dev);
  if (st != MOE_OK) return st;
  moe::RouteArgs ra{logits, T, E, k, ids, w, nullptr, 0, nullptr, 0};
  MOE_CUDA_TRY(moe::launch_route(ra, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status_t moe_sort_by_expert(const int32_t* ids, int64_t T, int E, int k, int32_t* counts, int64_t* offsets,
                                int32_t* sorted_pair, int32_t* inv, void* ws, size_t ws_bytes, void* stream) {
  if (!ids || !counts || !offsets || !sorted_pair || !inv || !ws) return MOE_ERR_INVALID_ARG;
  moe_workspace_layout_t L;
  moe_status_t st = layout(T, 128, 128, E, k, MOE_ACT_MXFP8, &L);
  if (st != MOE_OK) return st;
  if (!aligned(ws, 256) || !aligned(ids, 4) || !aligned(counts, 4) || !aligned(offsets, 8) ||
      !aligned(sorted_pair, 4) || !aligned(inv, 4))
    return MOE_ERR_MISALIGNED;
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo dev;
  st = device_info(&dev);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* W = static_cast<uint8_t*>(ws);
  uint32_t* status = reinterpret_cast<uint32_t*>(W + L.status);
  MOE_CUDA_TRY(cudaMemsetAsync(status, 0, sizeof(uint32_t), s));
  moe::SortArgs sa{ids, T, E, k, reinterpret_cast<int32_t*>(W + L.chunk_hist), L.nchunk, counts, offsets,
                   nullptr, nullptr, sorted_pair, inv, nullptr, status};
  if (T == 0) {
    MOE_CUDA_TRY(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s));
    MOE_CUDA_TRY(cudaMemsetAsync(offsets, 0, sizeof(int64_t) * (E + 1), s));
    return MOE_OK;
  }
  MOE_CUDA_TRY(moe::launch_histogram(sa, s));
  MOE_CUDA_TRY(moe::launch_sort(sa, s));
  return MOE_OK;
}

moe_status_t moe_quantize_mx(const void* x, int64_t rows, int K, moe_act_fmt_t fmt, uint8_t* codes,
                             uint8_t* scales, void* stream) {
  if (!x || !codes || !scales) return MOE_ERR_INVALID_ARG;
  if (rows < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (fmt != MOE_ACT_MXFP8 && fmt != MOE_ACT_MXFP4) return MOE_ERR_INVALID_ARG;
  if (K % 32 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(codes, 8)) return MOE_ERR_MISALIGNED;
  if (rows == 0) return MOE_OK;
  DeviceInfo dev;
  const moe_status_t st = device_info(&dev);
  if (st != MOE_OK) return st;
  moe::QuantArgs qa{static_cast<const uint16_t*>(x), rows, K, fmt == MOE_ACT_MXFP8 ? 0 : 1, codes, scales, nullptr, 1};
  MOE_CUDA_TRY(moe::launch_quant(qa, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status_t moe_a8w4_forward(const void* x, const float* logits, const uint8_t* w1, const uint8_t* w1s,
                              const uint8_t* w2, const uint8_t* w2s, void* out, int64_t T, int H, int I, int E, int k,
                              void* ws, size_t ws_bytes, void* stream) {
  return forward(x, nullptr, logits, w1, w1s, w2, w2s, out, T, H, I, E, k, ws, ws_bytes, stream, MOE_ACT_MXFP8, false);
}

moe_status_t moe_a8w4_forward_prepacked(const void* x, const float* logits, const uint8_t* w1, const uint8_t* w1s,
                                        const uint8_t* w2, const uint8_t* w2s, void* out, int64_t T, int H, int I,
                                        int E, int k, void* ws, size_t ws_bytes, void* stream) {
  return forward(x, nullptr, logits, w1, w1s, w2, w2s, out, T, H, I, E, k, ws, ws_bytes, stream, MOE_ACT_MXFP8, true);
}

moe_status_t moe_a4w4_forward_prepacked(const void* x, const float* logits, const uint8_t* w1, const uint8_t* w1s,
                                        const uint8_t* w2, const uint8_t* w2s, void* out, int64_t T, int H, int I,
                                        int E, int k, void* ws, size_t ws_bytes, void* stream) {
  return forward(x, nullptr, logits, w1, w1s, w2, w2s, out, T, H, I, E, k, ws, ws_bytes, stream, MOE_ACT_MXFP4, true);
}

moe_status_t moe_forward_ex(const moe_forward_args_t* a) {
  if (!a) return MOE_ERR_INVALID_ARG;
  if (a->act_fmt != MOE_ACT_MXFP8 && a->act_fmt != MOE_ACT_MXFP4) return MOE_ERR_INVALID_ARG;
  if (a->prequantized && a->T > 0 && !a->x_scale) return MOE_ERR_INVALID_ARG;
  return forward(a->x, a->prequantized ? a->x_scale : nullptr, a->gate_logits, a->w1, a->w1_scale, a->w2,
                 a->w2_scale, a->out, a->T, a->H, a->I, a->E, a->k, a->workspace, a->workspace_bytes, a->stream,
                 a->act_fmt, a->weight_scales_prepacked != 0, nullptr, a->schedule);
}

moe_status_t moe_a8w4_forward_prequant(const uint8_t* xq, const uint8_t* xq_scale, const float* logits,
                                       const uint8_t* w1, const uint8_t* w1s, const uint8_t* w2, const uint8_t* w2s,
                                       void* out, int64_t T, int H, int I, int E, int k, void* ws, size_t ws_bytes,
                                       void* stream) {
  if (T > 0 && !xq_scale) return MOE_ERR_INVALID_ARG;
  return forward(xq, T > 0 ? xq_scale : nullptr, logits, w1, w1s, w2, w2s, out, T, H, I, E, k, ws, ws_bytes,
                 stream, MOE_ACT_MXFP8, false);
}

moe_status_t moe_a4w4_forward_prequant(const uint8_t* xq, const uint8_t* xq_scale, const float* logits,
                                       const uint8_t* w1, const uint8_t* w1s, const uint8_t* w2, const uint8_t* w2s,
                                       void* out, int64_t T, int H, int I, int E, int k, void* ws, size_t ws_bytes,
                                       void* stream) {
  if (T > 0 && !xq_scale) return MOE_ERR_INVALID_ARG;
  return forward(xq, T > 0 ? xq_scale : nullptr, logits, w1, w1s, w2, w2s, out, T, H, I, E, k, ws, ws_bytes,
                 stream, MOE_ACT_MXFP4, false);
}

moe_status_t moe_prepack_scales(const uint8_t* scales, int64_t rows, int K, uint8_t* tiled, void* stream) {
  if (!scales || !tiled || rows < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (rows % 128 != 0 || K % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(scales, 4) || !aligned(tiled, 16)) return MOE_ERR_MISALIGNED;
  if (rows == 0) return MOE_OK;
  DeviceInfo dev;
  const moe_status_t st = device_info(&dev);
  if (st != MOE_OK) return st;
  MOE_CUDA_TRY(moe::launch_prepack_scales(scales, rows, K, tiled, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status_t moe_a4w4_forward(const void* x, const float* logits, const uint8_t* w1, const uint8_t* w1s,
                              const uint8_t* w2, const uint8_t* w2s, void* out, int64_t T, int H, int I, int E, int k,
                              void* ws, size_t ws_bytes, void* stream) {
  return forward(x, nullptr, logits, w1, w1s, w2, w2s, out, T, H, I, E, k, ws, ws_bytes, stream, MOE_ACT_MXFP4, false);
}

moe_status_t moe_read_device_status(const void* ws, void* stream, moe_status_t* status_out) {
  if (!ws || !status_out) return MOE_ERR_INVALID_ARG;
  uint32_t v = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  *status_out = (v & moe::kStatusTimeout) ? MOE_ERR_DEVICE_TIMEOUT
                : (v & moe::kStatusInvalidArg) ? MOE_ERR_INVALID_ARG
                                               : MOE_OK;
  return MOE_OK;
}

int moe_forward_launch_count(int64_t T, int H, int I) { return launch_count(T, H, I); }

int moe_forward_launch_count_ex(int64_t T, int H, int I, int schedule) {
  if (!valid_schedule(schedule)) return -1;
  return launch_count(T, H, I, schedule);
}

int moe_forward_launch_count_cfg(int64_t T, int H, int I, int E, int k, int fmt, int schedule,
                                 int prepacked_scales) {
  if (!valid_schedule(schedule) || (fmt != MOE_ACT_MXFP8 && fmt != MOE_ACT_MXFP4)) return -1;
  return launch_count_cfg(T, H, I, E, k, fmt == MOE_ACT_MXFP8 ? 0 : 1, schedule, prepacked_scales != 0);
}

int moe_forward_split_gemms(int64_t T, int H, int I, int E, int k, int fmt, int schedule, int prepacked_scales) {
  if (!valid_schedule(schedule) || (fmt != MOE_ACT_MXFP8 && fmt != MOE_ACT_MXFP4)) return -1;
  if (launch_count(T, H, I, schedule) <= 1) return 0;
  const int afmt = fmt == MOE_ACT_MXFP8 ? 0 : 1;
  const bool pp = prepacked_scales != 0;
  return (split_gemm(T, E, k, afmt, pp, schedule, 2 * I, H) ? 1 : 0) | (split_gemm(T, E, k, afmt, pp, schedule, H, I) ? 2 : 0);
}

moe_status_t moe_profile_forward(moe_act_fmt_t fmt, const void* x, const float* logits, const uint8_t* w1,
                                 const uint8_t* w1s, const uint8_t* w2, const uint8_t* w2s, void* out, int64_t T,
                                 int H, int I, int E, int k, void* ws, size_t ws_bytes, void* stream,
                                 int prepacked_scales, int schedule, float* kernel_us) {
  if (!kernel_us) return MOE_ERR_INVALID_ARG;
  if (fmt != MOE_ACT_MXFP8 && fmt != MOE_ACT_MXFP4) return MOE_ERR_INVALID_ARG;
  cudaEvent_t ev[kMaxForwardKernels + 1] = {};
  moe_status_t st = MOE_OK;
  for (int i = 0; i <= kMaxForwardKernels && st == MOE_OK; ++i)
    if (cudaEventCreate(&ev[i]) != cudaSuccess) st = MOE_ERR_CUDA;
  if (st == MOE_OK)
    st = forward(x, nullptr, logits, w1, w1s, w2, w2s, out, T, H, I, E, k, ws, ws_bytes, stream, fmt,
                 prepacked_scales != 0, ev, schedule);
  const int nk = launch_count_cfg(T, H, I, E, k, fmt == MOE_ACT_MXFP8 ? 0 : 1, schedule, prepacked_scales != 0);
  if (st == MOE_OK && T > 0) {
    if (cudaEventSynchronize(ev[nk]) != cudaSuccess) st = MOE_ERR_CUDA;
    for (int i = 0; i < nk && st == MOE_OK; ++i) {
      float ms = 0.0f;
      if (cudaEventElapsedTime(&ms, ev[i], ev[i + 1]) != cudaSuccess) st = MOE_ERR_CUDA;
      kernel_us[i] = ms * 1000.0f;
    }
  }
  for (int i = 0; i <= kMaxForwardKernels; ++i)
    if (ev[i]) cudaEventDestroy(ev[i]);
  return st;
}

}  // extern "C"
