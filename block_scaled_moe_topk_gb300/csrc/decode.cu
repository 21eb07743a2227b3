// decode.cu -- the whole expert layer for a small batch (T <= 64 tokens) in one persistent
// kernel: routing + sort, quantisation of x, GEMM1 with SwiGLU and the A2 requantisation,
// GEMM2 and the top-k combine.
//
// The pages replace the serial chain dispatch + gemm1 + quant + gemm2 + combine by one fused
// step ("feat(moe): FlyDSL MegaMoE fused EP-MoE integration", description; "add A4W4 and FP8
// P2P transport support to MegaMoE", Test Result: the fused kernel against the serial chain).
// On one GPU the exchange steps become the local permute and combine, and what fusion buys at
// decode sizes is time: one launch instead of five, and every SM streaming weights instead of
// the few that own a whole (expert, 256-column) tile.
//
// Schedule (identical in every CTA, derived from the routing each CTA computes itself):
//   prologue  every CTA routes all T tokens (a warp per token, top-k softmax) and sorts the T*k
//             pairs in shared memory (the chain's counting sort; CTA 0 also writes routing and
//             sort to the workspace): no CTA waits for another before its weights start to
//             stream.  CTA b < T then quantises token b into its k padded expert rows and
//             counts itself done; activation loads wait for that count.
//   GEMM1     items = (active expert, 256-column tile of 2I), K stages of 128 (256 for A4W4).
//             With at least as many items as SMs (and whenever cutting items would not pay for
//             its partial sums) whole items go round-robin to the CTAs.  Otherwise the stages of
//             all items, laid end to end, are cut into gridDim.x equal ranges (stream-K): a CTA
//             whose range covers a whole item runs the SwiGLU / requant epilogue itself;
//             items cut between CTAs leave fp32 partial accumulators in the
//             workspace, and the last contributor (an atomic ticket per item and epilogue warp)
//             sums them in CTA order -- the same order whoever arrives last -- and runs the
//             epilogue, one row at a time spread over the warp's lanes (every contributor's
//             load in flight at once).  Each finished part bumps its expert's ready counter.
//   GEMM2     the same over (active expert, 256-column tile of H) with K = I; the activation
//             producer waits for the expert's ready counter before loading A2, while the
//             weight producer runs ahead (the ring fills with W2 while GEMM1 finishes).
//             Final rows go to an fp32 y2 buffer.
//   combine   once every GEMM2 part is final (a counter), all CTAs form out = bf16(sum_j w_j *
//             y2_j) in slot order with fp32 accumulation, each a slice of (token, columns).
// Every wait (mbarriers, global counters) is bounded as in the GEMM kernel: on expiry the CTA
// records MOE_ERR_DEVICE_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns; any
// CTA waiting on its work then expires the same way.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "gemm_common.cuh"
#include "moe_internal.h"
#include "mx_device.cuh"
#include "ptx.cuh"
#include "route_device.cuh"

namespace moe {
namespace {

constexpr int kDThreads = 352;  // warp 0 activation producer, 1 MMA, 2..9 epilogue, 10 weight producer
constexpr int kDWarps = kDThreads / 32;
constexpr int kDEpiWarps = 8;
constexpr int kDWeightWarp = 10;
constexpr uint32_t kDTmemCols = 512;
constexpr uint32_t kDSfCol0 = 256;
constexpr uint32_t kDSfSlotCols = 32;
// A CTA is given at least this many K stages of a GEMM (fewer CTAs take part when the GEMM is
// small): each cut costs a partial write, a ticket and a read-back.
constexpr int kMinStagesPerCta = 2;

template <int ACT, int AROWS>
struct DGeo {
  static constexpr int kABytes = AROWS * 128;
  static constexpr int kBOff = kABytes;
  static constexpr int kBBytes = kNTile * 128;
  static constexpr int kSfaOff = kBOff + kBBytes;
  static constexpr int kSfaBytes = ActTraits<ACT>::kKPerStage / 128 * 512;
  static constexpr int kSfbOff = kSfaOff + kSfaBytes;
  static constexpr int kStageBytes = (kSfbOff + 2 * kSfaBytes + 1023) / 1024 * 1024;
  // as deep as shared memory allows: a decode step streams each weight byte once, so the bytes
  // in flight per SM (the ring) set the rate
  static constexpr int kStages = (AROWS == 16 && ACT == 0) ? 6 : 5;
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kTabOff = kBarOff + 256;
  // tables kept past the prologue [kDecodeMaxPairs]: per active expert its id, row count,
  // unpadded row offset and M-tile base (int16); per routed pair its weight (fp32) and
  // unpadded row (int16)
  static constexpr int kTabBytes = kDecodeMaxPairs * (4 * 2 + 4 + 2) + 128;  // + the two phase records
  static constexpr int kSmemBytes = kTabOff + kTabBytes + 1024;
  static_assert(kBOff % 1024 == 0 && kStageBytes % 1024 == 0, "SW128 tiles need 1024-byte alignment");
  static_assert(kSmemBytes <= 232448, "decode kernel shared memory");
  static_assert(kStages * 32 <= 256, "TMEM scale slots");
  // the prologue's scratch sits in the last ring slot, at these byte offsets: the expert
  // histogram (int [E+1]), the per-active-expert token masks (uint64), pair ids and padded rows
  // (int), then the staged quantised row of at most kDecodeMaxHidden elements and its scales
  static constexpr int kScrMaskOff = (4 * (kMaxExperts + 1) + 127) / 128 * 128;
  static constexpr int kScrPairIdOff = kScrMaskOff + 8 * kDecodeMaxPairs;
  static constexpr int kScrPairInvpOff = kScrPairIdOff + 4 * kDecodeMaxPairs;
  static constexpr int kStageCodesOff = (kScrPairInvpOff + 4 * kDecodeMaxPairs + 127) / 128 * 128;
  static_assert(kScrMaskOff % 8 == 0, "64-bit token masks");
  static_assert(kStageBytes >= kStageCodesOff + kDecodeMaxHidden + kDecodeMaxHidden / 32, "prologue scratch");
  static_assert(kStageCodesOff % 16 == 0, "16-byte accesses to the staged row");
};

struct DecodeParams {  // 64-byte aligned through its CUtensorMap members
  CUtensorMap tmap_x;   // xq [rows_cap, H or H/2], box 128 B x AROWS
  CUtensorMap tmap_w1;  // W1 [E, 2I, H/2]
  CUtensorMap tmap_a2;  // a2 [rows_cap, I or I/2], box 128 B x AROWS
  CUtensorMap tmap_w2;  // W2 [E, H, I/2]
  const uint16_t* x;
  const uint8_t* xq_in;
  const uint8_t* xs_in;
  const float* logits;
  const uint8_t* w1_sf;
  const uint8_t* w2_sf;
  uint8_t* xq;
  uint8_t* xs;
  uint8_t* a2;
  uint8_t* a2s;
  float* part;
  float* y2f;
  uint16_t* out;
  int32_t* ids;
  float* tw;
  int32_t* counts;
  int64_t* offsets;
  int64_t* padded_offsets;
  int32_t* mtile_base;
  int32_t* sorted_pair;
  int32_t* inv;
  int32_t* inv_padded;
  uint32_t* sync;
  uint32_t* status;
  uint64_t timeout_ns;
  int T, H, I, E, k;
  int w_sf_tiled;
  int test_stall;
};

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Poll a global counter until it reaches `target`, the CTA aborts, or the time limit passes
// (counted in SM cycles at 2 per nanosecond, as bounded_wait).  On expiry the first record
// names the counter as 1000 + its word offset in the sync region.
__device__ __noinline__ bool wait_counter(const uint32_t* ctr, uint32_t target, const uint32_t* sync_base,
                                          const Sync& s, uint64_t limit_ns) {
  const uint64_t limit_cycles = 2 * limit_ns;
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire_u32(ctr) >= target) return true;
    if ((it & 15u) == 15u) {
      if (*s.abort_flag) return false;
      const uint64_t now = clock64();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit_cycles) {
        *s.abort_flag = 1;
        atomicOr(s.status, kStatusTimeout);
        if (atomicCAS(s.status + 1, 0u, 1u) == 0u) {
          s.status[2] = 1000u + (uint32_t)(ctr - sync_base);
          s.status[3] = target;
          s.status[4] = blockIdx.x;
          s.status[5] = threadIdx.x / 32;
          s.status[6] = (uint32_t)((now - t0) / 2000);
        }
        return false;
      }
    }
    __nanosleep(64);
  }
}

// Per-GEMM schedule (the same in every CTA; computed once per CTA, kept in shared memory).
struct Phase {
  int nks;      // K stages per item
  int NT;       // N tiles per expert
  int N, K;
  int items;    // active experts x N tiles
  int Z;        // stages of all items
  int g;        // CTAs taking part
  int q, r;     // stream-K: Z = g * q + r; CTA b owns [b * q + min(b, r), ...), q + (b < r) stages
  int whole;    // whole items round-robin (item i on CTA i % g) instead of stream-K ranges
  int pad;
};
static_assert(sizeof(Phase) * 2 <= 128, "phase records");
// Cutting items pays for itself only if the stream-K ranges finish this many stages earlier
// than whole items would: the partial sums of a cut item (write, ticket, read-back by the last
// contributor) cost about as much latency as ten K stages.
constexpr int kCutCostStages = 10;

__device__ __forceinline__ int range_begin(const Phase& P, int b) { return b * P.q + min(b, P.r); }
// The CTA whose stream-K range holds stage z.
__device__ __forceinline__ int owner_of(const Phase& P, int z) {
  const int big = P.r * (P.q + 1);  // the first r ranges are one stage longer
  return z < big ? z / (P.q + 1) : P.r + (z - big) / P.q;
}

__device__ __forceinline__ void make_phase(Phase& P, int N, int K, int KPS, int n_act, int G) {
  P.N = N;
  P.K = K;
  P.nks = (K + KPS - 1) / KPS;
  P.NT = (N + kNTile - 1) / kNTile;
  P.items = n_act * P.NT;
  P.Z = P.items * P.nks;
  const int rr = (P.items + G - 1) / G * P.nks;        // stages of the busiest CTA, whole items
  const int sk = (P.Z + G - 1) / G + kCutCostStages;   // ... with stream-K ranges
  P.whole = 20 * sk >= 19 * rr ? 1 : 0;                // cut items only for a clear gain
  P.g = P.whole ? min(G, P.items) : max(1, min(G, P.Z / kMinStagesPerCta));
  P.q = P.Z / P.g;
  P.r = P.Z % P.g;
  P.pad = 0;
}

// Warp-uniform bounded wait for a shared-memory flag set by other warps of the CTA.
__device__ __noinline__ bool warp_wait_flag(volatile int* flag, const Sync& s, uint64_t limit_ns) {
  const uint64_t limit_cycles = 2 * limit_ns;
  uint64_t t0 = 0;
  bool ok = true;
  for (uint32_t it = 0;; ++it) {
    if (*flag != 0) break;
    if ((it & 15u) == 15u) {
      if (*s.abort_flag) {
        ok = false;
        break;
      }
      const uint64_t now = clock64();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit_cycles) {
        *s.abort_flag = 1;
        atomicOr(s.status, kStatusTimeout);
        if (atomicCAS(s.status + 1, 0u, 1u) == 0u) {
          s.status[2] = 999u;  // the prologue's scratch was never released
          s.status[3] = 0;
          s.status[4] = blockIdx.x;
          s.status[5] = threadIdx.x / 32;
          s.status[6] = (uint32_t)((now - t0) / 2000);
        }
        ok = false;
        break;
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}

// Named barriers of the prologue hand-off (id 0 is __syncthreads): the pair scatter (warp 0) is
// done before the quantiser (warps 2..9) reads the padded rows; the quantiser's warps meet
// before one of them signals.
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int ACT, int AROWS>
__global__ void __launch_bounds__(kDThreads, 1) moe_decode_kernel(const __grid_constant__ DecodeParams p) {
  using TR = ActTraits<ACT>;
  using G = DGeo<ACT, AROWS>;
  constexpr int kStages = G::kStages;
  constexpr int kStageBytes = G::kStageBytes;
  constexpr int kSfaOff = G::kSfaOff;
  constexpr int kSfbOff = G::kSfbOff;
  constexpr int kMmaPerStage = TR::kKPerStage / TR::kMmaK;
  constexpr int kAtomsPerStage = TR::kKPerStage / 128;
  constexpr uint32_t kSfaCols = kAtomsPerStage * 4;
  constexpr int KPS = TR::kKPerStage;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + G::kBarOff;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t tmem_full_bar = bar0 + 8u * (2 * kStages);
  const uint32_t tmem_empty_bar = tmem_full_bar + 8;
  const uint32_t drain_bar = tmem_full_bar + 16;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + G::kBarOff + 8 * (2 * kStages + 3));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* n_active_s = reinterpret_cast<int*>(tmem_holder + 2);
  int16_t* act_e = reinterpret_cast<int16_t*>(smem + G::kTabOff);
  int16_t* act_cnt = act_e + kDecodeMaxPairs;
  int16_t* act_off = act_e + 2 * kDecodeMaxPairs;
  int16_t* act_mtb = act_e + 3 * kDecodeMaxPairs;
  float* pair_w = reinterpret_cast<float*>(act_e + 4 * kDecodeMaxPairs);
  int16_t* pair_inv = reinterpret_cast<int16_t*>(pair_w + kDecodeMaxPairs);  // unpadded row of pair q
  Phase* phs = reinterpret_cast<Phase*>(pair_inv + kDecodeMaxPairs);
  // prologue scratch in the last ring slot: the scatter (warps 0, 2..9) and the quantiser (warps 2..9)
  // still read it after the producers start; the weight producer enters that slot only after
  // the quantiser's warps release it, the activation producer only after the quant count
  // (which includes this CTA's own quantiser)
  int* hist = reinterpret_cast<int*>(smem + (kStages - 1) * kStageBytes);
  // per active expert, the set of tokens routed to it (T <= 64: one bit per token); a pair's
  // rank inside its expert's group is the number of earlier tokens in that set
  unsigned long long* tok_mask = reinterpret_cast<unsigned long long*>(reinterpret_cast<uint8_t*>(hist) + G::kScrMaskOff);
  int* pair_id = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(hist) + G::kScrPairIdOff);
  int* pair_invp = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(hist) + G::kScrPairInvpOff);  // padded row of pair q

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int T = p.T, E = p.E, k = p.k, H = p.H, I = p.I;
  const int R = T * k;
  const int b = blockIdx.x;
  const Sync sync{abort_flag, p.status, p.timeout_ns, bar0};

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // activation producer's expect_tx + weight producer's expect_tx (+ its 32 lanes' cp.async
      // arrivals when the weight scales are gathered from the canonical layout)
      mbar_init(full_bar(s), p.w_sf_tiled ? 2 : 2 + 32);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tmem_full_bar, 1);
    mbar_init(tmem_empty_bar, kDEpiWarps);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    tmem_holder[3] = 0;  // set once the prologue's scratch (in the last ring slot) is free
    tmem_holder[4] = 1;  // routing available (cleared if the published routing never completes)
    fence_mbar_init();
    prefetch_tensormap(&p.tmap_x);
    prefetch_tensormap(&p.tmap_w1);
    prefetch_tensormap(&p.tmap_a2);
    prefetch_tensormap(&p.tmap_w2);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kDTmemCols);
    tmem_relinquish();
  }
  if (warp == kDWarps - 1 && lane == 0) {
    if (b < T && p.x != nullptr) bulk_prefetch_l2(p.x + (int64_t)b * H, (uint32_t)H * 2u);  // the row this CTA quantises
    // every token's logits (the 16-byte-aligned interior of the array) for the routing warps
    const uintptr_t lo = (reinterpret_cast<uintptr_t>(p.logits) + 15) & ~uintptr_t(15);
    const uintptr_t hi = (reinterpret_cast<uintptr_t>(p.logits + (int64_t)T * E)) & ~uintptr_t(15);
    if (hi > lo) bulk_prefetch_l2(reinterpret_cast<const void*>(lo), (uint32_t)(hi - lo));
  }
  for (int e = threadIdx.x; e < E; e += kDThreads) hist[e] = 0;
  for (int i = threadIdx.x; i < kDecodeMaxPairs; i += kDThreads) tok_mask[i] = 0;
  __syncthreads();

  // ---------------------------------------------------------------- quantise token b (b < T)
  // into shared memory (warps 2..9), while the other warps route: only the copy to the k padded
  // expert rows waits for the sort.  16 elements per thread, lanes 2m and 2m+1 share a block.
  // (16-byte stores and loads: the staging area starts on a 128-byte boundary of the slot)
  uint8_t* stage_codes = reinterpret_cast<uint8_t*>(hist) + G::kStageCodesOff;
  uint8_t* stage_sf = stage_codes + (ACT == 0 ? H : H / 2);
  const int row_bytes = ACT == 0 ? H : H / 2;
  if (b < T && warp >= 2 && warp < 2 + kDEpiWarps) {
    const int et = threadIdx.x - 64;
    if (p.x != nullptr) {
      const int chunks = H / 16;
      for (int base = et - lane; base < chunks; base += 32 * kDEpiWarps) {  // warp-uniform
        const int c = base + lane;
        const bool active = c < chunks;
        float v[16];
        if (active) {
          const uint4* src = reinterpret_cast<const uint4*>(p.x + (int64_t)b * H + c * 16);
          const uint4 r0 = src[0], r1 = src[1];
          const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            v[2 * q] = __uint_as_float(w[q] << 16);
            v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] = 0.0f;
        }
        float amax = 0.0f;
#pragma unroll
        for (int q = 0; q < 16; ++q) amax = fmaxf(amax, fabsf(v[q]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        if (!active) continue;
        const MxScale sc = mx_scale<ACT>(amax);
        if (ACT == 0) {
          const uint2 c0 = pack_e4m3x8(v, sc.mult), c1 = pack_e4m3x8(v + 8, sc.mult);
          *reinterpret_cast<uint4*>(stage_codes + c * 16) = make_uint4(c0.x, c0.y, c1.x, c1.y);
        } else {
          *reinterpret_cast<uint2*>(stage_codes + c * 8) = make_uint2(pack_e2m1x8(v, sc.mult), pack_e2m1x8(v + 8, sc.mult));
        }
        if ((c & 1) == 0) stage_sf[c / 2] = sc.byte;
      }
    } else {
      // prequantised input: token b's codes and canonical scales
      for (int c = et; c < row_bytes / 16; c += 32 * kDEpiWarps)
        *reinterpret_cast<uint4*>(stage_codes + c * 16) =
            *reinterpret_cast<const uint4*>(p.xq_in + (int64_t)b * row_bytes + c * 16);
      for (int kb = et; kb < H / 32; kb += 32 * kDEpiWarps) stage_sf[kb] = p.xs_in[(int64_t)b * (H / 32) + kb];
    }
  }

  // ---------------------------------------------------------------- routing
  // Up to 11 tokens every CTA routes the whole batch itself (a warp per token; warps 0, 1, 10
  // first, the quantising warps after): no CTA waits for another before its weights start to
  // stream.  Above that CTA b routes token b alone and publishes it (ids and weights in the
  // workspace, a counter), and every CTA reads the batch back once all T are published.
  const bool distributed = T > kDWarps;
  auto route_one = [&](int t, bool publish) {
    int id;
    float w;
    const float* l = p.logits + (int64_t)t * E;
    if (E <= 512) route_token_fast<16>(l, E, k, lane, id, w);
    else route_token_fast<kMaxExperts / 32>(l, E, k, lane, id, w);
    if (lane < k) {
      if (!distributed) {
        pair_id[t * k + lane] = id;
        pair_w[t * k + lane] = w;
        atomicAdd(&hist[id], 1);
      }
      if (publish) {
        p.ids[t * k + lane] = id;
        p.tw[t * k + lane] = w;
      }
    }
  };
  if (!distributed) {
    const int t = warp == 0 ? 0 : warp == 1 ? 1 : warp == kDWarps - 1 ? 2 : warp + 1;
    if (t < T) route_one(t, b == 0);
    __syncthreads();
  } else {
    if (warp == 0) {
      if (b < T) {
        route_one(b, true);
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(p.sync + kSyncRouted, 1u);
      }
      if (lane == 0 && !wait_counter(p.sync + kSyncRouted, (uint32_t)T, p.sync, sync, p.timeout_ns))
        tmem_holder[4] = 0;
    }
    __syncthreads();
    if (tmem_holder[4] != 0) {
      for (int q = threadIdx.x; q < R; q += kDThreads) {
        const int id = __ldcg(p.ids + q);
        pair_id[q] = id;
        pair_w[q] = __ldcg(p.tw + q);
        atomicAdd(&hist[id], 1);
      }
    }
    // (a routing wait that expired leaves the histogram empty: no expert is active, nothing is
    // scheduled, the scatter, copy and combine are skipped, and the status word carries the
    // timeout)
    __syncthreads();
  }
  const bool routed = tmem_holder[4] != 0;
  const bool writer = b == 0;  // CTA 0 writes the sort to the workspace
  // The stable scatter of the T*k pairs, on warp 0 and warps 2..9 (u = 0..287): token masks,
  // then every pair's rank and rows; named barrier 3 between the passes.
  auto scatter_pairs = [&](int u) {
    constexpr int kU = 32 + 32 * kDEpiWarps;
    if (routed)
      for (int q = u; q < R; q += kU) atomicOr(&tok_mask[hist[pair_id[q]]], 1ull << (q / k));
    named_barrier(3, kU);
    if (routed)
      for (int q = u; q < R; q += kU) {
        const int t = q / k;
        const int a = hist[pair_id[q]];
        const int local = __popcll(tok_mask[a] & ((1ull << t) - 1ull));
        const int r = act_off[a] + local;
        const int rp = kRowTile * act_mtb[a] + local;
        pair_inv[q] = (int16_t)r;
        pair_invp[q] = rp;
        if (writer) {
          p.sorted_pair[r] = q;
          p.inv[q] = r;
          p.inv_padded[q] = rp;
        }
      }
  };
  if (warp == 0) {
    // prefixes over experts (lane L owns experts [L * per, L * per + per)): unpadded rows,
    // 128-row tiles and the active-expert index; hist[e] becomes e's active index
    const int per = (E + 31) / 32;
    const int e0 = min(lane * per, E), e1 = min(e0 + per, E);
    int rows = 0, tiles = 0, nact = 0;
    for (int e = e0; e < e1; ++e) {
      const int c = hist[e];
      rows += c;
      tiles += (c + kRowTile - 1) / kRowTile;
      nact += c > 0;
    }
    int xr = rows, xt = tiles, xa = nact;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, xr, o), bb = __shfl_up_sync(0xffffffffu, xt, o),
                c = __shfl_up_sync(0xffffffffu, xa, o);
      if (lane >= o) {
        xr += a;
        xt += bb;
        xa += c;
      }
    }
    xr -= rows;
    xt -= tiles;
    xa -= nact;
    for (int e = e0; e < e1; ++e) {
      const int c = hist[e];
      if (writer) {
        p.counts[e] = c;
        p.offsets[e] = xr;
        p.padded_offsets[e] = (int64_t)kRowTile * xt;
        p.mtile_base[e] = xt;
      }
      if (c > 0) {
        act_e[xa] = (int16_t)e;
        act_cnt[xa] = (int16_t)c;
        act_off[xa] = (int16_t)xr;
        act_mtb[xa] = (int16_t)xt;
        hist[e] = xa++;
      } else {
        hist[e] = -1;
      }
      xr += c;
      xt += (c + kRowTile - 1) / kRowTile;
    }
    const int n_act = __shfl_sync(0xffffffffu, xa, 31);
    if (lane == 31) {
      if (writer) {
        p.offsets[E] = xr;
        p.padded_offsets[E] = (int64_t)kRowTile * xt;
        p.mtile_base[E] = xt;
      }
      *n_active_s = n_act;
    }
    if (lane == 0) {
      make_phase(phs[0], 2 * I, H, KPS, n_act, (int)gridDim.x);
      make_phase(phs[1], H, I, KPS, n_act, (int)gridDim.x);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int n_act = *n_active_s;
  // epilogue parts (warps) with rows per expert: one per live 32-row quadrant and column half
  auto quads_of = [&](int a) { return (act_cnt[a] + 31) / 32; };

  // Every role walks the same segments: (GEMM, item, first stage, end stage) of this CTA.
  // Whole-item phases walk items b, b + g, ...; stream-K phases walk the CTA's stage range.
#define MOE_FOR_EACH_SEGMENT(...)                                                          \
  _Pragma("unroll 1") for (int gi = 0; gi < 2; ++gi) {                                     \
    const Phase P = phs[gi];                                                               \
    if (b >= P.g) continue;                                                                \
    int z = P.whole ? b * P.nks : range_begin(P, b);                                       \
    const int zend = P.whole ? P.Z : range_begin(P, b + 1);                                \
    const int zstep = P.whole ? (P.g - 1) * P.nks : 0;                                     \
    while (z < zend) {                                                                     \
      const int item = z / P.nks;                                                          \
      const int ks0 = z - item * P.nks;                                                    \
      const int ks1 = min(P.nks, ks0 + (zend - z));                                        \
      const int a = item / P.NT, nt = item % P.NT;                                         \
      __VA_ARGS__                                                                          \
      z += ks1 - ks0 + zstep;                                                              \
    }                                                                                      \
  }

  if (warp == 0) {
    // ------------------------------------------------------------ pair scatter (with warps
    // 2..9), then the activation producer.  Pairs in (expert, token) order: pair q = (t, j) of
    // active expert a goes to row act_off[a] + (number of tokens below t routed to a).
    scatter_pairs(lane);
    named_barrier(1, 32 + 32 * kDEpiWarps);
    // converged loop, one elected lane issues the copies; lane 0 alone polls the global
    // counters and passes the result on (a warp barrier orders its acquire before the copies)
    {
      int slot = 0;
      uint32_t phase = 0;
      int armed[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) armed[s] = -1;
      bool ok = !p.test_stall, quant_seen = false;
      int ready_a = -1;
      MOE_FOR_EACH_SEGMENT({
        if (!ok) break;
        const int64_t row0 = (int64_t)kRowTile * act_mtb[a];
        const int K = P.K;
        for (int ks = ks0; ks < ks1; ++ks) {
          if (!warp_wait(empty_bar(slot), phase ^ 1u, sync, p.timeout_ns)) {
            ok = false;
            break;
          }
          if (gi == 0 && !quant_seen) {
            bool seen = true;
            if (lane == 0) seen = wait_counter(p.sync + kSyncQuant, (uint32_t)T, p.sync, sync, p.timeout_ns);
            seen = __shfl_sync(0xffffffffu, seen, 0);
            __syncwarp();
            if (!seen) {
              ok = false;
              break;
            }
            fence_proxy_async_global();
            quant_seen = true;
          }
          if (gi == 1 && ready_a != a) {
            const uint32_t need = (uint32_t)(phs[0].NT * 2 * quads_of(a));
            bool ready = true;
            if (lane == 0) ready = wait_counter(p.sync + kSyncReady + a, need, p.sync, sync, p.timeout_ns);
            ready = __shfl_sync(0xffffffffu, ready, 0);
            __syncwarp();
            if (!ready) {
              ok = false;
              break;
            }
            fence_proxy_async_global();
            ready_a = a;
          }
          const int katoms = min(KPS, K - ks * KPS) / 128;
          const uint32_t st = sbase + (uint32_t)slot * kStageBytes;
          if (elect_one()) {
            mbar_arrive_expect_tx(full_bar(slot), (uint32_t)(G::kABytes + katoms * 512));
            tma_load_2d(st, gi == 0 ? &p.tmap_x : &p.tmap_a2, full_bar(slot), ks * 128, (int)row0);
            bulk_load(st + kSfaOff,
                      (gi == 0 ? p.xs : p.a2s) + ((row0 / 128) * (K / 128) + (int64_t)ks * kAtomsPerStage) * 512,
                      (uint32_t)katoms * 512u, full_bar(slot));
          }
          __syncwarp();
          armed[slot] = (int)phase;
          if (++slot == kStages) {
            slot = 0;
            phase ^= 1u;
          }
        }
      })
      for (int s = 0; s < kStages; ++s)
        if (armed[s] >= 0) warp_wait(full_bar(s), (uint32_t)armed[s], sync, 100000000ull, true);
    }
    __syncwarp();
  } else if (warp == kDWeightWarp) {
    // ------------------------------------------------------------ weight producer
    // The last ring slot holds the prologue's scratch until the scatter and the quantiser are
    // done with it: the first pass over the ring waits there for their flag.
    int slot = 0;
    uint32_t phase = 0;
    int armed[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s) armed[s] = -1;
    bool ok = !p.test_stall;
    bool scratch_free = false;
    MOE_FOR_EACH_SEGMENT({
      if (!ok) break;
      const int e = act_e[a];
      const int N = P.N, K = P.K;
      const int n0 = nt * kNTile;
      const int n_rows = min(kNTile, N - n0);
      const uint8_t* wsf = gi == 0 ? p.w1_sf : p.w2_sf;
      const CUtensorMap* tmap = gi == 0 ? &p.tmap_w1 : &p.tmap_w2;
      const uint8_t* lane_sf = wsf + ((int64_t)e * N + n0 + lane) * (K / 32);
      const int64_t sf_row32 = (int64_t)32 * (K / 32);
      for (int ks = ks0; ks < ks1; ++ks) {
        if (!warp_wait(empty_bar(slot), phase ^ 1u, sync, p.timeout_ns)) {
          ok = false;
          break;
        }
        if (slot == kStages - 1 && !scratch_free) {
          if (!warp_wait_flag(reinterpret_cast<volatile int*>(tmem_holder + 3), sync, p.timeout_ns)) {
            ok = false;
            break;
          }
          scratch_free = true;
        }
        const int katoms = min(KPS, K - ks * KPS) / 128;
        const uint32_t st = sbase + (uint32_t)slot * kStageBytes;
        if (elect_one()) {
          if (p.w_sf_tiled) {
            const int halves = n_rows > 128 ? 2 : 1;
            mbar_arrive_expect_tx(full_bar(slot), (uint32_t)(TR::kBTxBytes + halves * katoms * 512));
            tma_load_3d(st + G::kBOff, tmap, full_bar(slot), ks * 128, n0, e);
            for (int na = 0; na < halves; ++na)
              bulk_load(st + kSfbOff + na * (kAtomsPerStage * 512),
                        wsf + ((((int64_t)e * N + n0) / 128 + na) * (K / 128) + (int64_t)ks * kAtomsPerStage) * 512,
                        (uint32_t)katoms * 512u, full_bar(slot));
          } else {
            mbar_arrive_expect_tx(full_bar(slot), (uint32_t)TR::kBTxBytes);
            tma_load_3d(st + G::kBOff, tmap, full_bar(slot), ks * 128, n0, e);
          }
        }
        if (!p.w_sf_tiled) {
          // weight scales from the canonical layout: rows lane + 32*jj of each k-atom, 4 bytes
          // each, into the 128x4 tile layout
          const uint8_t* src_k = lane_sf + ks * (KPS / 32);
          const uint32_t dst_k = st + kSfbOff + (uint32_t)lane * 16u;
#pragma unroll
          for (int j = 0; j < 8 * kAtomsPerStage; ++j) {
            const int jj = j & 7, ka = j >> 3;
            if (ka < katoms && jj * 32 + lane < n_rows)
              cp_async_4(dst_k + (jj >> 2) * (kAtomsPerStage * 512) + ka * 512 + (jj & 3) * 4,
                         src_k + jj * sf_row32 + ka * 4);
          }
          cp_async_arrive_noinc(full_bar(slot));
        }
        armed[slot] = (int)phase;
        if (++slot == kStages) {
          slot = 0;
          phase ^= 1u;
        }
      }
    })
    cp_async_wait_all();
    for (int s = 0; s < kStages; ++s)
      if (armed[s] >= 0) warp_wait(full_bar(s), (uint32_t)armed[s], sync, 100000000ull, true);
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer: the warp runs the
    // loop converged, one elected lane issues each tcgen05 instruction (from one divergent
    // lane the loop itself outlasted the stage's MMAs)
    {
      int slot = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true, issued = false;
      const uint64_t a_desc0 = smem_desc(sbase, 16, 1024, kLayoutSwizzle128B);
      const uint64_t b_desc0 = smem_desc(sbase + G::kBOff, 16, 1024, kLayoutSwizzle128B);
      const uint64_t sfa_desc0 = smem_desc(sbase + kSfaOff, 128, 128, kLayoutNone);
      const uint64_t sfb_desc0 = smem_desc(sbase + kSfbOff, 128, 128, kLayoutNone);
      constexpr uint64_t kSlotStep = kStageBytes >> 4;
      constexpr uint32_t kHalfStep = (kAtomsPerStage * 512) >> 4;
      const bool gathered = !p.w_sf_tiled;
      MOE_FOR_EACH_SEGMENT({
        if (!ok) break;
        if (!warp_wait(tmem_empty_bar, acc_phase ^ 1u, sync, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int K = P.K;
        for (int ks = ks0; ks < ks1; ++ks) {
          if (!warp_wait(full_bar(slot), phase, sync, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (gathered) fence_proxy_async_smem();
          const uint64_t so = (uint64_t)slot * kSlotStep;
          const uint32_t sf_col = tmem_base + kDSfCol0 + (uint32_t)slot * kDSfSlotCols;
          const int kvalid = min(KPS, K - ks * KPS);
          const int katoms = kvalid == KPS ? kAtomsPerStage : kvalid / 128;
          const int nmma = kvalid == KPS ? kMmaPerStage : kvalid / TR::kMmaK;
          if (elect_one()) {
#pragma unroll
            for (int ka = 0; ka < kAtomsPerStage; ++ka) {
              if (ka < katoms) {
                tc_cp_32x128b_warpx4(sf_col + ka * 4, sfa_desc0 + so + ka * 32);
                tc_cp_32x128b_warpx4(sf_col + kSfaCols + ka * 8, sfb_desc0 + so + ka * 32);
                tc_cp_32x128b_warpx4(sf_col + kSfaCols + ka * 8 + 4, sfb_desc0 + so + kHalfStep + ka * 32);
              }
            }
#pragma unroll
            for (int j = 0; j < kMmaPerStage; ++j) {
              if (j < nmma) {
                const int kblk = j * (TR::kMmaK / 32);
                const uint32_t idesc = make_idesc<ACT>((uint32_t)(kblk & 3), kRowTile);
                const uint32_t acc = (ks > ks0 || j > 0) ? 1u : 0u;
                if (ACT == 0)
                  tc_mma_mxf8f6f4(tmem_base, a_desc0 + so + 2 * j, b_desc0 + so + 2 * j, idesc,
                                  sf_col + (kblk >> 2) * 4, sf_col + kSfaCols + (kblk >> 2) * 8, acc);
                else
                  tc_mma_mxf4(tmem_base, a_desc0 + so + 2 * j, b_desc0 + so + 2 * j, idesc, sf_col + (kblk >> 2) * 4,
                              sf_col + kSfaCols + (kblk >> 2) * 8, acc);
              }
            }
            tc_commit(empty_bar(slot));
          }
          __syncwarp();
          issued = true;
          if (++slot == kStages) {
            slot = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one()) tc_commit(tmem_full_bar);
        __syncwarp();
        acc_phase ^= 1u;
      })
      if (issued) {
        if (elect_one()) tc_commit(drain_bar);
        __syncwarp();
        warp_wait(drain_bar, 0, sync, 100000000ull, true);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ warps 2..9
    const int et = threadIdx.x - 64;  // 0..255
    scatter_pairs(32 + et);
    named_barrier(1, 32 + 32 * kDEpiWarps);  // the pair scatter is done
    // token b's quantised row (staged at the start) into its k padded expert rows
    if (b < T && routed) {
      for (int c = et; c < row_bytes / 16; c += 32 * kDEpiWarps) {
        const uint4 v = *reinterpret_cast<const uint4*>(stage_codes + c * 16);
        for (int j = 0; j < k; ++j)
          *reinterpret_cast<uint4*>(p.xq + (int64_t)pair_invp[b * k + j] * row_bytes + c * 16) = v;
      }
      for (int kb = et; kb < H / 32; kb += 32 * kDEpiWarps) {
        const uint8_t v = stage_sf[kb];
        for (int j = 0; j < k; ++j) p.xs[sf_tile_offset(pair_invp[b * k + j], kb, H)] = v;
      }
    }
    // the warps' copies are ordered before the signal by the barrier and one gpu-scope fence of
    // the signalling thread (the usual last-arriver pattern)
    named_barrier(2, 32 * kDEpiWarps);
    if (et == 0) {
      if (b < T && routed) {
        __threadfence();
        fence_proxy_async_global();  // the codes are read by other CTAs' TMA loads
        atomicAdd(p.sync + kSyncQuant, 1u);
      }
      *reinterpret_cast<volatile int*>(tmem_holder + 3) = 1;  // prologue scratch free
    }

    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int ew = warp - 2;  // this warp's part of a tile: (quadrant, column half)
    const int row_local = quad * 32 + lane;
    uint32_t acc_phase = 0;
    bool ok = true;
    MOE_FOR_EACH_SEGMENT({
      if (!ok) break;
      const int cnt = act_cnt[a];
      const bool live = quad * 32 < cnt && nt * kNTile + half * 128 < P.N;
      const bool valid = live && row_local < cnt;
      if (!warp_wait(tmem_full_bar, acc_phase, sync, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (!live) {
        __syncwarp();
        if (lane == 0) mbar_arrive(tmem_empty_bar);
        acc_phase ^= 1u;
        z += ks1 - ks0 + zstep;
        continue;
      }
      float acc[128];
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(half * 128);
#pragma unroll
      for (int c = 0; c < 4; ++c) tc_ld_32x32b_x32(taddr + c * 32, acc + 32 * c);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_empty_bar);
      acc_phase ^= 1u;

      const int iz0 = item * P.nks;
      const int c_first = P.whole ? b : owner_of(P, iz0);
      const int c_last = P.whole ? b : owner_of(P, iz0 + P.nks - 1);
      const int64_t prow = (int64_t)kRowTile * act_mtb[a] + row_local;        // padded row (A2)
      float* y2_row = p.y2f + (int64_t)(act_off[a] + row_local) * H + nt * kNTile + half * 128;
      if (c_first == c_last) {
        // the whole item ran here
        if (gi == 0) {
          store_acc_rows<ACT, 0>(acc, valid, prow, nt, half, P.N, p.a2, p.a2s, nullptr);
        } else if (valid) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            __stcg(reinterpret_cast<float4*>(y2_row) + i,
                   make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]));
        }
      } else {
        // item cut between CTAs: leave the partial accumulator, take a ticket; the last
        // contributor sums every contributor's partial in CTA order (reading its own back
        // too, so the order does not depend on who came last) and finishes the part
        const int my_slot = range_begin(P, b) / P.nks == item ? 0 : 1;
        float* mine = p.part + ((((int64_t)b * 2 + gi) * 2 + my_slot) * AROWS + row_local) * kNTile + half * 128;
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            __stcg(reinterpret_cast<float4*>(mine) + i,
                   make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]));
        }
        __threadfence();
        __syncwarp();
        uint32_t ticket = 0;
        if (lane == 0) ticket = atomicAdd(p.sync + kSyncTicket + (gi * kDecodeMaxCtas + c_first) * 8 + ew, 1u);
        ticket = __shfl_sync(0xffffffffu, ticket, 0);
        if (ticket != (uint32_t)(c_last - c_first)) {
          z += ks1 - ks0 + zstep;
          continue;  // another contributor finishes this part
        }
        __threadfence();
        // Row by row over the warp's routed rows, the lanes splitting the 128 columns (lane l:
        // columns 4l..4l+3), four contributors' partials loaded before any is added.
        const int nrows = min(cnt - quad * 32, 32);
        const int cols = half * 128 + lane * 4;
        // every contributor after the first starts its range inside this item (slot 0); the
        // first one's slot depends on where its range starts
        const int cs_first = range_begin(P, c_first) / P.nks == item ? 0 : 1;
        for (int r = 0; r < nrows; ++r) {
          const int row = quad * 32 + r;
          float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          for (int c0 = c_first; c0 <= c_last; c0 += 4) {
            float4 f[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int c = c0 + u;
              if (c <= c_last) {
                const int slot_idx = (c * 2 + gi) * 2 + (c == c_first ? cs_first : 0);
                f[u] = __ldcg(reinterpret_cast<const float4*>(p.part + (size_t)slot_idx * (AROWS * kNTile)) +
                              (row * kNTile + cols) / 4);
              }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (c0 + u <= c_last) {
                if (c0 + u == c_first) {
                  sum = f[u];
                } else {
                  sum.x += f[u].x;
                  sum.y += f[u].y;
                  sum.z += f[u].z;
                  sum.w += f[u].w;
                }
              }
            }
          }
          if (gi == 0) {
            // SwiGLU on the two interleaved (gate, up) pairs of this lane; lanes 16*blk .. +15
            // hold one 32-wide block of h
            const float h[2] = {silu_mul(sum.x, sum.y), silu_mul(sum.z, sum.w)};
            float amax = fmaxf(fabsf(h[0]), fabsf(h[1]));
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const MxScale sc = mx_scale<ACT>(amax);
            const int kb = nt * 4 + half * 2 + lane / 16;
            const int64_t prow_r = (int64_t)kRowTile * act_mtb[a] + row;
            if (ACT == 0) {
              const __nv_fp8x2_storage_t c2 = __nv_cvt_float2_to_fp8x2(
                  make_float2(h[0] * sc.mult, h[1] * sc.mult), __NV_SATFINITE, __NV_E4M3);
              *reinterpret_cast<uint16_t*>(p.a2 + prow_r * I + kb * 32 + (lane % 16) * 2) = (uint16_t)c2;
            } else {
              const __nv_fp4x2_storage_t c2 = __nv_cvt_float2_to_fp4x2(
                  make_float2(h[0] * sc.mult, h[1] * sc.mult), __NV_E2M1, cudaRoundNearest);
              p.a2[prow_r * (I / 2) + kb * 16 + (lane % 16)] = (uint8_t)c2;
            }
            if (lane % 16 == 0) p.a2s[sf_tile_offset(prow_r, kb, I)] = sc.byte;
          } else {
            __stcg(reinterpret_cast<float4*>(p.y2f + (int64_t)(act_off[a] + row) * H + nt * kNTile + cols), sum);
          }
        }
      }
      // the part is final: count it (GEMM1: towards its expert's A2; GEMM2: towards the combine)
      __threadfence();
      if (gi == 0) fence_proxy_async_global();  // A2 is read by other CTAs' TMA loads
      __syncwarp();
      if (lane == 0) atomicAdd(p.sync + (gi == 0 ? kSyncReady + a : kSyncDone2), 1u);
    })
    // ------------------------------------------------------------ combine (every CTA)
    // out[t, n] = bf16(sum_j w[t, j] * y2[row(t, j), n]) in slot order with fp32 accumulation,
    // once every GEMM2 part is final; warp w of CTA b takes (token, 128-column block) units
    // b * 8 + w, + 8 * gridDim.x, ...; lane l owns 4 columns.
    if (ok && routed) {
      uint32_t parts = 0;
      for (int i = lane; i < n_act; i += 32) parts += (uint32_t)quads_of(i);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) parts += __shfl_xor_sync(0xffffffffu, parts, o);
      const uint32_t halves = (uint32_t)(2 * phs[1].NT - ((H % kNTile) != 0 ? 1 : 0));
      bool ready = true;
      if (lane == 0) ready = wait_counter(p.sync + kSyncDone2, halves * parts, p.sync, sync, p.timeout_ns);
      ready = __shfl_sync(0xffffffffu, ready, 0);
      if (ready) {
        __threadfence();
        const int cblocks = H / 128;
        const int units = T * cblocks;
        for (int u = b * kDEpiWarps + ew; u < units; u += (int)gridDim.x * kDEpiWarps) {
          const int t = u / cblocks;
          const int c = (u % cblocks) * 128 + lane * 4;
          float4 y[kMaxTopK];
#pragma unroll
          for (int j = 0; j < kMaxTopK; ++j)
            if (j < k) y[j] = __ldcg(reinterpret_cast<const float4*>(p.y2f + (int64_t)pair_inv[t * k + j] * H + c));
          float o0 = 0.0f, o1 = 0.0f, o2 = 0.0f, o3 = 0.0f;
#pragma unroll
          for (int j = 0; j < kMaxTopK; ++j) {
            if (j < k) {
              const float w = pair_w[t * k + j];
              o0 = fmaf(w, y[j].x, o0);
              o1 = fmaf(w, y[j].y, o1);
              o2 = fmaf(w, y[j].z, o2);
              o3 = fmaf(w, y[j].w, o3);
            }
          }
          const __nv_bfloat162 lo = __floats2bfloat162_rn(o0, o1), hi = __floats2bfloat162_rn(o2, o3);
          *reinterpret_cast<uint2*>(p.out + (int64_t)t * H + c) =
              make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
        }
      }
    }
  }
#undef MOE_FOR_EACH_SEGMENT

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kDTmemCols);
}

template <int ACT, int AROWS>
cudaError_t launch_decode_typed(const DecodeArgs& a, cudaStream_t s) {
  using G = DGeo<ACT, AROWS>;
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    err = cudaFuncSetAttribute(moe_decode_kernel<ACT, AROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               G::kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_set[dev].store(true, std::memory_order_release);
  }
  DecodeParams p;
  memset(&p, 0, sizeof(p));
  if (!encode_act_map(&p.tmap_x, a.xq, a.rows_cap, a.H, ACT, AROWS) ||
      !encode_weight_map(&p.tmap_w1, a.w1, a.E, 2 * a.I, a.H, ACT) ||
      !encode_act_map(&p.tmap_a2, a.a2, a.rows_cap, a.I, ACT, AROWS) ||
      !encode_weight_map(&p.tmap_w2, a.w2, a.E, a.H, a.I, ACT))
    return cudaErrorInvalidValue;
  p.x = a.x;
  p.xq_in = a.xq_in;
  p.xs_in = a.xs_in;
  p.logits = a.logits;
  p.w1_sf = a.w1_sf;
  p.w2_sf = a.w2_sf;
  p.xq = a.xq;
  p.xs = a.xs;
  p.a2 = a.a2;
  p.a2s = a.a2s;
  p.part = a.part;
  p.y2f = a.y2f;
  p.out = a.out;
  p.ids = a.ids;
  p.tw = a.tw;
  p.counts = a.counts;
  p.offsets = a.offsets;
  p.padded_offsets = a.padded_offsets;
  p.mtile_base = a.mtile_base;
  p.sorted_pair = a.sorted_pair;
  p.inv = a.inv;
  p.inv_padded = a.inv_padded;
  p.sync = a.sync;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  p.T = (int)a.T;
  p.H = a.H;
  p.I = a.I;
  p.E = a.E;
  p.k = a.k;
  p.w_sf_tiled = a.w_sf_tiled;
  p.test_stall = a.test_stall;
  const int grid = std::min(a.num_sms, kDecodeMaxCtas);
  // All CTAs must be resident together (later stages wait for other CTAs' results): one CTA per
  // SM (its shared memory allows no second), grid <= SMs, launched as a cooperative grid.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kDThreads);
  cfg.dynamicSmemBytes = G::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_decode_kernel<ACT, AROWS>, p);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (a.T > kDecodeMaxTokens) return cudaErrorInvalidValue;
  if (decode_arows(a.T) == 16)
    return a.act_fmt == 0 ? launch_decode_typed<0, 16>(a, s) : launch_decode_typed<1, 16>(a, s);
  return a.act_fmt == 0 ? launch_decode_typed<0, 64>(a, s) : launch_decode_typed<1, 64>(a, s);
}

}  // namespace moe
