// gemm_pair.cu -- the grouped block-scaled GEMMs of the expert layer on CTA pairs (A8W4, weight
// scales in the 128x4 tile layout): the pair kernel over the experts' whole pairs of M tiles, and
// the wide tail pass over their odd last M tiles (further below).
//
// Same contract as gemm.cu (GEMM1: SwiGLU + MX requant epilogue over the gate/up-interleaved
// W1 rows, "feat(moe): FlyDSL MegaMoE fused EP-MoE integration", description: INTERLEAVE(g1u1);
// GEMM2: bf16 rows).  An expert with m M tiles has m / 2 (rounded down) pair tiles in the pair
// kernel; its odd last M tile, if any, is left to the wide tail pass or to gemm.cu's tail pass
// (GemmArgs::tail_only), which runs right after the pair kernel on the same stream.
//
// A pair tile is 256 routed rows -- two consecutive 128-row M tiles of one expert -- by 256
// output columns, computed by a cluster of two CTAs on two SMs with tcgen05.mma.cta_group::2
// (M = 256):
//   * each CTA loads its own 128 activation rows and 128 of the 256 weight rows of the tile,
//     through two rings: 5 stages of activation rows and 8 of weight rows (16 KiB of shared
//     memory each), against the single kernel's 4 stages of 50 KiB holding both;
//   * each CTA stages the scales of all 256 weight rows of the tile (the MMA of each SM reads
//     the weight scales of every output column from its own TMEM);
//   * one elected lane of the even CTA's converged MMA warp issues the scale copies to TMEM and
//     the MMAs for both, once a stage's slots of both rings are full; each CTA's TMEM receives
//     the accumulator of its own 128 rows;
//   * every TMA load of either CTA completes on the even CTA's "full" barrier of its ring, whose
//     expected byte count the even CTA's producer posts for both CTAs (local arrivals only: a
//     remote arrive with release semantics stalls the issuing thread on a cluster-wide fence);
//     the MMA commits release the stage's slots in both CTAs (multicast), and the accumulator
//     hand-off goes to both epilogues, whose "TMEM free" arrivals go back to the even CTA.
// Measured (V4-Pro A8W4, T = 8192): a pair stage costs ~0.32 us per SM against ~0.42 for the
// single kernel's; the pairs plus the single-CTA tail pass ran GEMM1 in 1.94 ms against 2.13 ms
// for single-CTA tiles throughout, and with the wide tail pass in ~1.86 ms.
// Warp roles per CTA: 0 activation-side TMA, 10 weight-side TMA (both converged, copies issued
// by an elected lane), 1 TMEM (+ MMA issue in the even CTA), 2..9 epilogue (as in gemm.cu).
// Every wait is bounded; on expiry the CTA records MOE_ERR_DEVICE_TIMEOUT, lets its copies and
// MMAs drain, and both CTAs meet at the final cluster barrier before the pair's TMEM is freed.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "gemm_common.cuh"
#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

// Two rings: activation tiles (with their scale atom) and weight tiles (with theirs), each with
// its own full / empty barriers, so the weight ring can be deeper than the activation ring:
// the weight stream, which nothing else reads, is bound by its bytes in flight per SM (~2 us of
// loaded latency), and a CTA's activation tile (16 KiB a stage, mostly L2 hits: the expert's
// other N tiles read it too) would otherwise take as many slots.
constexpr int kPStagesA = 5;                       // activation ring
constexpr int kPThreads = 352;
constexpr int kPEpiWarps = 8;
constexpr int kPBWarp = 10;
constexpr int kPHalfRows = 128;                    // weight rows per CTA (half of kNTile)
constexpr int kPABytes = kRowTile * 128;           // 128 activation rows x 128 bytes
constexpr int kPBBytes = kPHalfRows * 128;         // 128 weight rows x 128 bytes (smem footprint)
constexpr int kPOutStageBytes = 32 * 32 * 2;       // GEMM2 epilogue staging: 32 rows x 32 bf16 per warp
constexpr uint32_t kPTmemCols = 512;
constexpr uint32_t kPSfCol0 = 256;                 // accumulator: columns [0, 256)
constexpr uint32_t kPSfSlotCols = 12;              // 4 A-scale + 8 weight-scale columns
// TMEM scale slots follow the activation ring: the copy for stage i + kPStagesA is issued only
// after the activation slot of stage i was released, i.e. after stage i's MMAs completed.
static_assert(kPSfCol0 + kPStagesA * kPSfSlotCols <= kPTmemCols, "pair GEMM TMEM scale slots");

// Shared memory: the activation ring, the weight ring (8 x 8 KiB of weights in flight; 7 for
// GEMM2, whose rows leave through a per-warp staging buffer as TMA stores -- direct 16-byte stores
// from every lane cost GEMM2's pairs ~5 % in competition with the weight stream), the scale
// atoms of both rings, the staging buffers, the barriers and the pair-tile prefix.
template <int EPI>
struct PairGeo {
  static constexpr bool kOutStaging = EPI == 1 || EPI == 3;  // GEMM2 rows: bf16, or FP8 transport codes
  static constexpr int kStagesW = kOutStaging ? 7 : 8;
  static constexpr int kWOff = kPStagesA * kPABytes;              // the weight ring after the activation ring
  static constexpr int kSfaOff = kWOff + kStagesW * kPBBytes;     // activation-scale atoms, 512 B a slot
  static constexpr int kSfbOff = kSfaOff + kPStagesA * 512;       // weight-scale atoms, 2 x 512 B a slot
  static constexpr int kOutOff = (kSfbOff + kStagesW * 1024 + 1023) / 1024 * 1024;
  static constexpr int kOutBytes = kOutStaging ? kPEpiWarps * kPOutStageBytes : 0;
  static constexpr int kBarOff = kOutStaging ? kOutOff + kOutBytes : kSfbOff + kStagesW * 1024;
  static constexpr int kBaseOff = kBarOff + 256;                  // pair-tile prefix over experts, int32 [E+1]
  static constexpr int kSmemBytes = kBaseOff + 4 * (kMaxExperts + 1) + 1024;
  static_assert(kSmemBytes <= 232448, "pair GEMM shared memory");
  static_assert(kWOff % 1024 == 0 && kSfaOff % 1024 == 0, "pair GEMM ring alignment");
  static_assert(8 * (2 * kPStagesA + 2 * kStagesW + 3) + 8 <= 256, "pair GEMM barriers");
};

struct PairParams {  // 64-byte aligned through its CUtensorMap members
  CUtensorMap tmap_act;  // activation codes [rows_cap, K or K/2], box 128 B x 128 rows
  CUtensorMap tmap_w;    // weights [E, N, K/2], box 128 K x 128 rows x 1
  CUtensorMap tmap_asf;  // activation scales as rows of 256 bytes, box 256 x (2 * atoms per stage)
  CUtensorMap tmap_wsf;  // prepacked weight scales as rows of 256 bytes, same box
  CUtensorMap tmap_out;  // GEMM2: y2 bf16 [rows_cap, N], box 32 columns x 32 rows, 64-byte swizzle
  const int32_t* counts;
  const int32_t* mtile_base;  // expert e's rows start at row 128 * mtile_base[e]
  const uint8_t* act_sf;      // activation scales, 128x4 tile layout
  uint8_t* act_sf_rot;        // or null: the tail pass's rotated A-scale atoms (written here)
  uint8_t* out_codes;
  uint8_t* out_sf;
  uint16_t* out_bf16;
  const float* row_w;         // epilogue 3: routing weight of each padded row
  uint32_t* status;
  uint64_t timeout_ns;
  int E, N, K;
  int test_stall;
};

struct PairTile {
  int e, pm, nt;
};

// Pair tiles of expert e occupy [base[e]*NT, base[e+1]*NT), pair index fastest.
__device__ __forceinline__ PairTile decode_pair_tile(int64_t tile, const int32_t* base, int E, int NT) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)base[mid] * NT <= tile) lo = mid;
    else hi = mid - 1;
  }
  const int pe = base[lo + 1] - base[lo];
  const int64_t local = tile - (int64_t)base[lo] * NT;
  PairTile t;
  t.e = lo;
  t.nt = (int)(local / pe);
  t.pm = (int)(local % pe);
  return t;
}

// Spin for about `cycles` SM clock cycles (used on the abort path only, to let copies that
// were issued but can no longer be waited for land before the CTA leaves).
__device__ __noinline__ void grace_spin(uint64_t cycles) {
  const uint64_t t0 = clock64();
  while (clock64() - t0 < cycles) {
  }
}

template <int ACT, int EPI>
__global__ void __launch_bounds__(kPThreads, 1) moe_gemm_pair_kernel(const __grid_constant__ PairParams p) {
  static_assert(ACT == 0, "the pair kernel serves A8W4 (E4M3 x E2M1)");
  using TR = ActTraits<ACT>;
  using G = PairGeo<EPI>;
  constexpr int kPStagesW = G::kStagesW;
  constexpr int kPWOff = G::kWOff, kPSfaOff = G::kSfaOff, kPSfbOff = G::kSfbOff, kPBarOff = G::kBarOff,
                kPBaseOff = G::kBaseOff;
  constexpr int kMmaPerStage = TR::kKPerStage / TR::kMmaK;  // 4
  constexpr uint32_t kSfaCols = 4;
  constexpr uint32_t kScaleBoxBytes = 512;                  // one k-atom a stage
  constexpr uint32_t kBHalfTx = TR::kBTxBytes / 2;          // global bytes of 128 weight rows

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kPBarOff;
  auto full_a = [&](int s) { return bar0 + 8u * s; };
  auto empty_a = [&](int s) { return bar0 + 8u * (kPStagesA + s); };
  auto full_w = [&](int s) { return bar0 + 8u * (2 * kPStagesA + s); };
  auto empty_w = [&](int s) { return bar0 + 8u * (2 * kPStagesA + kPStagesW + s); };
  const uint32_t tmem_full_bar = bar0 + 8u * (2 * kPStagesA + 2 * kPStagesW);
  const uint32_t tmem_empty_bar = tmem_full_bar + 8;
  const uint32_t drain_bar = tmem_full_bar + 16;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kPBarOff + 8 * (2 * kPStagesA + 2 * kPStagesW + 3));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int32_t* pair_base = reinterpret_cast<int32_t*>(smem + kPBaseOff);
  const int32_t* tile_base = p.mtile_base;  // M-tile prefix (read once per tile)

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int E = p.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStagesA; ++s) {
      mbar_init(full_a(s), 1);      // expect_tx arrival of warp 0 of the even CTA
      mbar_init(empty_a(s), 1);     // the pair's MMA commit
    }
    for (int s = 0; s < kPStagesW; ++s) {
      mbar_init(full_w(s), 1);      // expect_tx arrival of warp 10 of the even CTA
      mbar_init(empty_w(s), 1);
    }
    mbar_init(tmem_full_bar, 1);
    mbar_init(tmem_empty_bar, 2 * kPEpiWarps);  // epilogue warps of both CTAs
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Pair tiles per expert (whole pairs of M tiles), prefixed by warp 2 into shared memory.
  if (warp == 2) {
    int running = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? (p.mtile_base[e + 1] - p.mtile_base[e]) >> 1 : 0;  // whole pairs only
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < E) pair_base[e] = running + incl - v;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pair_base[E] = running;
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_holder), kPTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers initialised in both CTAs before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const Sync sync{abort_flag, p.status, p.timeout_ns, bar0};
  const int NT = p.N / kNTile;
  const int K = p.K;
  const int nks = (K + TR::kKPerStage - 1) / TR::kKPerStage;
  const int64_t total_tiles = (int64_t)pair_base[E] * NT;
  const int64_t first_tile = cluster_index();
  const int64_t tile_step = cluster_count();
  if (warp == 0 || warp == kPBWarp) {
    // ------------------------------------------------------------------ producers (converged)
    const bool act_warp = warp == 0;
    const int depth = act_warp ? kPStagesA : kPStagesW;
    // the even CTA's barriers of this producer's ring
    const uint32_t lfull0 = mapa_shared(act_warp ? full_a(0) : full_w(0), 0);
    {
      int slot = 0;
      uint32_t phase = 0;
      bool ok = !p.test_stall;  // the test hook leaves every stage unfilled
      for (int64_t tile = first_tile; ok && tile < total_tiles; tile += tile_step) {
        const PairTile pt = decode_pair_tile(tile, pair_base, E, NT);
        const int mt = 2 * pt.pm + (int)rank;
        const int mt_e = tile_base[pt.e + 1] - tile_base[pt.e];
        const bool real = mt < mt_e;
        const bool peer_real = 2 * pt.pm + 1 < mt_e;  // the odd CTA has rows in this tile
        const int64_t row0 = ((int64_t)tile_base[pt.e] + mt) * kRowTile;
        const int n0 = pt.nt * kNTile;
        const int asf_y0 = (int)(2 * ((row0 / 128) * (K / 128)));             // scale rows of 256 B
        const int wsf_y0 = (int)(2 * ((((int64_t)pt.e * p.N + n0) / 128) * (K / 128)));
        const int wsf_half = 2 * (K / 128);                                     // next 128 weight rows
        // bytes both CTAs land on the even CTA's barrier per stage, posted by the even CTA (a
        // load of the odd CTA may complete before the post, which the barrier's signed
        // transaction count allows: the phase cannot complete before both posts arrived)
        const uint32_t act_tx = ((uint32_t)kPABytes + kScaleBoxBytes) * (peer_real ? 2u : 1u);
        const uint32_t w_tx = 2u * (kBHalfTx + 2u * kScaleBoxBytes);
        for (int ks = 0; ks < nks; ++ks) {
          if (!warp_wait(act_warp ? empty_a(slot) : empty_w(slot), phase ^ 1u, sync, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t lfull = lfull0 + 8u * slot;
          const int ky = 2 * ks;
          if (elect_one()) {
            if (act_warp) {
              if (leader) mbar_arrive_expect_tx(full_a(slot), act_tx);
              if (real) {
                tma_load_2d_pair(sbase + (uint32_t)slot * kPABytes, &p.tmap_act, lfull, ks * 128, (int)row0);
                tma_load_2d_pair(sbase + kPSfaOff + (uint32_t)slot * 512u, &p.tmap_asf, lfull, 0, asf_y0 + ky);
              }
            } else {
              if (leader) mbar_arrive_expect_tx(full_w(slot), w_tx);
              const uint32_t sfb = sbase + kPSfbOff + (uint32_t)slot * 1024u;
              tma_load_3d_pair(sbase + kPWOff + (uint32_t)slot * kPBBytes, &p.tmap_w, lfull, ks * 128,
                               n0 + (int)rank * kPHalfRows, pt.e);
              tma_load_2d_pair(sfb, &p.tmap_wsf, lfull, 0, wsf_y0 + ky);
              tma_load_2d_pair(sfb + kScaleBoxBytes, &p.tmap_wsf, lfull, 0, wsf_y0 + wsf_half + ky);
            }
          }
          __syncwarp();
          if (++slot == depth) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (even CTA)
    // The warp runs the loop converged and one elected lane issues each tcgen05.cp / mma /
    // commit (see gemm.cu), with every descriptor and TMEM address precomputed.
    if (leader) {
      int sa = 0, sw = 0;             // activation and weight ring slots
      uint32_t pa = 0, pw = 0, acc_phase = 0;
      bool ok = true, issued = false;
      // descriptors of slot 0 of each ring; a slot adds its bytes, an MMA step 32 bytes (start
      // address field, in 16-byte units; shared-memory offsets stay below 2^18, so no carry)
      const uint64_t a_desc0 = smem_desc(sbase, 16, 1024, kLayoutSwizzle128B);
      const uint64_t b_desc0 = smem_desc(sbase + kPWOff, 16, 1024, kLayoutSwizzle128B);
      const uint64_t sfa_desc0 = smem_desc(sbase + kPSfaOff, 128, 128, kLayoutNone);
      const uint64_t sfb_desc0 = smem_desc(sbase + kPSfbOff, 128, 128, kLayoutNone);
      constexpr uint64_t kAStep = kPABytes >> 4, kBStep = kPBBytes >> 4;
      constexpr uint32_t kSfbCols = 8;  // TMEM columns of the 256 weight rows' scales
      for (int64_t tile = first_tile; ok && tile < total_tiles; tile += tile_step) {
        if (!warp_wait(tmem_empty_bar, acc_phase ^ 1u, sync, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < nks; ++ks) {
          if (!warp_wait(full_a(sa), pa, sync, p.timeout_ns) || !warp_wait(full_w(sw), pw, sync, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ao = (uint64_t)sa * kAStep, bo = (uint64_t)sw * kBStep;
          const uint32_t sf_col = tmem_base + kPSfCol0 + (uint32_t)sa * kPSfSlotCols;
          if (elect_one()) {
            tc_cp_pair_32x128b_warpx4(sf_col, sfa_desc0 + (uint64_t)sa * 32);
            tc_cp_pair_32x128b_warpx4(sf_col + kSfaCols, sfb_desc0 + (uint64_t)sw * 64);
            tc_cp_pair_32x128b_warpx4(sf_col + kSfaCols + 4, sfb_desc0 + (uint64_t)sw * 64 + (kScaleBoxBytes >> 4));
#pragma unroll
            for (int j = 0; j < kMmaPerStage; ++j) {
              const uint32_t idesc = make_idesc<ACT>((uint32_t)j, 2 * kRowTile);
              tc_mma_pair_mxf8f6f4(tmem_base, a_desc0 + ao + 2 * j, b_desc0 + bo + 2 * j, idesc, sf_col,
                                   sf_col + kSfaCols, (ks > 0 || j > 0) ? 1u : 0u);
            }
            tc_commit_pair_mc(empty_a(sa), 0x3);
            tc_commit_pair_mc(empty_w(sw), 0x3);
          }
          __syncwarp();
          (void)kSfbCols;
          issued = true;
          if (++sa == kPStagesA) {
            sa = 0;
            pa ^= 1u;
          }
          if (++sw == kPStagesW) {
            sw = 0;
            pw ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one()) tc_commit_pair_mc(tmem_full_bar, 0x3);
        __syncwarp();
        acc_phase ^= 1u;
      }
      if (issued) {
        // no MMA or TMEM copy of the pair may still run when TMEM is freed
        if (elect_one()) tc_commit_pair(drain_bar);
        __syncwarp();
        warp_wait(drain_bar, 0, sync, 100000000ull, true);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    if (p.act_sf_rot != nullptr) {
      // For the wide tail pass that follows: the A-scale atoms of each expert's odd last M tile
      // with their 8-byte halves swapped in every 16-byte lane chunk (rows r and r ^ 64 of the
      // 128-row block change places), the view its odd CTAs stage.  The epilogue threads of all
      // CTAs write them while the first stages load, 16 bytes a thread and eight loads in
      // flight before the stores (the loop is latency-bound: with one batch per load it cost a
      // pair kernel without pair tiles ~20 us).
      constexpr int kBatch = 8;
      const int atoms = K / 128;
      const int chunks = E * atoms * 32;  // 16-byte chunks of the atoms of one block per expert
      const int nthr = (int)gridDim.x * 32 * kPEpiWarps;
      const int tid = ((int)blockIdx.x * kPEpiWarps + (warp - 2)) * 32 + lane;
      for (int c0 = tid; c0 < chunks; c0 += kBatch * nthr) {
        int64_t off[kBatch];
        uint4 v[kBatch];
        bool on[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int c = c0 + u * nthr;
          on[u] = false;
          off[u] = 0;
          if (c < chunks) {
            const int e = c / (atoms * 32);
            const int m1 = tile_base[e + 1];
            on[u] = ((m1 - tile_base[e]) & 1) != 0;
            off[u] = (int64_t)(m1 - 1) * atoms * 512 + (int64_t)(c - e * atoms * 32) * 16;
          }
          if (on[u]) v[u] = *reinterpret_cast<const uint4*>(p.act_sf + off[u]);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          if (on[u]) *reinterpret_cast<uint4*>(p.act_sf_rot + off[u]) = make_uint4(v[u].z, v[u].w, v[u].x, v[u].y);
      }
    }
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t leader_tmem_empty = mapa_shared(tmem_empty_bar, 0);
    uint32_t acc_phase = 0;
    for (int64_t tile = first_tile; tile < total_tiles; tile += tile_step) {
      const PairTile pt = decode_pair_tile(tile, pair_base, E, NT);
      const int mt = 2 * pt.pm + (int)rank;
      const int row_local = mt * kRowTile + quad * 32 + lane;
      const bool valid = row_local < p.counts[pt.e];  // false for every row of a missing M tile
      const int64_t prow = (int64_t)tile_base[pt.e] * kRowTile + row_local;
      if (!warp_wait(tmem_full_bar, acc_phase, sync, p.timeout_ns)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(half * 128);
      float acc[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc_ld_32x32b_x32(taddr + c * 32, acc + 32 * c);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(leader_tmem_empty);  // registers hold the tile
      acc_phase ^= 1u;
      if (EPI == 1 && G::kOutStaging && __all_sync(0xffffffffu, valid)) {
        // GEMM2 rows as bf16 (nearest even) through shared memory when all 32 rows of this warp
        // are routed rows: each 32-column chunk leaves as one TMA store (as in gemm.cu)
        const uint32_t buf = sbase + G::kOutOff + (uint32_t)(warp - 2) * kPOutStageBytes;
        const int x0 = pt.nt * kNTile + half * 128;
        const int y0 = (int)(prow - lane);
        const uint32_t swz = (uint32_t)((lane >> 1) & 3);  // 64-byte swizzle: 16-byte chunk ^= (row/2)%4
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (lane == 0) bulk_wait_read_all();  // the previous store has read the buffer
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const __nv_bfloat162 b = __floats2bfloat162_rn(acc[32 * c + 8 * i + 2 * q], acc[32 * c + 8 * i + 2 * q + 1]);
              w[q] = *reinterpret_cast<const uint32_t*>(&b);
            }
            st_shared_v4(buf + (uint32_t)lane * 64u + (((uint32_t)i ^ swz) << 4), w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();  // generic-proxy writes -> visible to the TMA engine
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&p.tmap_out, buf, x0 + 32 * c, y0);
            bulk_commit_group();
          }
        }
      } else if (EPI == 3 && G::kOutStaging && __all_sync(0xffffffffu, valid)) {
        // FP8 transport: the weighted row's four 32-column blocks as E4M3 codes, staged like the
        // bf16 rows (32 rows x 64 bytes a chunk, 64-byte swizzle, one TMA store), two chunks; the
        // four scale bytes of the row leave as one 4-byte store
        const uint32_t buf = sbase + G::kOutOff + (uint32_t)(warp - 2) * kPOutStageBytes;
        const int x0 = pt.nt * kNTile + half * 128;
        const int y0 = (int)(prow - lane);
        const uint32_t swz = (uint32_t)((lane >> 1) & 3);
        // the routing weight w >= 0 folds into the block maximum and the quantiser's power-of-two
        // multiplier: max |w * acc| = w * max |acc| and (w * mult) * acc = (w * acc) * mult in fp32
        // (exact while w * acc is a normal fp32 number: rounding is monotone, mult a power of two)
        const float wgt = p.row_w[prow];
        uint32_t sbytes = 0;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float mult[2];  // the chunk's two 32-column blocks, times w
#pragma unroll
          for (int bb = 0; bb < 2; ++bb) {
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(acc[64 * c + 32 * bb + i]));
            const MxScale sc = mx_scale<0>(amax * wgt);
            mult[bb] = sc.mult * wgt;
            sbytes |= (uint32_t)sc.byte << (8 * (2 * c + bb));
          }
          if (lane == 0) bulk_wait_read_all();  // the previous store has read the buffer
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {  // 16 columns a chunk piece: block 2c + i/2
            const float* v = acc + 64 * c + 16 * i;
            const uint2 q0 = pack_e4m3x8(v, mult[i / 2]), q1 = pack_e4m3x8(v + 8, mult[i / 2]);
            st_shared_v4(buf + (uint32_t)lane * 64u + (((uint32_t)i ^ swz) << 4), q0.x, q0.y, q1.x, q1.y);
          }
          fence_proxy_async_smem();  // generic-proxy writes -> visible to the TMA engine
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&p.tmap_out, buf, x0 + 64 * c, y0);
            bulk_commit_group();
          }
        }
        *reinterpret_cast<uint32_t*>(p.out_sf + prow * (p.N / 32) + x0 / 32) = sbytes;
      } else {
        store_acc_rows<ACT, EPI>(acc, valid, prow, pt.nt, half, p.N, p.out_codes, p.out_sf, p.out_bf16, p.row_w);
      }
    }
    if (G::kOutStaging && lane == 0) bulk_wait_all();  // this warp's y2 stores have completed
  }

  tc_fence_before();
  cluster_sync();  // both CTAs done with the pair's TMEM
  // Without an abort every stage a producer filled was consumed by the pair's MMAs, so no copy
  // is in flight.  After an abort in either CTA, loads that were issued but never waited for
  // may still be landing in this CTA's shared memory or on the even CTA's barriers: give them
  // time (they complete within microseconds) before either CTA can leave.
  const uint32_t peer_abort = ld_shared_cluster_u32(mapa_shared(smem_u32((const void*)abort_flag), rank ^ 1u));
  if (*abort_flag || peer_abort) grace_spin(2000000ull);
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kPTmemCols);
}

// ---------------------------------------------------------------------- host side
// Scale arrays in the 128x4 tile layout viewed as rows of 256 bytes; a stage's k-atoms of one
// 128-row block are 2 * atoms consecutive rows.
CUresult encode_scale_rows(EncodeTiledFn encode, CUtensorMap* m, const uint8_t* base, uint64_t bytes, int atoms) {
  const cuuint64_t dims[2] = {256, (cuuint64_t)(bytes / 256)};
  const cuuint64_t strides[1] = {256};
  const cuuint32_t box[2] = {256, (cuuint32_t)(2 * atoms)};
  const cuuint32_t es[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int ACT, int EPI>
cudaError_t launch_pair_typed(const GemmArgs& a, cudaStream_t s) {
  // per device, computed once; host threads racing here compute and store the same value
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = PairGeo<EPI>::kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters[dev].load(std::memory_order_acquire) == 0) {
    err = cudaFuncSetAttribute(moe_gemm_pair_kernel<ACT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               PairGeo<EPI>::kSmemBytes);
    if (err != cudaSuccess) return err;
    int n = 0;
    cfg.gridDim = dim3(2 * a.num_sms / 2);
    err = cudaOccupancyMaxActiveClusters(&n, moe_gemm_pair_kernel<ACT, EPI>, &cfg);
    if (err != cudaSuccess) return err;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    max_clusters[dev].store(n, std::memory_order_release);
  }
  EncodeTiledFn encode = get_encode_fn();
  if (!encode) return cudaErrorNotSupported;

  PairParams p;
  memset(&p, 0, sizeof(p));
  const int K = a.K;
  const int atoms = ActTraits<ACT>::kKPerStage / 128;
  const uint64_t act_row_bytes = ACT == 0 ? (uint64_t)K : (uint64_t)K / 2;
  {
    const cuuint64_t dims[2] = {act_row_bytes, (cuuint64_t)a.rows_cap};
    const cuuint64_t strides[1] = {act_row_bytes};
    const cuuint32_t box[2] = {128, (cuuint32_t)kRowTile};
    const cuuint32_t es[2] = {1, 1};
    if (encode(&p.tmap_act, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.act), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t row_bytes = (uint64_t)K / 2;
    const cuuint64_t strides[2] = {row_bytes, row_bytes * (uint64_t)a.N};
    const cuuint32_t box[3] = {128, (cuuint32_t)kPHalfRows, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    CUresult r;
    if (ACT == 0) {
      const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)a.N, (cuuint64_t)a.E};
      r = encode(&p.tmap_w, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<uint8_t*>(a.w), dims, strides, box,
                 es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
      const cuuint64_t dims[3] = {row_bytes, (cuuint64_t)a.N, (cuuint64_t)a.E};
      r = encode(&p.tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(a.w), dims, strides, box, es,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  const uint64_t asf_bytes = (uint64_t)(a.rows_cap / 128) * (uint64_t)(K / 128) * 512u;
  const uint64_t wsf_bytes = (uint64_t)a.E * (uint64_t)(a.N / 128) * (uint64_t)(K / 128) * 512u;
  if (encode_scale_rows(encode, &p.tmap_asf, a.act_sf, asf_bytes, atoms) != CUDA_SUCCESS ||
      encode_scale_rows(encode, &p.tmap_wsf, a.w_sf, wsf_bytes, atoms) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (EPI == 1) {
    const cuuint64_t dims[2] = {(cuuint64_t)a.N, (cuuint64_t)a.rows_cap};
    const cuuint64_t strides[1] = {(cuuint64_t)a.N * 2};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t es[2] = {1, 1};
    if (encode(&p.tmap_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.out_bf16, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (EPI == 3) {  // FP8 transport codes [rows_cap, N] bytes, box 64 bytes x 32 rows
    const cuuint64_t dims[2] = {(cuuint64_t)a.N, (cuuint64_t)a.rows_cap};
    const cuuint64_t strides[1] = {(cuuint64_t)a.N};
    const cuuint32_t box[2] = {64, 32};
    const cuuint32_t es[2] = {1, 1};
    if (encode(&p.tmap_out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.out_codes, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  p.counts = a.counts;
  p.mtile_base = a.mtile_base;
  p.act_sf = a.act_sf;
  p.act_sf_rot = a.act_sf_rot;
  p.out_codes = a.out_codes;
  p.out_sf = a.out_sf;
  p.out_bf16 = a.out_bf16;
  p.row_w = a.row_w;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  p.E = a.E;
  p.N = a.N;
  p.K = a.K;
  p.test_stall = a.test_stall;
  // pair tiles <= M tiles / 2: a bound on the clusters that can find work
  const int64_t clusters = std::min<int64_t>(std::min<int64_t>(max_clusters[dev].load(std::memory_order_acquire), a.num_sms / 2), a.max_tiles);
  if (clusters <= 0) return cudaSuccess;
  cfg.gridDim = dim3((unsigned)(2 * clusters));
  err = cudaLaunchKernelEx(&cfg, moe_gemm_pair_kernel<ACT, EPI>, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// ====================================================================== the wide tail pass
// Each expert's odd last M tile (at most 128 rows) by 512 output columns (two 256-column N tiles)
// on a cluster of two CTAs, tcgen05.mma.cta_group::2 with M = 128.  Each CTA stages 64 of the
// tile's activation rows and, for each N tile, 128 of its 256 weight rows: 8 KiB of activations
// and 32 KiB of weights (16 KiB read from HBM) per K stage, so five stages keep 80 KiB of weight
// bytes in flight per SM, where a single-CTA tail tile (one 128-row activation tile per 256
// weight rows, four stages) keeps 64 KiB.  Tail tiles share their weights with no other tile, and
// their weight stream is bound by those bytes in flight (loaded latency ~2 us).
// TMEM layouts (probed on the GB300 for M = 128 on a CTA pair): a CTA's 64 rows land in lanes
// 0-63 for output columns 0-127 of an N tile and in lanes 64-127 for columns 128-255, over 128
// TMEM columns per N tile; row m reads its A scale from lane m, column sfa + m/32, so the odd CTA,
// whose rows are rows 64-127 of their 128-row scale block, stages that block's atom with its two
// halves swapped (act_sf_rot, written by the pair kernel that runs just before); lanes 64-127
// read the weight scales of rows 128-255 from the same four columns where lanes 0-63 read rows
// 0-127: one .64x128b.warpx2::01_23 copy of the two atoms places them, per N tile.
constexpr int kWStages = 5;
constexpr int kWARows = 64;
constexpr int kWABytes = kWARows * 128;             // 64 activation rows x 128 bytes
constexpr int kWBOff = kWABytes;                    // N tile 0's weight rows, then N tile 1's
constexpr int kWBBytes = kPHalfRows * 128;          // 128 weight rows x 128 bytes (smem footprint)
constexpr int kWSfaOff = kWBOff + 2 * kWBBytes;     // one A-scale atom (A8W4: one k-atom a stage)
constexpr int kWSfbOff = kWSfaOff + 512;            // four weight-scale atoms, two per N tile
constexpr int kWStageBytes = (kWSfbOff + 4 * 512 + 1023) / 1024 * 1024;  // 43 KiB
constexpr int kWBarOff = kWStages * kWStageBytes;
constexpr int kWBaseOff = kWBarOff + 256;           // tail-tile prefix over experts, int32 [E+1]
constexpr int kWTileBaseOff = kWBaseOff + 4 * (kMaxExperts + 1);  // M-tile prefix, int32 [E+1]
constexpr int kWSmemBytes = kWTileBaseOff + 4 * (kMaxExperts + 1) + 1024;
constexpr uint32_t kWTmemCols = 512;
constexpr uint32_t kWSfCol0 = 256;                  // accumulators: N tile t in columns [128t, 128t + 128)
constexpr uint32_t kWSfSlotCols = 12;               // 4 A-scale columns, 4 + 4 weight-scale columns
static_assert(kWSmemBytes <= 232448, "wide tail pass shared memory");
static_assert(kWSfCol0 + kWStages * kWSfSlotCols <= kWTmemCols, "wide tail pass TMEM");

struct TailParams {  // 64-byte aligned through its CUtensorMap members
  CUtensorMap tmap_act;      // activation codes [rows_cap, K], box 128 B x 64 rows
  CUtensorMap tmap_w;        // weights [E, N, K/2], box 128 K x 128 rows x 1
  CUtensorMap tmap_asf;      // activation scales as rows of 256 bytes, box 256 x 2
  CUtensorMap tmap_asf_rot;  // their rotated atoms (act_sf_rot), same view
  CUtensorMap tmap_wsf;      // prepacked weight scales as rows of 256 bytes, box 256 x 2
  const int32_t* counts;
  const int32_t* mtile_base;
  uint8_t* out_codes;
  uint8_t* out_sf;
  uint16_t* out_bf16;
  const float* row_w;         // epilogue 3: routing weight of each padded row
  uint32_t* status;
  uint64_t timeout_ns;
  int E, N, K;
  int test_stall;
};

template <int EPI>
__global__ void __launch_bounds__(kPThreads, 1) moe_gemm_tail_wide_kernel(const __grid_constant__ TailParams p) {
  constexpr int ACT = 0;
  using TR = ActTraits<ACT>;
  constexpr int kMmaPerStage = TR::kKPerStage / TR::kMmaK;  // 4
  constexpr uint32_t kBHalfTx = TR::kBTxBytes / 2;          // global bytes of 128 weight rows

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kWBarOff;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kWStages + s); };
  const uint32_t tmem_full_bar = bar0 + 8u * (2 * kWStages);
  const uint32_t tmem_empty_bar = tmem_full_bar + 8;
  const uint32_t drain_bar = tmem_full_bar + 16;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kWBarOff + 8 * (2 * kWStages + 3));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int32_t* tail_base = reinterpret_cast<int32_t*>(smem + kWBaseOff);
  int32_t* tile_base = reinterpret_cast<int32_t*>(smem + kWTileBaseOff);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int E = p.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(full_bar(s), 2);    // expect_tx arrivals of warps 0 and 10 of the even CTA
      mbar_init(empty_bar(s), 1);   // the pair's MMA commit
    }
    mbar_init(tmem_full_bar, 1);
    mbar_init(tmem_empty_bar, 2 * kPEpiWarps);  // epilogue warps of both CTAs
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int e = threadIdx.x; e <= E; e += blockDim.x) tile_base[e] = p.mtile_base[e];
  if (warp == 2) {  // tail tiles per expert: 1 when its M-tile count is odd
    int running = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? ((p.mtile_base[e + 1] - p.mtile_base[e]) & 1) : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < E) tail_base[e] = running + incl - v;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tail_base[E] = running;
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_holder), kWTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers initialised in both CTAs before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const Sync sync{abort_flag, p.status, p.timeout_ns, bar0};
  const int NT2 = p.N / kTailWideN;
  const int K = p.K;
  const int nks = K / TR::kKPerStage;  // K % 128 == 0
  const int64_t total_tiles = (int64_t)tail_base[E] * NT2;
  const int64_t first_tile = cluster_index();
  const int64_t tile_step = cluster_count();
  const uint32_t leader_full0 = mapa_shared(full_bar(0), 0);

  if (warp == 0 || warp == kPBWarp) {
    // ------------------------------------------------------------------ producers (converged)
    const bool act_warp = warp == 0;
    int slot = 0;
    uint32_t phase = 0;
    bool ok = !p.test_stall;  // the test hook leaves every stage unfilled
    for (int64_t tile = first_tile; ok && tile < total_tiles; tile += tile_step) {
      const PairTile pt = decode_pair_tile(tile, tail_base, E, NT2);  // pm = 0: one tail per expert
      const int64_t row0 = (int64_t)(tile_base[pt.e + 1] - 1) * kRowTile;  // the last M tile
      const int n0 = pt.nt * kTailWideN;
      const int asf_y0 = (int)(2 * ((row0 / 128) * (K / 128)));              // scale rows of 256 B
      const int wsf_y0 = (int)(2 * ((((int64_t)pt.e * p.N + n0) / 128) * (K / 128)));
      const int wsf_next = 2 * (K / 128);                                      // next 128 weight rows
      const uint32_t act_tx = 2u * ((uint32_t)kWABytes + 512u);
      const uint32_t w_tx = 2u * (2u * kBHalfTx + 4u * 512u);
      for (int ks = 0; ks < nks; ++ks) {
        if (!warp_wait(empty_bar(slot), phase ^ 1u, sync, p.timeout_ns)) {
          ok = false;
          break;
        }
        const uint32_t st = sbase + (uint32_t)slot * kWStageBytes;
        const uint32_t lfull = leader_full0 + 8u * slot;
        const int ky = 2 * ks;
        if (elect_one()) {
          if (act_warp) {
            if (leader) mbar_arrive_expect_tx(full_bar(slot), act_tx);
            tma_load_2d_pair(st, &p.tmap_act, lfull, ks * 128, (int)(row0 + (int64_t)rank * kWARows));
            tma_load_2d_pair(st + kWSfaOff, leader ? &p.tmap_asf : &p.tmap_asf_rot, lfull, 0, asf_y0 + ky);
          } else {
            if (leader) mbar_arrive_expect_tx(full_bar(slot), w_tx);
#pragma unroll
            for (int t = 0; t < 2; ++t)
              tma_load_3d_pair(st + kWBOff + t * kWBBytes, &p.tmap_w, lfull, ks * 128,
                               n0 + t * kNTile + (int)rank * kPHalfRows, pt.e);
#pragma unroll
            for (int b = 0; b < 4; ++b)  // weight rows n0 + 128 b .. + 127
              tma_load_2d_pair(st + kWSfbOff + b * 512, &p.tmap_wsf, lfull, 0, wsf_y0 + b * wsf_next + ky);
          }
        }
        __syncwarp();
        if (++slot == kWStages) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (even CTA)
    if (leader) {
      int slot = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true, issued = false;
      const uint64_t a_desc0 = smem_desc(sbase, 16, 1024, kLayoutSwizzle128B);
      const uint64_t b_desc0 = smem_desc(sbase + kWBOff, 16, 1024, kLayoutSwizzle128B);
      const uint64_t sfa_desc0 = smem_desc(sbase + kWSfaOff, 128, 128, kLayoutNone);
      const uint64_t sfb_desc0 = smem_desc(sbase + kWSfbOff, 128, 128, kLayoutNone);
      constexpr uint64_t kSlotStep = kWStageBytes >> 4;
      constexpr uint64_t kBTileStep = kWBBytes >> 4;
      for (int64_t tile = first_tile; ok && tile < total_tiles; tile += tile_step) {
        if (!warp_wait(tmem_empty_bar, acc_phase ^ 1u, sync, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = 0; ks < nks; ++ks) {
          if (!warp_wait(full_bar(slot), phase, sync, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t so = (uint64_t)slot * kSlotStep;
          const uint32_t sf_col = tmem_base + kWSfCol0 + (uint32_t)slot * kWSfSlotCols;
          if (elect_one()) {
            tc_cp_pair_32x128b_warpx4(sf_col, sfa_desc0 + so);
            tc_cp_pair_64x128b_warpx2_0123(sf_col + 4, sfb_desc0 + so);
            tc_cp_pair_64x128b_warpx2_0123(sf_col + 8, sfb_desc0 + so + (1024 >> 4));
#pragma unroll
            for (int j = 0; j < kMmaPerStage; ++j) {
              const uint32_t idesc = make_idesc<ACT>((uint32_t)j, kRowTile);  // M = 128 over the pair
              const uint32_t acc = (ks > 0 || j > 0) ? 1u : 0u;
#pragma unroll
              for (int t = 0; t < 2; ++t)
                tc_mma_pair_mxf8f6f4(tmem_base + (uint32_t)t * 128u, a_desc0 + so + 2 * j,
                                     b_desc0 + so + (uint64_t)t * kBTileStep + 2 * j, idesc, sf_col,
                                     sf_col + 4 + 4 * t, acc);
            }
            tc_commit_pair_mc(empty_bar(slot), 0x3);
          }
          __syncwarp();
          issued = true;
          if (++slot == kWStages) {
            slot = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one()) tc_commit_pair_mc(tmem_full_bar, 0x3);
        __syncwarp();
        acc_phase ^= 1u;
      }
      if (issued) {
        // no MMA or TMEM copy of the pair may still run when TMEM is freed
        if (elect_one()) tc_commit_pair(drain_bar);
        __syncwarp();
        warp_wait(drain_bar, 0, sync, 100000000ull, true);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    // lane quadrant q: rows (q & 1) * 32 + lane of this CTA's 64, output columns of half q / 2 of
    // the N tile; warps 2-5 take N tile 0 of the pair tile, warps 6-9 N tile 1
    const int quad = warp & 3;
    const int ntl = (warp - 2) >> 2;
    const uint32_t leader_tmem_empty = mapa_shared(tmem_empty_bar, 0);
    uint32_t acc_phase = 0;
    for (int64_t tile = first_tile; tile < total_tiles; tile += tile_step) {
      const PairTile pt = decode_pair_tile(tile, tail_base, E, NT2);
      const int mt = tile_base[pt.e + 1] - tile_base[pt.e] - 1;
      const int row_local = mt * kRowTile + (int)rank * kWARows + (quad & 1) * 32 + lane;
      const bool valid = row_local < p.counts[pt.e];
      const int64_t prow = (int64_t)tile_base[pt.e] * kRowTile + row_local;
      if (!warp_wait(tmem_full_bar, acc_phase, sync, p.timeout_ns)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(ntl * 128);
      float acc[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc_ld_32x32b_x32(taddr + c * 32, acc + 32 * c);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(leader_tmem_empty);  // registers hold the tile
      acc_phase ^= 1u;
      store_acc_rows<ACT, EPI>(acc, valid, prow, 2 * pt.nt + ntl, quad >> 1, p.N, p.out_codes, p.out_sf,
                               p.out_bf16, p.row_w);
    }
  }

  tc_fence_before();
  cluster_sync();  // both CTAs done with the pair's TMEM
  // as in the pair kernel: after an abort, let copies that were issued but never waited for land
  const uint32_t peer_abort = ld_shared_cluster_u32(mapa_shared(smem_u32((const void*)abort_flag), rank ^ 1u));
  if (*abort_flag || peer_abort) grace_spin(2000000ull);
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kWTmemCols);
}

template <int EPI>
cudaError_t launch_tail_wide_typed(const GemmArgs& a, cudaStream_t s) {
  // per device, computed once; host threads racing here compute and store the same value
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kWSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters[dev].load(std::memory_order_acquire) == 0) {
    err = cudaFuncSetAttribute(moe_gemm_tail_wide_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kWSmemBytes);
    if (err != cudaSuccess) return err;
    int n = 0;
    cfg.gridDim = dim3(2 * (a.num_sms / 2));
    err = cudaOccupancyMaxActiveClusters(&n, moe_gemm_tail_wide_kernel<EPI>, &cfg);
    if (err != cudaSuccess) return err;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    max_clusters[dev].store(n, std::memory_order_release);
  }
  EncodeTiledFn encode = get_encode_fn();
  if (!encode) return cudaErrorNotSupported;
  TailParams p;
  memset(&p, 0, sizeof(p));
  const int K = a.K;
  if (!encode_act_map(&p.tmap_act, a.act, a.rows_cap, K, 0, kWARows)) return cudaErrorInvalidValue;
  {
    const uint64_t row_bytes = (uint64_t)K / 2;
    const cuuint64_t strides[2] = {row_bytes, row_bytes * (uint64_t)a.N};
    const cuuint32_t box[3] = {128, (cuuint32_t)kPHalfRows, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)a.N, (cuuint64_t)a.E};
    if (encode(&p.tmap_w, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<uint8_t*>(a.w), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const uint64_t asf_bytes = (uint64_t)(a.rows_cap / 128) * (uint64_t)(K / 128) * 512u;
  const uint64_t wsf_bytes = (uint64_t)a.E * (uint64_t)(a.N / 128) * (uint64_t)(K / 128) * 512u;
  if (encode_scale_rows(encode, &p.tmap_asf, a.act_sf, asf_bytes, 1) != CUDA_SUCCESS ||
      encode_scale_rows(encode, &p.tmap_asf_rot, a.act_sf_rot, asf_bytes, 1) != CUDA_SUCCESS ||
      encode_scale_rows(encode, &p.tmap_wsf, a.w_sf, wsf_bytes, 1) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  p.counts = a.counts;
  p.mtile_base = a.mtile_base;
  p.out_codes = a.out_codes;
  p.out_sf = a.out_sf;
  p.out_bf16 = a.out_bf16;
  p.row_w = a.row_w;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  p.E = a.E;
  p.N = a.N;
  p.K = a.K;
  p.test_stall = a.test_stall;
  // tail tiles <= M tiles x 512-column tiles
  const int64_t clusters = std::min<int64_t>(
      std::min<int64_t>(max_clusters[dev].load(std::memory_order_acquire), a.num_sms / 2), a.max_tiles);
  if (clusters <= 0) return cudaSuccess;
  cfg.gridDim = dim3((unsigned)(2 * clusters));
  err = cudaLaunchKernelEx(&cfg, moe_gemm_tail_wide_kernel<EPI>, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_pair(const GemmArgs& a, cudaStream_t s) {
  // A8W4, prepacked weight scales, K a multiple of 128
  if (!a.w_sf_tiled || a.act_fmt != 0 || a.K % 128 != 0) return cudaErrorInvalidValue;
  switch (a.epilogue) {
    case 0: return launch_pair_typed<0, 0>(a, s);
    case 1: return launch_pair_typed<0, 1>(a, s);
    case 3: return launch_pair_typed<0, 3>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_tail_wide(const GemmArgs& a, cudaStream_t s) {
  // A8W4 with prepacked weight scales, N a multiple of 512, the rotated atoms written
  if (!a.w_sf_tiled || a.act_fmt != 0 || a.N % kTailWideN != 0 || a.K % 128 != 0 || a.act_sf_rot == nullptr)
    return cudaErrorInvalidValue;
  switch (a.epilogue) {
    case 0: return launch_tail_wide_typed<0>(a, s);
    case 1: return launch_tail_wide_typed<1>(a, s);
    case 3: return launch_tail_wide_typed<3>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
