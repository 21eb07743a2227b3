// gemm.cu -- grouped block-scaled GEMMs of the expert layer on the tcgen05 tensor cores.
//
// One persistent kernel; its epilogues:
//   GEMM1 (EPI=0): acc[r, n] = sum_K xq[r, K] * W1[e, n, K], n in [0, 2I) with rows 2j = gate_j,
//                  2j+1 = up_j ("feat(moe): FlyDSL MegaMoE fused EP-MoE integration", description:
//                  INTERLEAVE(g1u1)); the epilogue forms h_j = silu(gate_j) * up_j and requantises
//                  h to MX: the intermediate activation A2 leaves as FP4 codes with E8M0 scales
//                  for A4W4 ("add A4W4 and FP8 P2P transport support to MegaMoE", Technical
//                  Details) and as E4M3 codes for A8W4.
//   GEMM2 (EPI=1): y2[r, n] = sum_I a2[r, I] * W2[e, n, I], accumulated in fp32, stored as bf16.
//   GEMM2 (EPI=3, FP8 transport): the same rows times their routing weights, stored as E4M3
//                  codes with one E8M0 scale per 1x32 block (same page, Technical Details).
//   GEMM1 (EPI=2, bf16-out form): h as bf16 rows for a separate requantisation kernel.
//
// Tiles are 128 routed rows (one expert's padded segment) x 256 output columns.  Per CTA:
//   warp 0      producer: TMA (activation tile 128x128B, weight tile 256x128B) and a bulk copy
//               of the activation scales (already in the 128x4 tile layout);
//   warp 10     producer: with canonical weight scales, 4-byte cp.async copies that rearrange
//               them into that layout; with prepacked scales, the TMA of the weight tile and
//               the bulk copies of its scales (so the two halves of a stage issue in parallel);
//   warp 1      TMEM owner; converged, with one elected lane issuing tcgen05.cp of the scales
//               to TMEM, then tcgen05.mma kind::mxf8f6f4 (E4M3 x E2M1, scale_vec 1X) or
//               kind::mxf4 (E2M1 x E2M1, scale_vec 2X) into a 128x256 fp32 accumulator in
//               TMEM, from precomputed descriptors;
//   warps 2..9  epilogue: tcgen05.ld of the accumulator, one TMEM lane (= one routed row) per
//               thread; warps 2-5 take columns [0, 128), warps 6-9 columns [128, 256).  Each
//               thread pulls its 128 columns into registers, releases TMEM at once, and only
//               then runs the SwiGLU / requant / store work, so that work overlaps the next
//               tile's MMAs.  GEMM2 rows leave through shared memory as TMA stores.
// A 4-deep shared-memory ring with full/empty mbarriers overlaps the weight stream with the
// MMAs; each tile's canonical weight-scale block is prefetched into L2 at the tile start.
// The experts' M-tile prefix is staged in shared memory for the per-tile lookups.  Every wait
// is bounded: on expiry the kernel records MOE_ERR_DEVICE_TIMEOUT in the status word, lets its
// own copies and MMAs drain (again bounded), frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "gemm_common.cuh"
#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 352;    // TMA producer, MMA, 8 epilogue warps, weight-scale copier
constexpr int kEpiWarps = 8;
constexpr int kScaleWarp = 10;
constexpr int kOutStageBytes = 32 * 32 * 2;  // GEMM2 epilogue staging: 32 rows x 32 bf16 per warp

// Shared-memory geometry of one CTA.  Regular tiles stage all 128 activation rows of a tile
// per K stage.  Small batches stage fewer, which leaves room for more stages of the
// latency-bound weight stream: AROWS = 16 when T <= 16 (no tile then has more routed rows: a
// token routes to an expert at most once), AROWS = 64 when experts average few rows -- work
// units are then 64-row halves of the 128-row tiles, an expert with more than 64 rows taking
// two.  The MMA still reads 128 rows: rows past AROWS come from the following bytes of the
// stage and only reach accumulator rows that are never stored.
template <int ACT, int AROWS>
struct Geo {
  static constexpr int kUnitRows = AROWS == 64 ? 64 : kRowTile;  // rows of one work unit
  static constexpr int kABytes = AROWS * 128;              // activation slot
  static constexpr int kBOff = kABytes;                    // weight tile, 1024-aligned (SW128)
  static constexpr int kBBytes = kNTile * 128;             // 256 rows x 128 bytes of shared memory
  static constexpr int kSfaOff = kBOff + kBBytes;
  static constexpr int kSfaBytes = ActTraits<ACT>::kKPerStage / 128 * 512;
  static constexpr int kSfbOff = kSfaOff + kSfaBytes;      // two 128-row halves of kSfaBytes each
  static constexpr int kStageBytes = (kSfbOff + 2 * kSfaBytes + 1023) / 1024 * 1024;
  static constexpr int kStages = AROWS == kRowTile ? 4 : (AROWS == 16 && ACT == 0 ? 6 : 5);
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kTileBaseOff = kBarOff + 256;      // M-tile prefix over experts, int32 [E+1]
  // 64-row units, and the tail pass of A8W4 128-row tiles: their own prefix over experts,
  // int32 [E+1] (else the M-tile prefix serves)
  static constexpr bool kUnitTable = kUnitRows == 64 || (AROWS == kRowTile && ACT == 0);
  static constexpr int kUnitBaseOff = kTileBaseOff + 4 * (kMaxExperts + 1);
  static constexpr int kTablesEnd = kUnitBaseOff + (kUnitTable ? 4 * (kMaxExperts + 1) : 0);
  static constexpr bool kOutStaging = AROWS == kRowTile;  // GEMM2 rows leave as TMA stores
  static constexpr int kOutStageOff = (kTablesEnd + 1023) / 1024 * 1024;
  static constexpr int kSmemBytes =
      (kOutStaging ? kOutStageOff + kEpiWarps * kOutStageBytes : kTablesEnd) + 1024;  // + alignment slack
  static_assert(kBOff % 1024 == 0 && kStageBytes % 1024 == 0, "SW128 tiles need 1024-byte alignment");
  static_assert(kSmemBytes <= 232448, "single-CTA GEMM shared memory");
  static_assert(kStages * 32 <= 256, "TMEM scale slots");
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;   // accumulator uses columns [0, 256)
constexpr uint32_t kSfSlotCols = 32;

struct GemmParams {  // 64-byte aligned through its CUtensorMap members
  CUtensorMap tmap_act;   // activation codes, box 128 B x AROWS rows
  CUtensorMap tmap_w;
  CUtensorMap tmap_out;   // GEMM2: y2 bf16 [rows_cap, N], box 32 columns x 32 rows, 64-byte swizzle
  const uint8_t* act_sf;
  const uint8_t* w_sf;    // canonical [E, N, K/32], or the 128x4 tile layout when w_sf_tiled
  const int32_t* counts;
  const int32_t* mtile_base;  // expert e's rows start at row 128 * mtile_base[e]
  uint8_t* out_codes;
  uint8_t* out_sf;
  uint16_t* out_bf16;
  const float* row_w;     // epilogue 3: routing weight of each padded row
  uint32_t* status;
  uint64_t timeout_ns;
  int E, N, K;
  int w_sf_tiled;
  int test_stall;
  int tail_only;  // only the odd last M tile of each expert (the pair kernel took the rest)
};

template <int ACT, int EPI, int AROWS>
__global__ void __launch_bounds__(kThreads, 1) moe_gemm_kernel(const __grid_constant__ GemmParams p) {
  using TR = ActTraits<ACT>;
  using G = Geo<ACT, AROWS>;
  constexpr int kStages = G::kStages;
  constexpr int kStageBytes = G::kStageBytes;
  constexpr int kSfaOff = G::kSfaOff;
  constexpr int kSfbOff = G::kSfbOff;
  constexpr int kMmaPerStage = TR::kKPerStage / TR::kMmaK;  // 4
  constexpr int kAtomsPerStage = TR::kKPerStage / 128;      // k-atoms of 4 scale blocks
  constexpr uint32_t kSfaCols = kAtomsPerStage * 4;

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
  int32_t* tile_base = reinterpret_cast<int32_t*>(smem + G::kTileBaseOff);
  // work units per expert: its M tiles, (64-row units) ceil(count / 64), or (tail pass) its odd
  // last M tile
  const bool unit_table = G::kUnitRows == 64 || (G::kUnitTable && p.tail_only);
  int32_t* unit_base = unit_table ? reinterpret_cast<int32_t*>(smem + G::kUnitBaseOff) : tile_base;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // the per-tile expert lookup (a binary search) reads shared memory, not global memory: it
  // sits on the producer's path at every tile boundary
  for (int e = threadIdx.x; e <= p.E; e += blockDim.x) tile_base[e] = p.mtile_base[e];
  if (unit_table && threadIdx.x / 32 == 2) {  // exclusive prefix of the units per expert, warp 2
    const int ln = threadIdx.x % 32;
    int running = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + ln;
      const int v = e >= p.E ? 0
                    : G::kUnitRows == 64 ? (p.counts[e] + 63) / 64
                                         : ((p.mtile_base[e + 1] - p.mtile_base[e]) & 1);
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (ln >= o) incl += n;
      }
      if (e < p.E) unit_base[e] = running + incl - v;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (ln == 0) unit_base[p.E] = running;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // canonical scales: warp 0's expect_tx arrive + 32 cp.async arrivals of the scale warp;
      // prepacked scales: one expect_tx arrive from each of warps 0 and 10
      mbar_init(full_bar(s), p.w_sf_tiled ? 2 : 1 + 32);
      mbar_init(empty_bar(s), 1);      // tcgen05.commit
    }
    mbar_init(tmem_full_bar, 1);
    mbar_init(tmem_empty_bar, kEpiWarps);  // one arrival per epilogue warp
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const Sync sync{abort_flag, p.status, p.timeout_ns, bar0};
  // N is a multiple of 128: when it is not one of 256 the last N tile has 128 columns.  Its
  // weight rows past N come from the TMA's out-of-bounds zero fill, its scale copies stop at N
  // and the epilogue warps of the missing half store nothing.
  const int NT = (p.N + kNTile - 1) / kNTile;
  const int K = p.K;
  const int nks = (K + TR::kKPerStage - 1) / TR::kKPerStage;
  const int64_t total_tiles = (int64_t)unit_base[p.E] * NT;  // work units

  if (warp == 0 || warp == kScaleWarp) {
    // ------------------------------------------------------------------ producers
    // Warp 0 issues the TMA loads of a stage; warp 10 gathers the stage's weight scales
    // with 4-byte cp.async copies.  Both walk the same stages and wait for the same free
    // slots, so the two kinds of copy are issued in parallel.
    const bool tma_warp = warp == 0;
    int slot = 0;
    uint32_t phase = 0;
    int armed_parity[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s) armed_parity[s] = -1;
    bool ok = !p.test_stall;  // the test hook leaves every stage unfilled
    for (int64_t tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      Tile tc = decode_tile(tile, unit_base, p.E, NT);  // tc.mt: unit index inside the expert
      if (G::kUnitTable && p.tail_only) tc.mt = tile_base[tc.e + 1] - tile_base[tc.e] - 1;  // the last M tile
      const int64_t row0 = (int64_t)tile_base[tc.e] * kRowTile + (int64_t)tc.mt * G::kUnitRows;
      const int n0 = tc.nt * kNTile;
      const uint8_t* wsf_rows = p.w_sf + ((int64_t)tc.e * p.N + n0) * (K / 32);
      const int64_t sf_row32 = (int64_t)32 * (K / 32);        // 32 weight rows of scales
      const uint8_t* lane_sf = wsf_rows + (int64_t)lane * (K / 32);
      const int n_rows = min(kNTile, p.N - n0);  // weight rows of this tile inside [0, N)
      if (!tma_warp && !p.w_sf_tiled && lane == 0) {
        // warm L2 with this tile's whole (contiguous) weight-scale block
        const uint32_t sf_bytes = (uint32_t)n_rows * (uint32_t)(K / 32);
        if ((reinterpret_cast<uintptr_t>(wsf_rows) & 15) == 0 && (sf_bytes & 15) == 0)
          bulk_prefetch_l2(wsf_rows, sf_bytes);
      }
      for (int ks = 0; ks < nks; ++ks) {
        if (!warp_wait(empty_bar(slot), phase ^ 1u, sync, p.timeout_ns)) {
          ok = false;
          break;
        }
        const int katoms = min(TR::kKPerStage, K - ks * TR::kKPerStage) / 128;
        const uint32_t st = sbase + (uint32_t)slot * kStageBytes;
        // one elected lane of the converged warp issues the copies (as for the MMAs, this keeps
        // their operands in uniform registers and the loop short)
        if (elect_one()) {
          if (tma_warp) {
            // activation side, plus the weight codes when the scale warp is busy gathering
            mbar_arrive_expect_tx(full_bar(slot),
                                  (uint32_t)(G::kABytes + katoms * 512 + (p.w_sf_tiled ? 0 : TR::kBTxBytes)));
            tma_load_2d(st, &p.tmap_act, full_bar(slot), ks * 128, (int)row0);
            bulk_load(st + kSfaOff, p.act_sf + ((row0 / 128) * (K / 128) + (int64_t)ks * kAtomsPerStage) * 512,
                      (uint32_t)katoms * 512u, full_bar(slot));
            if (!p.w_sf_tiled) tma_load_3d(st + G::kBOff, &p.tmap_w, full_bar(slot), ks * 128, n0, tc.e);
          } else if (p.w_sf_tiled) {
            // weight side with prepacked scales: codes + one contiguous run of k-atoms per
            // 128-row half of the tile, issued in parallel with warp 0
            const int halves = n_rows > 128 ? 2 : 1;
            mbar_arrive_expect_tx(full_bar(slot), (uint32_t)(TR::kBTxBytes + halves * katoms * 512));
            tma_load_3d(st + G::kBOff, &p.tmap_w, full_bar(slot), ks * 128, n0, tc.e);
            for (int na = 0; na < halves; ++na)
              bulk_load(st + kSfbOff + na * (kAtomsPerStage * 512),
                        p.w_sf + ((((int64_t)tc.e * p.N + n0) / 128 + na) * (K / 128) + (int64_t)ks * kAtomsPerStage) * 512,
                        (uint32_t)katoms * 512u, full_bar(slot));
          }
        }
        // weight scales: this lane copies rows lane + 32*jj (jj < 8) of each k-atom, 4 bytes each,
        // into the 128x4 tile layout (row r -> byte (r%32)*16 + ((r%128)/32)*4 of tile r/128)
        if (!tma_warp && !p.w_sf_tiled) {
          const uint8_t* src_k = lane_sf + ks * (TR::kKPerStage / 32);
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
        armed_parity[slot] = (int)phase;
        if (++slot == kStages) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
    // Let every copy this warp started land before the CTA can exit.
    cp_async_wait_all();
    // both warps that issued TMA / bulk copies (warp 10 does with prepacked scales) let
    // them land before the CTA can exit
    if (tma_warp || p.w_sf_tiled)
      for (int s = 0; s < kStages; ++s)
        if (armed_parity[s] >= 0) warp_wait(full_bar(s), (uint32_t)armed_parity[s], sync, 100000000ull, true);
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The warp runs the loop converged (waits, descriptor arithmetic) and one elected lane
    // issues each tcgen05.cp / tcgen05.mma / tcgen05.commit.  From one divergent lane the same
    // loop took longer per stage than the four MMAs it issues (the pipe then idled between
    // stages); from the converged warp the stage runs at the MMAs' own rate.
    int slot = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true, issued = false;
    // descriptors of slot 0; a slot adds kStageBytes, an MMA step 32 bytes (start address
    // field, in 16-byte units; shared-memory offsets stay below 2^18, so no carry)
    const uint64_t a_desc0 = smem_desc(sbase, 16, 1024, kLayoutSwizzle128B);
    const uint64_t b_desc0 = smem_desc(sbase + G::kBOff, 16, 1024, kLayoutSwizzle128B);
    const uint64_t sfa_desc0 = smem_desc(sbase + kSfaOff, 128, 128, kLayoutNone);
    const uint64_t sfb_desc0 = smem_desc(sbase + kSfbOff, 128, 128, kLayoutNone);
    constexpr uint64_t kSlotStep = kStageBytes >> 4;
    constexpr uint32_t kHalfStep = (kAtomsPerStage * 512) >> 4;  // second 128 weight rows
    const bool gathered = !p.w_sf_tiled;
    for (int64_t tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      // A 64-row unit over rows 64..127 of its 128-row block: the block's scale tile lands in
      // TMEM as a whole and row m reads lane m, column sfa + m/32, so the unit's rows 0..63
      // take the scales of block rows 64..127 two columns further on.
      uint32_t sfa_shift = 0;
      if (G::kUnitRows == 64) sfa_shift = 2u * (uint32_t)(decode_tile(tile, unit_base, p.E, NT).mt & 1);
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
        if (gathered) fence_proxy_async_smem();  // scales written by cp.async, read by tcgen05.cp
        const uint64_t so = (uint64_t)slot * kSlotStep;
        const uint32_t sf_col = tmem_base + kSfCol0 + (uint32_t)slot * kSfSlotCols;
        const int kvalid = min(TR::kKPerStage, K - ks * TR::kKPerStage);
        const int katoms = kvalid == TR::kKPerStage ? kAtomsPerStage : kvalid / 128;
        const int nmma = kvalid == TR::kKPerStage ? kMmaPerStage : kvalid / TR::kMmaK;
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
              const int kblk = j * (TR::kMmaK / 32);  // first 32-block of this MMA inside the stage
              const uint32_t idesc = make_idesc<ACT>((uint32_t)(kblk & 3), kRowTile);
              const uint32_t acc = (ks > 0 || j > 0) ? 1u : 0u;
              if (ACT == 0)
                tc_mma_mxf8f6f4(tmem_base, a_desc0 + so + 2 * j, b_desc0 + so + 2 * j, idesc,
                                sf_col + (kblk >> 2) * 4 + sfa_shift, sf_col + kSfaCols + (kblk >> 2) * 8, acc);
              else
                tc_mma_mxf4(tmem_base, a_desc0 + so + 2 * j, b_desc0 + so + 2 * j, idesc,
                            sf_col + (kblk >> 2) * 4 + sfa_shift, sf_col + kSfaCols + (kblk >> 2) * 8, acc);
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
    }
    // Make sure no MMA or TMEM copy of this CTA is still running before TMEM is freed.
    if (issued) {
      if (elect_one()) tc_commit(drain_bar);
      __syncwarp();
      warp_wait(drain_bar, 0, sync, 100000000ull, true);
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int quad = warp & 3;         // TMEM lane quadrant this warp may read
    const int half = (warp - 2) >> 2;  // accumulator columns [half*128, half*128 + 128)
    uint32_t acc_phase = 0;
    for (int64_t tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      Tile tc = decode_tile(tile, unit_base, p.E, NT);
      if (G::kUnitTable && p.tail_only) tc.mt = tile_base[tc.e + 1] - tile_base[tc.e] - 1;
      const int row_local = tc.mt * G::kUnitRows + quad * 32 + lane;
      // a 64-row unit fills accumulator lanes 0..63 only: the warps of quadrants 2 and 3 keep
      // step with the tile hand-off (wait, release) and store nothing; so do the warps of
      // columns [128, 256) of a 128-column last N tile
      const bool lanes_used = (G::kUnitRows == kRowTile || quad < 2) && tc.nt * kNTile + half * 128 < p.N;
      const bool valid = lanes_used && row_local < p.counts[tc.e];
      const int64_t prow = (int64_t)tile_base[tc.e] * kRowTile + row_local;
      if (!warp_wait(tmem_full_bar, acc_phase, sync, p.timeout_ns)) break;
      tc_fence_after();
      if (!lanes_used) {
        __syncwarp();
        if (lane == 0) mbar_arrive(tmem_empty_bar);
        acc_phase ^= 1u;
        continue;
      }
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(half * 128);
      float acc[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc_ld_32x32b_x32(taddr + c * 32, acc + 32 * c);
      tc_wait_ld();
      // the accumulator is in registers: hand TMEM back to the MMA warp before the math
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_empty_bar);
      acc_phase ^= 1u;
      if (EPI == 1 && G::kOutStaging && __all_sync(0xffffffffu, valid)) {
        // GEMM2 rows as bf16 (round to nearest even) through shared memory when all 32 rows of
        // this warp are routed rows: each 32-column chunk leaves as one TMA store.  (Every lane
        // storing 16-byte pieces of its own row kept the load/store pipe so busy that the MMA
        // warp's barrier polls queued behind the stores: GEMM2 ran 25 % slower at large T.)
        // A warp with padding rows stores its valid rows directly (few such warps at large T;
        // at small T most rows are padding, and skipping them saves HBM writes).
        const uint32_t buf = sbase + G::kOutStageOff + (uint32_t)(warp - 2) * kOutStageBytes;
        const int x0 = tc.nt * kNTile + half * 128;
        const int y0 = (tile_base[tc.e] + tc.mt) * kRowTile + quad * 32;
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
      } else {
        store_acc_rows<ACT, EPI>(acc, valid, prow, tc.nt, half, p.N, p.out_codes, p.out_sf, p.out_bf16, p.row_w);
      }
    }
  }

  if (EPI == 1 && G::kOutStaging && warp >= 2 && warp < 2 + kEpiWarps && lane == 0) bulk_wait_all();  // y2 stores

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------- host side
template <int ACT, int EPI, int AROWS>
cudaError_t launch_typed(const GemmArgs& a, cudaStream_t s) {
  using G = Geo<ACT, AROWS>;
  // per device, set once; host threads racing here both set the same attribute
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    err = cudaFuncSetAttribute(moe_gemm_kernel<ACT, EPI, AROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               G::kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_set[dev].store(true, std::memory_order_release);
  }
  EncodeTiledFn encode = get_encode_fn();
  if (!encode) return cudaErrorNotSupported;

  GemmParams p;
  memset(&p, 0, sizeof(p));
  if (!encode_act_map(&p.tmap_act, a.act, a.rows_cap, a.K, ACT, AROWS) ||
      !encode_weight_map(&p.tmap_w, a.w, a.E, a.N, a.K, ACT))
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
  p.act_sf = a.act_sf;
  p.w_sf = a.w_sf;
  p.w_sf_tiled = a.w_sf_tiled;
  p.test_stall = a.test_stall;
  p.tail_only = a.tail_only;
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
  // 64-row units: at most two per 128-row tile
  const int64_t grid = std::min<int64_t>(a.num_sms, G::kUnitRows == 64 ? 2 * a.max_tiles : a.max_tiles);
  if (grid <= 0) return cudaSuccess;
  moe_gemm_kernel<ACT, EPI, AROWS><<<(unsigned)grid, kThreads, G::kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

// a_rows = 16: no tile has more routed rows; 64: 64-row work units (any routing); else 128.
// A4W4's larger stages gain no extra stage from a 64-row slot.
template <int EPI>
cudaError_t launch_epi(const GemmArgs& a, cudaStream_t s) {
  if (a.a_rows <= 16) return a.act_fmt == 0 ? launch_typed<0, EPI, 16>(a, s) : launch_typed<1, EPI, 16>(a, s);
  if (a.a_rows <= 64 && a.act_fmt == 0) return launch_typed<0, EPI, 64>(a, s);
  return a.act_fmt == 0 ? launch_typed<0, EPI, kRowTile>(a, s) : launch_typed<1, EPI, kRowTile>(a, s);
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s) {
  switch (a.epilogue) {
    case 0: return launch_epi<0>(a, s);
    case 1: return launch_epi<1>(a, s);
    case 2: return launch_epi<2>(a, s);  // GEMM1 writing bf16 h (the bf16-out form)
    case 3: return launch_epi<3>(a, s);  // GEMM2 rows as weighted FP8 (FP8 transport)
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
