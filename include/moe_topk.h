/*
 * moe_topk.h -- C ABI of the GB300 (sm_103a) block-scaled MoE top-k expert layer.
 *
 * The layer (all steps run in this library's CUDA kernels, on the caller's stream):
 *   1. top-k softmax gating over E experts;
 *   2. a stable sort of the T*k (token, slot) pairs by expert, 64-bit offsets;
 *   3. BF16 -> MXFP8 (E4M3) or MXFP4 (E2M1) activation quantisation, one E8M0
 *      scale per 1x32 block;
 *   4. grouped GEMM1 against gate/up-interleaved MXFP4 weights on the tcgen05
 *      block-scaled tensor cores, with SwiGLU and the requantisation of the
 *      intermediate activation (A2) fused into its epilogue;
 *   5. grouped GEMM2 against MXFP4 weights;
 *   6. the top-k-weighted FP32 combine back to token order, rounded to BF16.
 *
 * Sources for the operation (page titles and sections):
 *   - "feat(moe): FlyDSL MegaMoE fused EP-MoE integration" (ATOM PR #1666),
 *     description: the expert step is dispatch+gemm1+quant+gemm2+combine;
 *     w1 gate/up rows are INTERLEAVE(g1u1) (row 2j gate_j, row 2j+1 up_j);
 *     the expert count is passed explicitly, never inferred from weight shapes;
 *     per-layer weight pointers are swapped per call; the forward must be
 *     CUDA-graph capturable; more than 8192 batched tokens overflowed an int32
 *     kernel argument (hence 64-bit offsets here).
 *   - "add A4W4 and FP8 P2P transport support to MegaMoE" (FlyDSL PR #972),
 *     Technical Details: BF16 activations quantised with per-1x32 E8M0 scales,
 *     FP4 A2 activations and scales emitted for an FP4 x FP4 GEMM2, top-k
 *     contributions accumulated in FP32; Test Plan: "prequant" and "BF16"
 *     end-to-end variants.
 *   - "[HIP] gfx950 A8W4 fused_moe configs for DSv4.1 TP-sharded experts"
 *     (aiter PR #6125), Motivation/Changes: MXFP4 routed experts run with
 *     MXFP8 activations (A8W4); the top-k softmax kernel.
 *
 * Data formats (OCP Microscaling v1.0):
 *   MXFP4 weights: E2M1 codes, two per byte, element 2i in the LOW nibble of
 *   byte i; one E8M0 scale byte (value 2^(s-127)) per 32 consecutive elements
 *   along K, row-major [rows, K/32].  MXFP8 activations: one E4M3 byte per
 *   element with the same scales.  Scale rule: s = floor(log2 amax) - emax +
 *   127 clamped to [0, 254] (emax 8 for E4M3, 2 for E2M1); elements rounded to
 *   nearest even and saturated; a block whose amax is zero or fp32-subnormal
 *   gets s = 0 and signed-zero codes.
 *
 * Ownership and execution:
 *   - The caller owns every buffer (inputs, outputs, weights, workspace); all
 *     pointers are DEVICE pointers unless stated otherwise.  The library never
 *     allocates, frees or synchronises inside a compute call; it only enqueues
 *     kernels on `stream` (a cudaStream_t passed as void*, NULL = legacy
 *     default stream).
 *   - Arguments are validated before anything is launched.  On any error the
 *     call returns a non-zero moe_status_t, launches nothing and leaves the
 *     outputs untouched.  A launch failure returns MOE_ERR_CUDA.
 *   - Conditions only the device can see (a bounded wait that expired inside a
 *     kernel) are recorded in a status word inside the workspace; read it with
 *     moe_read_device_status after the stream has finished.
 *   - No call throws, traps or aborts.  Kernels never __trap().
 *   - Environment (read once per process): MOE_WAIT_TIMEOUT_NS bounds every in-kernel wait
 *     (default 4 s); MOE_TEST_STALL_PRODUCER=1 is a test hook that makes the GEMM producers
 *     issue nothing, so a forward ends with MOE_ERR_DEVICE_TIMEOUT in its status word.
 *   - The forward calls may be captured into a CUDA graph; a captured graph is
 *     valid only for the pointers and sizes it was captured with.
 *   - Supported device: compute capability 10.3 (sm_103a) only.
 */
#ifndef MOE_TOPK_H_
#define MOE_TOPK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,          /* null pointer, negative size, k > E, ... */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,    /* H or I not a multiple of 128, E > 1024, k > 8 */
  MOE_ERR_UNSUPPORTED_DEVICE = 3,   /* current device is not compute capability 10.3 */
  MOE_ERR_WORKSPACE_TOO_SMALL = 4,  /* workspace_bytes < moe_workspace_bytes(...) */
  MOE_ERR_CUDA = 5,                 /* a CUDA runtime/driver call or a launch failed */
  MOE_ERR_DEVICE_TIMEOUT = 6,       /* a bounded in-kernel wait expired (device status) */
  MOE_ERR_MISALIGNED = 7            /* a pointer misses its required alignment */
} moe_status_t;

typedef enum {
  MOE_ACT_MXFP8 = 0, /* E4M3 activation codes, one byte per element (A8W4) */
  MOE_ACT_MXFP4 = 1  /* E2M1 activation codes, two per byte (A4W4)         */
} moe_act_fmt_t;

/*
 * How a forward call schedules its work (moe_forward_ex, moe_profile_forward).
 *   MOE_SCHEDULE_CHAIN  the kernel chain: routing + sort, quantiser, GEMM1, GEMM2, combine;
 *                       each GEMM runs one CTA per 128-row x 256-column tile over the whole K;
 *                       GEMM2 rows are stored as bf16 before the combine.  With A8W4,
 *                       prepacked weight scales, 128-row tiles and an N (2I for GEMM1, H for
 *                       GEMM2) that is a multiple of 256, a GEMM runs as two kernels -- the
 *                       experts' whole pairs of M tiles on CTA pairs (cta_group::2), then a tail
 *                       pass over each expert's odd last M tile -- when either
 *                         N is a multiple of 512, K (H for GEMM1, I for GEMM2) at least 2048 and
 *                         T * k > 16 * E: the tail pass runs 512-column tiles on CTA pairs; or
 *                         T * k >= 128 * E: otherwise the tail pass runs on single CTAs.
 *                       Bit-identical to CHAIN_SINGLE_CTA, and faster.
 *   MOE_SCHEDULE_CHAIN_SINGLE_CTA  the kernel chain with single-CTA GEMM tiles throughout.
 *   MOE_SCHEDULE_FUSED  T <= 64 and H <= 16384 only (else MOE_ERR_UNSUPPORTED_SHAPE): the whole layer in one
 *                       persistent kernel on every SM ("feat(moe): FlyDSL MegaMoE fused EP-MoE
 *                       integration", description: one fused step for dispatch + gemm1 + quant
 *                       + gemm2 + combine).  Each CTA routes and sorts the batch itself; the
 *                       K stages of each GEMM are split evenly over the CTAs, partial
 *                       accumulators of an item cut between CTAs are summed in CTA order by
 *                       the last contributor (deterministic); GEMM2 rows stay fp32 up to the
 *                       combine.  Preceded by a memset of the workspace's status and sync words.
 *   MOE_SCHEDULE_CHAIN_BF16_H  the kernel chain with GEMM1 in its bf16-out form: the GEMM1
 *                       epilogue writes h = SwiGLU(acc) as bf16 rows and a separate kernel
 *                       requantises them into A2 ("[HIP] gfx950 A8W4 fused_moe configs for
 *                       DSv4.1 TP-sharded experts", How the rows were chosen: the bf16-out stage-1
 *                       family against the fused-quant one).  h is rounded to bf16 before its MX
 *                       quantisation, so A2 can differ from the fused epilogue's in a few codes.
 *                       Needs I <= H and I <= 16384 (h is kept in the y2 region), else
 *                       MOE_ERR_UNSUPPORTED_SHAPE.  One kernel more than CHAIN.
 *   MOE_SCHEDULE_CHAIN_FP8_Y2  the kernel chain with the GEMM2 rows in FP8 transport form ("add
 *                       A4W4 and FP8 P2P transport support to MegaMoE", Technical Details): GEMM2's
 *                       epilogue multiplies each row by its routing weight and writes it as E4M3
 *                       codes with one E8M0 scale per 1x32 block; the combine sums the dequantised
 *                       rows in fp32 in slot order.  Half the bytes of the bf16 rows, at E4M3
 *                       precision: the output differs from the other schedules by ~3 % (relative
 *                       Frobenius error) and matches the FP8-transport form of the layer.  The
 *                       GEMMs split as in CHAIN; the same number of kernels.
 *   MOE_SCHEDULE_AUTO   the library's choice (every named entry point uses this rule): FUSED
 *                       for T <= 2, and for T <= 16 when I >= 1024 (H <= 16384 in both cases),
 *                       CHAIN otherwise -- the faster of the two on the GB300 over the shapes
 *                       measured (with I = 640 the chain wins from 4-8 tokens on).
 * Every schedule computes the same routing, permutation and quantised activations bit for
 * bit; outputs agree within the parity tolerance of the layer (CHAIN_FP8_Y2: of its FP8
 * transport form), and each schedule is deterministic (repeated calls give the same bits).
 */
typedef enum {
  MOE_SCHEDULE_AUTO = 0,
  MOE_SCHEDULE_CHAIN = 1,
  MOE_SCHEDULE_FUSED = 2,
  MOE_SCHEDULE_CHAIN_BF16_H = 3,
  MOE_SCHEDULE_CHAIN_SINGLE_CTA = 4,
  MOE_SCHEDULE_CHAIN_FP8_Y2 = 5
} moe_schedule_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(moe_status_t status);

/*
 * Byte offsets of the intermediates inside the forward's workspace, so that
 * tests and tools can read the forward's own routing, permutation and
 * quantised activations.  All offsets are 256-byte aligned.
 *   topk_ids     int32 [T, k]      expert of slot j of token t
 *   topk_w       fp32  [T, k]      renormalised routing weight
 *   counts       int32 [E]         rows routed to each expert
 *   offsets      int64 [E+1]       exclusive prefix of counts (unpadded)
 *   padded_offsets int64 [E+1]     prefix of counts rounded up to 128 rows
 *   mtile_base   int32 [E+1]       prefix of 128-row tiles per expert
 *   chunk_hist   int32 [E, nchunk] per-chunk expert histogram (sort scratch)
 *   sorted_pair  int32 [T*k]       pair q = t*k+j of the r-th row in (expert, q) order
 *   inv          int32 [T*k]       inverse of sorted_pair: unpadded row of pair q
 *   inv_padded   int32 [T*k]       padded row of pair q (row index into xq/a2/y2)
 *   xq           u8 [rows_cap, H or H/2]   activation codes in padded expert order
 *   xs           u8 [rows_cap/128][H/128][512]  their E8M0 scales, 128x4 tile layout
 *   a2           u8 [rows_cap, I or I/2]   requantised SwiGLU output codes
 *   a2s          u8 [rows_cap/128][I/128][512]  their scales, same tile layout
 *   y2           bf16 [rows_cap, H]        GEMM2 output rows (unweighted; fp32-accumulated,
 *                                          rounded to bf16 like the pages' reduced-precision
 *                                          stage-2 transport)
 *                MOE_SCHEDULE_CHAIN_FP8_Y2 lays out the same bytes as E4M3 codes of the
 *                weighted rows [rows_cap, H], then their E8M0 scales [rows_cap, H/32]
 *                (row-major), then at the next 256-byte boundary each padded row's routing
 *                weight, fp32 [rows_cap]
 *   sf_rot       u8 [rows_cap/128][max(H, I)/128][512]  scratch of the split GEMMs: the A-scale
 *                atoms of each expert's odd last M tile with their two 64-row halves swapped
 *                (GEMM1's, then GEMM2's); empty unless A8W4 and T * k > 16 * E
 *   part         fp32 partial accumulators of the fused schedule (T <= 64 only, else empty)
 *   y2f          fp32 [T*k, H] GEMM2 rows of the fused schedule, unpadded row order
 *                (T <= 64 only, else empty)
 *   sync         uint32 counters of the fused schedule, zeroed by the forward before its launch
 *   status       uint32[8]: [0] device status bits (read them with moe_read_device_status);
 *                [1..6] the first expired in-kernel wait, if any: [1] = 1 when recorded,
 *                [2] barrier index (1000 + word offset in `sync` for a counter of the fused
 *                schedule), [3] phase parity (counter target), [4] CTA, [5] warp,
 *                [6] microseconds waited
 * The 128x4 tile layout stores the scale of (row r, 32-block kb) at byte
 *   ((r/128)*(K/128) + kb/4)*512 + (r%32)*16 + ((r%128)/32)*4 + kb%4.
 */
typedef struct {
  size_t status, sync, topk_ids, topk_w, counts, offsets, padded_offsets, mtile_base, chunk_hist;
  size_t sorted_pair, inv, inv_padded, xq, xs, a2, a2s, y2, sf_rot, part, y2f;
  size_t total;      /* bytes needed == moe_workspace_bytes(...) */
  int64_t rows_cap;  /* padded row capacity (multiple of 128) */
  int64_t nchunk;    /* number of routing chunks (sort scratch width) */
} moe_workspace_layout_t;

/* Fill *layout for a problem size.  Returns MOE_ERR_INVALID_ARG /
 * MOE_ERR_UNSUPPORTED_SHAPE for sizes the forward would reject. */
moe_status_t moe_get_workspace_layout(int64_t T, int H, int I, int E, int k, moe_act_fmt_t fmt,
                                      moe_workspace_layout_t* layout);

/* Workspace bytes the forward needs for this size (0 for rejected sizes). */
size_t moe_workspace_bytes(int64_t T, int H, int I, int E, int k, moe_act_fmt_t fmt);

/*
 * Top-k softmax gating ("[HIP] gfx950 A8W4 fused_moe configs ...", Changes:
 * the top-k softmax kernel).  For each token t: experts ranked by fp32 logit,
 * descending, ties to the lower expert index; topk_ids[t, j] is the j-th
 * ranked expert; topk_w[t, j] = p_j / sum_{i<k} p_i with p the softmax of the
 * logits (the full softmax denominator cancels).
 *   gate_logits  fp32 [T, E] row-major, device
 *   topk_ids     int32 [T, k] out, device;  topk_w fp32 [T, k] out, device
 * 1 <= k <= 8, k <= E <= 1024, T >= 0 (T = 0 is a no-op).  A NaN logit ranks as
 * -inf (the method defines none), so topk_ids always holds k distinct experts;
 * the forward entry points route the same way.
 */
moe_status_t moe_topk_route(const float* gate_logits, int64_t T, int E, int k, int32_t* topk_ids,
                            float* topk_w, void* stream);

/*
 * Stable sort of the T*k routed pairs by expert (the local form of the
 * dispatch step of "feat(moe): FlyDSL MegaMoE fused EP-MoE integration").
 *   topk_ids     int32 [T, k] in, device (every id in [0, E))
 *   counts       int32 [E] out;  offsets int64 [E+1] out (offsets[E] = T*k)
 *   sorted_pair  int32 [T*k] out: pair q = t*k+j at row r, rows ordered by
 *                (expert ascending, q ascending)
 *   inv          int32 [T*k] out: inv[sorted_pair[r]] = r
 *   workspace    device scratch of at least moe_workspace_bytes(T, 128, 128, E, k,
 *                MOE_ACT_MXFP8) bytes (only its routing-size part is used)
 * Ids outside [0, E) are an error the device detects: they are skipped and
 * MOE_ERR_INVALID_ARG is written to the workspace status word.
 */
moe_status_t moe_sort_by_expert(const int32_t* topk_ids, int64_t T, int E, int k, int32_t* counts,
                                int64_t* offsets, int32_t* sorted_pair, int32_t* inv, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * moe_sort_by_expert without a workspace argument.  The pages have no counterpart to
 * this entry point; it exists for callers that cannot give the library scratch memory:
 * runtimes that plan every device buffer ahead of time and hand a kernel only its
 * inputs and outputs (fixed arenas in embedded or real-time deployments, plugin
 * interfaces of other frameworks that expose no allocator), and latency-critical hosts
 * that must not call cudaMalloc, which can synchronise the whole device.
 *   Same arguments, results and errors as moe_sort_by_expert, minus the workspace.
 *   Scratch: a fixed 4 MiB array inside the library, present on every GPU that loads
 *   it until the process exits.  It must hold 256 + 4 * E * ceil(T / 32) bytes;
 *   larger T * E is rejected with MOE_ERR_WORKSPACE_TOO_SMALL before anything runs
 *   (with E = 384 that allows T up to 87,360 tokens).
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call before any
 *   stream capture.  The address is cached per device and context: after
 *   cudaDeviceReset the next call looks it up again (again outside any capture).
 *   The call allocates nothing.
 *   Every call on a device shares the array: two calls whose kernels overlap on the
 *   GPU (different streams, or several host threads) race on it and must be
 *   serialised by the caller.  Ids outside [0, E) are skipped as in
 *   moe_sort_by_expert, but the flag they raise stays inside the library.
 */
moe_status_t moe_sort_by_expert_noalloc(const int32_t* topk_ids, int64_t T, int E, int k, int32_t* counts,
                                        int64_t* offsets, int32_t* sorted_pair, int32_t* inv, void* stream);

/*
 * MX quantisation of BF16 rows ("add A4W4 and FP8 P2P transport support to
 * MegaMoE", Technical Details: per-1x32 E8M0 scales).
 *   x_bf16   bf16 [rows, K] in, device, 16-byte aligned, K % 32 == 0
 *   codes    u8 out: MOE_ACT_MXFP8 -> [rows, K]; MOE_ACT_MXFP4 -> [rows, K/2]
 *   scales   u8 [rows, K/32] out, row-major E8M0
 */
moe_status_t moe_quantize_mx(const void* x_bf16, int64_t rows, int K, moe_act_fmt_t fmt, uint8_t* codes,
                             uint8_t* scales, void* stream);

/*
 * The whole expert layer with MXFP8 activations and MXFP4 weights (A8W4).
 *   x_bf16       bf16 [T, H]                       16-byte aligned
 *   gate_logits  fp32 [T, E]
 *   w1           MXFP4 [E, 2I, H/2]  row 2j = gate_j, row 2j+1 = up_j; 32-byte aligned
 *   w1_scale     E8M0  [E, 2I, H/32]               4-byte aligned
 *   w2           MXFP4 [E, H, I/2]                 32-byte aligned
 *   w2_scale     E8M0  [E, H, I/32]                4-byte aligned
 *   out_bf16     bf16 [T, H] out                   16-byte aligned
 *   T >= 0 tokens (0: no-op; x, logits and out may then be NULL), H and I
 *   multiples of 128, 1 <= k <= 8,
 *   k <= E <= 1024; E is the true expert count (never inferred).
 *   workspace    device, 256-byte aligned, >= moe_workspace_bytes(T,H,I,E,k,MOE_ACT_MXFP8)
 * Weights are read in place (canonical layout); nothing is cached between
 * calls, so per-layer weight pointers may change on every call.
 */
moe_status_t moe_a8w4_forward(const void* x_bf16, const float* gate_logits, const uint8_t* w1,
                              const uint8_t* w1_scale, const uint8_t* w2, const uint8_t* w2_scale,
                              void* out_bf16, int64_t T, int H, int I, int E, int k, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * As moe_a8w4_forward with MXFP4 activations and MXFP4 A2 (A4W4: "add A4W4
 * and FP8 P2P transport support to MegaMoE", Technical Details).  Needs
 * moe_workspace_bytes(..., MOE_ACT_MXFP4).
 */
moe_status_t moe_a4w4_forward(const void* x_bf16, const float* gate_logits, const uint8_t* w1,
                              const uint8_t* w1_scale, const uint8_t* w2, const uint8_t* w2_scale,
                              void* out_bf16, int64_t T, int H, int I, int E, int k, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * One-time rearrangement of MXFP4 weight scales for the *_prepacked forwards, the
 * analogue of the load-time scale shuffle of "feat(moe): FlyDSL MegaMoE fused EP-MoE
 * integration" (description: shuffle_scale_w4 for w1/w1_scale).  Only the scale bytes
 * move; the FP4 codes stay in their canonical layout.
 *   scales  E8M0 [rows, K/32] row-major in, device, 4-byte aligned (rows = E*2I for W1,
 *           E*H for W2; K = H for W1, I for W2)
 *   tiled   out, device, 16-byte aligned, rows*K/32 bytes: the 128x4 tile layout, the
 *           scale of (row r, 32-block kb) at ((r/128)*(K/128) + kb/4)*512 + (r%32)*16 +
 *           ((r%128)/32)*4 + kb%4
 *   rows % 128 == 0 and K % 128 == 0, else MOE_ERR_UNSUPPORTED_SHAPE.
 */
moe_status_t moe_prepack_scales(const uint8_t* scales, int64_t rows, int K, uint8_t* tiled, void* stream);

/*
 * moe_a8w4_forward / moe_a4w4_forward with w1_scale and w2_scale already in the tile
 * layout of moe_prepack_scales (16-byte aligned).  Identical results; the weight scales
 * then stream with two 512-byte bulk copies per pipeline stage instead of 4-byte gathers.
 */
moe_status_t moe_a8w4_forward_prepacked(const void* x_bf16, const float* gate_logits, const uint8_t* w1,
                                        const uint8_t* w1_scale_tiled, const uint8_t* w2,
                                        const uint8_t* w2_scale_tiled, void* out_bf16, int64_t T, int H, int I,
                                        int E, int k, void* workspace, size_t workspace_bytes, void* stream);
moe_status_t moe_a4w4_forward_prepacked(const void* x_bf16, const float* gate_logits, const uint8_t* w1,
                                        const uint8_t* w1_scale_tiled, const uint8_t* w2,
                                        const uint8_t* w2_scale_tiled, void* out_bf16, int64_t T, int H, int I,
                                        int E, int k, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The "prequant" forward ("add A4W4 and FP8 P2P transport support to MegaMoE", Test
 * Plan: prequant end-to-end, i.e. without the activation quantisation): x arrives already
 * quantised, as moe_quantize_mx writes it.
 *   xq        A8W4: E4M3 codes [T, H]; A4W4: E2M1 codes [T, H/2]; 16-byte aligned
 *   xq_scale  E8M0 [T, H/32] row-major
 * Everything else as moe_a8w4_forward / moe_a4w4_forward (canonical weight scales).  The
 * quantiser kernel is replaced by a copy of each token's codes to its k expert rows.
 */
moe_status_t moe_a8w4_forward_prequant(const uint8_t* xq, const uint8_t* xq_scale, const float* gate_logits,
                                       const uint8_t* w1, const uint8_t* w1_scale, const uint8_t* w2,
                                       const uint8_t* w2_scale, void* out_bf16, int64_t T, int H, int I, int E,
                                       int k, void* workspace, size_t workspace_bytes, void* stream);
moe_status_t moe_a4w4_forward_prequant(const uint8_t* xq, const uint8_t* xq_scale, const float* gate_logits,
                                       const uint8_t* w1, const uint8_t* w1_scale, const uint8_t* w2,
                                       const uint8_t* w2_scale, void* out_bf16, int64_t T, int H, int I, int E,
                                       int k, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Every forward variant through one argument block: activation format, bf16 or
 * prequantised input (x_scale then required), canonical or prepacked weight scales.
 * Fields and rules as in the named entry points above.
 */
typedef struct {
  moe_act_fmt_t act_fmt;
  int prequantized;             /* 0: x is bf16 [T, H]; 1: x is codes, x_scale their E8M0 scales */
  int weight_scales_prepacked;  /* 0: canonical [rows, K/32]; 1: moe_prepack_scales layout */
  const void* x;
  const uint8_t* x_scale;
  const float* gate_logits;
  const uint8_t* w1;
  const uint8_t* w1_scale;
  const uint8_t* w2;
  const uint8_t* w2_scale;
  void* out;
  int64_t T;
  int H, I, E, k;
  void* workspace;
  size_t workspace_bytes;
  void* stream;
  int schedule;                 /* moe_schedule_t; any other value is MOE_ERR_INVALID_ARG */
} moe_forward_args_t;
moe_status_t moe_forward_ex(const moe_forward_args_t* args);

/*
 * Read the device status word a forward (or sort) left in `workspace`.
 * Synchronises `stream`, then copies 4 bytes to the host.  *status_out gets
 * MOE_OK or the moe_status_t a kernel recorded (MOE_ERR_DEVICE_TIMEOUT,
 * MOE_ERR_INVALID_ARG).  Returns MOE_ERR_CUDA if the copy fails.
 */
moe_status_t moe_read_device_status(const void* workspace, void* stream, moe_status_t* status_out);

/* Number of kernels one forward call of T tokens, hidden size H and intermediate size I
 * launches under MOE_SCHEDULE_AUTO with canonical weight scales: 0 for T = 0, 1 when the fused
 * kernel is chosen, else the kernel chain's 5 (T <= 64: routing and sort in one kernel) or 7. */
int moe_forward_launch_count(int64_t T, int H, int I);

/* The same for a given schedule (moe_schedule_t), canonical weight scales; -1 for an unknown
 * schedule. */
int moe_forward_launch_count_ex(int64_t T, int H, int I, int schedule);

/* The exact count for any forward: E experts, top-k, activation format `fmt`, the schedule, and
 * whether the weight scales are prepacked (a GEMM split into its pair kernel and tail pass
 * counts as two launches, see MOE_SCHEDULE_CHAIN); -1 for an unknown schedule or format. */
int moe_forward_launch_count_cfg(int64_t T, int H, int I, int E, int k, int fmt, int schedule,
                                 int prepacked_scales);

/* Which GEMMs of that forward run split into their pair kernel and tail pass: bit 0 GEMM1,
 * bit 1 GEMM2 (0 for the fused schedule); -1 for an unknown schedule or format. */
int moe_forward_split_gemms(int64_t T, int H, int I, int E, int k, int fmt, int schedule, int prepacked_scales);

/*
 * Profiling form of the forward: enqueues exactly the launch sequence of
 * moe_a8w4_forward (fmt = MOE_ACT_MXFP8) or moe_a4w4_forward (MOE_ACT_MXFP4),
 * or of their *_prepacked forms when prepacked_scales != 0, under the
 * schedule `schedule` (moe_schedule_t, as in moe_forward_ex),
 * with a CUDA event recorded before the first kernel and after each kernel,
 * waits for the last event, and writes the duration of each kernel in
 * microseconds to kernel_us[moe_forward_launch_count_cfg(T, H, I, E, k, fmt, schedule,
 * prepacked_scales)] (HOST array), in launch order: route, scan, scatter, quant, gemm1, gemm2,
 * combine (chain, T > 64), route_sort, quant, gemm1, gemm2, combine (chain, T <= 64) or decode
 * (fused); the bf16-out chain adds requant after gemm1, and a split GEMM contributes two
 * entries (its pair kernel, then its tail pass).
 * Arguments and errors as for the forward; additionally synchronises on its
 * own events (so it is not graph-capturable) and creates/destroys them.
 */
moe_status_t moe_profile_forward(moe_act_fmt_t fmt, const void* x_bf16, const float* gate_logits,
                                 const uint8_t* w1, const uint8_t* w1_scale, const uint8_t* w2,
                                 const uint8_t* w2_scale, void* out_bf16, int64_t T, int H, int I, int E,
                                 int k, void* workspace, size_t workspace_bytes, void* stream,
                                 int prepacked_scales, int schedule, float* kernel_us);

#ifdef __cplusplus
}
#endif
#endif /* MOE_TOPK_H_ */
