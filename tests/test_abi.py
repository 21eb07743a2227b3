"""The C-ABI library on the host: it loads without a GPU, exports every entry point the
public header declares, and its host-side validation and workspace sizing behave as
documented.  No call here launches a kernel."""
import ctypes
import os
import re

import pytest

import block_scaled_moe_topk_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _declared():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert {"moe_topk_route", "moe_a8w4_forward", "moe_a4w4_forward"} <= names
    lib = ctypes.CDLL(moe.LIB_PATH)
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings():
    for code, name in moe.STATUS_NAMES.items():
        assert moe.moe_status_string(code) == name
    assert moe.moe_status_string(99) == "MOE_UNKNOWN_STATUS"


def test_workspace_layout_and_bytes():
    L = moe.moe_get_workspace_layout(8192, 7168, 3072, 384, 6)
    R = 8192 * 6
    assert L.rows_cap % 128 == 0 and L.rows_cap >= R and L.rows_cap <= R + 127 * 384 + 127
    offs = [L.status, L.sync, L.topk_ids, L.topk_w, L.counts, L.offsets, L.padded_offsets, L.mtile_base,
            L.chunk_hist, L.sorted_pair, L.inv, L.inv_padded, L.xq, L.xs, L.a2, L.a2s, L.y2, L.sf_rot, L.part, L.y2f]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    assert L.y2 + 2 * 7168 * L.rows_cap <= L.sf_rot  # bf16 GEMM2 rows
    assert L.sf_rot + 7168 // 32 * L.rows_cap <= L.total  # rotated A-scale atoms of the split GEMMs
    assert L.part == L.y2f == L.total  # the fused schedule's buffers exist only for T <= 64
    assert L.sync == 256  # right after the status words (one memset clears both)
    small = moe.moe_get_workspace_layout(64, 7168, 3072, 384, 6)
    assert small.y2f - small.part >= 160 * 4 * 64 * 256 * 4  # partial slots: CTAs x 4 x 64 rows x 256
    assert small.total - small.y2f >= 64 * 6 * 7168 * 4      # fp32 GEMM2 rows
    assert moe.moe_workspace_bytes(8192, 7168, 3072, 384, 6) == L.total
    a4 = moe.moe_get_workspace_layout(8192, 7168, 3072, 384, 6, moe.MOE_ACT_MXFP4)
    assert a4.total < L.total and a4.part == a4.sf_rot  # A4W4 never splits: no rotated scales
    few = moe.moe_get_workspace_layout(1024, 7168, 3072, 384, 6)
    assert few.part == few.sf_rot  # at most 16 rows per expert on average: 64-row units, no split
    # rows_cap never exceeds R + 127 per active expert: T=1 routes to k experts
    L1 = moe.moe_get_workspace_layout(1, 7168, 3072, 384, 6)
    assert L1.rows_cap == 6 * 128
    assert moe.moe_workspace_bytes(0, 7168, 3072, 384, 6) > 0


@pytest.mark.parametrize("args,status", [
    ((16, 250, 128, 8, 2), 2),      # H not a multiple of 128
    ((16, 256, 96, 8, 2), 2),       # I not a multiple of 128
    ((16, 256, 128, 8, 9), 1),      # k > E
    ((16, 256, 128, 2048, 2), 2),   # E > 1024
    ((16, 256, 128, 16, 9), 2),     # k > 8
    ((-1, 256, 128, 8, 2), 1),      # negative T
])
def test_layout_rejects_bad_sizes(args, status):
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_get_workspace_layout(*args)
    assert ei.value.status == status
    assert moe.moe_workspace_bytes(*args) == 0


def test_forward_validation_before_any_launch():
    lib = moe.lib()
    f = lib.moe_a8w4_forward
    ok = ctypes.c_void_p(1 << 20)  # aligned dummy addresses: validation fails before any use
    # Only argument lists that fail host-side validation are ever passed: none of these
    # calls reaches a CUDA API call or a launch.
    args = [ok] * 7 + [16, 256, 128, 8, 2, ok, 1 << 30, None]
    bad = list(args)
    bad[0] = None
    assert f(*bad) == 1  # null x
    bad = list(args)
    bad[0] = ctypes.c_void_p((1 << 20) + 8)
    assert f(*bad) == 7  # misaligned x
    bad = list(args)
    bad[13] = 16
    assert f(*bad) == 4  # workspace too small
    bad = list(args)
    bad[8] = 250
    assert f(*bad) == 2  # H % 128
    bad = list(args)
    bad[11] = 9
    assert f(*bad) == 1  # k > E


def test_forward_launch_count():
    pro, flash = (7168, 3072), (5120, 640)
    assert moe.moe_forward_launch_count(0, *pro) == 0
    assert moe.moe_forward_launch_count(1, *pro) == 1      # fused decode kernel
    assert moe.moe_forward_launch_count(16, *pro) == 1
    assert moe.moe_forward_launch_count(17, *pro) == 5     # kernel chain, routing + sort in one kernel
    assert moe.moe_forward_launch_count(65, *pro) == 7
    assert moe.moe_forward_launch_count(2, *flash) == 1    # small I: fused only for T <= 2
    assert moe.moe_forward_launch_count(3, *flash) == 5
    assert moe.moe_forward_launch_count(1, 32768, 256) == 5  # H beyond the fused kernel's staged row
    assert moe.moe_forward_launch_count_ex(64, *pro, moe.MOE_SCHEDULE_CHAIN) == 5
    assert moe.moe_forward_launch_count_ex(65, *pro, moe.MOE_SCHEDULE_CHAIN) == 7
    assert moe.moe_forward_launch_count_ex(3, *flash, moe.MOE_SCHEDULE_FUSED) == 1
    assert moe.moe_forward_launch_count_ex(3, *flash, 9) == -1
    assert moe.moe_forward_launch_count_ex(3, *flash, moe.MOE_SCHEDULE_CHAIN_BF16_H) == 6
    assert moe.moe_forward_launch_count_ex(100, *pro, moe.MOE_SCHEDULE_CHAIN_BF16_H) == 8
    assert moe.moe_forward_launch_count_ex(65, *pro, moe.MOE_SCHEDULE_CHAIN_SINGLE_CTA) == 7
    # FP8 transport of the GEMM2 rows: the chain's kernels, its epilogue and combine in FP8 form
    assert moe.moe_forward_launch_count_ex(65, *pro, moe.MOE_SCHEDULE_CHAIN_FP8_Y2) == 7
    assert moe.moe_forward_launch_count_ex(3, *flash, moe.MOE_SCHEDULE_CHAIN_FP8_Y2) == 5


def test_forward_launch_count_with_split_gemms():
    """The exact count: a GEMM split into its pair kernel and tail pass (A8W4, prepacked scales,
    128-row tiles, N % 256 == 0, and N % 512 == 0 with T * k > 16 * E or T * k >= 128 * E) counts
    twice."""
    pro, a8, a4 = (7168, 3072), moe.MOE_ACT_MXFP8, moe.MOE_ACT_MXFP4
    auto, chain = moe.MOE_SCHEDULE_AUTO, moe.MOE_SCHEDULE_CHAIN
    cfg, split = moe.moe_forward_launch_count_cfg, moe.moe_forward_split_gemms
    assert (cfg(8192, *pro, 384, 6, a8, auto, True), split(8192, *pro, 384, 6, a8, auto, True)) == (9, 3)
    assert (cfg(8192, *pro, 384, 6, a8, chain, True), split(8192, *pro, 384, 6, a8, chain, True)) == (9, 3)
    assert (cfg(8191, *pro, 384, 6, a8, auto, True), split(8191, *pro, 384, 6, a8, auto, True)) == (9, 3)  # wide tails
    assert (cfg(1025, *pro, 384, 6, a8, auto, True), split(1025, *pro, 384, 6, a8, auto, True)) == (9, 3)
    assert (cfg(1024, *pro, 384, 6, a8, auto, True), split(1024, *pro, 384, 6, a8, auto, True)) == (7, 0)  # 64-row units
    # V4.1-Flash (5120/640): GEMM1's N = 1280 is no multiple of 512 and GEMM2's K = 640 is 5 stages,
    # so neither takes the wide tails: both split from 128 rows per expert on; the draft shape's GEMM1
    # (N = 2304, K = 5120) neither; GEMM2 of I = 2048 (K = 16 stages) does
    flash, draft = (5120, 640), (5120, 1152)
    assert (cfg(2048, *flash, 384, 6, a8, auto, True), split(2048, *flash, 384, 6, a8, auto, True)) == (7, 0)
    assert split(8192, *flash, 384, 6, a8, auto, True) == 3
    assert split(2048, *draft, 128, 3, a8, auto, True) == 0
    assert split(2048, 5120, 2048, 128, 3, a8, auto, True) == 3
    assert cfg(8192, *pro, 384, 6, a8, auto, False) == 7                     # canonical weight scales
    assert cfg(8192, *pro, 384, 6, a4, auto, True) == 7                      # A4W4
    assert cfg(8192, *pro, 384, 6, a8, moe.MOE_SCHEDULE_CHAIN_SINGLE_CTA, True) == 7
    assert cfg(8192, *pro, 384, 6, a8, moe.MOE_SCHEDULE_CHAIN_BF16_H, True) == 8
    fp8 = moe.MOE_SCHEDULE_CHAIN_FP8_Y2
    assert (cfg(8192, *pro, 384, 6, a8, fp8, True), split(8192, *pro, 384, 6, a8, fp8, True)) == (9, 3)
    assert (cfg(1, *pro, 384, 6, a8, auto, True), split(1, *pro, 384, 6, a8, auto, True)) == (1, 0)  # fused
    assert (cfg(0, *pro, 384, 6, a8, auto, True), split(0, *pro, 384, 6, a8, auto, True)) == (0, 0)
    # GEMM2 of H = 384 has a 128-column last N tile: only GEMM1 (N = 2I = 256) splits
    assert (cfg(512, 384, 128, 8, 2, a8, auto, True), split(512, 384, 128, 8, 2, a8, auto, True)) == (8, 1)
    assert split(512, 256, 128, 8, 2, a8, auto, True) == 3
    assert cfg(512, 256, 128, 8, 2, a8, 9, True) == -1 and split(512, 256, 128, 8, 2, 5, auto, True) == -1


def test_forward_ex_schedule_validation():
    """An unknown schedule value is rejected by host-side validation, before any CUDA call."""
    ok = (1 << 20)
    a = moe.ForwardArgs(act_fmt=0, prequantized=0, weight_scales_prepacked=0, x=ok, x_scale=None, gate_logits=ok,
                        w1=ok, w1_scale=ok, w2=ok, w2_scale=ok, out=ok, T=16, H=256, I=128, E=8, k=2, workspace=ok,
                        workspace_bytes=1 << 30, stream=None, schedule=7)
    assert moe.lib().moe_forward_ex(ctypes.byref(a)) == 1
    a.schedule = -1
    assert moe.lib().moe_forward_ex(ctypes.byref(a)) == 1
    a.schedule = moe.MOE_SCHEDULE_CHAIN_BF16_H
    a.I = 512  # h lives in the y2 region: I <= H
    a.workspace_bytes = moe.moe_workspace_bytes(16, 256, 512, 8, 2)
    assert moe.lib().moe_forward_ex(ctypes.byref(a)) == 2
    a.I = 128
    a.schedule = moe.MOE_SCHEDULE_FUSED
    a.T = 65  # the fused schedule takes at most 64 tokens
    a.workspace_bytes = moe.moe_workspace_bytes(65, 256, 128, 8, 2)
    assert moe.lib().moe_forward_ex(ctypes.byref(a)) == 2
