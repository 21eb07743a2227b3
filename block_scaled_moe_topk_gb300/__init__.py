"""GB300-native block-scaled MoE top-k expert layer (A8W4 / A4W4).

A thin ctypes binding over ``libmoe_topk.so`` (the C ABI declared in
``include/moe_topk.h``).  Every function here only marshals torch tensors to
device pointers and sizes and raises on a non-zero status; every step of the
layer runs in the library's CUDA kernels.  There is no fallback: if the
library is missing the functions raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "MoeError", "MOE_ACT_MXFP8", "MOE_ACT_MXFP4", "MOE_SCHEDULE_AUTO", "MOE_SCHEDULE_CHAIN", "MOE_SCHEDULE_FUSED",
    "MOE_SCHEDULE_CHAIN_BF16_H", "MOE_SCHEDULE_CHAIN_SINGLE_CTA", "MOE_SCHEDULE_CHAIN_FP8_Y2", "lib", "moe_status_string", "moe_workspace_bytes",
    "moe_get_workspace_layout", "moe_topk_route", "moe_sort_by_expert", "moe_sort_by_expert_noalloc",
    "moe_quantize_mx", "moe_a8w4_forward",
    "moe_a4w4_forward", "moe_forward_ex", "moe_a8w4_forward_prequant", "moe_a4w4_forward_prequant", "moe_prepack_scales", "moe_a8w4_forward_prepacked", "moe_a4w4_forward_prepacked",
    "moe_read_device_status", "moe_forward_launch_count", "moe_forward_launch_count_ex", "moe_forward_launch_count_cfg",
    "moe_forward_split_gemms", "moe_profile_forward",
    "workspace_views",
]

MOE_ACT_MXFP8 = 0
MOE_ACT_MXFP4 = 1
MOE_SCHEDULE_AUTO = 0   # the library's choice for the shape and T
MOE_SCHEDULE_CHAIN = 1  # kernel chain, one CTA per 128 x 256 GEMM tile over the whole K
MOE_SCHEDULE_FUSED = 2  # T <= 64: the whole layer in one persistent kernel
MOE_SCHEDULE_CHAIN_BF16_H = 3  # kernel chain, GEMM1 writes bf16 h, a separate kernel requantises
MOE_SCHEDULE_CHAIN_SINGLE_CTA = 4  # kernel chain with single-CTA GEMM tiles only (no pair split)
MOE_SCHEDULE_CHAIN_FP8_Y2 = 5  # kernel chain, GEMM2 rows travel as weighted E4M3 + E8M0 scales
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_topk.so")

STATUS_NAMES = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE", 3: "MOE_ERR_UNSUPPORTED_DEVICE",
    4: "MOE_ERR_WORKSPACE_TOO_SMALL", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_DEVICE_TIMEOUT", 7: "MOE_ERR_MISALIGNED",
}


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")
        self.status = status


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "status", "sync", "topk_ids", "topk_w", "counts", "offsets", "padded_offsets", "mtile_base", "chunk_hist",
        "sorted_pair", "inv", "inv_padded", "xq", "xs", "a2", "a2s", "y2", "sf_rot", "part", "y2f", "total")] + [
        ("rows_cap", ctypes.c_int64), ("nchunk", ctypes.c_int64)]


class ForwardArgs(ctypes.Structure):
    _fields_ = [("act_fmt", ctypes.c_int), ("prequantized", ctypes.c_int), ("weight_scales_prepacked", ctypes.c_int),
                ("x", ctypes.c_void_p), ("x_scale", ctypes.c_void_p), ("gate_logits", ctypes.c_void_p),
                ("w1", ctypes.c_void_p), ("w1_scale", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("w2_scale", ctypes.c_void_p), ("out", ctypes.c_void_p), ("T", ctypes.c_int64), ("H", ctypes.c_int),
                ("I", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("stream", ctypes.c_void_p), ("schedule", ctypes.c_int)]


_lib = None


def lib():
    """Load libmoe_topk.so (built in-tree by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "(there is no non-CUDA fallback)")
    L = ctypes.CDLL(LIB_PATH)
    P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_status_string.argtypes = [i32]
    L.moe_get_workspace_layout.restype = i32
    L.moe_get_workspace_layout.argtypes = [i64, i32, i32, i32, i32, i32, ctypes.POINTER(WorkspaceLayout)]
    L.moe_workspace_bytes.restype = sz
    L.moe_workspace_bytes.argtypes = [i64, i32, i32, i32, i32, i32]
    L.moe_topk_route.restype = i32
    L.moe_topk_route.argtypes = [P, i64, i32, i32, P, P, P]
    L.moe_sort_by_expert.restype = i32
    L.moe_sort_by_expert.argtypes = [P, i64, i32, i32, P, P, P, P, P, sz, P]
    L.moe_quantize_mx.restype = i32
    L.moe_quantize_mx.argtypes = [P, i64, i32, i32, P, P, P]
    for name in ("moe_a8w4_forward", "moe_a4w4_forward", "moe_a8w4_forward_prepacked",
                 "moe_a4w4_forward_prepacked"):
        f = getattr(L, name)
        f.restype = i32
        f.argtypes = [P, P, P, P, P, P, P, i64, i32, i32, i32, i32, P, sz, P]
    L.moe_read_device_status.restype = i32
    L.moe_read_device_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_int)]
    L.moe_forward_launch_count.restype = i32
    L.moe_forward_launch_count.argtypes = [i64, i32, i32]
    L.moe_forward_launch_count_ex.restype = i32
    L.moe_forward_launch_count_ex.argtypes = [i64, i32, i32, i32]
    L.moe_forward_launch_count_cfg.restype = i32
    L.moe_forward_launch_count_cfg.argtypes = [i64, i32, i32, i32, i32, i32, i32, i32]
    L.moe_forward_split_gemms.restype = i32
    L.moe_forward_split_gemms.argtypes = [i64, i32, i32, i32, i32, i32, i32, i32]
    L.moe_profile_forward.restype = i32
    L.moe_profile_forward.argtypes = [i32, P, P, P, P, P, P, P, i64, i32, i32, i32, i32, P, sz, P, i32, i32,
                                      ctypes.POINTER(ctypes.c_float)]
    for name in ("moe_a8w4_forward_prequant", "moe_a4w4_forward_prequant"):
        f = getattr(L, name)
        f.restype = i32
        f.argtypes = [P, P, P, P, P, P, P, P, i64, i32, i32, i32, i32, P, sz, P]
    L.moe_forward_ex.restype = i32
    L.moe_forward_ex.argtypes = [ctypes.POINTER(ForwardArgs)]
    L.moe_prepack_scales.restype = i32
    L.moe_prepack_scales.argtypes = [P, i64, i32, P, P]
    _lib = L
    return L


def _check(status: int, where: str):
    if status != 0:
        raise MoeError(status, where)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def moe_get_workspace_layout(T, H, I, E, k, fmt=MOE_ACT_MXFP8) -> WorkspaceLayout:
    lay = WorkspaceLayout()
    _check(lib().moe_get_workspace_layout(int(T), int(H), int(I), int(E), int(k), int(fmt), ctypes.byref(lay)),
           "moe_get_workspace_layout")
    return lay


def moe_workspace_bytes(T, H, I, E, k, fmt=MOE_ACT_MXFP8) -> int:
    return int(lib().moe_workspace_bytes(int(T), int(H), int(I), int(E), int(k), int(fmt)))


def moe_forward_launch_count(T, H, I) -> int:
    return int(lib().moe_forward_launch_count(int(T), int(H), int(I)))


def moe_forward_launch_count_ex(T, H, I, schedule) -> int:
    return int(lib().moe_forward_launch_count_ex(int(T), int(H), int(I), int(schedule)))


def moe_forward_launch_count_cfg(T, H, I, E, k, fmt, schedule, prepacked_scales) -> int:
    return int(lib().moe_forward_launch_count_cfg(int(T), int(H), int(I), int(E), int(k), int(fmt), int(schedule),
                                                  int(bool(prepacked_scales))))


def moe_forward_split_gemms(T, H, I, E, k, fmt, schedule, prepacked_scales) -> int:
    return int(lib().moe_forward_split_gemms(int(T), int(H), int(I), int(E), int(k), int(fmt), int(schedule),
                                             int(bool(prepacked_scales))))


def moe_topk_route(gate_logits, k, topk_ids, topk_w, stream=None):
    """gate_logits fp32 [T, E] -> topk_ids int32 [T, k], topk_w fp32 [T, k] (outputs given)."""
    T, E = gate_logits.shape
    _check(lib().moe_topk_route(_p(gate_logits), T, E, int(k), _p(topk_ids), _p(topk_w), _stream(stream)),
           "moe_topk_route")


def moe_sort_by_expert(topk_ids, E, counts, offsets, sorted_pair, inv, workspace, stream=None):
    T, k = topk_ids.shape
    _check(lib().moe_sort_by_expert(_p(topk_ids), T, int(E), k, _p(counts), _p(offsets), _p(sorted_pair), _p(inv),
                                    _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_sort_by_expert")


def moe_sort_by_expert_noalloc(topk_ids, E, counts, offsets, sorted_pair, inv, stream=None):
    """moe_sort_by_expert for callers that cannot provide scratch memory: the library uses
    its own fixed 4 MiB device array instead of a workspace (see include/moe_topk.h)."""
    f = lib().moe_sort_by_expert_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    T, k = topk_ids.shape
    _check(f(_p(topk_ids), T, int(E), k, _p(counts), _p(offsets), _p(sorted_pair), _p(inv), _stream(stream)),
           "moe_sort_by_expert_noalloc")


def moe_quantize_mx(x, fmt, codes, scales, stream=None):
    rows, K = x.shape
    _check(lib().moe_quantize_mx(_p(x), rows, K, int(fmt), _p(codes), _p(scales), _stream(stream)),
           "moe_quantize_mx")


def _forward(name, x, gate_logits, w1, w1_scale, w2, w2_scale, out, E, k, workspace, stream):
    T, H = x.shape
    I = w2.shape[-1] * 2
    f = getattr(lib(), name)
    _check(f(_p(x), _p(gate_logits), _p(w1), _p(w1_scale), _p(w2), _p(w2_scale), _p(out), T, H, I, int(E), int(k),
             _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)), name)


def moe_a8w4_forward(x, gate_logits, w1, w1_scale, w2, w2_scale, out, E, k, workspace, stream=None):
    """x bf16 [T, H], gate_logits fp32 [T, E], w1 u8 [E, 2I, H/2], w1_scale u8 [E, 2I, H/32],
    w2 u8 [E, H, I/2], w2_scale u8 [E, H, I/32] -> out bf16 [T, H]."""
    _forward("moe_a8w4_forward", x, gate_logits, w1, w1_scale, w2, w2_scale, out, E, k, workspace, stream)


def moe_a4w4_forward(x, gate_logits, w1, w1_scale, w2, w2_scale, out, E, k, workspace, stream=None):
    _forward("moe_a4w4_forward", x, gate_logits, w1, w1_scale, w2, w2_scale, out, E, k, workspace, stream)


def _forward_prequant(name, xq, xq_scale, gate_logits, w1, w1_scale, w2, w2_scale, out, E, k, workspace, stream):
    T, H = out.shape
    I = w2.shape[-1] * 2
    f = getattr(lib(), name)
    _check(f(_p(xq), _p(xq_scale), _p(gate_logits), _p(w1), _p(w1_scale), _p(w2), _p(w2_scale), _p(out), T, H, I,
             int(E), int(k), _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)), name)


def moe_a8w4_forward_prequant(xq, xq_scale, gate_logits, w1, w1_scale, w2, w2_scale, out, E, k, workspace,
                              stream=None):
    """The A8W4 layer from prequantised activations: xq u8 [T, H] E4M3, xq_scale u8 [T, H/32]."""
    _forward_prequant("moe_a8w4_forward_prequant", xq, xq_scale, gate_logits, w1, w1_scale, w2, w2_scale, out, E, k,
                      workspace, stream)


def moe_a4w4_forward_prequant(xq, xq_scale, gate_logits, w1, w1_scale, w2, w2_scale, out, E, k, workspace,
                              stream=None):
    """The A4W4 layer from prequantised activations: xq u8 [T, H/2] E2M1, xq_scale u8 [T, H/32]."""
    _forward_prequant("moe_a4w4_forward_prequant", xq, xq_scale, gate_logits, w1, w1_scale, w2, w2_scale, out, E, k,
                      workspace, stream)


def moe_forward_ex(x, gate_logits, w1, w1_scale, w2, w2_scale, out, E, k, workspace, act_fmt=MOE_ACT_MXFP8,
                   x_scale=None, weight_scales_prepacked=False, stream=None, schedule=MOE_SCHEDULE_AUTO):
    """Any forward variant: bf16 x (x_scale None) or prequantised codes + scales; canonical or
    prepacked weight scales; the schedule (MOE_SCHEDULE_*)."""
    T, H = out.shape
    a = ForwardArgs(act_fmt=int(act_fmt), prequantized=int(x_scale is not None),
                    weight_scales_prepacked=int(bool(weight_scales_prepacked)), x=x.data_ptr(),
                    x_scale=None if x_scale is None else x_scale.data_ptr(), gate_logits=gate_logits.data_ptr(),
                    w1=w1.data_ptr(), w1_scale=w1_scale.data_ptr(), w2=w2.data_ptr(), w2_scale=w2_scale.data_ptr(),
                    out=out.data_ptr(), T=T, H=H, I=w2.shape[-1] * 2, E=int(E), k=int(k),
                    workspace=workspace.data_ptr(), workspace_bytes=workspace.numel() * workspace.element_size(),
                    stream=_stream(stream).value, schedule=int(schedule))
    _check(lib().moe_forward_ex(ctypes.byref(a)), "moe_forward_ex")


def moe_prepack_scales(scales, tiled, stream=None):
    """E8M0 scales [..., rows, K/32] (any leading dims) -> 128x4 tile layout into ``tiled`` (same bytes)."""
    K = scales.shape[-1] * 32
    rows = scales.numel() // (K // 32)
    _check(lib().moe_prepack_scales(_p(scales), rows, K, _p(tiled), _stream(stream)), "moe_prepack_scales")


def moe_a8w4_forward_prepacked(x, gate_logits, w1, w1_scale_tiled, w2, w2_scale_tiled, out, E, k, workspace,
                               stream=None):
    """moe_a8w4_forward with both weight-scale tensors prepacked by moe_prepack_scales."""
    _forward("moe_a8w4_forward_prepacked", x, gate_logits, w1, w1_scale_tiled, w2, w2_scale_tiled, out, E, k,
             workspace, stream)


def moe_a4w4_forward_prepacked(x, gate_logits, w1, w1_scale_tiled, w2, w2_scale_tiled, out, E, k, workspace,
                               stream=None):
    _forward("moe_a4w4_forward_prepacked", x, gate_logits, w1, w1_scale_tiled, w2, w2_scale_tiled, out, E, k,
             workspace, stream)


KERNEL_NAMES = ("route", "scan", "scatter", "quant", "gemm1", "gemm2", "combine")
KERNEL_NAMES_SMALL = ("route_sort", "quant", "gemm1", "gemm2", "combine")  # kernel chain, T <= 64
KERNEL_NAMES_FUSED = ("decode",)  # fused schedule
KERNEL_NAMES_BF16_H = ("route", "scan", "scatter", "quant", "gemm1", "requant", "gemm2", "combine")
KERNEL_NAMES_BF16_H_SMALL = ("route_sort", "quant", "gemm1", "requant", "gemm2", "combine")


def moe_profile_forward(fmt, x, gate_logits, w1, w1_scale, w2, w2_scale, out, E, k, workspace, stream=None,
                        prepacked_scales=False, schedule=MOE_SCHEDULE_AUTO):
    """One forward with a CUDA event between kernels; returns {kernel name: microseconds}."""
    T, H = x.shape
    I = w2.shape[-1] * 2
    n = moe_forward_launch_count_cfg(T, H, I, E, k, fmt, schedule, prepacked_scales)
    split = moe_forward_split_gemms(T, H, I, E, k, fmt, schedule, prepacked_scales)
    us = (ctypes.c_float * max(n, 1))()
    _check(lib().moe_profile_forward(int(fmt), _p(x), _p(gate_logits), _p(w1), _p(w1_scale), _p(w2), _p(w2_scale),
                                     _p(out), T, H, I, int(E), int(k), _p(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream),
                                     int(bool(prepacked_scales)), int(schedule), us),
           "moe_profile_forward")
    n_base = n - bin(max(split, 0)).count("1")
    if schedule == MOE_SCHEDULE_CHAIN_BF16_H:
        names = KERNEL_NAMES_BF16_H if n_base == len(KERNEL_NAMES_BF16_H) else KERNEL_NAMES_BF16_H_SMALL
    else:
        names = {len(KERNEL_NAMES): KERNEL_NAMES, len(KERNEL_NAMES_SMALL): KERNEL_NAMES_SMALL,
                 1: KERNEL_NAMES_FUSED}[n_base]
    # a split GEMM: its pair kernel, then its tail pass
    expand = {"gemm1": ("gemm1_pairs", "gemm1_tails") if split & 1 else ("gemm1",),
              "gemm2": ("gemm2_pairs", "gemm2_tails") if split & 2 else ("gemm2",)}
    names = [m for nm in names for m in expand.get(nm, (nm,))]
    assert len(names) == n
    return {names[i]: float(us[i]) for i in range(n)}


def moe_read_device_status(workspace, stream=None) -> int:
    st = ctypes.c_int(0)
    _check(lib().moe_read_device_status(_p(workspace), _stream(stream), ctypes.byref(st)), "moe_read_device_status")
    return int(st.value)


def workspace_views(workspace, T, H, I, E, k, fmt=MOE_ACT_MXFP8):
    """Typed views of the forward's intermediates inside a uint8 workspace tensor."""
    L = moe_get_workspace_layout(T, H, I, E, k, fmt)
    R = T * k
    hb = H if fmt == MOE_ACT_MXFP8 else H // 2
    ib = I if fmt == MOE_ACT_MXFP8 else I // 2
    rc = L.rows_cap

    def v(off, n, dtype):
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return workspace[off:off + nbytes].view(dtype)

    return dict(
        layout=L,
        topk_ids=v(L.topk_ids, R, torch.int32).view(T, k), topk_w=v(L.topk_w, R, torch.float32).view(T, k),
        counts=v(L.counts, E, torch.int32), offsets=v(L.offsets, E + 1, torch.int64),
        padded_offsets=v(L.padded_offsets, E + 1, torch.int64), mtile_base=v(L.mtile_base, E + 1, torch.int32),
        sorted_pair=v(L.sorted_pair, R, torch.int32), inv=v(L.inv, R, torch.int32),
        inv_padded=v(L.inv_padded, R, torch.int32), xq=v(L.xq, rc * hb, torch.uint8).view(rc, hb),
        xs=v(L.xs, rc * H // 32, torch.uint8), a2=v(L.a2, rc * ib, torch.uint8).view(rc, ib),
        a2s=v(L.a2s, rc * I // 32, torch.uint8), y2=v(L.y2, rc * H, torch.bfloat16).view(rc, H),
        status=v(L.status, 8, torch.int32))
