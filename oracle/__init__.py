"""CPU oracle for the block-scaled MoE top-k expert layer -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never loads it, and it
never loads the CUDA library: the two share no code.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64 accumulation, explicit
codebooks).  This module only compiles it with gcc and marshals numpy arrays
through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

FMT_E4M3 = 0  # MXFP8 activations (A8W4)
FMT_E2M1 = 1  # MXFP4 activations (A4W4) and all weights

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/liboracle.so (gcc, OpenMP if present)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", _LIB_PATH + ".tmp", _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)  # no OpenMP: single thread
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i64, i32, d = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_e2m1_decode.restype = d
        lib.oracle_e2m1_decode.argtypes = [i32]
        lib.oracle_e4m3_decode.restype = d
        lib.oracle_e4m3_decode.argtypes = [i32]
        lib.oracle_e8m0_decode.restype = d
        lib.oracle_e8m0_decode.argtypes = [i32]
        lib.oracle_mx_encode.restype = i32
        lib.oracle_mx_encode.argtypes = [d, i32]
        lib.oracle_mx_scale_byte.restype = i32
        lib.oracle_mx_scale_byte.argtypes = [ctypes.c_float, i32]
        lib.oracle_mx_quantize_block.restype = None
        lib.oracle_mx_quantize_block.argtypes = [P, i32, P, P]
        lib.oracle_quantize_rows_f32.restype = None
        lib.oracle_quantize_rows_f32.argtypes = [P, i64, i32, i32, P, P]
        lib.oracle_quantize_rows_bf16.restype = None
        lib.oracle_quantize_rows_bf16.argtypes = [P, i64, i32, i32, P, P]
        lib.oracle_dequantize_rows.restype = None
        lib.oracle_dequantize_rows.argtypes = [P, P, i64, i32, i32, P]
        lib.oracle_route.restype = None
        lib.oracle_route.argtypes = [P, i64, i32, i32, P, P]
        lib.oracle_sort.restype = None
        lib.oracle_sort.argtypes = [P, i64, i32, i32, P, P, P, P]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        lib.oracle_f64_to_bf16.argtypes = [d]
        lib.oracle_moe_forward.restype = i32
        lib.oracle_moe_forward.argtypes = [P, P, P, P, P, P, i64, i32, i32, i32, i32, i32, P, i64,
                                           P, P, P, P, P, i32]
        lib.oracle_moe_forward_opts.restype = i32
        lib.oracle_moe_forward_opts.argtypes = [P, P, P, P, P, P, i64, i32, i32, i32, i32, i32, P, i64,
                                                P, P, P, P, P, i32, i32]
        lib.oracle_max_threads.restype = i32
        lib.oracle_max_threads.argtypes = []
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return a


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def e2m1_decode(code: int) -> float:
    return float(_load().oracle_e2m1_decode(int(code)))


def e4m3_decode(code: int) -> float:
    return float(_load().oracle_e4m3_decode(int(code)))


def e8m0_decode(s: int) -> float:
    return float(_load().oracle_e8m0_decode(int(s)))


def mx_encode(y: float, fmt: int) -> int:
    """Nearest code (RNE, satfinite, signed zero kept) of an already-scaled value."""
    return int(_load().oracle_mx_encode(float(y), int(fmt)))


def mx_scale_byte(amax: float, fmt: int) -> int:
    return int(_load().oracle_mx_scale_byte(float(amax), int(fmt)))


def quantize_block(v, fmt: int):
    """32 fp32 values -> (codes uint8[32], one code per byte; scale byte)."""
    v = _c(np.asarray(v, dtype=np.float32), np.float32)
    assert v.size == 32
    codes = np.zeros(32, np.uint8)
    scale = np.zeros(1, np.uint8)
    _load().oracle_mx_quantize_block(_ptr(v), fmt, _ptr(codes), _ptr(scale))
    return codes, int(scale[0])


def code_bytes(K: int, fmt: int) -> int:
    return K if fmt == FMT_E4M3 else K // 2


def quantize_rows_f32(v, fmt: int):
    """fp32 [rows, K] -> (codes uint8 [rows, K or K/2], scales uint8 [rows, K/32])."""
    v = _c(np.asarray(v, dtype=np.float32), np.float32)
    rows, K = v.shape
    codes = np.zeros((rows, code_bytes(K, fmt)), np.uint8)
    scales = np.zeros((rows, K // 32), np.uint8)
    _load().oracle_quantize_rows_f32(_ptr(v), rows, K, fmt, _ptr(codes), _ptr(scales))
    return codes, scales


def quantize_rows_bf16(x_bits, fmt: int):
    """bf16 bit patterns uint16 [rows, K] -> (codes, scales) as quantize_rows_f32."""
    x_bits = _c(x_bits, np.uint16)
    rows, K = x_bits.shape
    codes = np.zeros((rows, code_bytes(K, fmt)), np.uint8)
    scales = np.zeros((rows, K // 32), np.uint8)
    _load().oracle_quantize_rows_bf16(_ptr(x_bits), rows, K, fmt, _ptr(codes), _ptr(scales))
    return codes, scales


def dequantize_rows(codes, scales, K: int, fmt: int):
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    rows = scales.shape[0]
    out = np.zeros((rows, K), np.float64)
    _load().oracle_dequantize_rows(_ptr(codes), _ptr(scales), rows, K, fmt, _ptr(out))
    return out


def route(logits, k: int):
    """fp32 [T, E] -> (ids int32 [T, k], w fp32 [T, k])."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    _load().oracle_route(_ptr(logits), T, E, k, _ptr(ids), _ptr(w))
    return ids, w


def sort(ids, E: int):
    """ids int32 [T, k] -> (counts int32[E], offsets int64[E+1], sorted_pair int32[R], inv int32[R])."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    R = T * k
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int64)
    sorted_pair = np.zeros(R, np.int32)
    inv = np.zeros(R, np.int32)
    _load().oracle_sort(_ptr(ids), T, k, E, _ptr(counts), _ptr(offsets), _ptr(sorted_pair), _ptr(inv))
    return counts, offsets, sorted_pair, inv


def f64_to_bf16(v: float) -> int:
    return int(_load().oracle_f64_to_bf16(float(v)))


def moe_forward(x_bits, logits, w1, w1s, w2, w2s, E: int, k: int, act_fmt: int, tokens=None,
                diagnostics: bool = False, nthreads: int | None = None, h_bf16: bool = False,
                y2_fp8: bool = False):
    """The whole expert layer for the listed tokens (all tokens if None).

    h_bf16: round the SwiGLU output h to bf16 before its MX quantisation (the bf16-out stage-1
    form of "[HIP] gfx950 A8W4 fused_moe configs for DSv4.1 TP-sharded experts", How the rows
    were chosen); by default h is quantised from fp32, as the fused stage-1 epilogue does.
    y2_fp8: the weighted GEMM2 rows w_j * y2 (fp32 product) travel as E4M3 codes with one E8M0
    scale per 1x32 block and the combine sums their dequantised values (the FP8 transport of the
    stage-2 rows in "add A4W4 and FP8 P2P transport support to MegaMoE", Technical Details);
    by default the fp32 rows are weighted and summed directly.

    x_bits uint16 [T, H] (bf16 bit patterns), logits fp32 [T, E],
    w1 uint8 [E, 2I, H/2], w1s uint8 [E, 2I, H/32], w2 uint8 [E, H, I/2], w2s uint8 [E, H, I/32].
    Returns out bf16 bits uint16 [n_tok, H]; with diagnostics also a dict of
    h fp32 [n_tok, k, I], a2 codes, a2 scales and y2 fp32 [n_tok, k, H].
    """
    x_bits = _c(x_bits, np.uint16)
    logits = _c(logits, np.float32)
    w1, w1s, w2, w2s = (_c(a, np.uint8) for a in (w1, w1s, w2, w2s))
    T, H = x_bits.shape
    I = w2.shape[2] * 2
    assert logits.shape == (T, E) and w1.shape == (E, 2 * I, H // 2) and w1s.shape == (E, 2 * I, H // 32)
    assert w2.shape == (E, H, I // 2) and w2s.shape == (E, H, I // 32)
    if tokens is None:
        tok = None
        n = T
    else:
        tok = _c(np.asarray(tokens, dtype=np.int64), np.int64)
        n = tok.size
        assert n == 0 or (tok.min() >= 0 and tok.max() < T)
    out = np.zeros((n, H), np.uint16)
    diag = None
    if diagnostics:
        diag = dict(h=np.zeros((n, k, I), np.float32),
                    a2=np.zeros((n, k, code_bytes(I, act_fmt)), np.uint8),
                    a2s=np.zeros((n, k, I // 32), np.uint8),
                    y2=np.zeros((n, k, H), np.float32))
    if nthreads is None:
        nthreads = max_threads()
    rc = _load().oracle_moe_forward_opts(
        _ptr(x_bits), _ptr(logits), _ptr(w1), _ptr(w1s), _ptr(w2), _ptr(w2s), T, H, I, E, k, act_fmt,
        _ptr(tok), n, _ptr(out),
        _ptr(diag["h"]) if diag else None, _ptr(diag["a2"]) if diag else None,
        _ptr(diag["a2s"]) if diag else None, _ptr(diag["y2"]) if diag else None, int(nthreads),
        (1 if h_bf16 else 0) | (2 if y2_fp8 else 0))
    if rc != 0:
        raise ValueError("oracle_moe_forward rejected its arguments")
    return (out, diag) if diagnostics else out


def bf16_bits_to_f32(bits):
    """uint16 bf16 patterns -> float32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
