"""Shared helpers for the parity tests: inputs, oracle runs and comparisons.

Inputs come from ``synth`` (seeded random numbers only).  Weights for the tiny
shape are bf16 draws quantised by the ORACLE's quantiser; larger shapes draw
MXFP4 codes directly.  Expected values always come from ``oracle``.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

TOL_REL = 5e-3       # relative Frobenius error of the bf16 output
TOL_COS = 0.9999     # per-row cosine similarity


def tile_sf_to_rows(buf, rows, K):
    """Scales stored in the 128x4 tile layout -> canonical [rows, K/32]."""
    buf = np.asarray(buf, dtype=np.uint8)
    r = np.arange(rows, dtype=np.int64)[:, None]
    kb = np.arange(K // 32, dtype=np.int64)[None, :]
    off = ((r // 128) * (K // 128) + kb // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4
    return buf[off]


def oracle_weights_from_bf16(E, H, I, seed=0):
    """bf16 N(0, 0.02) draws quantised to MXFP4 by the oracle (numpy arrays)."""
    w1b, w2b = synth.weights_bf16(E, H, I, seed)
    w1, w1s = oracle.quantize_rows_bf16(synth.bf16_bits(w1b).reshape(E * 2 * I, H), oracle.FMT_E2M1)
    w2, w2s = oracle.quantize_rows_bf16(synth.bf16_bits(w2b).reshape(E * H, I), oracle.FMT_E2M1)
    return (w1.reshape(E, 2 * I, H // 2), w1s.reshape(E, 2 * I, H // 32),
            w2.reshape(E, H, I // 2), w2s.reshape(E, H, I // 32))


class Weights:
    """MXFP4 weights resident on the GPU, with host copies for the oracle."""

    def __init__(self, E, H, I, seed=0, device="cuda", from_bf16=False):
        self.E, self.H, self.I = E, H, I
        if from_bf16:
            host = oracle_weights_from_bf16(E, H, I, seed)
            self.host = host
            self.dev = tuple(torch.from_numpy(np.ascontiguousarray(a)).to(device) for a in host)
        else:
            self.dev = synth.weights_codes(E, H, I, seed, device=device)
            self.host = tuple(t.cpu().numpy() for t in self.dev)
        self._prepacked = None

    def dev_prepacked(self):
        """The device weights with both scale tensors in the library's prepacked tile layout."""
        if self._prepacked is None:
            import block_scaled_moe_topk_gb300 as moe
            w1, w1s, w2, w2s = self.dev
            t1, t2 = torch.empty_like(w1s), torch.empty_like(w2s)
            moe.moe_prepack_scales(w1s, t1)
            moe.moe_prepack_scales(w2s, t2)
            self._prepacked = (w1, t1, w2, t2)
        return self._prepacked


def compare(got_bits, want_bits):
    """bf16 bit patterns (uint16) -> (relative Frobenius error, min per-row cosine)."""
    got = oracle.bf16_bits_to_f32(got_bits).astype(np.float64)
    want = oracle.bf16_bits_to_f32(want_bits).astype(np.float64)
    rel = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))
    ng, nw = np.linalg.norm(got, axis=1), np.linalg.norm(want, axis=1)
    ok = (ng > 0) & (nw > 0)
    cos = (got[ok] * want[ok]).sum(1) / (ng[ok] * nw[ok])
    assert np.array_equal(ng > 0, nw > 0), "zero rows differ"
    return rel, float(cos.min()) if cos.size else 1.0


def bits(t: torch.Tensor):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
