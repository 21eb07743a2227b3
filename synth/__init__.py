"""Seeded synthetic inputs for the block-scaled MoE expert layer.

This module only draws random numbers.  It holds none of the layer's
arithmetic: no quantiser, no routing, no GEMM.  Both the CUDA path and the CPU
oracle consume exactly the tensors it returns.

Workload shapes follow the pages' layer shapes:
  * tiny:         H=256,  I=128,  E=8,   k=2  (T=16)
  * flash_decode: H=5120, I=640,  E=384, k=6  (DeepSeek-V4.1-Flash routed experts, TP4 shard;
                  "[HIP] gfx950 A8W4 fused_moe configs for DSv4.1 TP-sharded experts", Changes)
  * draft:        H=5120, I=1152, E=128, k=3  (DSpark draft experts, TP2 shard; same page)
  * pro:          H=7168, I=3072, E=384, k=6  (DeepSeek-V4-Pro; "add A4W4 and FP8 P2P transport
                  support to MegaMoE", Test Result: hidden/intermediate 7168/3072, experts/top-k 384/6)
  * flash_tp2:    H=5120, I=1152, E=384, k=6  and
  * draft_tp4:    H=5120, I=640,  E=128, k=3  -- the other two pairs of the tuned-shape grid
                  (per-rank inter 640 / 1152 x experts 384x6 / 128x3) of the aiter page, Changes

Sub-seeds, one per tensor: x = seed, logits = seed+1, expert bias = seed+2,
W1 = seed+3, W2 = seed+4.

Weights come in two forms:
  * ``weights_bf16``: raw bf16 draws N(0, 0.02) of W1 [E, 2I, H] and W2 [E, H, I]; the caller
    quantises them (the tests do so with the oracle's quantiser).
  * ``weights_codes``: MXFP4 weights drawn directly as codes -- every FP4 nibble uniform over the
    16 E2M1 codes, every E8M0 scale byte uniform over {119, 120, 121} (2^-8 .. 2^-6).  The
    resulting weight standard deviation is about 0.02, the spread of the N(0, 0.02) draws after
    quantisation.  This is the stand-in used where drawing and quantising gigabytes of bf16 on
    the host would take minutes (the 2-13.5 GB layer shapes).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

SCALE_BYTES = (119, 122)  # E8M0 scale bytes drawn uniformly from [119, 122)


@dataclass(frozen=True)
class Shape:
    name: str
    H: int
    I: int
    E: int
    k: int
    skew: bool = False  # add a per-expert N(0, 1.5) bias to the logits


SHAPES = {
    "tiny": Shape("tiny", 256, 128, 8, 2),
    # both GEMMs' N (2I, H) multiples of 512 and K (H, I) of 16 stages: the wide tail pass
    "tiny_wide": Shape("tiny_wide", 2048, 2048, 8, 2),
    "flash_decode": Shape("flash_decode", 5120, 640, 384, 6),
    "draft": Shape("draft", 5120, 1152, 128, 3, skew=True),
    "pro": Shape("pro", 7168, 3072, 384, 6),
    "pro_skew": Shape("pro_skew", 7168, 3072, 384, 6, skew=True),
    "flash_tp2": Shape("flash_tp2", 5120, 1152, 384, 6),
    "draft_tp4": Shape("draft_tp4", 5120, 640, 128, 3, skew=True),
}

TOKEN_SWEEPS = {
    "tiny": [16],
    "flash_decode": [1, 2, 4, 8, 16, 32, 64],
    "draft": [2 ** i for i in range(16)] + [3072, 24576],
    "pro": [1, 16, 128, 512, 1024, 4096, 8192, 16384, 32768],
    "pro_a4w4": [512, 1024, 8192],
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def x_bf16(T: int, H: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Token activations, bf16 N(0, 1), [T, H]."""
    g = _gen(seed, device)
    return torch.randn((T, H), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def gate_logits(T: int, E: int, seed: int = 0, skew: bool = False, device="cpu") -> torch.Tensor:
    """Router logits fp32 N(0, 1), [T, E]; with ``skew`` a per-expert N(0, 1.5) bias
    (drawn once from seed+2) is added, which concentrates load on a few experts."""
    g = _gen(seed + 1, device)
    lg = torch.randn((T, E), generator=g, device=device, dtype=torch.float32)
    if skew:
        gb = _gen(seed + 2, device)
        bias = torch.randn((E,), generator=gb, device=device, dtype=torch.float32) * 1.5
        lg = lg + bias[None, :]
    return lg


def weights_bf16(E: int, H: int, I: int, seed: int = 0, device="cpu", std: float = 0.02):
    """Raw bf16 weights N(0, std): W1 [E, 2I, H] (rows 2j gate_j, 2j+1 up_j) and W2 [E, H, I]."""
    g1 = _gen(seed + 3, device)
    w1 = (torch.randn((E, 2 * I, H), generator=g1, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    g2 = _gen(seed + 4, device)
    w2 = (torch.randn((E, H, I), generator=g2, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    return w1, w2


def _codes(shape_rows, K, gen, device):
    packed = torch.randint(0, 256, (*shape_rows, K // 2), generator=gen, device=device, dtype=torch.uint8)
    scales = torch.randint(SCALE_BYTES[0], SCALE_BYTES[1], (*shape_rows, K // 32), generator=gen,
                           device=device, dtype=torch.uint8)
    return packed, scales


def weights_codes(E: int, H: int, I: int, seed: int = 0, device="cpu"):
    """MXFP4 weights drawn directly as codes.

    Returns (w1 uint8 [E, 2I, H/2], w1s uint8 [E, 2I, H/32], w2 uint8 [E, H, I/2],
    w2s uint8 [E, H, I/32]); FP4 element 2i sits in the low nibble of byte i.
    """
    w1, w1s = _codes((E, 2 * I), H, _gen(seed + 3, device), device)
    w2, w2s = _codes((E, H), I, _gen(seed + 4, device), device)
    return w1, w1s, w2, w2s


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
