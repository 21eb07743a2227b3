"""Failure detection without a GPU fault.

A wait that can never complete (the test hook MOE_TEST_STALL_PRODUCER stops the GEMM
producers from issuing, so no stage is ever filled) must expire after the short limit
MOE_WAIT_TIMEOUT_NS, be reported through the workspace status words, and leave the CUDA
context usable.  Runs in a child process because both variables are read once
per process.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
import torch
import block_scaled_moe_topk_gb300 as moe
import synth
dev = torch.device("cuda", 0)
s = synth.SHAPES[sys.argv[5]]
T = int(sys.argv[3])
W = synth.weights_codes(s.E, s.H, s.I, seed=0, device=dev)
prepacked = sys.argv[4] == "1"
if prepacked:
    t1, t2 = torch.empty_like(W[1]), torch.empty_like(W[3])
    moe.moe_prepack_scales(W[1], t1)
    moe.moe_prepack_scales(W[3], t2)
    W = (W[0], t1, W[2], t2)
x, lg = synth.x_bf16(T, s.H, 0, device=dev), synth.gate_logits(T, s.E, 0, device=dev)
out = torch.zeros(T, s.H, dtype=torch.bfloat16, device=dev)
ws = torch.zeros(moe.moe_workspace_bytes(T, s.H, s.I, s.E, s.k), dtype=torch.uint8, device=dev)
t0 = time.time()
moe.moe_forward_ex(x, lg, *W, out, s.E, s.k, ws, schedule=int(sys.argv[2]), weight_scales_prepacked=prepacked)
torch.cuda.synchronize()
dt = time.time() - t0
status = moe.moe_read_device_status(ws)
words = moe.workspace_views(ws, T, s.H, s.I, s.E, s.k)["status"].cpu().tolist()
alive = float((torch.arange(1000, device=dev, dtype=torch.float32) * 2).sum().item())
print(json.dumps({"status": status, "words": words, "alive": alive, "seconds": dt}))
"""


@pytest.mark.parametrize("schedule", ["chain", "fused", "split", "split_wide"])
def test_expired_wait_is_reported_and_the_context_survives(schedule):
    import __graft_entry__
    __graft_entry__.build()
    env = dict(os.environ, MOE_TEST_STALL_PRODUCER="1", MOE_WAIT_TIMEOUT_NS="50000000")  # 50 ms
    # split: T = 512 on the tiny shape with prepacked scales runs GEMM1 as the CTA-pair kernel
    # split_wide: the same on tiny_wide (N = 512), whose tail pass is the wide CTA-pair kernel
    sched, T, pp, shape = {"chain": (1, 16, 0, "tiny"), "fused": (2, 16, 0, "tiny"), "split": (1, 512, 1, "tiny"),
                           "split_wide": (1, 512, 1, "tiny_wide")}[schedule]
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, str(sched), str(T), str(pp), shape], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["status"] == 6  # MOE_ERR_DEVICE_TIMEOUT
    words = d["words"]
    assert words[1] == 1                 # an expiry was recorded
    # the first expiry: stage 0's full barrier in the MMA warp (index 0, warp 1) or the
    # accumulator-ready barrier in an epilogue warp (index 2 * stages = 12: the chain and fused
    # schedules run a 6-stage ring for 16-row slots; 2 * (5 + 8) = 26 in the CTA-pair kernel of a
    # split GEMM, which runs a 5-stage activation ring and an 8-stage weight ring), warps 2-9, or
    # -- fused schedule -- the combine's wait for every GEMM2 part in a CTA with no work of its own
    # (1000 + its sync word offset 1), whichever came first
    acc_ready = 26 if schedule.startswith("split") else 12
    ok = (words[2], words[5]) == (0, 1) or (words[2] == acc_ready and 2 <= words[5] <= 9)
    if schedule == "fused":
        ok = ok or (words[2] == 1001 and 2 <= words[5] <= 9)
    assert ok, words
    assert words[6] >= 25000             # it waited the limit (>= 50 ms at <= 2 GHz), in us
    assert d["alive"] == 999000.0        # the context still runs kernels
    assert d["seconds"] < 60
