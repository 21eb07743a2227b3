"""The allocation-free expert sort against the workspace one.

moe_sort_by_expert_noalloc serves callers that cannot hand the library scratch memory
(pre-planned device arenas, allocator-less plugin interfaces, hosts that must not pay
cudaMalloc's device-wide synchronisation).  Its scratch is a fixed array inside the
library that every call shares, so the check runs two different sorts back to back and
compares each, bit for bit, with moe_sort_by_expert given its own workspace.  This file
is collected last so that a run stopping at the first failure has run everything else.
"""
import numpy as np
import pytest
import torch

import block_scaled_moe_topk_gb300 as moe
import oracle
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()
    yield


def _outputs(T, E, k):
    return (torch.empty(E, dtype=torch.int32, device=DEV), torch.empty(E + 1, dtype=torch.int64, device=DEV),
            torch.empty(T * k, dtype=torch.int32, device=DEV), torch.empty(T * k, dtype=torch.int32, device=DEV))


def test_noalloc_sort_matches_workspace_sort_on_two_calls_in_a_row():
    # the larger sort first, so the second call runs over the first one's leftovers
    cases = [(32768, 384, 6, True, 1), (5000, 128, 3, False, 2)]
    for T, E, k, skew, seed in cases:
        ids_h, _ = oracle.route(synth.gate_logits(T, E, seed=seed, skew=skew).numpy(), k)
        ids = torch.from_numpy(ids_h).to(DEV)
        want = _outputs(T, E, k)
        ws = torch.empty(moe.moe_workspace_bytes(T, 128, 128, E, k), dtype=torch.uint8, device=DEV)
        moe.moe_sort_by_expert(ids, E, *want, ws)
        got = _outputs(T, E, k)
        for g in got:
            g.fill_(-7)
        moe.moe_sort_by_expert_noalloc(ids, E, *got)
        torch.cuda.synchronize()
        for a, b in zip(got, want):
            assert torch.equal(a, b), (T, E, k)
        assert moe.moe_read_device_status(ws) == 0


def test_noalloc_sort_skips_out_of_range_ids_like_the_workspace_sort():
    """Ids outside [0, E) are skipped by both sorts: counts, offsets and every written row of
    sorted_pair / inv agree; the pairs with bad ids are left untouched in both."""
    T, E, k = 3000, 128, 4
    ids_h, _ = oracle.route(synth.gate_logits(T, E, seed=11).numpy(), k)
    ids_h = ids_h.copy()
    bad = [(0, 0), (7, 3), (100, 1), (2999, 2)]
    for n, (t, j) in enumerate(bad):
        ids_h[t, j] = E + n if n % 2 == 0 else -1 - n
    ids = torch.from_numpy(ids_h).to(DEV)
    want, got = _outputs(T, E, k), _outputs(T, E, k)
    for a, b in zip(want, got):
        a.fill_(-7)
        b.fill_(-7)
    ws = torch.empty(moe.moe_workspace_bytes(T, 128, 128, E, k), dtype=torch.uint8, device=DEV)
    moe.moe_sort_by_expert(ids, E, *want, ws)
    moe.moe_sort_by_expert_noalloc(ids, E, *got)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 1  # MOE_ERR_INVALID_ARG from the workspace sort
    for a, b in zip(got, want):
        assert torch.equal(a, b)
    R = T * k - len(bad)
    assert int(got[1][-1].item()) == R
    inv = got[3].cpu().numpy()
    for t, j in bad:
        assert inv[t * k + j] == -7
    # a valid sort right after still matches (nothing of the bad call lingers)
    ids_ok = torch.from_numpy(oracle.route(synth.gate_logits(T, E, seed=12).numpy(), k)[0]).to(DEV)
    want, got = _outputs(T, E, k), _outputs(T, E, k)
    moe.moe_sort_by_expert(ids_ok, E, *want, ws)
    moe.moe_sort_by_expert_noalloc(ids_ok, E, *got)
    torch.cuda.synchronize()
    for a, b in zip(got, want):
        assert torch.equal(a, b)


def test_noalloc_sort_rejects_sizes_beyond_its_scratch():
    T, E, k = 300000, 1024, 1  # 4 * 1024 * ceil(300000 / 32) bytes > 4 MiB
    ids = torch.zeros(T, k, dtype=torch.int32, device=DEV)
    out = _outputs(T, E, k)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_sort_by_expert_noalloc(ids, E, *out)
    assert ei.value.status == 4  # MOE_ERR_WORKSPACE_TOO_SMALL, nothing launched
