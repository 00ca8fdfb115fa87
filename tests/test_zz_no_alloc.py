"""GPU check of moe_assign_slots_static, the slot assignment for callers that
cannot allocate device memory (an operator inside a framework that owns all
device allocations, or a path that must avoid cudaMalloc's synchronisation).

Its scratch is a static device array shared by every call, so this file is
collected last: it must pass on its own in a fresh process and after every
other test.  Two calls in a row on the same stream (the second finds the
first one's leftovers in the array) must both reproduce, bit for bit, what
moe_assign_slots computes with a caller workspace.  The same holds for an
empty batch (T = 0: zero counts and offsets) and for a batch holding an
expert id outside [0, E), which both entry points count as no assignment and
report through their status words: moe_device_status for the workspace,
moe_assign_slots_static_status for the static array.
"""
import numpy as np
import pytest
import torch

import expert_parallelism_gemm_b300 as moe
import moe_inputs

pytestmark = pytest.mark.gpu

OUTS = ("slot_pos", "counts_routed", "counts_kept", "expert_offsets", "shard_offsets", "shard_routed",
        "shard_overflow", "row_token", "dropped")


def _outputs(wl, rows_max):
    i32 = torch.int32
    z = lambda n: torch.full(n, -7, dtype=i32, device="cuda")
    return dict(slot_pos=z((wl.T, wl.k)), counts_routed=z((wl.E,)), counts_kept=z((wl.E,)),
                expert_offsets=z((wl.E + 1,)), shard_offsets=z((wl.D + 1,)), shard_routed=z((wl.D,)),
                shard_overflow=z((wl.D,)), row_token=z((max(rows_max, 1),)), dropped=z((1,)))


@pytest.mark.parametrize("wl", [
    moe_inputs.Workload("static_skew", T=3000, d=128, E=64, D=8, k=2, ffn=128, capacity_factor=1.0,
                        seed=41, zipf_s=1.2),
    moe_inputs.Workload("static_top1", T=5000, d=128, E=128, D=8, k=1, ffn=128, capacity_factor=1.25,
                        seed=42),
], ids=lambda w: w.name)
def test_static_scratch_matches_workspace_version(wl):
    inp = moe_inputs.make_inputs(wl, device="cuda")
    p = moe.problem_of(wl)
    C, Cs, rows_max = moe.moe_capacity(p)
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    gate = torch.empty(wl.T, wl.k, dtype=torch.float32, device="cuda")
    moe.moe_route(p, inp.x, inp.Wg, inp.bias, idx, gate, None, None, 0)
    ws = moe.alloc_workspace(p, "cuda")
    ref = _outputs(wl, rows_max)
    moe.moe_assign_slots(p, idx, *[ref[n] for n in OUTS], ws, ws.numel())
    torch.cuda.synchronize()
    kept = int(ref["expert_offsets"][-1].item())
    for call in range(2):
        got = _outputs(wl, rows_max)
        moe.moe_assign_slots_static(p, idx, *[got[n] for n in OUTS])
        torch.cuda.synchronize()
        for n in OUTS:
            a, b = got[n], ref[n]
            if n == "row_token":
                a, b = a[:kept], b[:kept]
            assert torch.equal(a, b), f"call {call}: {n} differs"
    assert ref["dropped"].item() >= 0
    assert moe.moe_assign_slots_static_status() == moe.MOE_OK


def _compare_with_workspace_version(wl, idx):
    p = moe.problem_of(wl)
    C, Cs, rows_max = moe.moe_capacity(p)
    ws = moe.alloc_workspace(p, "cuda")
    ref = _outputs(wl, rows_max)
    moe.moe_assign_slots(p, idx, *[ref[n] for n in OUTS], ws, ws.numel())
    ws_status = moe.moe_device_status(ws)
    got = _outputs(wl, rows_max)
    moe.moe_assign_slots_static(p, idx, *[got[n] for n in OUTS])
    static_status = moe.moe_assign_slots_static_status()
    kept = int(ref["expert_offsets"][-1].item())
    for n in OUTS:
        a, b = got[n], ref[n]
        if n == "row_token":
            a, b = a[:kept], b[:kept]
        assert torch.equal(a, b), f"{n} differs"
    return ref, ws_status, static_status


def test_static_scratch_empty_batch():
    wl = moe_inputs.Workload("static_empty", T=0, d=64, E=16, D=4, k=2, ffn=64, capacity_factor=1.0)
    idx = torch.empty(0, wl.k, dtype=torch.int32, device="cuda")
    ref, ws_status, static_status = _compare_with_workspace_version(wl, idx)
    assert ws_status == static_status == moe.MOE_OK
    assert ref["counts_routed"].abs().sum().item() == 0 and ref["expert_offsets"].abs().sum().item() == 0
    assert int(ref["dropped"].item()) == 0


def test_static_scratch_reports_an_out_of_range_expert():
    # token 5's rank-1 choice names expert E, one past the last: both entry
    # points skip that assignment, and each reports it through its status
    wl = moe_inputs.Workload("static_bad_id", T=70, d=64, E=8, D=4, k=2, ffn=64, capacity_factor=1.0)
    g = torch.Generator().manual_seed(3)
    idx = torch.stack([torch.randperm(wl.E, generator=g)[:wl.k] for _ in range(wl.T)]).to(torch.int32)
    idx[5, 1] = wl.E
    idx = idx.cuda()
    assert moe.moe_assign_slots_static_status() == moe.MOE_OK  # nothing pending from earlier tests
    ref, ws_status, static_status = _compare_with_workspace_version(wl, idx)
    assert ws_status == moe.MOE_ERR_DEVICE
    assert static_status == moe.MOE_ERR_DEVICE
    assert int(ref["slot_pos"][5, 1].item()) == -1
    assert int(ref["counts_routed"].sum().item()) == wl.T * wl.k - 1
    # the read cleared the word, and a clean call leaves it clear
    assert moe.moe_assign_slots_static_status() == moe.MOE_OK
    idx[5, 1] = (int(idx[5, 0].item()) + 1) % wl.E
    _, ws_status, static_status = _compare_with_workspace_version(wl, idx)
    assert ws_status == static_status == moe.MOE_OK


def test_static_scratch_rejects_problems_beyond_its_size():
    # E * k * ceil(T / 32) = 256 * 8 * 1024 > 2^20 histogram entries
    p = moe.make_problem(T=32768, d=64, E=256, D=8, k=8, ffn=64, capacity_factor=1.0)
    A = torch.empty(1, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_assign_slots_static(p, *([A] * 10))
    assert ei.value.status == moe.MOE_ERR_WORKSPACE
