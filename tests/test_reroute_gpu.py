"""Parity of overflow rerouting (MOE_FLAG_REROUTE) through the C ABI against
the CPU oracle.

A choice over its expert's capacity moves once to the token's next-best
expert (its j-th overflowing choice to its rank k+j expert) and takes the
capacity the k choices left, in (rank, token) priority.  Expert ids,
positions, counts, offsets and rows are bit-exact; gates within 1e-5
relative (rerouted gates are copied, so they match the router's bit for
bit); the layer output within the layer-dtype tolerance of the fp64 oracle
(1e-2 + 2e-2|o| bf16, 1e-5 + 1e-4|o| fp32).  Small cases check every
output; the 64-expert skewed shape checks every integer output and the
layer output on a seeded token sample.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import expert_parallelism_gemm_b300 as moe
import moe_inputs
import oracle
from moe_inputs import Workload
from tests.gpu_steps import Device, assert_close, assert_probs, host, t_dev

pytestmark = pytest.mark.gpu

CASES = {
    "rr_skew_8e": Workload("rr_skew_8e", T=1000, d=256, E=8, D=4, k=2, ffn=384, capacity_factor=1.0,
                           seed=81, zipf_s=1.5, reroute=True),
    "rr_top1_64e": Workload("rr_top1_64e", T=777, d=128, E=64, D=8, k=1, ffn=192, capacity_factor=1.0,
                            seed=82, zipf_s=1.2, reroute=True),
    "rr_k4_32e_shared": Workload("rr_k4_32e_shared", T=513, d=200, E=32, D=4, k=4, ffn=136,
                                 capacity_factor=0.5, seed=83, zipf_s=1.5, reroute=True, ffn_shared=136),
    "rr_fp32_gelu": Workload("rr_fp32_gelu", T=130, d=32, E=8, D=4, k=2, ffn=64, capacity_factor=0.6,
                             dtype="f32", act="gelu", seed=84, zipf_s=1.0, reroute=True),
    "rr_no_overflow": Workload("rr_no_overflow", T=300, d=64, E=8, D=2, k=2, ffn=64,
                               capacity_factor=math.inf, seed=85, reroute=True),
}
BIG = moe_inputs.WORKLOADS["skewed_64e"].with_(name="skewed_64e_reroute", reroute=True)


@pytest.fixture(scope="module", params=list(CASES) + ["skewed_64e_reroute"])
def case(request):
    wl = CASES.get(request.param) or BIG
    inp = moe_inputs.make_inputs(wl, device="cuda")
    cpu = inp.to("cpu")
    g, probs, idx, gate, fidx, fgate = oracle.route_fallback(cpu.x, cpu.Wg, cpu.bias, wl.k)
    rr = oracle.assign_reroute(idx, gate, fidx, fgate, wl.E, wl.D, wl.capacity_factor)
    yield wl, Device(inp), cpu, dict(probs=probs, idx=idx, gate=gate, fidx=fidx, fgate=fgate, rr=rr)
    torch.cuda.empty_cache()


def test_cases_exercise_rerouting(case):
    wl, dev, cpu, o = case
    rr = o["rr"]
    if math.isinf(wl.capacity_factor):
        assert rr.rerouted == 0 and rr.dropped == 0
    else:
        assert rr.rerouted > 0, "the case should overflow some expert"


def test_route_fallback(case):
    wl, dev, cpu, o = case
    T, k = wl.T, wl.k
    i32, f32 = torch.int32, torch.float32
    idx, gate = dev.empty((T, k), i32), dev.empty((T, k), f32)
    fidx, fgate = dev.empty((T, k), i32), dev.empty((T, k), f32)
    probs = dev.empty((T, wl.E), f32)
    moe.moe_route_fallback(dev.p, dev.inp.x, dev.inp.Wg, dev.inp.bias, idx, gate, fidx, fgate, probs)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), o["idx"])
    np.testing.assert_array_equal(fidx.cpu().numpy(), o["fidx"])
    assert_probs(gate.cpu().numpy(), o["gate"], "gate")
    assert_probs(fgate.cpu().numpy(), o["fgate"], "fallback gate")
    assert_probs(probs.cpu().numpy(), o["probs"], "probs")
    # the plain router's choices are the same
    idx2, _, _ = dev.route(want_probs=False)
    assert torch.equal(idx2, idx)


def _assign(dev, o, in_place):
    wl = dev.wl
    T, k, E, D = wl.T, wl.k, wl.E, wl.D
    i32 = torch.int32
    topk_idx, topk_gate = t_dev(o["idx"]), t_dev(o["gate"])
    out = dict(route_idx=topk_idx if in_place else torch.full((T, k), -7, dtype=i32, device="cuda"),
               route_gate=topk_gate if in_place else torch.full((T, k), -7.0, device="cuda"),
               slot_pos=torch.full((T, k), -7, dtype=i32, device="cuda"),
               counts_routed=dev.empty(E, i32), counts_kept=dev.empty(E, i32),
               expert_offsets=dev.empty(E + 1, i32), shard_offsets=dev.empty(D + 1, i32),
               shard_routed=dev.empty(D, i32), shard_overflow=dev.empty(D, i32),
               row_token=torch.full((max(dev.rows_max, 1),), -7, dtype=i32, device="cuda"),
               dropped=dev.empty(1, i32), rerouted=dev.empty(1, i32))
    moe.moe_assign_slots_reroute(dev.p, topk_idx, topk_gate, t_dev(o["fidx"]), t_dev(o["fgate"]),
                                 out["route_idx"], out["route_gate"], out["slot_pos"], out["counts_routed"],
                                 out["counts_kept"], out["expert_offsets"], out["shard_offsets"],
                                 out["shard_routed"], out["shard_overflow"], out["row_token"], out["dropped"],
                                 out["rerouted"], dev.ws, dev.ws_bytes)
    torch.cuda.synchronize()
    assert dev.status() == moe.MOE_OK
    return {n: v.cpu().numpy() for n, v in out.items()}


@pytest.mark.parametrize("in_place", [False, True])
def test_assign_slots_reroute(case, in_place):
    wl, dev, cpu, o = case
    rr = o["rr"]
    for _ in range(2):  # the second call reuses the workspace's histogram and ticket
        got = _assign(dev, o, in_place)
        for f in ("route_idx", "slot_pos", "counts_routed", "counts_kept", "expert_offsets", "shard_offsets",
                  "shard_routed", "shard_overflow"):
            np.testing.assert_array_equal(got[f], getattr(rr, f), err_msg=f)
        np.testing.assert_array_equal(got["route_gate"].view(np.uint32), rr.route_gate.view(np.uint32))
        n = int(rr.expert_offsets[-1])
        np.testing.assert_array_equal(got["row_token"][:n], rr.row_token)
        assert int(got["dropped"][0]) == rr.dropped and int(got["rerouted"][0]) == rr.rerouted


def test_layer_forward_reroute(case):
    wl, dev, cpu, o = case
    rr = o["rr"]
    resid = torch.randn(wl.T, wl.d, generator=torch.Generator().manual_seed(19)).to(dev.dtype)
    inp = dev.inp
    ys = []
    for _ in range(2):
        y = torch.empty(wl.T, wl.d, dtype=dev.dtype, device="cuda")
        moe.moe_layer_forward_shared(dev.p, inp.x, inp.Wg, inp.bias, inp.W1, inp.W3, inp.W2, inp.Ws1, inp.Ws3,
                                     inp.Ws2, resid.cuda(), y, dev.ws, dev.ws_bytes)
        torch.cuda.synchronize()
        assert dev.status() == moe.MOE_OK
        ys.append(y)
    # deterministic: the second step is the first bit for bit
    assert torch.equal(ys[0].view(torch.int16 if ys[0].dtype == torch.bfloat16 else torch.int32),
                       ys[1].view(torch.int16 if ys[1].dtype == torch.bfloat16 else torch.int32))
    Tk = wl.T * wl.k
    reg = lambda name, dt, n: dev.region(name, dt, n).cpu().numpy()
    np.testing.assert_array_equal(reg("topk_idx", torch.int32, Tk).reshape(wl.T, wl.k), rr.route_idx)
    np.testing.assert_array_equal(reg("slot_pos", torch.int32, Tk).reshape(wl.T, wl.k), rr.slot_pos)
    assert_probs(reg("topk_gate", torch.float32, Tk).reshape(wl.T, wl.k), rr.route_gate, "route gate")
    np.testing.assert_array_equal(reg("counts_kept", torch.int32, wl.E), rr.counts_kept)
    np.testing.assert_array_equal(reg("expert_offsets", torch.int32, wl.E + 1), rr.expert_offsets)
    n = int(rr.expert_offsets[-1])
    np.testing.assert_array_equal(reg("row_token", torch.int32, n), rr.row_token)
    assert int(reg("rerouted", torch.int32, 1)[0]) == rr.rerouted
    assert int(reg("dropped", torch.int32, 1)[0]) == rr.dropped
    if wl.name in CASES:
        toks = np.arange(wl.T)
    else:
        rng = np.random.default_rng(23)
        moved = np.unique(np.nonzero((rr.route_idx != o["idx"]).any(axis=1))[0])
        toks = np.unique(np.concatenate([rng.choice(wl.T, size=48, replace=False),
                                         rng.choice(moved, size=min(48, moved.size), replace=False),
                                         [0, wl.T - 1]]))
    act = oracle.act_code(wl.act)
    shared = (cpu.Ws1, cpu.Ws3, cpu.Ws2) if wl.ffn_shared else None
    want = oracle.token_outputs(toks, cpu.x, rr.route_idx, rr.slot_pos, rr.route_gate, cpu.W1, cpu.W3, cpu.W2,
                                act, residual=resid, shared=shared)
    assert_close(host(ys[0][torch.from_numpy(toks).cuda()]), want, wl.dtype, "y")
