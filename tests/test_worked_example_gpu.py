"""The pages' worked example through the CUDA path (C ABI), fp32 and bf16.

"Expert Parallelism" (theinfinity.ai, Systems / Distributed), caption of the
capacity figure: 6 tokens, 8 experts on 4 devices, top-2, capacity 2; two
assignments are dropped and experts 1 and 8 (1-indexed) stay unused.  The
caption gives no per-token choices; tests/golden/worked_example.txt holds the
hand-built instance (logits 3 and 2 at a token's two choices, 0 elsewhere,
Wg = identity, so every logit is exact) and the values worked out by hand
from the capacity rule.  Every integer the fixture lists must come out of
moe_route, moe_assign_slots and moe_layer_forward bit for bit, the gates must
be e^3/(e^3+e^2+6) and e^2/(e^3+e^2+6), and the routing statistics must
reproduce their closed forms.  tests/golden/worked_example_reroute.txt is the
same instance with the notes page's fallback (a choice over capacity goes to
the token's next-best expert), rerouted by hand.
"""
import math

import numpy as np
import pytest
import torch

import expert_parallelism_gemm_b300 as moe
import oracle
from tests.conftest import read_golden
from tests.gpu_steps import assert_close

pytestmark = pytest.mark.gpu

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def _fixture(name):
    kv, lists = {}, {}
    for r in read_golden(name):
        if r[0] in ("choice", "dropped", "fallback", "rerouted"):
            lists.setdefault(r[0], []).append(tuple(int(v) for v in r[1:]))
        else:
            kv[r[0]] = r[1:]
    return kv, lists


def _instance(dtype, act="swiglu", ffn=64):
    kv, lists = _fixture("worked_example.txt")
    T, d, E, D, k = (int(kv[n][0]) for n in ("T", "d", "E", "D", "k"))
    c = float(kv["c"][0])
    x = torch.zeros(T, d)
    for t, e0, e1 in lists["choice"]:
        x[t, e0], x[t, e1] = 3.0, 2.0
    Wg = torch.eye(E, d)
    g = torch.Generator().manual_seed(7)
    W1 = torch.randn(E, ffn, d, generator=g) / math.sqrt(d)
    W3 = torch.randn(E, ffn, d, generator=g) / math.sqrt(d)
    W2 = torch.randn(E, d, ffn, generator=g) / math.sqrt(ffn)
    dt = DTYPES[dtype]
    tens = {n: v.to(dt).cuda() for n, v in dict(x=x, Wg=Wg, W1=W1, W3=W3, W2=W2).items()}
    p = moe.make_problem(T=T, d=d, E=E, D=D, k=k, ffn=ffn, capacity_factor=c, dtype=dtype, act=act)
    return kv, lists, p, tens


def _ints(v):
    return [int(a) for a in v]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_route_and_assign_reproduce_the_caption(dtype):
    kv, lists, p, t = _instance(dtype)
    T, E, k = p.T, p.E, p.k
    C, C_shard, rows_max = moe.moe_capacity(p)
    assert (C, C_shard) == (int(kv["C"][0]), int(kv["C_shard"][0]))
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    gate = torch.empty(T, k, dtype=torch.float32, device="cuda")
    probs = torch.empty(T, E, dtype=torch.float32, device="cuda")
    moe.moe_route(p, t["x"], t["Wg"], None, idx, gate, probs, None, 0)
    torch.cuda.synchronize()
    assert [tuple(r) for r in idx.cpu().tolist()] == [(e0, e1) for _, e0, e1 in lists["choice"]]
    z = math.exp(3) + math.exp(2) + 6
    np.testing.assert_allclose(gate[:, 0].cpu().numpy(), math.exp(3) / z, rtol=1e-5)
    np.testing.assert_allclose(gate[:, 1].cpu().numpy(), math.exp(2) / z, rtol=1e-5)
    # the printed values carry 7 decimals (rounding error up to 5e-8)
    np.testing.assert_allclose(gate[:, 0].cpu().numpy(), float(kv["gate0"][0]), rtol=1e-5, atol=5e-8)
    np.testing.assert_allclose(gate[:, 1].cpu().numpy(), float(kv["gate1"][0]), rtol=1e-5, atol=5e-8)

    ws = moe.alloc_workspace(p, "cuda")
    i32 = torch.int32
    o = dict(slot_pos=torch.empty(T, k, dtype=i32, device="cuda"),
             counts_routed=torch.empty(E, dtype=i32, device="cuda"),
             counts_kept=torch.empty(E, dtype=i32, device="cuda"),
             expert_offsets=torch.empty(E + 1, dtype=i32, device="cuda"),
             shard_offsets=torch.empty(p.D + 1, dtype=i32, device="cuda"),
             shard_routed=torch.empty(p.D, dtype=i32, device="cuda"),
             shard_overflow=torch.empty(p.D, dtype=i32, device="cuda"),
             row_token=torch.full((rows_max,), -7, dtype=i32, device="cuda"),
             dropped=torch.empty(1, dtype=i32, device="cuda"))
    moe.moe_assign_slots(p, idx, *o.values(), ws, ws.numel())
    assert moe.moe_device_status(ws) == moe.MOE_OK
    got = {n: v.cpu() for n, v in o.items()}
    for n in ("counts_routed", "counts_kept", "expert_offsets", "shard_offsets", "shard_routed", "shard_overflow"):
        assert got[n].tolist() == _ints(kv[n]), n
    assert [e for e in range(E) if got["counts_routed"][e] == 0] == _ints(kv["unused_experts"])
    dropped = sorted((tt, r) for tt in range(T) for r in range(k) if got["slot_pos"][tt, r] < 0)
    assert dropped == sorted(lists["dropped"])
    assert int(got["dropped"].item()) == len(lists["dropped"]) == 2
    # every kept (t, r) sits at its expert's offset + position
    off = got["expert_offsets"]
    for tt in range(T):
        for r in range(k):
            pos = int(got["slot_pos"][tt, r])
            if pos >= 0:
                assert int(got["row_token"][int(off[int(idx[tt, r])]) + pos]) == tt

    # routing statistics: load-balancing term (16 e^3 + 12 e^2 + 44) / (9 S),
    # entropy of (e^3, e^2, 1 x 6) / S, 2 of 12 dropped, imbalance 3 / 1.5
    stats = torch.empty(moe.MOE_NUM_STATS, dtype=torch.float32, device="cuda")
    mean_prob = torch.empty(E, dtype=torch.float32, device="cuda")
    moe.moe_routing_stats(p, probs, o["counts_routed"], o["counts_kept"], stats, mean_prob, ws, ws.numel())
    torch.cuda.synchronize()
    e3, e2 = math.exp(3.0), math.exp(2.0)
    a, b, cc = e3 / z, e2 / z, 1.0 / z
    want = [(16 * e3 + 12 * e2 + 44) / (9 * z), -(a * math.log(a) + b * math.log(b) + 6 * cc * math.log(cc)),
            2 / 12, 3 / (12 / 8)]
    np.testing.assert_allclose(stats.cpu().numpy(), want, rtol=1e-5)
    np.testing.assert_allclose(mean_prob.cpu().numpy()[[0, 7]], cc, rtol=1e-5)


@pytest.mark.parametrize("dtype,act", [("f32", "swiglu"), ("bf16", "swiglu"), ("f32", "gelu")])
def test_layer_forward_reproduces_the_caption(dtype, act):
    kv, lists, p, t = _instance(dtype, act)
    T, E, k = p.T, p.E, p.k
    ws = moe.alloc_workspace(p, "cuda")
    y = torch.empty(T, p.d, dtype=DTYPES[dtype], device="cuda")
    W3 = t["W3"] if act == "swiglu" else None
    moe.moe_layer_forward(p, t["x"], t["Wg"], None, t["W1"], W3, t["W2"], None, y, ws, ws.numel())
    assert moe.moe_device_status(ws) == moe.MOE_OK
    view = lambda n, c: moe.workspace_view(ws, p, n, torch.int32, c).cpu()
    idx = view("topk_idx", T * k).reshape(T, k)
    assert [tuple(r) for r in idx.tolist()] == [(e0, e1) for _, e0, e1 in lists["choice"]]
    for n, c in (("counts_routed", E), ("counts_kept", E), ("expert_offsets", E + 1), ("shard_offsets", p.D + 1),
                 ("shard_routed", p.D), ("shard_overflow", p.D)):
        assert view(n, c).tolist() == _ints(kv[n]), n
    slot = view("slot_pos", T * k).reshape(T, k)
    assert sorted((tt, r) for tt in range(T) for r in range(k) if slot[tt, r] < 0) == sorted(lists["dropped"])
    assert int(view("dropped", 1).item()) == 2
    # the layer output against the oracle's, which drops the same two choices
    cpu = {n: v.cpu() for n, v in t.items()}
    ref = oracle.layer_forward(cpu["x"], cpu["Wg"], None, cpu["W1"], cpu["W3"] if act == "swiglu" else None,
                               cpu["W2"], k, p.D, p.capacity_factor, oracle.act_code(act))
    assert ref.slots.dropped == 2
    assert_close(y.float().cpu().numpy(), ref.y, dtype, "worked-example layer output")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rerouting_reproduces_the_hand_rerouted_example(dtype):
    rkv, rlists = _fixture("worked_example_reroute.txt")
    kv, lists, p, t = _instance(dtype)
    p.flags |= moe.MOE_FLAG_REROUTE
    T, E, k = p.T, p.E, p.k
    i32, f32 = torch.int32, torch.float32
    idx = torch.empty(T, k, dtype=i32, device="cuda")
    gate = torch.empty(T, k, dtype=f32, device="cuda")
    fidx = torch.empty(T, k, dtype=i32, device="cuda")
    fgate = torch.empty(T, k, dtype=f32, device="cuda")
    moe.moe_route_fallback(p, t["x"], t["Wg"], None, idx, gate, fidx, fgate, None)
    torch.cuda.synchronize()
    assert [tuple(r) for r in fidx.cpu().tolist()] == [tuple(f[1:]) for f in rlists["fallback"]]
    z = math.exp(3) + math.exp(2) + 6
    np.testing.assert_allclose(fgate.cpu().numpy(), 1.0 / z, rtol=1e-5)
    ws = moe.alloc_workspace(p, "cuda")
    C, C_shard, rows_max = moe.moe_capacity(p)
    ridx = torch.empty(T, k, dtype=i32, device="cuda")
    rgate = torch.empty(T, k, dtype=f32, device="cuda")
    o = dict(slot_pos=torch.empty(T, k, dtype=i32, device="cuda"),
             counts_routed=torch.empty(E, dtype=i32, device="cuda"),
             counts_kept=torch.empty(E, dtype=i32, device="cuda"),
             expert_offsets=torch.empty(E + 1, dtype=i32, device="cuda"),
             shard_offsets=torch.empty(p.D + 1, dtype=i32, device="cuda"),
             shard_routed=torch.empty(p.D, dtype=i32, device="cuda"),
             shard_overflow=torch.empty(p.D, dtype=i32, device="cuda"),
             row_token=torch.full((rows_max,), -7, dtype=i32, device="cuda"),
             dropped=torch.empty(1, dtype=i32, device="cuda"), rerouted=torch.empty(1, dtype=i32, device="cuda"))
    moe.moe_assign_slots_reroute(p, idx, gate, fidx, fgate, ridx, rgate, o["slot_pos"], o["counts_routed"],
                                 o["counts_kept"], o["expert_offsets"], o["shard_offsets"], o["shard_routed"],
                                 o["shard_overflow"], o["row_token"], o["dropped"], o["rerouted"], ws, ws.numel())
    assert moe.moe_device_status(ws) == moe.MOE_OK
    got = {n: v.cpu() for n, v in o.items()}
    for n in ("counts_routed", "counts_kept", "expert_offsets", "shard_offsets", "shard_routed", "shard_overflow"):
        assert got[n].tolist() == _ints(rkv[n]), n
    kept = int(got["expert_offsets"][-1])
    assert got["row_token"][:kept].tolist() == _ints(rkv["row_token"])
    assert int(got["dropped"].item()) == int(rkv["dropped_after"][0]) == 0
    assert int(got["rerouted"].item()) == len(rlists["rerouted"]) == 2
    ri, sp = ridx.cpu(), got["slot_pos"]
    for tt, r, e, pos in rlists["rerouted"]:
        assert (int(ri[tt, r]), int(sp[tt, r])) == (e, pos)
        assert abs(float(rgate.cpu()[tt, r]) - 1.0 / z) <= 1e-5 / z
