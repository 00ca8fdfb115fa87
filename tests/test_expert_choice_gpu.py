"""Parity of expert-choice routing (MOE_FLAG_EXPERT_CHOICE) through the C ABI
against the CPU oracle.

Each expert takes its min(C, T) tokens of largest fp32 router logit (ties:
lower token first): router logits, rows, offsets and the selection map are
bit-exact; probabilities within 1e-5 relative; the layer output within the
layer-dtype tolerance of the fp64 oracle (1e-2 + 2e-2|o| for bf16,
1e-5 + 1e-4|o| for fp32).  Small cases check every output; the Mixtral-style
shape checks the selection in full and the output on a seeded token sample.
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
from tests.gpu_steps import Device, assert_close, assert_probs, host, oracle_dtype_tensor, t_dev

pytestmark = pytest.mark.gpu

CASES = {
    "ec_bf16": Workload("ec_bf16", T=1000, d=256, E=8, D=4, k=2, ffn=384, capacity_factor=1.0, seed=71,
                        expert_choice=True),
    "ec_odd_shared": Workload("ec_odd_shared", T=333, d=200, E=16, D=4, k=1, ffn=136, capacity_factor=2.0,
                              seed=72, expert_choice=True, ffn_shared=136),
    "ec_64e_skew": Workload("ec_64e_skew", T=777, d=128, E=64, D=8, k=2, ffn=192, capacity_factor=1.0,
                            seed=73, zipf_s=1.2, expert_choice=True),
    "ec_every_token": Workload("ec_every_token", T=200, d=64, E=4, D=2, k=1, ffn=64,
                               capacity_factor=math.inf, seed=74, expert_choice=True),
    "ec_fp32_gelu": Workload("ec_fp32_gelu", T=130, d=32, E=8, D=4, k=2, ffn=64, capacity_factor=1.0,
                             dtype="f32", act="gelu", seed=75, expert_choice=True),
}
BIG = moe_inputs.WORKLOADS["mixtral_scaled"].with_(name="mixtral_scaled_ec", expert_choice=True)


@pytest.fixture(scope="module", params=list(CASES) + ["mixtral_scaled_ec"])
def case(request):
    wl = CASES.get(request.param) or BIG
    inp = moe_inputs.make_inputs(wl, device="cuda")
    cpu = inp.to("cpu")
    g, probs, _, _ = oracle.route(cpu.x, cpu.Wg, cpu.bias, wl.k)
    ec = oracle.expert_choice(g, wl.capacity_factor, wl.k, wl.D)
    yield wl, Device(inp), cpu, dict(logits=g, probs=probs, ec=ec)
    torch.cuda.empty_cache()


def _select(dev, logits):
    wl = dev.wl
    rows = wl.E * dev.C
    row_token = torch.full((max(rows, 1),), -7, dtype=torch.int32, device="cuda")
    off = torch.full((wl.E + 1,), -7, dtype=torch.int32, device="cuda")
    sel = torch.full((wl.T, wl.E), -7, dtype=torch.int32, device="cuda")
    moe.moe_expert_choice_assign(dev.p, logits, row_token, off, sel)
    torch.cuda.synchronize()
    return row_token, off, sel


def test_router_logits(case):
    wl, dev, cpu, o = case
    logits = torch.empty(wl.T, wl.E, dtype=torch.float32, device="cuda")
    probs = torch.empty(wl.T, wl.E, dtype=torch.float32, device="cuda")
    moe.moe_router_logits(dev.p, dev.inp.x, dev.inp.Wg, dev.inp.bias, logits, probs)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(logits.cpu().numpy().view(np.uint32), o["logits"].view(np.uint32))
    assert_probs(probs.cpu().numpy(), o["probs"], "probs")


def test_expert_choice_select(case):
    wl, dev, cpu, o = case
    ec = o["ec"]
    assert dev.C == ec.C and dev.rows_max == wl.E * ec.C
    row_token, off, sel = _select(dev, t_dev(o["logits"]))
    np.testing.assert_array_equal(row_token[: wl.E * ec.C].cpu().numpy(), ec.row_token)
    np.testing.assert_array_equal(off.cpu().numpy(), ec.expert_offsets)
    np.testing.assert_array_equal(sel.cpu().numpy(), ec.sel_row)


def test_expert_choice_combine(case):
    wl, dev, cpu, o = case
    if wl.name not in CASES:
        pytest.skip("checked through the layer on the large shape")
    ec = o["ec"]
    act = oracle.act_code(wl.act)
    xd = oracle.dispatch(cpu.x, ec.row_token)
    yd_t = oracle_dtype_tensor(oracle.expert_ffn(xd, ec.expert_offsets, cpu.W1, cpu.W3, cpu.W2, act), wl.dtype)
    resid = torch.randn(wl.T, wl.d, generator=torch.Generator().manual_seed(9)).to(dev.dtype)
    y = torch.empty(wl.T, wl.d, dtype=dev.dtype, device="cuda")
    moe.moe_combine_expert_choice(dev.p, yd_t.cuda(), t_dev(o["probs"]), t_dev(ec.sel_row), None, resid.cuda(), y)
    torch.cuda.synchronize()
    want = oracle.combine_expert_choice(host(yd_t), o["probs"], ec.sel_row, resid,
                                        oracle.BF16 if wl.dtype == "bf16" else oracle.F32)
    assert_close(host(y), want, wl.dtype, "y")


def _oracle_tokens(wl, cpu, o, toks, resid):
    """y[t] for the listed tokens from the definition: the sum over the experts
    that took t (ascending) of probs[t, e] * FFN_e(x[t]), plus the shared
    expert and the residual."""
    ec, probs = o["ec"], o["probs"]
    act = oracle.act_code(wl.act)
    pairs = [(t, e) for e in range(wl.E) for t in toks if ec.sel_row[t, e] >= 0]
    y = np.zeros((len(toks), wl.d))
    where = {t: i for i, t in enumerate(toks)}
    if pairs:
        xs = cpu.x[torch.tensor([t for t, _ in pairs])]
        counts = np.bincount([e for _, e in pairs], minlength=wl.E)
        offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        yd = oracle.expert_ffn(xs, offs, cpu.W1, cpu.W3, cpu.W2, act)
        contrib = {}
        for row, (t, e) in enumerate(pairs):
            contrib.setdefault(t, []).append((e, row))
        for t, lst in contrib.items():
            for e, row in sorted(lst):
                y[where[t]] += float(probs[t, e]) * yd[row]
    if wl.ffn_shared:
        y += oracle.shared_expert(cpu.x[torch.from_numpy(np.asarray(toks))], cpu.Ws1, cpu.Ws3, cpu.Ws2, act)
    y += resid.double().numpy()[np.asarray(toks)]
    return y


def test_expert_choice_layer(case):
    wl, dev, cpu, o = case
    ec = o["ec"]
    resid = torch.randn(wl.T, wl.d, generator=torch.Generator().manual_seed(13)).to(dev.dtype)
    y = torch.empty(wl.T, wl.d, dtype=dev.dtype, device="cuda")
    inp = dev.inp
    moe.moe_layer_forward_shared(dev.p, inp.x, inp.Wg, inp.bias, inp.W1, inp.W3, inp.W2, inp.Ws1, inp.Ws3,
                                 inp.Ws2, resid.cuda(), y, dev.ws, dev.ws_bytes)
    torch.cuda.synchronize()
    assert dev.status() == moe.MOE_OK
    # the selection the layer took is the oracle's, bit for bit
    np.testing.assert_array_equal(dev.region("sel_row", torch.int32, wl.T * wl.E).cpu().numpy(),
                                  ec.sel_row.reshape(-1))
    np.testing.assert_array_equal(dev.region("row_token", torch.int32, wl.E * ec.C).cpu().numpy(), ec.row_token)
    if wl.name in CASES:
        toks = list(range(wl.T))
    else:
        rng = np.random.default_rng(17)
        toks = sorted(set(rng.choice(wl.T, size=64, replace=False).tolist()) | {0, wl.T - 1})
    want = _oracle_tokens(wl, cpu, o, toks, resid)
    assert_close(host(y[torch.tensor(toks).cuda()]), want, wl.dtype, "y")


def test_expert_choice_ties_take_the_lower_tokens():
    # x = 0: every logit is its expert's bias, so each expert sees T equal
    # scores and must take tokens 0 .. C-1
    wl = Workload("ec_ties", T=96, d=64, E=8, D=4, k=2, ffn=64, capacity_factor=1.0, seed=76,
                  expert_choice=True)
    inp = moe_inputs.make_inputs(wl, device="cuda")
    inp.x.zero_()
    inp.bias = torch.tensor([1, 2, 2, 0, -1, 1, 3, 0], dtype=torch.float32, device="cuda")
    dev = Device(inp)
    logits = torch.empty(wl.T, wl.E, dtype=torch.float32, device="cuda")
    moe.moe_router_logits(dev.p, inp.x, inp.Wg, inp.bias, logits, None)
    row_token, off, sel = _select(dev, logits)
    C = dev.C
    for e in range(wl.E):
        assert row_token[e * C:(e + 1) * C].cpu().tolist() == list(range(C))
    g = oracle.router_logits(inp.x.cpu(), inp.Wg.cpu(), inp.bias.cpu())
    np.testing.assert_array_equal(sel.cpu().numpy(), oracle.expert_choice(g, 1.0, 2, 4).sel_row)
