"""Parity of the two layer options beyond the plain capacity-limited top-k
layer, through the C ABI, against the CPU oracle:

* renormalised gates (MOE_FLAG_RENORM): a token's k gates are the softmax over
  its k chosen logits -- choices bit-exact, gates within 1e-5 relative;
* a shared expert (ffn_shared > 0): a dense FFN every token goes through,
  added after the routed sum and before the residual -- bf16 within
  1e-2 + 2e-2|o|, fp32 within 1e-5 + 1e-4|o| of the fp64 oracle.

Small cases run the whole oracle (ragged T, K and N tails, both FFN paths);
the Mixtral-style shape with a shared expert as wide as a routed one is
checked on a seeded token sample.
"""
from __future__ import annotations

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
    "renorm_shared_bf16": Workload("renorm_shared_bf16", T=1000, d=256, E=8, D=4, k=2, ffn=384,
                                   capacity_factor=1.0, seed=51, renorm=True, ffn_shared=384),
    "shared_odd_bf16": Workload("shared_odd_bf16", T=333, d=200, E=8, D=2, k=2, ffn=136,
                                capacity_factor=1.25, seed=52, ffn_shared=264),
    "renorm_64e_bf16": Workload("renorm_64e_bf16", T=777, d=128, E=64, D=8, k=4, ffn=192,
                                capacity_factor=1.0, seed=53, zipf_s=1.2, renorm=True, ffn_shared=128),
    "renorm_top1": Workload("renorm_top1", T=300, d=64, E=16, D=4, k=1, ffn=64, capacity_factor=1.0,
                            seed=54, renorm=True),
    "shared_fp32_gelu": Workload("shared_fp32_gelu", T=130, d=32, E=8, D=4, k=2, ffn=64,
                                 capacity_factor=1.0, dtype="f32", act="gelu", seed=55, renorm=True,
                                 ffn_shared=48),
}
BIG = moe_inputs.WORKLOADS["mixtral_scaled"].with_(name="mixtral_scaled_shared", renorm=True,
                                                    ffn_shared=3584)


def _shared_args(inp):
    return inp.Ws1, inp.Ws3, inp.Ws2


@pytest.fixture(scope="module", params=list(CASES) + ["mixtral_scaled_shared"])
def case(request):
    wl = CASES.get(request.param) or BIG
    inp = moe_inputs.make_inputs(wl, device="cuda")
    cpu = inp.to("cpu")
    g, probs, idx, gate = oracle.route(cpu.x, cpu.Wg, cpu.bias, wl.k, renorm=wl.renorm)
    slots = oracle.assign(idx, wl.E, wl.D, wl.capacity_factor)
    yield wl, Device(inp), cpu, dict(probs=probs, idx=idx, gate=gate, slots=slots)
    torch.cuda.empty_cache()


def test_route_renorm(case):
    wl, dev, cpu, o = case
    idx, gate, probs = dev.route(want_probs=True)
    np.testing.assert_array_equal(idx.cpu().numpy(), o["idx"])
    assert_probs(gate.cpu().numpy(), o["gate"], "gate")
    assert_probs(probs.cpu().numpy(), o["probs"], "probs")
    if wl.renorm:
        np.testing.assert_allclose(gate.double().sum(dim=1).cpu().numpy(), 1.0, rtol=1e-6)


def test_shared_expert_ffn(case):
    wl, dev, cpu, o = case
    if not wl.ffn_shared:
        pytest.skip("no shared expert")
    ys = torch.full((wl.T, wl.d), float("nan"), dtype=dev.dtype, device="cuda")
    for _ in range(2):  # the second call reuses the workspace's release counters
        moe.moe_shared_expert_ffn(dev.p, dev.inp.x, *_shared_args(dev.inp), ys, dev.ws, dev.ws_bytes)
        torch.cuda.synchronize()
        assert dev.status() == moe.MOE_OK
        act = oracle.act_code(wl.act)
        if wl.name in CASES:
            want = oracle.shared_expert(cpu.x, *_shared_args(cpu), act)
            assert_close(host(ys), want, wl.dtype, "ys")
        else:
            rows = np.random.default_rng(7).choice(wl.T, size=64, replace=False)
            rows = np.unique(np.concatenate([rows, [0, wl.T - 1]]))
            want = oracle.shared_expert(cpu.x[torch.from_numpy(rows)], *_shared_args(cpu), act)
            assert_close(host(ys[torch.from_numpy(rows).cuda()]), want, wl.dtype, "ys sample")


def test_combine_shared(case):
    wl, dev, cpu, o = case
    if wl.name not in CASES:
        pytest.skip("checked through the layer on the large shape")
    s = o["slots"]
    act = oracle.act_code(wl.act)
    xd = oracle.dispatch(cpu.x, s.row_token)
    yd_t = oracle_dtype_tensor(oracle.expert_ffn(xd, s.expert_offsets, cpu.W1, cpu.W3, cpu.W2, act),
                               wl.dtype)
    yd = torch.zeros((max(dev.rows_max, 1), wl.d), dtype=dev.dtype, device="cuda")
    yd[: yd_t.shape[0]] = yd_t
    sh = None
    if wl.ffn_shared:
        sh = oracle_dtype_tensor(oracle.shared_expert(cpu.x, *_shared_args(cpu), act), wl.dtype)
    resid = torch.randn(wl.T, wl.d, generator=torch.Generator().manual_seed(3)).to(dev.dtype)
    y = torch.empty(wl.T, wl.d, dtype=dev.dtype, device="cuda")
    moe.moe_combine_shared(dev.p, yd, t_dev(o["idx"]), t_dev(s.slot_pos), t_dev(s.expert_offsets),
                           t_dev(o["gate"]), None if sh is None else sh.cuda(), resid.cuda(), y)
    torch.cuda.synchronize()
    want = oracle.combine(host(yd_t), o["idx"], s.slot_pos, o["gate"], s.expert_offsets, resid,
                          oracle.BF16 if wl.dtype == "bf16" else oracle.F32,
                          shared=None if sh is None else host(sh))
    assert_close(host(y), want, wl.dtype, "y")


def test_layer_forward_shared(case):
    wl, dev, cpu, o = case
    s = o["slots"]
    act = oracle.act_code(wl.act)
    resid = torch.randn(wl.T, wl.d, generator=torch.Generator().manual_seed(5)).to(dev.dtype)
    y = torch.empty(wl.T, wl.d, dtype=dev.dtype, device="cuda")
    inp = dev.inp
    moe.moe_layer_forward_shared(dev.p, inp.x, inp.Wg, inp.bias, inp.W1, inp.W3, inp.W2,
                                 *_shared_args(inp), resid.cuda(), y, dev.ws, dev.ws_bytes)
    torch.cuda.synchronize()
    assert dev.status() == moe.MOE_OK
    shared = _shared_args(cpu) if wl.ffn_shared else None
    if wl.name in CASES:
        toks = np.arange(wl.T)
    else:
        rng = np.random.default_rng(11)
        toks = np.unique(np.concatenate([rng.choice(wl.T, size=96, replace=False), [0, wl.T - 1]]))
    want = oracle.token_outputs(toks, cpu.x, o["idx"], s.slot_pos, o["gate"], cpu.W1, cpu.W3, cpu.W2, act,
                                residual=resid, shared=shared)
    assert_close(host(y[torch.from_numpy(toks).cuda()]), want, wl.dtype, "y")
    if not wl.ffn_shared:
        # without a shared expert the two entry points agree bit for bit
        y2 = dev.layer(resid.cuda())
        assert torch.equal(y.view(torch.int32 if y.dtype == torch.float32 else torch.int16),
                           y2.view(torch.int32 if y2.dtype == torch.float32 else torch.int16))


def _bits(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16)


def test_layer_forward_shared_matches_its_calls(case):
    """moe_layer_forward_shared lets its shared-expert FFN start on the SMs the
    routed FFN's CTAs leave and wait for the routed launch at its end; its
    output equals, bit for bit, that of the same steps as separate calls with
    a synchronisation after each, and stays so over back-to-back layers on
    one workspace with no synchronisation between them."""
    wl, dev, cpu, o = case
    if not wl.ffn_shared:
        pytest.skip("no shared expert")
    inp = dev.inp
    resid = torch.randn(wl.T, wl.d, generator=torch.Generator().manual_seed(6)).to(dev.dtype).cuda()
    idx, gate, _ = dev.route(want_probs=False)
    a = dev.assign(idx)
    xd = dev.dispatch(a["row_token"], a["expert_offsets"])
    yd = dev.expert_ffn(xd, a["expert_offsets"])
    ys = torch.empty(wl.T, wl.d, dtype=dev.dtype, device="cuda")
    moe.moe_shared_expert_ffn(dev.p, inp.x, *_shared_args(inp), ys, dev.ws, dev.ws_bytes)
    torch.cuda.synchronize()
    want = torch.empty(wl.T, wl.d, dtype=dev.dtype, device="cuda")
    moe.moe_combine_shared(dev.p, yd, idx, a["slot_pos"], a["expert_offsets"], gate, ys, resid, want)
    torch.cuda.synchronize()
    ys_layer = [torch.empty(wl.T, wl.d, dtype=dev.dtype, device="cuda") for _ in range(3)]
    for y in ys_layer:
        moe.moe_layer_forward_shared(dev.p, inp.x, inp.Wg, inp.bias, inp.W1, inp.W3, inp.W2,
                                     *_shared_args(inp), resid, y, dev.ws, dev.ws_bytes)
    torch.cuda.synchronize()
    assert dev.status() == moe.MOE_OK
    for i, y in enumerate(ys_layer):
        assert torch.equal(_bits(y), _bits(want)), f"layer {i} differs from the separate calls"


def test_plain_entry_points_reject_a_shared_expert():
    wl = CASES["shared_odd_bf16"]
    p = moe.problem_of(wl)
    A = 1 << 20
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward(p, A, A, None, A, A, A, None, A, A, 1 << 40, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
