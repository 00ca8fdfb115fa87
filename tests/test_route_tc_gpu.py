"""The bf16 router's tensor-core path against the oracle on inputs built to
put many tokens inside its error band.

moe_route without the probability output (and the layer forward) computes
the logits on the tensor cores, bounds their distance from the fixed-order
logits per token, and recomputes in the fixed order every expert that could
still be in the token's top-k ("Expert Parallelism" notes page, "Formal
Algorithm: Expert Parallelism Forward Pass": gate computation and expert
selection).  Its top-k indices must equal the oracle's bit for bit on every
input; gates must be within 1e-5 relative.  The cases below make that
recompute path do the work: experts with identical or nearly identical router
rows (exact and near ties in every token), rows that are scaled copies of
each other, heavy-tailed activations, a bias that forces ties, and shapes
across the kernel's instances (k <= 2 or <= 8; 24 to 128 experts, padded
and unpadded; ragged tiles; one token).  The tensor-core path serves 17 to
128 experts; the 256-expert case checks the fixed-order router that takes
over above that range.  Each case prints the share of tokens whose fixed-order top-(k+1)
gaps lie inside twice the bound, i.e. roughly the share of tokens the kernel
had to re-rank.
"""
import math
import zlib

import numpy as np
import pytest
import torch

import expert_parallelism_gemm_b300 as moe
import moe_inputs
import oracle
from moe_inputs import Workload
from tests.gpu_steps import Device, assert_close, assert_probs, host

pytestmark = pytest.mark.gpu


def _bf16_ulp_up(t):
    """The next bf16 value away from zero (one unit in the last place)."""
    b = t.to(torch.bfloat16).view(torch.int16)
    return (b + torch.where(t == 0, torch.zeros_like(b), torch.ones_like(b))).view(torch.bfloat16)


def _case(name):
    g = torch.Generator().manual_seed(zlib.crc32(name.encode()))
    if name == "duplicate_rows":
        wl = Workload(name, T=1000, d=256, E=24, D=4, k=2, ffn=64, capacity_factor=1.0, seed=60)
        inp = moe_inputs.make_inputs(wl)
        inp.Wg[5] = inp.Wg[3]
        inp.Wg[6] = inp.Wg[0]
    elif name == "near_duplicate_rows":
        wl = Workload(name, T=1500, d=512, E=64, D=8, k=2, ffn=64, capacity_factor=1.0, seed=61)
        inp = moe_inputs.make_inputs(wl)
        for a, b in ((1, 0), (9, 8), (33, 32), (63, 62)):
            inp.Wg[a] = inp.Wg[b]
            cols = torch.randint(0, wl.d, (3,), generator=g)
            inp.Wg[a, cols] = _bf16_ulp_up(inp.Wg[b, cols].float())
    elif name == "scaled_copies":
        # every odd expert is its even neighbour scaled by 1 + 2^-7: exact
        # logits differ by under 1% and the order flips with the sign
        wl = Workload(name, T=2048, d=1024, E=32, D=4, k=4, ffn=64, capacity_factor=1.0, seed=62)
        inp = moe_inputs.make_inputs(wl)
        for e in range(1, wl.E, 2):
            inp.Wg[e] = (inp.Wg[e - 1].float() * (1 + 2.0**-7)).to(torch.bfloat16)
    elif name == "heavy_tailed_x":
        wl = Workload(name, T=777, d=2048, E=128, D=8, k=1, ffn=64, capacity_factor=1.0, seed=63)
        inp = moe_inputs.make_inputs(wl)
        scale = torch.pow(10.0, torch.empty(wl.T, wl.d).uniform_(-3, 3, generator=g))
        inp.x = (inp.x.float() * scale).to(torch.bfloat16)
    elif name == "bias_ties":
        # two equal biases far above the rest: ties decided by tiny logits
        wl = Workload(name, T=640, d=128, E=32, D=4, k=2, ffn=64, capacity_factor=1.0, seed=64)
        inp = moe_inputs.make_inputs(wl)
        inp.x = (inp.x.float() * 1e-3).to(torch.bfloat16)
        inp.bias = torch.zeros(wl.E)
        inp.bias[[4, 20, 21]] = 5.0
    elif name == "e256_k8":
        wl = Workload(name, T=300, d=192, E=256, D=8, k=8, ffn=64, capacity_factor=2.0, seed=65)
        inp = moe_inputs.make_inputs(wl)
        inp.Wg[200:] = inp.Wg[100:156]
    elif name == "one_token":
        wl = Workload(name, T=1, d=64, E=24, D=4, k=2, ffn=64, capacity_factor=1.0, seed=66)
        inp = moe_inputs.make_inputs(wl)
    elif name == "ragged_129":
        wl = Workload(name, T=129, d=4096, E=40, D=8, k=2, ffn=64, capacity_factor=math.inf, seed=67)
        inp = moe_inputs.make_inputs(wl)
        inp.Wg[7] = inp.Wg[2]
    else:
        raise KeyError(name)
    return wl, inp


CASES = ["duplicate_rows", "near_duplicate_rows", "scaled_copies", "heavy_tailed_x", "bias_ties", "e256_k8",
         "one_token", "ragged_129"]


def _band_share(x, Wg, bias, g, k):
    """Share of tokens whose fixed-order top-(k+1) gaps lie within twice a
    bound of the kernel's form (tensor-core steps at 2^-18 each plus the
    fixed order's rounding, through ||x|| max ||w||)."""
    xf, wf = x.double().numpy(), Wg.double().numpy()
    d = xf.shape[1]
    steps = 4 * math.ceil(d / 64)
    c_d = 2 * steps * 2.0**-18 + (8 * math.ceil(d / 256) + 5) * 2.0**-24
    theta = c_d * np.linalg.norm(xf, axis=1) * np.linalg.norm(wf, axis=1).max() + 2.4e-7 * np.abs(g).max(1)
    top = -np.sort(-g.astype(np.float64), axis=1)[:, : k + 1]
    gaps = top[:, :-1] - top[:, 1:]
    return float(((gaps <= 2 * theta[:, None]).any(axis=1)).mean()) if top.shape[1] > 1 else 0.0


@pytest.mark.parametrize("name", CASES)
def test_tensor_core_router_matches_the_fixed_order(name):
    wl, inp = _case(name)
    logits, probs, o_idx, o_gate = oracle.route(inp.x, inp.Wg, inp.bias, wl.k)
    share = _band_share(inp.x, inp.Wg, inp.bias, logits, wl.k)
    print(f"{name}: {100 * share:.1f}% of tokens inside the band")
    dev = Device(inp.to("cuda"))
    idx, gate, _ = dev.route(want_probs=False)
    np.testing.assert_array_equal(idx.cpu().numpy(), o_idx)
    assert_probs(gate.cpu().numpy(), o_gate, "gate")
    # with the probability output the SIMT router runs: the same indices
    idx_p, gate_p, probs_p = dev.route(want_probs=True)
    assert torch.equal(idx_p, idx)
    assert_probs(probs_p.cpu().numpy(), probs, "probs")
    assert dev.status() == moe.MOE_OK


@pytest.mark.parametrize("name", ["near_duplicate_rows", "scaled_copies", "bias_ties"])
def test_layer_forward_on_near_ties(name):
    wl, inp = _case(name)
    _, _, o_idx, o_gate = oracle.route(inp.x, inp.Wg, inp.bias, wl.k)
    slots = oracle.assign(o_idx, wl.E, wl.D, wl.capacity_factor)
    dev = Device(inp.to("cuda"))
    y = dev.layer()
    assert dev.status() == moe.MOE_OK
    Tk = wl.T * wl.k
    np.testing.assert_array_equal(dev.region("topk_idx", torch.int32, Tk).cpu().numpy().reshape(wl.T, wl.k), o_idx)
    np.testing.assert_array_equal(dev.region("slot_pos", torch.int32, Tk).cpu().numpy().reshape(wl.T, wl.k),
                                  slots.slot_pos)
    np.testing.assert_array_equal(dev.region("expert_offsets", torch.int32, wl.E + 1).cpu().numpy(),
                                  slots.expert_offsets)
    cpu = inp
    xd = oracle.dispatch(cpu.x, slots.row_token)
    yd = oracle.expert_ffn(xd, slots.expert_offsets, cpu.W1, cpu.W3, cpu.W2, oracle.act_code(wl.act))
    want = oracle.combine(yd, o_idx, slots.slot_pos, o_gate, slots.expert_offsets, None, oracle.BF16)
    assert_close(host(y), want, wl.dtype, "y")


def test_renormalised_gates_on_the_tensor_core_path():
    wl, inp = _case("scaled_copies")
    wl = wl.with_(renorm=True)
    inp.wl = wl
    _, _, o_idx, o_gate = oracle.route(inp.x, inp.Wg, inp.bias, wl.k, renorm=True)
    dev = Device(inp.to("cuda"))
    idx, gate, _ = dev.route(want_probs=False)
    np.testing.assert_array_equal(idx.cpu().numpy(), o_idx)
    assert_probs(gate.cpu().numpy(), o_gate, "renormalised gate")
    np.testing.assert_allclose(gate.cpu().numpy().astype(np.float64).sum(1), 1.0, rtol=1e-6)
