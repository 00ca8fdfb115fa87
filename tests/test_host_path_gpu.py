"""The layer forward from host buffers (moe_layer_forward_host): several steps
with different inputs, copies overlapped with the layers through two staging
buffers each way.  Every step's host output must equal, bit for bit, the
device-path layer forward on the same input (the same kernels run), and the
device path is itself checked against the oracle elsewhere; one step is also
checked against the oracle here."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import expert_parallelism_gemm_b300 as moe
import moe_inputs
import oracle
from moe_inputs import Workload
from tests.gpu_steps import assert_close

pytestmark = pytest.mark.gpu

CASES = [
    Workload("host_bf16", T=1000, d=256, E=8, D=4, k=2, ffn=384, capacity_factor=1.0, seed=101),
    Workload("host_fp32_gelu", T=130, d=32, E=8, D=4, k=2, ffn=64, capacity_factor=0.8, dtype="f32",
             act="gelu", seed=102),
    Workload("host_reroute", T=513, d=128, E=16, D=4, k=2, ffn=128, capacity_factor=1.0, seed=103,
             zipf_s=1.5, reroute=True),
    Workload("host_expert_choice", T=400, d=128, E=8, D=4, k=2, ffn=128, capacity_factor=1.0, seed=104,
             expert_choice=True),
]


@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
@pytest.mark.parametrize("n_steps", [1, 5])
def test_layer_forward_host_matches_the_device_path(wl, n_steps):
    inp = moe_inputs.make_inputs(wl, device="cuda")
    p = moe.problem_of(wl)
    ws = moe.alloc_workspace(p, "cuda")
    dt = moe_inputs.torch_dtype(wl.dtype)
    staging_bytes = moe.moe_host_staging_size(p)
    staging = torch.empty(staging_bytes, dtype=torch.uint8, device="cuda")
    nbytes = wl.T * wl.d * torch.empty((), dtype=dt).element_size()
    xs_ptr = [moe.moe_host_alloc(nbytes) for _ in range(n_steps)]
    ys_ptr = [moe.moe_host_alloc(nbytes) for _ in range(n_steps)]
    try:
        xs = [moe.host_tensor(a, (wl.T, wl.d), dt) for a in xs_ptr]
        ys = [moe.host_tensor(a, (wl.T, wl.d), dt) for a in ys_ptr]
        for i, x in enumerate(xs):
            g = torch.Generator().manual_seed(1000 + i)
            x.copy_(torch.randn(wl.T, wl.d, generator=g).to(dt))
            ys[i].fill_(float("nan"))
        moe.moe_layer_forward_host(p, xs_ptr, inp.Wg, inp.bias, inp.W1, inp.W3, inp.W2, ys_ptr, staging,
                                   staging_bytes, ws, ws.numel())
        torch.cuda.synchronize()
        assert moe.moe_device_status(ws) == moe.MOE_OK
        bits = torch.int16 if dt == torch.bfloat16 else torch.int32
        for i in range(n_steps):
            y_dev = torch.empty(wl.T, wl.d, dtype=dt, device="cuda")
            moe.moe_layer_forward(p, xs[i].cuda(), inp.Wg, inp.bias, inp.W1, inp.W3, inp.W2, None, y_dev, ws,
                                  ws.numel())
            torch.cuda.synchronize()
            assert torch.equal(ys[i].view(bits), y_dev.cpu().view(bits)), f"step {i}"
        if wl.expert_choice:
            return  # the device path it equals is checked against the expert-choice oracle elsewhere
        # and the last step against the oracle, on a token sample
        cpu = inp.to("cpu")
        x_last = xs[-1].clone()
        _, _, idx, gate = oracle.route(x_last, cpu.Wg, cpu.bias, wl.k)
        if wl.reroute:
            _, _, idx, gate, fidx, fgate = oracle.route_fallback(x_last, cpu.Wg, cpu.bias, wl.k)
            s = oracle.assign_reroute(idx, gate, fidx, fgate, wl.E, wl.D, wl.capacity_factor)
            idx, gate = s.route_idx, s.route_gate
        else:
            s = oracle.assign(idx, wl.E, wl.D, wl.capacity_factor)
        toks = np.unique(np.concatenate([np.random.default_rng(7).choice(wl.T, size=min(64, wl.T),
                                                                         replace=False), [0, wl.T - 1]]))
        want = oracle.token_outputs(toks, x_last, idx, s.slot_pos, gate, cpu.W1, cpu.W3, cpu.W2,
                                    oracle.act_code(wl.act))
        assert_close(ys[-1][torch.from_numpy(toks)].double().numpy(), want, wl.dtype, "y from host path")
    finally:
        for a in xs_ptr + ys_ptr:
            moe.moe_host_free(a)
