"""Failure detection on the GPU without a fault: a bounded wait of the expert
FFN kernel is made to run out, and the host reads the error.

The tensor-core FFN kernel's down tiles wait on release counters that the
gate/up epilogues bump.  Here the counters start far below zero, so no
number of releases reaches the target: nothing ever sets the flag the wait
needs.  Every wait of the kernel is bounded (2 s), so it records
MOE_ERR_TIMEOUT in the workspace status word, stops issuing work, drains its
own copies and MMAs, frees its tensor memory and returns; the last CTA out
zeroes the counters.  The test checks the status, the clean counters and
that the same context then computes the FFN correctly.
"""
from __future__ import annotations

import time

import pytest
import torch

import expert_parallelism_gemm_b300 as moe
import moe_inputs
import oracle
from moe_inputs import Workload
from tests.gpu_steps import Device, assert_close, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl", [
    # capacity 250: 2-SM pair tiles
    Workload("timeout_pairs", T=1000, d=256, E=8, D=4, k=2, ffn=384, capacity_factor=1.0, seed=91),
    # capacity 125: every expert within one 128-row tile, one-CTA tiles
    Workload("timeout_single", T=1000, d=256, E=16, D=4, k=2, ffn=384, capacity_factor=1.0, seed=92),
], ids=lambda w: w.name)
def test_ffn_release_wait_times_out_and_the_context_stays_usable(wl):
    inp = moe_inputs.make_inputs(wl, device="cuda")
    dev = Device(inp)
    cpu = inp.to("cpu")
    _, _, idx, _ = oracle.route(cpu.x, cpu.Wg, cpu.bias, wl.k, want_probs=False)
    s = oracle.assign(idx, wl.E, wl.D, wl.capacity_factor)
    rows = int(s.expert_offsets[-1])
    xd_host = oracle.dispatch(cpu.x, s.row_token)  # bf16 bits
    xd = torch.zeros((dev.rows_max, wl.d), dtype=dev.dtype)
    xd[:rows] = torch.from_numpy(xd_host).view(torch.bfloat16)
    xd = xd.cuda()
    offs = torch.from_numpy(s.expert_offsets).cuda()

    # the region holds the exit ticket, a counter per (expert, 128-row m-tile)
    # and the progress window; the pair form uses one counter per (expert,
    # m-tile pair), the one-CTA form (capacity within one tile, or within two
    # with a mean load within one) one per m-tile
    m_tiles = -(-dev.C // 128)
    one_cta = dev.C <= 128 or (dev.C <= 256 and wl.T * wl.k <= wl.E * 128)
    n_used = 1 + wl.E * (m_tiles if one_cta else -(-m_tiles // 2))
    sync = dev.region("ffn_sync", torch.int32, 2 + wl.E * m_tiles)
    assert int(sync.abs().sum()) == 0
    sync[1:n_used] = -(1 << 30)  # release counters that can never reach their target
    torch.cuda.synchronize()

    yd = torch.zeros((dev.rows_max, wl.d), dtype=dev.dtype, device="cuda")
    t0 = time.monotonic()
    moe.moe_expert_ffn(dev.p, xd, offs, inp.W1, inp.W3, inp.W2, yd, dev.ws, dev.ws_bytes)
    status = moe.moe_device_status(dev.ws)  # synchronises the stream
    elapsed = time.monotonic() - t0
    assert status == moe.MOE_ERR_TIMEOUT
    assert 1.5 < elapsed < 60, elapsed  # the 2 s limit, not a hang and not an early exit
    assert int(sync.abs().sum()) == 0  # the last CTA out cleaned up
    assert moe.moe_device_status(dev.ws) == moe.MOE_OK  # reading cleared the word

    # the context is intact: the same call now gives the oracle's result
    yd2 = dev.expert_ffn(xd, offs)
    assert dev.status() == moe.MOE_OK
    want = oracle.expert_ffn(xd_host, s.expert_offsets, cpu.W1, cpu.W3, cpu.W2, oracle.act_code(wl.act))
    assert_close(host(yd2[:rows]), want, wl.dtype, "yd after the timeout")
