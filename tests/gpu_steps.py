"""Helpers of the GPU parity tests: run the C-ABI steps on device tensors and
bring the results back, and the tolerance checks shared by the tests.

Inputs flow only from the oracle (or the seeded generator) to the CUDA path,
never the other way: each per-step check feeds the CUDA step with the
oracle's result of the previous step.
"""
from __future__ import annotations

import numpy as np
import torch

import expert_parallelism_gemm_b300 as moe
import oracle
import moe_inputs

# bf16 layer outputs against the fp64 oracle: |a - o| <= 1e-2 + 2e-2 |o|;
# fp32 outputs: |a - o| <= 1e-5 + 1e-4 |o|; router probabilities 1e-5 relative.
TOL = {"bf16": (1e-2, 2e-2), "f32": (1e-5, 1e-4)}
PROB_RTOL, PROB_ATOL = 1e-5, 1e-12


def assert_close(actual, expected, dtype: str, what: str):
    atol, rtol = TOL[dtype]
    a = np.asarray(actual, dtype=np.float64)
    o = np.asarray(expected, dtype=np.float64)
    assert a.shape == o.shape, (what, a.shape, o.shape)
    err = np.abs(a - o)
    bad = err > atol + rtol * np.abs(o)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(o))), err.shape)
        where = [tuple(int(v) for v in w) for w in np.argwhere(bad)[:8]]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {i}: "
                             f"got {a[i]!r} want {o[i]!r}; first bad {where}")


def assert_probs(actual, expected, what: str):
    np.testing.assert_allclose(actual, expected, rtol=PROB_RTOL, atol=PROB_ATOL, err_msg=what)


def raw(t: torch.Tensor) -> np.ndarray:
    """Exact storage bytes on the host (bf16 as uint16, others as numpy)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def host(t: torch.Tensor) -> np.ndarray:
    """Exact host copy (bf16 as float64 values, others as numpy)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.float().numpy().astype(np.float64)
    return t.numpy()


class Device:
    """Device copies of one layer's inputs plus a zeroed workspace."""

    def __init__(self, inp: moe_inputs.LayerInputs, device="cuda"):
        wl = inp.wl
        self.wl = wl
        self.p = moe.problem_of(wl)
        self.C, self.C_shard, self.rows_max = moe.moe_capacity(self.p)
        d = torch.device(device)
        self.inp = inp if inp.x.device == d else inp.to(d)
        self.ws = moe.alloc_workspace(self.p, d)
        self.ws_bytes = self.ws.numel()
        self.dtype = moe_inputs.torch_dtype(wl.dtype)
        self.dev = d

    def empty(self, shape, dtype):
        return torch.empty(shape, dtype=dtype, device=self.dev)

    # -- one C-ABI call per step ------------------------------------------
    def route(self, want_probs=True):
        wl = self.wl
        idx = self.empty((wl.T, wl.k), torch.int32)
        gate = self.empty((wl.T, wl.k), torch.float32)
        probs = self.empty((wl.T, wl.E), torch.float32) if want_probs else None
        moe.moe_route(self.p, self.inp.x, self.inp.Wg, self.inp.bias, idx, gate, probs, None, 0)
        torch.cuda.synchronize()
        return idx, gate, probs

    def assign(self, topk_idx):
        wl = self.wl
        i32 = torch.int32
        out = dict(slot_pos=self.empty((wl.T, wl.k), i32), counts_routed=self.empty(wl.E, i32),
                   counts_kept=self.empty(wl.E, i32), expert_offsets=self.empty(wl.E + 1, i32),
                   shard_offsets=self.empty(wl.D + 1, i32), shard_routed=self.empty(wl.D, i32),
                   shard_overflow=self.empty(wl.D, i32),
                   row_token=torch.full((max(self.rows_max, 1),), -7, dtype=i32, device=self.dev),
                   dropped=self.empty(1, i32))
        moe.moe_assign_slots(self.p, topk_idx, out["slot_pos"], out["counts_routed"],
                             out["counts_kept"], out["expert_offsets"], out["shard_offsets"],
                             out["shard_routed"], out["shard_overflow"], out["row_token"],
                             out["dropped"], self.ws, self.ws_bytes)
        torch.cuda.synchronize()
        return out

    def dispatch(self, row_token, expert_offsets):
        xd = torch.zeros((max(self.rows_max, 1), self.wl.d), dtype=self.dtype, device=self.dev)
        moe.moe_dispatch(self.p, self.inp.x, row_token, expert_offsets, xd)
        torch.cuda.synchronize()
        return xd

    def expert_ffn(self, xd, expert_offsets):
        yd = torch.zeros((max(self.rows_max, 1), self.wl.d), dtype=self.dtype, device=self.dev)
        moe.moe_expert_ffn(self.p, xd, expert_offsets, self.inp.W1, self.inp.W3, self.inp.W2, yd,
                           self.ws, self.ws_bytes)
        torch.cuda.synchronize()
        return yd

    def combine(self, yd, topk_idx, slot_pos, expert_offsets, topk_gate, residual=None):
        y = self.empty((self.wl.T, self.wl.d), self.dtype)
        moe.moe_combine(self.p, yd, topk_idx, slot_pos, expert_offsets, topk_gate, residual, y)
        torch.cuda.synchronize()
        return y

    def layer(self, residual=None):
        y = self.empty((self.wl.T, self.wl.d), self.dtype)
        moe.moe_layer_forward(self.p, self.inp.x, self.inp.Wg, self.inp.bias, self.inp.W1,
                              self.inp.W3, self.inp.W2, residual, y, self.ws, self.ws_bytes)
        torch.cuda.synchronize()
        return y

    def region(self, name, dtype, count):
        return moe.workspace_view(self.ws, self.p, name, dtype, count)

    def status(self):
        return moe.moe_device_status(self.ws)


def t_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def oracle_dtype_tensor(a_f64: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Round oracle fp64 values to the layer dtype on the host, then upload."""
    t = torch.from_numpy(np.ascontiguousarray(a_f64))
    return t.to(moe_inputs.torch_dtype(dtype)).to(device)


def sample_rows(expert_offsets: np.ndarray, per_expert: int, rng) -> np.ndarray:
    """Sorted packed-row sample: first, last and random rows of every expert."""
    rows = []
    E = len(expert_offsets) - 1
    for e in range(E):
        a, b = int(expert_offsets[e]), int(expert_offsets[e + 1])
        if b <= a:
            continue
        pick = {a, b - 1}
        n = b - a
        if n > 2:
            pick.update(rng.choice(np.arange(a, b), size=min(per_expert, n), replace=False).tolist())
        rows.extend(sorted(pick))
    return np.array(sorted(set(rows)), dtype=np.int64)


def oracle_ffn_rows(xd_host_rows, row_expert, inp, act_code, wl):
    """Oracle FFN of selected packed rows: repack them per expert and run the
    oracle's expert FFN on the small packed matrix."""
    order = np.argsort(row_expert, kind="stable")
    xs = xd_host_rows[order]
    counts = np.bincount(row_expert, minlength=wl.E)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    yd = oracle.expert_ffn(xs, offs, inp.W1, inp.W3, inp.W2, act_code)
    out = np.empty_like(yd)
    out[order] = yd
    return out
