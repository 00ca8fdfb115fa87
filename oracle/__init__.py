"""CPU oracle of the capacity-limited top-k MoE layer forward.

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/``, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline / reference leg, never by the CUDA
library or its Python binding.  The arithmetic lives in ``moe_oracle.c``
(plain loops, one function per step of the method, each citing the passage of
the expert-parallelism pages it follows); this module only builds that file
with gcc, marshals arrays through ctypes and strings the steps together in
the pages' order (route, capacity, slots, dispatch, expert FFN, combine).

Parity status: every step is pinned by ``tests/test_oracle_*.py`` against
values fixed by the pages or by mathematics (worked example, closed forms,
invariants, brute force, textbook special cases).  The exact floating-point
values of the expert FFN on random inputs have no printed counterpart on the
pages; they are pinned only through the special cases and the dense brute
force.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

F32, BF16 = 0, 1
SWIGLU, GELU = 0, 1

_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into libmoe_oracle.so (gcc, OpenMP, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_capacity.argtypes = [i64, i32, i32, i32, dbl, P, P, P]
        lib.oracle_capacity.restype = i32
        lib.oracle_router_logits.argtypes = [i64, i32, i32, i32, P, P, P, P]
        lib.oracle_softmax_topk.argtypes = [i64, i32, i32, i32, P, P, P, P]
        lib.oracle_assign.argtypes = [i64, i32, i32, i32, i64, i64] + [P] * 10
        lib.oracle_assign_reroute.argtypes = [i64, i32, i32, i32, i64, i64] + [P] * 16
        lib.oracle_dispatch.argtypes = [i64, i32, i32, P, P, P]
        lib.oracle_expert_ffn.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P]
        lib.oracle_combine.argtypes = [i64, i32, i32, i32, P, P, P, P, P, P, P, P]
        lib.oracle_token_outputs.argtypes = [i64, P, i32, i32, i32, i32, i32] + [P] * 9
        lib.oracle_routing_stats.argtypes = [i64, i32, i32, P, P, P, P, P]
        lib.oracle_expert_choice.argtypes = [i64, i32, i64, P, P, P]
        lib.oracle_combine_expert_choice.argtypes = [i64, i32, i32, i32, P, P, P, P, P, P]
        _lib = lib
    return _lib


def _host(t) -> Optional[np.ndarray]:
    """Contiguous host array with the tensor's exact bytes (bf16 as uint16)."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return np.ascontiguousarray(t)
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _host_values(t) -> np.ndarray:
    """Values of a fp32 or bf16 tensor as float64 on the host (exact)."""
    a = _host(t)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _dtype_code(t) -> int:
    a = _host(t)
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    raise TypeError(f"oracle takes fp32 or bf16 tensors, got {a.dtype}")


def capacity(T: int, k: int, E: int, D: int, c: float):
    """(C_expert, C_shard, rows_max) from the capacity rule."""
    out = [ctypes.c_int64() for _ in range(3)]
    rc = _load().oracle_capacity(T, k, E, D, float(c), *[ctypes.byref(o) for o in out])
    if rc != 0:
        raise ValueError("invalid capacity arguments")
    return tuple(o.value for o in out)


def router_logits(x, Wg, bias=None) -> np.ndarray:
    xa, wa, ba = _host(x), _host(Wg), _host(bias)
    T, d = xa.shape
    E = wa.shape[0]
    if ba is not None:
        ba = np.ascontiguousarray(ba, dtype=np.float32)
    g = np.empty((T, E), dtype=np.float32)
    _load().oracle_router_logits(T, d, E, _dtype_code(x), _ptr(xa), _ptr(wa), _ptr(ba), _ptr(g))
    return g


def softmax_topk(logits: np.ndarray, k: int, want_probs: bool = True, renorm: bool = False):
    g = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = g.shape
    probs = np.empty((T, E), dtype=np.float32) if want_probs else None
    idx = np.empty((T, k), dtype=np.int32)
    gate = np.empty((T, k), dtype=np.float32)
    _load().oracle_softmax_topk(T, E, k, int(renorm), _ptr(g), _ptr(probs), _ptr(idx), _ptr(gate))
    return probs, idx, gate


@dataclass
class Slots:
    slot_pos: np.ndarray
    counts_routed: np.ndarray
    counts_kept: np.ndarray
    expert_offsets: np.ndarray
    shard_offsets: np.ndarray
    shard_routed: np.ndarray
    shard_overflow: np.ndarray
    row_token: np.ndarray  # [total kept]
    dropped: int
    C: int
    C_shard: int
    rows_max: int


def assign(topk_idx: np.ndarray, E: int, D: int, capacity_factor: float) -> Slots:
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    C, Cs, rows_max = capacity(T, k, E, D, capacity_factor)
    slot_pos = np.empty((T, k), np.int32)
    cr, ck = np.empty(E, np.int32), np.empty(E, np.int32)
    eo, so = np.empty(E + 1, np.int32), np.empty(D + 1, np.int32)
    sr, sov = np.empty(D, np.int32), np.empty(D, np.int32)
    row_token = np.full(max(rows_max, 1), -1, np.int32)
    dropped = ctypes.c_int64()
    _load().oracle_assign(T, E, D, k, C, Cs, _ptr(idx), _ptr(slot_pos), _ptr(cr), _ptr(ck),
                          _ptr(eo), _ptr(so), _ptr(sr), _ptr(sov), _ptr(row_token),
                          ctypes.byref(dropped))
    return Slots(slot_pos, cr, ck, eo, so, sr, sov, row_token[: int(eo[E])].copy(),
                 dropped.value, C, Cs, rows_max)


@dataclass
class Rerouted(Slots):
    route_idx: np.ndarray   # [T, k] expert that serves (t, r): the choice, or its fallback
    route_gate: np.ndarray  # [T, k] weight of (t, r): that expert's gate
    rerouted: int           # rerouted assignments that got a slot


def assign_reroute(topk_idx: np.ndarray, topk_gate: np.ndarray, fallback_idx: np.ndarray,
                   fallback_gate: np.ndarray, E: int, D: int, capacity_factor: float) -> Rerouted:
    """Slot assignment where an overflowing choice goes once to the token's
    next-best expert (fallback j for its j-th overflowing choice) and takes
    the capacity the first pass left."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    gate = np.ascontiguousarray(topk_gate, dtype=np.float32)
    fidx = np.ascontiguousarray(fallback_idx, dtype=np.int32)
    fgate = np.ascontiguousarray(fallback_gate, dtype=np.float32)
    assert gate.shape == fidx.shape == fgate.shape == (T, k)
    C, Cs, rows_max = capacity(T, k, E, D, capacity_factor)
    ridx, rgate = np.empty((T, k), np.int32), np.empty((T, k), np.float32)
    slot_pos = np.empty((T, k), np.int32)
    cr, ck = np.empty(E, np.int32), np.empty(E, np.int32)
    eo, so = np.empty(E + 1, np.int32), np.empty(D + 1, np.int32)
    sr, sov = np.empty(D, np.int32), np.empty(D, np.int32)
    row_token = np.full(max(rows_max, 1), -1, np.int32)
    rerouted, dropped = ctypes.c_int64(), ctypes.c_int64()
    _load().oracle_assign_reroute(T, E, D, k, C, Cs, _ptr(idx), _ptr(gate), _ptr(fidx), _ptr(fgate),
                                  _ptr(ridx), _ptr(rgate), _ptr(slot_pos), _ptr(cr), _ptr(ck), _ptr(eo),
                                  _ptr(so), _ptr(sr), _ptr(sov), _ptr(row_token), ctypes.byref(rerouted),
                                  ctypes.byref(dropped))
    return Rerouted(slot_pos, cr, ck, eo, so, sr, sov, row_token[: int(eo[E])].copy(), dropped.value, C, Cs,
                    rows_max, ridx, rgate, rerouted.value)


def dispatch(x, row_token: np.ndarray) -> np.ndarray:
    xa = _host(x)
    rows = int(row_token.shape[0])
    d = xa.shape[1]
    xd = np.empty((rows, d), dtype=xa.dtype)
    rt = np.ascontiguousarray(row_token, dtype=np.int32)
    _load().oracle_dispatch(rows, d, xa.itemsize, _ptr(xa), _ptr(rt), _ptr(xd))
    return xd


def expert_ffn(xd, expert_offsets: np.ndarray, W1, W3, W2, act: int) -> np.ndarray:
    xa, w1, w3, w2 = _host(xd), _host(W1), _host(W3), _host(W2)
    E, f, d = w1.shape
    eo = np.ascontiguousarray(expert_offsets, dtype=np.int32)
    yd = np.zeros((xa.shape[0], d), dtype=np.float64)
    _load().oracle_expert_ffn(E, d, f, act, _dtype_code(xd), _ptr(xa), _ptr(eo), _ptr(w1),
                              _ptr(w3), _ptr(w2), _ptr(yd))
    return yd


def combine(yd: np.ndarray, topk_idx, slot_pos, topk_gate, expert_offsets,
            residual=None, dtype: int = F32, shared=None) -> np.ndarray:
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    d = yd.shape[1]
    y = np.empty((T, d), dtype=np.float64)
    ra = _host(residual)
    # converted copies stay referenced here until the C call returns
    sp = np.ascontiguousarray(slot_pos, np.int32)
    gt = np.ascontiguousarray(topk_gate, np.float32)
    eo = np.ascontiguousarray(expert_offsets, np.int32)
    ydd = np.ascontiguousarray(yd, np.float64)
    sh = None if shared is None else np.ascontiguousarray(shared, np.float64)
    _load().oracle_combine(T, d, k, dtype, _ptr(idx), _ptr(sp), _ptr(gt), _ptr(eo), _ptr(ydd),
                           _ptr(sh), _ptr(ra), _ptr(y))
    return y


def routing_stats(probs, counts_routed, counts_kept, k: int):
    """Routing statistics in double: (aux, entropy, drop_fraction,
    load_imbalance), and the per-expert mean router probability."""
    pa = np.ascontiguousarray(probs, dtype=np.float32)
    T, E = pa.shape
    cr = np.ascontiguousarray(counts_routed, dtype=np.int32)
    ck = np.ascontiguousarray(counts_kept, dtype=np.int32)
    out = np.zeros(4, dtype=np.float64)
    mp = np.zeros(E, dtype=np.float64)
    _load().oracle_routing_stats(T, E, k, _ptr(pa), _ptr(cr), _ptr(ck), _ptr(out), _ptr(mp))
    return out, mp


def shared_expert(x, Ws1, Ws3, Ws2, act: int) -> np.ndarray:
    """A shared expert: the expert FFN applied to every token (one expert
    whose rows are all T tokens in order)."""
    xa = _host(x)
    T = xa.shape[0]
    w1, w3, w2 = _host(Ws1), _host(Ws3), _host(Ws2)
    add = lambda a: None if a is None else a[None]  # one expert
    return expert_ffn(xa, np.array([0, T], np.int32), add(w1), add(w3), add(w2), act)


@dataclass
class ExpertChoice:
    C: int                  # tokens per expert, min(C_expert, T)
    row_token: np.ndarray   # [E * C]: expert e's tokens, ascending, at rows e*C ...
    expert_offsets: np.ndarray  # [E + 1] = e * C
    sel_row: np.ndarray     # [T, E]: row of (t, e), or -1


def expert_choice(scores, capacity_factor: float, k: int, D: int = 1) -> ExpertChoice:
    """Expert-choice routing: each expert takes its min(C, T) tokens of highest
    score -- the fp32 router logit -- (ties: lower token first), C from the
    capacity rule."""
    pa = np.ascontiguousarray(scores, dtype=np.float32)
    T, E = pa.shape
    C, _, _ = capacity(T, k, E, D, capacity_factor)
    Cc = min(C, T)
    row_token = np.empty(E * Cc, dtype=np.int32)
    sel_row = np.empty((T, E), dtype=np.int32)
    _load().oracle_expert_choice(T, E, C, _ptr(pa), _ptr(row_token), _ptr(sel_row))
    return ExpertChoice(Cc, row_token, np.arange(E + 1, dtype=np.int32) * Cc, sel_row)


def combine_expert_choice(yd, probs, sel_row, residual=None, dtype: int = F32, shared=None) -> np.ndarray:
    pa = np.ascontiguousarray(probs, dtype=np.float32)
    T, E = pa.shape
    sr = np.ascontiguousarray(sel_row, dtype=np.int32)
    ydd = np.ascontiguousarray(yd, np.float64)
    d = ydd.shape[1]
    sh = None if shared is None else np.ascontiguousarray(shared, np.float64)
    ra = _host(residual)
    y = np.empty((T, d), dtype=np.float64)
    _load().oracle_combine_expert_choice(T, d, E, dtype, _ptr(pa), _ptr(sr), _ptr(ydd), _ptr(sh), _ptr(ra),
                                         _ptr(y))
    return y


def token_outputs(tokens, x, topk_idx, slot_pos, topk_gate, W1, W3, W2, act: int,
                  residual=None, shared=None) -> np.ndarray:
    """y[t] for the listed tokens, evaluated from the definition; `shared`
    = (Ws1, Ws3, Ws2) adds a shared expert after the routed sum, before the
    residual."""
    toks = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    if shared is not None:
        y = token_outputs(toks, x, topk_idx, slot_pos, topk_gate, W1, W3, W2, act)
        y += shared_expert(_host(x)[toks], *shared, act)
        if residual is not None:
            y += _host_values(residual)[toks]
        return y
    xa, w1, w3, w2, ra = _host(x), _host(W1), _host(W3), _host(W2), _host(residual)
    E, f, d = w1.shape
    k = topk_idx.shape[1]
    y = np.empty((toks.shape[0], d), dtype=np.float64)
    ti = np.ascontiguousarray(topk_idx, np.int32)
    sp = np.ascontiguousarray(slot_pos, np.int32)
    gt = np.ascontiguousarray(topk_gate, np.float32)
    _load().oracle_token_outputs(toks.shape[0], _ptr(toks), d, f, k, act, _dtype_code(x),
                                 _ptr(xa), _ptr(ti), _ptr(sp), _ptr(gt),
                                 _ptr(w1), _ptr(w3), _ptr(w2), _ptr(ra), _ptr(y))
    return y


@dataclass
class LayerResult:
    logits: np.ndarray
    probs: np.ndarray
    topk_idx: np.ndarray
    topk_gate: np.ndarray
    slots: Slots
    xd: Optional[np.ndarray]
    yd: Optional[np.ndarray]
    y: Optional[np.ndarray]


def route(x, Wg, bias, k: int, want_probs: bool = True, renorm: bool = False):
    g = router_logits(x, Wg, bias)
    probs, idx, gate = softmax_topk(g, k, want_probs, renorm)
    return g, probs, idx, gate


def route_fallback(x, Wg, bias, k: int, want_probs: bool = True):
    """Router with the k choices and the token's next k experts in the same
    descending-logit order (its fallbacks), each with its softmax probability."""
    g = router_logits(x, Wg, bias)
    probs, idx2, gate2 = softmax_topk(g, 2 * k, want_probs)
    return g, probs, idx2[:, :k].copy(), gate2[:, :k].copy(), idx2[:, k:].copy(), gate2[:, k:].copy()


def layer_forward(x, Wg, bias, W1, W3, W2, k: int, D: int, capacity_factor: float,
                  act: int, residual=None, with_ffn: bool = True) -> LayerResult:
    """The whole layer, step by step in the pages' order."""
    g, probs, idx, gate = route(x, Wg, bias, k)
    E = _host(Wg).shape[0]
    slots = assign(idx, E, D, capacity_factor)
    if not with_ffn:
        return LayerResult(g, probs, idx, gate, slots, None, None, None)
    xd = dispatch(x, slots.row_token)
    yd = expert_ffn(xd, slots.expert_offsets, W1, W3, W2, act)
    y = combine(yd, idx, slots.slot_pos, gate, slots.expert_offsets, residual,
                _dtype_code(x))
    return LayerResult(g, probs, idx, gate, slots, xd, yd, y)


def act_code(act: str) -> int:
    return {"swiglu": SWIGLU, "gelu": GELU}[act]
