"""Python binding of libmoe_b300.so, the B300 (sm_103a) MoE layer forward.

Argument marshalling only: every function here has the name and argument
order of the C entry point in ``include/moe.h`` and forwards to it through
ctypes.  Tensor arguments may be ``torch.Tensor`` (their ``data_ptr()`` is
passed), plain integer device addresses, or None for nullable pointers.  The
``stream`` argument takes a ``torch.cuda.Stream``, a raw handle, or None for
torch's current stream.  A non-zero status raises :class:`MoeError`.

The CUDA library must have been built (``python -m
expert_parallelism_gemm_b300.build``); importing the functions without it
raises immediately -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_F32, MOE_BF16 = 0, 1
MOE_FLAG_RENORM, MOE_FLAG_EXPERT_CHOICE, MOE_FLAG_REROUTE = 1, 2, 4
MOE_ACT_SWIGLU, MOE_ACT_GELU = 0, 1
MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE = 4, 5, 6

EXPORTS = ("moe_capacity", "moe_workspace_size", "moe_workspace_layout_of", "moe_route",
           "moe_assign_slots", "moe_dispatch", "moe_dispatch_by_token", "moe_expert_ffn", "moe_combine",
           "moe_layer_forward", "moe_device_status", "moe_status_string",
           "moe_assign_slots_static", "moe_routing_stats", "moe_shared_expert_ffn",
           "moe_combine_shared", "moe_layer_forward_shared", "moe_expert_choice_assign",
           "moe_combine_expert_choice", "moe_router_logits", "moe_route_fallback",
           "moe_assign_slots_reroute", "moe_host_alloc", "moe_host_free", "moe_host_staging_size",
           "moe_layer_forward_host", "moe_layer_launch_count", "moe_assign_slots_static_status")


class moe_problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("D", ctypes.c_int32), ("k", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("capacity_factor", ctypes.c_double), ("dtype", ctypes.c_int32),
                ("act", ctypes.c_int32), ("flags", ctypes.c_int32), ("ffn_shared", ctypes.c_int32)]


_LAYOUT_FIELDS = ("status", "topk_idx", "topk_gate", "slot_pos", "counts_routed", "counts_kept",
                  "expert_offsets", "shard_offsets", "shard_routed", "shard_overflow", "dropped",
                  "hist", "row_token", "xd", "h", "yd", "ffn_sync", "stats", "hs", "ys", "shared_sync",
                  "probs", "logits", "sel_row", "fallback_idx", "fallback_gate", "rerouted", "total")


class moe_workspace_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in _LAYOUT_FIELDS]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {moe_status_string(status)} (status {status})")


_lib = None


def load() -> ctypes.CDLL:
    """Load libmoe_b300.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoe_b300.so not built at {LIB_PATH}: run "
                          "`python -m expert_parallelism_gemm_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I = ctypes.c_void_p, ctypes.c_int
    PP = ctypes.POINTER(moe_problem)
    sz = ctypes.c_size_t
    lib.moe_capacity.argtypes = [PP, P, P, P]
    lib.moe_workspace_size.argtypes = [PP, P]
    lib.moe_workspace_layout_of.argtypes = [PP, ctypes.POINTER(moe_workspace_layout)]
    lib.moe_route.argtypes = [PP, P, P, P, P, P, P, P, sz, P]
    lib.moe_assign_slots.argtypes = [PP] + [P] * 11 + [sz, P]
    lib.moe_dispatch.argtypes = [PP, P, P, P, P, P]
    lib.moe_dispatch_by_token.argtypes = [PP, P, P, P, P, P, P]
    lib.moe_expert_ffn.argtypes = [PP, P, P, P, P, P, P, P, sz, P]
    lib.moe_combine.argtypes = [PP, P, P, P, P, P, P, P, P]
    lib.moe_layer_forward.argtypes = [PP, P, P, P, P, P, P, P, P, P, sz, P]
    lib.moe_assign_slots_static.argtypes = [PP] + [P] * 11
    lib.moe_assign_slots_static_status.argtypes = [P]
    lib.moe_device_status.argtypes = [P, P]
    lib.moe_routing_stats.argtypes = [PP, P, P, P, P, P, P, sz, P]
    lib.moe_shared_expert_ffn.argtypes = [PP, P, P, P, P, P, P, sz, P]
    lib.moe_combine_shared.argtypes = [PP, P, P, P, P, P, P, P, P, P]
    lib.moe_layer_forward_shared.argtypes = [PP, P, P, P, P, P, P, P, P, P, P, P, P, sz, P]
    lib.moe_expert_choice_assign.argtypes = [PP, P, P, P, P, P]
    lib.moe_router_logits.argtypes = [PP, P, P, P, P, P, P]
    lib.moe_combine_expert_choice.argtypes = [PP, P, P, P, P, P, P, P]
    lib.moe_route_fallback.argtypes = [PP] + [P] * 9
    lib.moe_assign_slots_reroute.argtypes = [PP] + [P] * 17 + [sz, P]
    lib.moe_host_alloc.argtypes = [sz, ctypes.POINTER(ctypes.c_void_p)]
    lib.moe_host_free.argtypes = [P]
    lib.moe_host_staging_size.argtypes = [PP, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_layer_forward_host.argtypes = [PP, ctypes.c_int64, P, P, P, P, P, P, P, P, sz, P, sz, P]
    lib.moe_layer_launch_count.argtypes = [PP, ctypes.POINTER(ctypes.c_int)]
    lib.moe_status_string.argtypes = [I]
    lib.moe_status_string.restype = ctypes.c_char_p
    for n in EXPORTS:
        if n != "moe_status_string":
            getattr(lib, n).restype = I
    _lib = lib
    return lib


# ------------------------------------------------------------ marshalling --
def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def make_problem(T, d, E, D, k, ffn, capacity_factor, dtype="bf16", act="swiglu", renorm=False,
                 ffn_shared=0, expert_choice=False, reroute=False) -> moe_problem:
    """moe_problem from plain values; dtype 'bf16'|'f32' (or code), act 'swiglu'|'gelu'."""
    dt = {"bf16": MOE_BF16, "f32": MOE_F32}.get(dtype, dtype)
    ac = {"swiglu": MOE_ACT_SWIGLU, "gelu": MOE_ACT_GELU}.get(act, act)
    return moe_problem(int(T), int(d), int(E), int(D), int(k), int(ffn), float(capacity_factor),
                       int(dt), int(ac),
                       (MOE_FLAG_RENORM if renorm else 0) | (MOE_FLAG_EXPERT_CHOICE if expert_choice else 0)
                       | (MOE_FLAG_REROUTE if reroute else 0),
                       int(ffn_shared))


def problem_of(wl) -> moe_problem:
    """moe_problem from any object with T, d, E, D, k, ffn, capacity_factor, dtype, act
    (and optionally renorm, ffn_shared, expert_choice, reroute)."""
    return make_problem(wl.T, wl.d, wl.E, wl.D, wl.k, wl.ffn, wl.capacity_factor, wl.dtype, wl.act,
                        getattr(wl, "renorm", False), getattr(wl, "ffn_shared", 0),
                        getattr(wl, "expert_choice", False), getattr(wl, "reroute", False))


# -------------------------------------------------------------- entries --
def moe_status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def moe_capacity(problem: moe_problem):
    out = [ctypes.c_int64() for _ in range(3)]
    _check(load().moe_capacity(ctypes.byref(problem), *[ctypes.byref(o) for o in out]), "moe_capacity")
    return tuple(o.value for o in out)


def moe_workspace_size(problem: moe_problem) -> int:
    n = ctypes.c_size_t()
    _check(load().moe_workspace_size(ctypes.byref(problem), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_workspace_layout_of(problem: moe_problem) -> dict:
    L = moe_workspace_layout()
    _check(load().moe_workspace_layout_of(ctypes.byref(problem), ctypes.byref(L)),
           "moe_workspace_layout_of")
    return {n: getattr(L, n) for n in _LAYOUT_FIELDS}


def moe_route(problem, x, Wg, bias, topk_idx, topk_gate, probs, ws, ws_bytes, stream=None):
    _check(load().moe_route(ctypes.byref(problem), _p(x), _p(Wg), _p(bias), _p(topk_idx),
                            _p(topk_gate), _p(probs), _p(ws), int(ws_bytes), _stream(stream)),
           "moe_route")


def moe_assign_slots(problem, topk_idx, slot_pos, counts_routed, counts_kept, expert_offsets,
                     shard_offsets, shard_routed, shard_overflow, row_token, dropped, ws, ws_bytes,
                     stream=None):
    _check(load().moe_assign_slots(ctypes.byref(problem), _p(topk_idx), _p(slot_pos),
                                   _p(counts_routed), _p(counts_kept), _p(expert_offsets),
                                   _p(shard_offsets), _p(shard_routed), _p(shard_overflow),
                                   _p(row_token), _p(dropped), _p(ws), int(ws_bytes),
                                   _stream(stream)),
           "moe_assign_slots")


def moe_route_fallback(problem, x, Wg, bias, topk_idx, topk_gate, fallback_idx, fallback_gate, probs,
                       stream=None):
    _check(load().moe_route_fallback(ctypes.byref(problem), _p(x), _p(Wg), _p(bias), _p(topk_idx),
                                     _p(topk_gate), _p(fallback_idx), _p(fallback_gate), _p(probs),
                                     _stream(stream)),
           "moe_route_fallback")


def moe_assign_slots_reroute(problem, topk_idx, topk_gate, fallback_idx, fallback_gate, route_idx,
                             route_gate, slot_pos, counts_routed, counts_kept, expert_offsets, shard_offsets,
                             shard_routed, shard_overflow, row_token, dropped, rerouted, ws, ws_bytes,
                             stream=None):
    _check(load().moe_assign_slots_reroute(ctypes.byref(problem), _p(topk_idx), _p(topk_gate),
                                           _p(fallback_idx), _p(fallback_gate), _p(route_idx),
                                           _p(route_gate), _p(slot_pos), _p(counts_routed),
                                           _p(counts_kept), _p(expert_offsets), _p(shard_offsets),
                                           _p(shard_routed), _p(shard_overflow), _p(row_token),
                                           _p(dropped), _p(rerouted), _p(ws), int(ws_bytes),
                                           _stream(stream)),
           "moe_assign_slots_reroute")


def moe_assign_slots_static(problem, topk_idx, slot_pos, counts_routed, counts_kept, expert_offsets,
                            shard_offsets, shard_routed, shard_overflow, row_token, dropped,
                            stream=None):
    """moe_assign_slots without a workspace, for callers that cannot allocate
    device memory; scratch is a static device array shared by all calls (see
    include/moe.h for its size limit and the rule that overlapping calls race)."""
    _check(load().moe_assign_slots_static(ctypes.byref(problem), _p(topk_idx), _p(slot_pos),
                                          _p(counts_routed), _p(counts_kept), _p(expert_offsets),
                                          _p(shard_offsets), _p(shard_routed), _p(shard_overflow),
                                          _p(row_token), _p(dropped), _stream(stream)),
           "moe_assign_slots_static")


def moe_assign_slots_static_status(stream=None) -> int:
    """Status code of moe_assign_slots_static's device word on the current
    device (synchronises the stream, then reads and clears it); no raise."""
    return load().moe_assign_slots_static_status(_stream(stream))


def moe_dispatch(problem, x, row_token, expert_offsets, xd, stream=None):
    _check(load().moe_dispatch(ctypes.byref(problem), _p(x), _p(row_token), _p(expert_offsets),
                               _p(xd), _stream(stream)), "moe_dispatch")


def moe_dispatch_by_token(problem, x, topk_idx, slot_pos, expert_offsets, xd, stream=None):
    _check(load().moe_dispatch_by_token(ctypes.byref(problem), _p(x), _p(topk_idx), _p(slot_pos),
                                        _p(expert_offsets), _p(xd), _stream(stream)), "moe_dispatch_by_token")


def moe_expert_ffn(problem, xd, expert_offsets, W1, W3, W2, yd, ws, ws_bytes, stream=None):
    _check(load().moe_expert_ffn(ctypes.byref(problem), _p(xd), _p(expert_offsets), _p(W1), _p(W3),
                                 _p(W2), _p(yd), _p(ws), int(ws_bytes), _stream(stream)),
           "moe_expert_ffn")


def moe_combine(problem, yd, topk_idx, slot_pos, expert_offsets, topk_gate, residual, y,
                stream=None):
    _check(load().moe_combine(ctypes.byref(problem), _p(yd), _p(topk_idx), _p(slot_pos),
                              _p(expert_offsets), _p(topk_gate), _p(residual), _p(y),
                              _stream(stream)), "moe_combine")


def moe_layer_forward(problem, x, Wg, bias, W1, W3, W2, residual, y, ws, ws_bytes, stream=None):
    _check(load().moe_layer_forward(ctypes.byref(problem), _p(x), _p(Wg), _p(bias), _p(W1),
                                    _p(W3), _p(W2), _p(residual), _p(y), _p(ws), int(ws_bytes),
                                    _stream(stream)), "moe_layer_forward")


MOE_STAT_AUX, MOE_STAT_ENTROPY, MOE_STAT_DROP, MOE_STAT_IMBALANCE, MOE_NUM_STATS = 0, 1, 2, 3, 4


def moe_shared_expert_ffn(problem, x, Ws1, Ws3, Ws2, ys, ws, ws_bytes, stream=None):
    _check(load().moe_shared_expert_ffn(ctypes.byref(problem), _p(x), _p(Ws1), _p(Ws3), _p(Ws2), _p(ys),
                                        _p(ws), int(ws_bytes), _stream(stream)), "moe_shared_expert_ffn")


def moe_combine_shared(problem, yd, topk_idx, slot_pos, expert_offsets, topk_gate, shared, residual, y,
                       stream=None):
    _check(load().moe_combine_shared(ctypes.byref(problem), _p(yd), _p(topk_idx), _p(slot_pos),
                                     _p(expert_offsets), _p(topk_gate), _p(shared), _p(residual), _p(y),
                                     _stream(stream)), "moe_combine_shared")


def moe_router_logits(problem, x, Wg, bias, logits, probs, stream=None):
    _check(load().moe_router_logits(ctypes.byref(problem), _p(x), _p(Wg), _p(bias), _p(logits), _p(probs),
                                    _stream(stream)), "moe_router_logits")


def moe_expert_choice_assign(problem, logits, row_token, expert_offsets, sel_row, stream=None):
    _check(load().moe_expert_choice_assign(ctypes.byref(problem), _p(logits), _p(row_token), _p(expert_offsets),
                                           _p(sel_row), _stream(stream)), "moe_expert_choice_assign")


def moe_combine_expert_choice(problem, yd, probs, sel_row, shared, residual, y, stream=None):
    _check(load().moe_combine_expert_choice(ctypes.byref(problem), _p(yd), _p(probs), _p(sel_row), _p(shared),
                                            _p(residual), _p(y), _stream(stream)), "moe_combine_expert_choice")


def moe_layer_forward_shared(problem, x, Wg, bias, W1, W3, W2, Ws1, Ws3, Ws2, residual, y, ws, ws_bytes,
                             stream=None):
    _check(load().moe_layer_forward_shared(ctypes.byref(problem), _p(x), _p(Wg), _p(bias), _p(W1), _p(W3),
                                           _p(W2), _p(Ws1), _p(Ws3), _p(Ws2), _p(residual), _p(y), _p(ws),
                                           int(ws_bytes), _stream(stream)), "moe_layer_forward_shared")


def moe_routing_stats(problem, probs, counts_routed, counts_kept, stats, mean_prob, ws, ws_bytes,
                      stream=None):
    _check(load().moe_routing_stats(ctypes.byref(problem), _p(probs), _p(counts_routed),
                                    _p(counts_kept), _p(stats), _p(mean_prob), _p(ws), int(ws_bytes),
                                    _stream(stream)), "moe_routing_stats")


def moe_host_alloc(nbytes: int) -> int:
    """Page-locked host memory (address as an int; 0 for nbytes == 0)."""
    ptr = ctypes.c_void_p()
    _check(load().moe_host_alloc(int(nbytes), ctypes.byref(ptr)), "moe_host_alloc")
    return ptr.value or 0


def moe_host_free(ptr: int):
    _check(load().moe_host_free(ptr or None), "moe_host_free")


def host_tensor(ptr: int, shape, dtype):
    """CPU tensor viewing host memory at `ptr` (e.g. from moe_host_alloc)."""
    import torch
    n = 1
    for v in shape:
        n *= int(v)
    item = torch.empty((), dtype=dtype).element_size()
    buf = (ctypes.c_char * (n * item)).from_address(ptr)
    return torch.frombuffer(buf, dtype=torch.uint8).view(dtype).view(*shape)


def moe_host_staging_size(problem: moe_problem) -> int:
    n = ctypes.c_size_t()
    _check(load().moe_host_staging_size(ctypes.byref(problem), ctypes.byref(n)), "moe_host_staging_size")
    return n.value


def moe_layer_forward_host(problem, x_hosts, Wg, bias, W1, W3, W2, y_hosts, staging, staging_bytes, ws,
                           ws_bytes, stream=None):
    """len(x_hosts) steps of the layer from host buffers (addresses or CPU
    tensors), copies overlapped with the layers; see include/moe.h."""
    n = len(x_hosts)
    if len(y_hosts) != n:
        raise ValueError("x_hosts and y_hosts differ in length")
    xs = (ctypes.c_void_p * max(n, 1))(*[_p(t) for t in x_hosts])
    ys = (ctypes.c_void_p * max(n, 1))(*[_p(t) for t in y_hosts])
    _check(load().moe_layer_forward_host(ctypes.byref(problem), n, xs, _p(Wg), _p(bias), _p(W1), _p(W3),
                                         _p(W2), ys, _p(staging), int(staging_bytes), _p(ws), int(ws_bytes),
                                         _stream(stream)),
           "moe_layer_forward_host")


def moe_layer_launch_count(problem: moe_problem) -> int:
    """Kernels one moe_layer_forward launches for this problem (host-only)."""
    n = ctypes.c_int()
    _check(load().moe_layer_launch_count(ctypes.byref(problem), ctypes.byref(n)), "moe_layer_launch_count")
    return n.value


def moe_device_status(ws, stream=None) -> int:
    """Status code of the kernels' device word (synchronises the stream); no raise."""
    return load().moe_device_status(_p(ws), _stream(stream))


# ------------------------------------------------------ torch plumbing --
def alloc_workspace(problem: moe_problem, device="cuda"):
    """Zero-filled uint8 torch tensor of moe_workspace_size bytes."""
    import torch
    return torch.zeros(moe_workspace_size(problem), dtype=torch.uint8, device=device)


def workspace_view(ws, problem: moe_problem, region: str, dtype, count: int):
    """torch view of `count` elements of one workspace region."""
    import torch
    off = moe_workspace_layout_of(problem)[region]
    item = torch.empty((), dtype=dtype).element_size()
    return ws[off: off + count * item].view(dtype)
