"""Host-side checks of the C ABI; no GPU and no kernel launch.

* libmoe_b300.so loads and exports every function include/moe.h declares;
* argument validation rejects bad problems and pointers before launching;
* moe_capacity reproduces the capacity rule's values for every workload;
* the workspace layout is aligned, disjoint and sized as documented;
* the binding fails loudly when the library is missing.
"""
import math
import os
import re

import pytest

import expert_parallelism_gemm_b300 as moe
from expert_parallelism_gemm_b300 import build as moe_build
from tests.conftest import ROOT, read_golden
import moe_inputs


@pytest.fixture(scope="module", autouse=True)
def built_library():
    moe_build.build()
    moe.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?(?:int|char\s*\*|const char\s*\*)\s+(moe_\w+)\s*\(",
                                 src, flags=re.M)))


def test_every_declared_symbol_is_exported():
    names = _declared_functions()
    assert len(names) == 28, names
    assert sorted(moe.EXPORTS) == names
    lib = moe.load()
    for n in names:
        assert hasattr(lib, n), n


def test_route_doc_states_the_fixed_logit_order():
    # the order the router and the oracle both use: 32 slices of runs of 8
    # consecutive elements, one ascending fused multiply-add chain each, then
    # the xor butterfly over offsets 16, 8, 4, 2, 1, then the bias
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    doc = src[:src.index("int moe_route(")]
    doc = doc[doc.rindex("/*"):]
    flat = " ".join(doc.replace("*", " ").split())
    for phrase in ("32 slices of runs of 8 consecutive elements", "i = 256 m + 8 j + q",
                   "q = 0..7", "ascending from +0", "xor butterfly o = 16, 8, 4, 2, 1",
                   "s[j] + s[j ^ o]", "then the bias add"):
        assert phrase in flat, phrase
    assert "one fused multiply-add chain over i ascending" not in flat


def test_status_strings():
    for code in range(7):
        assert moe.moe_status_string(code) not in ("", "unknown status")
    assert moe.moe_status_string(99) == "unknown status"


def _problem(**kw):
    base = dict(T=128, d=64, E=8, D=4, k=2, ffn=64, capacity_factor=1.0, dtype="bf16", act="swiglu")
    base.update(kw)
    return moe.make_problem(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(k=9, E=16, D=4), moe.MOE_ERR_UNSUPPORTED),
    (dict(k=3, E=2, D=1), moe.MOE_ERR_INVALID_ARG),
    (dict(k=0), moe.MOE_ERR_INVALID_ARG),
    (dict(E=6, D=4), moe.MOE_ERR_INVALID_ARG),
    (dict(d=60), moe.MOE_ERR_INVALID_ARG),
    (dict(ffn=12), moe.MOE_ERR_INVALID_ARG),
    (dict(capacity_factor=0.0), moe.MOE_ERR_INVALID_ARG),
    (dict(capacity_factor=-1.0), moe.MOE_ERR_INVALID_ARG),
    (dict(capacity_factor=math.nan), moe.MOE_ERR_INVALID_ARG),
    (dict(T=-1), moe.MOE_ERR_INVALID_ARG),
    (dict(E=512, D=4), moe.MOE_ERR_UNSUPPORTED),
    (dict(T=1 << 30, k=2), moe.MOE_ERR_UNSUPPORTED),
    (dict(dtype=7), moe.MOE_ERR_INVALID_ARG),
    (dict(act=5), moe.MOE_ERR_INVALID_ARG),
    (dict(reroute=True, E=8, D=4, k=5), moe.MOE_ERR_INVALID_ARG),    # needs 2k <= E
    (dict(reroute=True, renorm=True), moe.MOE_ERR_INVALID_ARG),
    (dict(reroute=True, expert_choice=True), moe.MOE_ERR_INVALID_ARG),
])
def test_invalid_problems_rejected(kw, code):
    p = _problem(**kw)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_workspace_size(p)
    assert ei.value.status == code
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward(p, 16, 16, None, 16, 16, 16, None, 16, 16, 1 << 30, stream=0)
    assert ei.value.status == code


def test_capacity_matches_the_rule_for_every_workload():
    for name, T, k, E, D, c, C, Cs, rm in read_golden("capacities.txt"):
        wl = moe_inputs.WORKLOADS[name]
        assert moe.moe_capacity(moe.problem_of(wl)) == (int(C), int(Cs), int(rm))
    assert moe.moe_capacity(_problem(T=6, d=8, E=8, D=4, k=2)) == (2, 3, 12)
    assert moe.moe_capacity(_problem(T=0)) == (0, 0, 0)


def test_workspace_layout_is_aligned_and_disjoint():
    for wl in moe_inputs.WORKLOADS.values():
        p = moe.problem_of(wl)
        L = moe.moe_workspace_layout_of(p)
        assert L["total"] == moe.moe_workspace_size(p)
        C, Cs, rows_max = moe.moe_capacity(p)
        eb = 2 if wl.dtype == "bf16" else 4
        Tk = wl.T * wl.k
        nblk = -(-wl.T // 32)
        sizes = dict(status=16, topk_idx=4 * Tk, topk_gate=4 * Tk, slot_pos=4 * Tk,
                     counts_routed=4 * wl.E, counts_kept=4 * wl.E, expert_offsets=4 * (wl.E + 1),
                     shard_offsets=4 * (wl.D + 1), shard_routed=4 * wl.D, shard_overflow=4 * wl.D,
                     dropped=4, hist=4 * wl.E * wl.k * nblk, row_token=4 * rows_max,
                     xd=eb * rows_max * wl.d, h=eb * rows_max * wl.ffn, yd=eb * rows_max * wl.d,
                     ffn_sync=4 * (2 + wl.E * -(-C // 128)),
                     stats=8 * (wl.E + 1))
        spans = sorted((L[n], L[n] + s) for n, s in sizes.items())
        # rerouting adds the fallback choices (and the rerouted count) to the same layout
        Lr = moe.moe_workspace_layout_of(moe.problem_of(wl.with_(reroute=True))) if 2 * wl.k <= wl.E else None
        if Lr is not None:
            assert all(Lr[n] == L[n] for n in sizes)
            assert Lr["fallback_gate"] - Lr["fallback_idx"] >= 4 * Tk
            assert Lr["rerouted"] - Lr["fallback_gate"] >= 4 * Tk and Lr["total"] >= Lr["rerouted"] + 4
        assert spans[0][0] == 0 == L["status"]
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            assert a1 <= b0
        assert spans[-1][1] <= L["total"]
        assert all(L[n] % 256 == 0 for n in sizes)


def test_bad_pointers_and_workspace_rejected_before_launch():
    p = _problem()
    need = moe.moe_workspace_size(p)
    A = 1 << 20  # an aligned fake address; nothing is launched on these paths
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward(p, A, A, None, A, A, A, None, A, A, need - 1, stream=0)
    assert ei.value.status == moe.MOE_ERR_WORKSPACE
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward(p, A, A, None, A, None, A, None, A, A, need, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG  # SwiGLU needs W3
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward(p, A + 4, A, None, A, A, A, None, A, A, need, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG  # misaligned x
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_expert_ffn(p, A, A, A, A, A, A, None, need, stream=0)
    assert ei.value.status == moe.MOE_ERR_WORKSPACE
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_assign_slots(p, A, A, A, A, A, A, A, A, A, None, A + 8, need, stream=0)
    assert ei.value.status == moe.MOE_ERR_WORKSPACE  # misaligned workspace
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route(p, None, A, None, A, A, None, None, 0, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_combine(p, A, A, A, A, A, A + 2, A, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG  # misaligned residual
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_dispatch_by_token(p, A, A, None, A, A, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG  # slot_pos missing
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_dispatch_by_token(p, A, A, A, A, A + 8, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG  # misaligned xd
    # rerouting: the plain slot calls refuse the flag, the rerouting calls need it
    pr = _problem(reroute=True)
    need_r = moe.moe_workspace_size(pr)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_assign_slots(pr, A, A, A, A, A, A, A, A, A, None, A, need_r, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_assign_slots_static(pr, A, A, A, A, A, A, A, A, A, None, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_assign_slots_reroute(p, *([A] * 14), None, None, A, need, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route_fallback(p, A, A, None, A, A, A, A, None, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route_fallback(pr, A, A, None, A, A, None, A, None, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG  # fallback_idx missing
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_assign_slots_reroute(pr, *([A] * 14), None, None, A, need_r - 1, stream=0)
    assert ei.value.status == moe.MOE_ERR_WORKSPACE


def test_host_path_rejects_bad_arguments_before_any_cuda_call():
    p = _problem()
    need = moe.moe_workspace_size(p)
    stg = moe.moe_host_staging_size(p)
    assert stg == 4 * (-(-(128 * 64 * 2) // 256) * 256)
    A = 1 << 20
    for kw, code in [(dict(staging_bytes=stg - 1), moe.MOE_ERR_WORKSPACE),
                     (dict(ws_bytes=need - 1), moe.MOE_ERR_WORKSPACE),
                     (dict(x=[None]), moe.MOE_ERR_INVALID_ARG)]:
        args = dict(x=[A], y=[A], staging_bytes=stg, ws_bytes=need)
        args.update(kw)
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_layer_forward_host(p, args["x"], A, None, A, A, A, args["y"], A, args["staging_bytes"], A,
                                       args["ws_bytes"], stream=0)
        assert ei.value.status == code
    with pytest.raises(moe.MoeError) as ei:  # a shared expert needs the device entry point
        moe.moe_layer_forward_host(_problem(ffn_shared=64), [A], A, None, A, A, A, [A], A, stg, A, need, stream=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    # no steps: nothing to do
    moe.moe_layer_forward_host(p, [], A, None, A, A, A, [], A, stg, A, need, stream=0)


def test_layer_launch_count():
    count = lambda **kw: moe.moe_layer_launch_count(_problem(**kw))
    # T=128: 4 blocks, small histogram -> router, slot-and-pack, FFN, combine
    assert count() == 4
    assert count(dtype="f32", act="gelu") == 5          # two-kernel SIMT FFN
    assert count(ffn_shared=64) == 5                    # + the shared expert's FFN
    assert count(expert_choice=True) == 5
    assert count(reroute=True) == 6
    assert count(T=0) == 0
    # the slot-and-pack limit: E*k*ceil(T/32) = 16384 entries, and one block past it
    assert count(T=8192, E=64, D=8, k=1) == 4
    assert count(T=8224, E=64, D=8, k=1) == 5
    # redundant histogram reads above 32 MB take the other path too
    assert count(T=32768, d=4096, E=8, D=8, k=2, ffn=14336, capacity_factor=math.inf) == 5


def test_empty_batch_is_a_no_op():
    p = _problem(T=0)
    need = moe.moe_workspace_size(p)
    A = 1 << 20
    # T = 0: validated, nothing to launch, success
    moe.moe_layer_forward(p, A, A, None, A, A, A, None, A, A, need, stream=0)
    moe.moe_route(p, A, A, None, A, A, None, None, 0, stream=0)
    moe.moe_dispatch(p, A, A, A, A, stream=0)
    moe.moe_combine(p, A, A, A, A, A, None, A, stream=0)


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(moe, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libmoe_b300.so"))
    monkeypatch.setattr(moe, "_lib", None)
    with pytest.raises(ImportError):
        moe.moe_workspace_size(_problem())
