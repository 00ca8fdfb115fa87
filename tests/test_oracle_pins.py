"""Pins of the CPU oracle against what the pages and mathematics fix.

No GPU.  Each test is chosen so that a plausible slip in the oracle (dropped
term, wrong index or sign, transposed operand, wrong priority) fails it:

* the worked example of the capacity figure ("Expert Parallelism",
  theinfinity.ai) reproduced exactly, from a fixture under tests/golden;
* the capacity rule's closed forms for every workload;
* router logits against exact integer dot products and an fp64 error bound;
* softmax against a library softmax and the worked example's closed form;
* top-k and slot assignment against brute-force sorts;
* the expert FFN and combine against dense evaluation of every expert with
  library matmuls and activations (dense soft mixture, plain MLP, no drops).
"""
import math

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

import oracle
from tests.conftest import read_golden
import moe_inputs


# --------------------------------------------------------------------------
# worked example
# --------------------------------------------------------------------------
def _worked_example():
    rows = read_golden("worked_example.txt")
    kv = {}
    choices, dropped = [], []
    for r in rows:
        if r[0] == "choice":
            choices.append((int(r[1]), int(r[2]), int(r[3])))
        elif r[0] == "dropped":
            dropped.append((int(r[1]), int(r[2])))
        else:
            kv[r[0]] = r[1:]
    return kv, choices, dropped


def test_worked_example_reproduces_caption():
    kv, choices, dropped = _worked_example()
    T, d, E, D, k = (int(kv[n][0]) for n in ("T", "d", "E", "D", "k"))
    c = float(kv["c"][0])
    x = np.zeros((T, d), np.float32)
    for t, e0, e1 in choices:
        x[t, e0] = 3.0
        x[t, e1] = 2.0
    Wg = np.eye(E, d, dtype=np.float32)
    for dt in (torch.float32, torch.bfloat16):
        xt, wt = torch.from_numpy(x).to(dt), torch.from_numpy(Wg).to(dt)
        res = oracle.layer_forward(xt, wt, None, None, None, None, k, D, c, oracle.SWIGLU,
                                   with_ffn=False)
        s = res.slots
        assert (s.C, s.C_shard) == (int(kv["C"][0]), int(kv["C_shard"][0]))
        assert [tuple(r) for r in res.topk_idx.tolist()] == [(e0, e1) for _, e0, e1 in choices]
        assert s.counts_routed.tolist() == [int(v) for v in kv["counts_routed"]]
        assert s.counts_kept.tolist() == [int(v) for v in kv["counts_kept"]]
        unused = [e for e in range(E) if s.counts_routed[e] == 0]
        assert unused == [int(v) for v in kv["unused_experts"]]
        got_dropped = sorted((t, r) for t in range(T) for r in range(k) if s.slot_pos[t, r] < 0)
        assert got_dropped == sorted(dropped)
        assert s.dropped == 2
        assert s.expert_offsets.tolist() == [int(v) for v in kv["expert_offsets"]]
        assert s.shard_offsets.tolist() == [int(v) for v in kv["shard_offsets"]]
        assert s.shard_routed.tolist() == [int(v) for v in kv["shard_routed"]]
        assert s.shard_overflow.tolist() == [int(v) for v in kv["shard_overflow"]]
        np.testing.assert_allclose(res.topk_gate[:, 0], float(kv["gate0"][0]), rtol=0, atol=1e-7)
        np.testing.assert_allclose(res.topk_gate[:, 1], float(kv["gate1"][0]), rtol=0, atol=1e-7)
        # the closed form behind the printed gates
        z = math.exp(3) + math.exp(2) + 6
        assert abs(res.topk_gate[0, 0] - math.exp(3) / z) < 1e-7


# --------------------------------------------------------------------------
# capacity
# --------------------------------------------------------------------------
def test_capacity_closed_forms_of_every_workload():
    for name, T, k, E, D, c, C, Cs, rm in read_golden("capacities.txt"):
        wl = moe_inputs.WORKLOADS[name]
        assert (wl.T, wl.k, wl.E, wl.D) == (int(T), int(k), int(E), int(D))
        cf = math.inf if c == "inf" else float(c)
        assert wl.capacity_factor == cf
        assert oracle.capacity(int(T), int(k), int(E), int(D), cf) == (int(C), int(Cs), int(rm))


def test_capacity_edge_cases():
    # ceil rounds a fractional mean load up; tiny c still gives one slot
    assert oracle.capacity(6, 2, 8, 4, 1.0)[0] == 2          # 1.5 -> 2
    assert oracle.capacity(10, 1, 4, 2, 1e-9)[0] == 1
    # never more than T per expert, never more than T*k per shard
    assert oracle.capacity(5, 2, 2, 1, 100.0)[:2] == (5, 10)
    assert oracle.capacity(0, 2, 8, 4, 1.0) == (0, 0, 0)
    with pytest.raises(ValueError):
        oracle.capacity(4, 2, 8, 4, 0.0)


def test_active_parameter_fraction():
    # "Expert Parallelism" glossary (inferensys.com): 128 experts, top-2,
    # about 1.6% of the expert parameters active per token.  Each token reads
    # the weights of exactly k distinct experts.
    wl = moe_inputs.Workload("p", T=64, d=16, E=128, D=8, k=2, ffn=16, capacity_factor=math.inf)
    inp = moe_inputs.make_inputs(wl)
    _, _, idx, _ = oracle.route(inp.x, inp.Wg, None, wl.k)
    per_token = np.array([len(set(r)) for r in idx.tolist()])
    assert (per_token == 2).all()
    frac = per_token.mean() / wl.E
    assert frac == 2 / 128 and round(100 * frac, 1) == 1.6


# --------------------------------------------------------------------------
# router
# --------------------------------------------------------------------------
def test_logits_exact_on_small_integers():
    # Every partial sum is an integer below 2^24, so any order is exact: the
    # oracle must equal the integer dot product (pins operand pairing and bias).
    rng = np.random.default_rng(11)
    T, d, E = 37, 96, 13
    xi = rng.integers(-8, 9, size=(T, d))
    wi = rng.integers(-8, 9, size=(E, d))
    b = rng.integers(-50, 51, size=E).astype(np.float32)
    for dt in (torch.float32, torch.bfloat16):
        g = oracle.router_logits(torch.tensor(xi, dtype=dt), torch.tensor(wi, dtype=dt),
                                 torch.from_numpy(b))
        exact = xi @ wi.T + b.astype(np.int64)
        assert np.array_equal(g.astype(np.int64), exact)
        assert np.array_equal(g, exact.astype(np.float32))


def test_logits_within_fp32_bound_of_fp64():
    rng = np.random.default_rng(12)
    T, d, E = 50, 512, 16
    x = rng.standard_normal((T, d)).astype(np.float32)
    w = (rng.standard_normal((E, d)) / math.sqrt(d)).astype(np.float32)
    g = oracle.router_logits(x, w)
    exact = x.astype(np.float64) @ w.astype(np.float64).T
    bound = d * 2.0**-24 * (np.abs(x).astype(np.float64) @ np.abs(w).astype(np.float64).T)
    assert (np.abs(g - exact) <= bound).all()
    # and not trivially: the bound is far below the logit scale
    assert bound.max() < 1e-3


def test_logit_order_rounding_cases_derived_by_hand():
    # The summation order is a reading (the pages give none): 32 slices of
    # runs of 8 consecutive hidden elements (slice j: i = 256m + 8j + q), one
    # ascending fmaf chain per slice from +0, then the xor butterfly over
    # o = 16, 8, 4, 2, 1.  These inputs make fp32 rounding depend on the order,
    # and the expected values were worked out by hand from that definition.
    d = 256
    # (a) slice 0 holds 2^12 * 2^12 = 2^24, slices 1..31 hold 1 each (at
    # i = 8j).  Butterfly: round 16: 2^24 + 1 -> 2^24 (ties to even), every
    # other slice pair -> 2; round 8: 2^24 + 2; round 4: + 4; round 2: + 8;
    # round 1: + 16.  Result 2^24 + 30.  (One ascending chain would give 2^24,
    # slices of single elements i mod 32 would give 2^24 + 24.)
    x = np.zeros((1, d), np.float32)
    w = np.zeros((1, d), np.float32)
    x[0, 0] = w[0, 0] = 2.0**12
    for j in range(1, 32):
        x[0, 8 * j] = w[0, 8 * j] = 1.0
    # (b) within one slice the chain is ascending: products 1, 1, 2^24 at
    # i = 0, 1, 2 give 1, 2, 2^24 + 2 (exact); descending would give 2^24.
    x2 = np.zeros((1, d), np.float32)
    w2 = np.zeros((1, d), np.float32)
    x2[0, 0] = w2[0, 0] = x2[0, 1] = w2[0, 1] = 1.0
    x2[0, 2] = w2[0, 2] = 2.0**12
    for dt in (torch.float32, torch.bfloat16):
        g = oracle.router_logits(torch.tensor(x, dtype=dt), torch.tensor(w, dtype=dt))
        assert float(g[0, 0]) == 16777246.0
        g2 = oracle.router_logits(torch.tensor(x2, dtype=dt), torch.tensor(w2, dtype=dt))
        assert float(g2[0, 0]) == 16777218.0


def test_softmax_matches_library_and_sums_to_one():
    rng = np.random.default_rng(13)
    g = (3 * rng.standard_normal((200, 64))).astype(np.float32)
    probs, idx, gate = oracle.softmax_topk(g, 4)
    ref = scipy.special.softmax(g.astype(np.float64), axis=1)
    np.testing.assert_allclose(probs, ref, rtol=1e-6, atol=1e-12)
    np.testing.assert_allclose(probs.astype(np.float64).sum(1), 1.0, atol=1e-6)
    np.testing.assert_array_equal(gate, np.take_along_axis(probs, idx, 1))


def _brute_topk(g, k):
    # stable sort on (-logit, expert): largest first, equal -> lower index
    T, E = g.shape
    out = np.empty((T, k), np.int64)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(g[t, e]), e))
        out[t] = order[:k]
    return out


@pytest.mark.parametrize("E,k", [(8, 2), (16, 1), (64, 2), (13, 4), (4, 4)])
def test_topk_brute_force(E, k):
    rng = np.random.default_rng(E * 10 + k)
    g = rng.standard_normal((300, E)).astype(np.float32)
    _, idx, _ = oracle.softmax_topk(g, k)
    np.testing.assert_array_equal(idx, _brute_topk(g, k))


def test_topk_exact_ties_prefer_lower_expert():
    # x = 0 makes every logit exactly the bias, so ties are exact.
    E, k, T, d = 12, 3, 20, 8
    rng = np.random.default_rng(14)
    bias = rng.integers(0, 3, size=E).astype(np.float32)
    x = torch.zeros(T, d, dtype=torch.bfloat16)
    w = torch.from_numpy(rng.standard_normal((E, d)).astype(np.float32)).to(torch.bfloat16)
    g, _, idx, _ = oracle.route(x, w, torch.from_numpy(bias), k)
    assert np.array_equal(g, np.broadcast_to(bias, (T, E)))
    np.testing.assert_array_equal(idx, _brute_topk(g, k))
    top = sorted(range(E), key=lambda e: (-bias[e], e))[:k]
    assert idx[0].tolist() == top


# --------------------------------------------------------------------------
# slot assignment
# --------------------------------------------------------------------------
def _random_routing(rng, T, E, k, skew=0.0):
    w = np.exp(-skew * np.log(np.arange(1, E + 1)))
    w = w / w.sum()
    idx = np.empty((T, k), np.int32)
    for t in range(T):
        idx[t] = rng.choice(E, size=k, replace=False, p=w)
    return idx


def _brute_assign(idx, E, C):
    # literal sort of all assignments by (expert, rank, token); the first C of
    # each expert are kept at positions 0..C-1
    T, k = idx.shape
    items = sorted(((int(idx[t, r]), r, t) for t in range(T) for r in range(k)))
    pos = np.full((T, k), -1, np.int64)
    seen = {}
    for e, r, t in items:
        p = seen.get(e, 0)
        seen[e] = p + 1
        if p < C:
            pos[t, r] = p
    return pos


@pytest.mark.parametrize("T,E,D,k,c,skew", [
    (50, 8, 4, 2, 1.0, 0.0), (64, 8, 4, 2, 1.0, 1.5), (97, 16, 4, 1, 1.25, 2.0),
    (33, 12, 3, 3, 0.5, 1.0), (40, 4, 2, 4, 1.0, 0.0), (128, 64, 8, 2, 1.0, 1.2)])
def test_assign_brute_force_and_invariants(T, E, D, k, c, skew):
    rng = np.random.default_rng(T + E + k)
    idx = _random_routing(rng, T, E, k, skew)
    s = oracle.assign(idx, E, D, c)
    C = s.C
    np.testing.assert_array_equal(s.slot_pos, _brute_assign(idx, E, C))
    # counts
    routed = np.bincount(idx.ravel(), minlength=E)
    np.testing.assert_array_equal(s.counts_routed, routed)
    assert s.counts_routed.sum() == T * k
    assert (s.counts_kept <= C).all()
    np.testing.assert_array_equal(s.counts_kept, np.minimum(routed, C))
    kept = int((s.slot_pos >= 0).sum())
    assert kept + s.dropped == T * k
    assert kept == s.counts_kept.sum() == s.expert_offsets[E]
    assert kept <= s.rows_max
    # per expert, kept positions are exactly 0..kept_e-1
    for e in range(E):
        p = sorted(s.slot_pos[idx == e][s.slot_pos[idx == e] >= 0].tolist())
        assert p == list(range(s.counts_kept[e]))
    # shard statistics: contiguous blocks of E/D experts
    per = E // D
    for sh in range(D):
        es = range(sh * per, (sh + 1) * per)
        assert s.shard_routed[sh] == routed[list(es)].sum()
        assert s.shard_offsets[sh] == s.expert_offsets[sh * per]
        # assignments dropped on the shard are at least what a shard holding
        # (E/D)*C slots must refuse
        dropped_on_shard = sum(int((s.slot_pos[idx == e] < 0).sum()) for e in es)
        assert dropped_on_shard >= max(0, s.shard_routed[sh] - per * C)
        if per * C == s.C_shard:
            # per-expert capacity is at least as strict as the pooled shard one
            assert dropped_on_shard >= s.shard_overflow[sh]
    assert s.shard_offsets[D] == kept
    # row_token inverts (t, r) -> row
    hit = np.zeros(kept, np.int64)
    for t in range(T):
        for r in range(k):
            if s.slot_pos[t, r] >= 0:
                row = s.expert_offsets[idx[t, r]] + s.slot_pos[t, r]
                assert s.row_token[row] == t
                hit[row] += 1
    assert (hit == 1).all()


def test_priority_rank_before_token():
    # a kept assignment implies every earlier assignment (rank, then token) to
    # the same expert is kept too
    rng = np.random.default_rng(21)
    idx = _random_routing(rng, 80, 6, 2, 1.0)
    s = oracle.assign(idx, 6, 3, 0.7)
    for e in range(6):
        order = [(r, t) for r in range(2) for t in range(80) if idx[t, r] == e]
        kept_flags = [s.slot_pos[t, r] >= 0 for r, t in order]
        assert kept_flags == sorted(kept_flags, reverse=True)


def test_more_capacity_never_drops_more():
    rng = np.random.default_rng(22)
    idx = _random_routing(rng, 100, 8, 2, 1.5)
    drops = [oracle.assign(idx, 8, 4, c).dropped for c in (0.25, 0.5, 1.0, 1.25, 2.0, 4.0)]
    assert drops == sorted(drops, reverse=True)
    assert oracle.assign(idx, 8, 4, math.inf).dropped == 0


def test_shard_overflow_is_the_capacity_formula():
    # the per-device rule of the capacity paragraph: a device receiving the
    # fraction p of the T*k assignments overflows by max(0, p*T*k - C_shard)
    rng = np.random.default_rng(23)
    T, E, D, k, c = 120, 8, 4, 2, 1.0
    idx = _random_routing(rng, T, E, k, 2.0)
    s = oracle.assign(idx, E, D, c)
    Cs = math.ceil(T * k / D * c)
    for sh in range(D):
        p = np.isin(idx, np.arange(sh * E // D, (sh + 1) * E // D)).sum() / (T * k)
        assert s.shard_overflow[sh] == max(0, round(p * T * k) - Cs)


# --------------------------------------------------------------------------
# dispatch, FFN, combine
# --------------------------------------------------------------------------
def test_dispatch_is_the_inverse_permutation():
    wl = moe_inputs.Workload("d", T=70, d=24, E=8, D=4, k=2, ffn=16, capacity_factor=0.8)
    inp = moe_inputs.make_inputs(wl)
    res = oracle.layer_forward(inp.x, inp.Wg, None, inp.W1, inp.W3, inp.W2, wl.k, wl.D,
                               wl.capacity_factor, oracle.SWIGLU)
    x16 = inp.x.view(torch.int16).numpy()
    xd16 = res.xd.view(np.int16)
    s = res.slots
    for t in range(wl.T):
        for r in range(wl.k):
            if s.slot_pos[t, r] >= 0:
                row = s.expert_offsets[res.topk_idx[t, r]] + s.slot_pos[t, r]
                assert np.array_equal(xd16[row], x16[t])


def _dense_ffn(x, W1, W3, W2, act):
    """Every expert on every token with library matmuls: [E, T, d] in fp64."""
    x = x.double()
    a = torch.einsum("td,efd->etf", x, W1.double())
    if act == "swiglu":
        h = F.silu(a) * torch.einsum("td,efd->etf", x, W3.double())
    else:
        h = F.gelu(a)  # exact erf form
    return torch.einsum("etf,edf->etd", h, W2.double())


@pytest.mark.parametrize("dtype,act", [("bf16", "swiglu"), ("f32", "gelu"), ("f32", "swiglu"),
                                       ("bf16", "gelu")])
def test_layer_equals_dense_evaluation_without_drops(dtype, act):
    wl = moe_inputs.Workload("n", T=48, d=32, E=8, D=4, k=2, ffn=40, capacity_factor=math.inf,
                             dtype=dtype, act=act, seed=5)
    inp = moe_inputs.make_inputs(wl)
    res = oracle.layer_forward(inp.x, inp.Wg, None, inp.W1, inp.W3, inp.W2, wl.k, wl.D,
                               wl.capacity_factor, oracle.act_code(act))
    assert res.slots.dropped == 0
    dense = _dense_ffn(inp.x, inp.W1, inp.W3, inp.W2, act).numpy()
    probs = res.probs.astype(np.float64)
    want = np.zeros((wl.T, wl.d))
    for t in range(wl.T):
        for e in res.topk_idx[t]:
            want[t] += probs[t, e] * dense[e, t]
    np.testing.assert_allclose(res.y, want, rtol=1e-12, atol=1e-12)


def test_drops_contribute_nothing_and_residual_passes():
    wl = moe_inputs.Workload("r", T=64, d=16, E=4, D=2, k=2, ffn=24, capacity_factor=0.25,
                             seed=6, zipf_s=3.0)
    inp = moe_inputs.make_inputs(wl)
    resid = torch.randn(wl.T, wl.d, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    res = oracle.layer_forward(inp.x, inp.Wg, inp.bias, inp.W1, inp.W3, inp.W2, wl.k, wl.D,
                               wl.capacity_factor, oracle.SWIGLU, residual=resid)
    assert res.slots.dropped > 0
    dense = _dense_ffn(inp.x, inp.W1, inp.W3, inp.W2, "swiglu").numpy()
    want = resid.double().numpy().copy()
    all_dropped = 0
    for t in range(wl.T):
        kept_any = False
        for r in range(wl.k):
            if res.slots.slot_pos[t, r] >= 0:
                kept_any = True
                want[t] += float(res.topk_gate[t, r]) * dense[res.topk_idx[t, r], t]
        all_dropped += not kept_any
    assert all_dropped > 0  # some tokens pass through the residual only
    np.testing.assert_allclose(res.y, want, rtol=1e-12, atol=1e-12)
    # sampled evaluation from the definition agrees with the step-by-step layer
    toks = [0, 5, 17, 63]
    y_tok = oracle.token_outputs(toks, inp.x, res.topk_idx, res.slots.slot_pos, res.topk_gate,
                                 inp.W1, inp.W3, inp.W2, oracle.SWIGLU, residual=resid)
    np.testing.assert_allclose(y_tok, res.y[toks], rtol=1e-12, atol=1e-12)


def test_dense_soft_mixture_when_every_expert_is_chosen():
    # k = E and no capacity limit: the layer is the dense soft mixture
    # sum_e p_e FFN_e(x)
    wl = moe_inputs.Workload("s", T=30, d=16, E=4, D=2, k=4, ffn=20, capacity_factor=math.inf,
                             dtype="f32", seed=7)
    inp = moe_inputs.make_inputs(wl)
    res = oracle.layer_forward(inp.x, inp.Wg, None, inp.W1, inp.W3, inp.W2, wl.k, wl.D,
                               wl.capacity_factor, oracle.SWIGLU)
    dense = _dense_ffn(inp.x, inp.W1, inp.W3, inp.W2, "swiglu")
    p = torch.softmax(inp.x.double() @ inp.Wg.double().T, dim=1)
    want = torch.einsum("te,etd->td", p, dense).numpy()
    # the oracle's gates are fp32 (rounded once), the reference's fp64
    np.testing.assert_allclose(res.y, want, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
def test_single_expert_is_a_plain_mlp(act):
    wl = moe_inputs.Workload("m", T=25, d=24, E=1, D=1, k=1, ffn=36, capacity_factor=1.0,
                             dtype="f32", act=act, seed=8)
    inp = moe_inputs.make_inputs(wl)
    res = oracle.layer_forward(inp.x, inp.Wg, None, inp.W1, inp.W3, inp.W2, 1, 1, 1.0,
                               oracle.act_code(act))
    assert (res.topk_gate == 1.0).all() and res.slots.dropped == 0
    x = inp.x.double()
    a = F.linear(x, inp.W1[0].double())
    h = F.silu(a) * F.linear(x, inp.W3[0].double()) if act == "swiglu" else F.gelu(a)
    want = F.linear(h, inp.W2[0].double()).numpy()
    np.testing.assert_allclose(res.y, want, rtol=1e-12, atol=1e-12)


def test_combine_converted_inputs_stay_alive():
    # inputs that need a dtype conversion (fp32 yd, int64 indices, fp64 gates)
    # must give the same result as inputs passed in the oracle's own dtypes
    rng = np.random.default_rng(31)
    T, d, k, E = 64, 32, 2, 8
    idx = _random_routing(rng, T, E, k)
    s = oracle.assign(idx, E, 4, 1.0)
    kept = int(s.expert_offsets[-1])
    yd64 = rng.standard_normal((kept, d))
    gate = rng.random((T, k)).astype(np.float32)
    want = oracle.combine(yd64, idx, s.slot_pos, gate, s.expert_offsets)
    for _ in range(20):
        got = oracle.combine(yd64.astype(np.float32), idx.astype(np.int64), s.slot_pos.astype(np.int64),
                             gate.astype(np.float64), s.expert_offsets.astype(np.int64))
        np.testing.assert_allclose(got, oracle.combine(yd64.astype(np.float32).astype(np.float64), idx,
                                                       s.slot_pos, gate, s.expert_offsets), rtol=0, atol=0)
    np.testing.assert_allclose(want, got, rtol=1e-6, atol=1e-6)


# --------------------------------------------------------------------------
# routing statistics (load-balancing term, entropy, drops, imbalance)
# --------------------------------------------------------------------------
def test_routing_stats_worked_example_closed_form():
    # The [TI] worked example (6 tokens, 8 experts, top-2): every token has
    # logit 3 at its rank-0 expert, 2 at its rank-1 expert, 0 elsewhere, so
    # p = (e^3, e^2, 1 x 6) / S with S = e^3 + e^2 + 6.  Per expert, the mean
    # probability times 6 is (#rank-0) e^3/S + (#rank-1) e^2/S + (#other)/S;
    # with the routed counts (0, 3, 3, 2, 2, 1, 1, 0) over 12 assignments the
    # load-balancing term E * sum f_e P_e works out by hand to
    # (16 e^3 + 12 e^2 + 44) / (9 S).
    rows = read_golden("worked_example.txt")
    choices = [tuple(int(v) for v in r[2:4]) for r in rows if r[0] == "choice"]
    assert len(choices) == 6
    E, k = 8, 2
    g = np.zeros((6, E), np.float32)
    for t, (a, b) in enumerate(choices):
        g[t, a], g[t, b] = 3.0, 2.0
    probs, idx, _ = oracle.softmax_topk(g, k)
    s = oracle.assign(idx, E, 4, 1.0)
    out, mp = oracle.routing_stats(probs, s.counts_routed, s.counts_kept, k)
    e3, e2 = math.exp(3.0), math.exp(2.0)
    S = e3 + e2 + 6.0
    assert out[0] == pytest.approx((16 * e3 + 12 * e2 + 44) / (9 * S), rel=1e-6)
    a, b, c = e3 / S, e2 / S, 1.0 / S
    assert out[1] == pytest.approx(-(a * math.log(a) + b * math.log(b) + 6 * c * math.log(c)), rel=1e-6)
    assert out[2] == pytest.approx(2 / 12)             # the two dropped assignments
    assert out[3] == pytest.approx(3 / (12 / 8))       # experts 1 and 2 carry 3 of a mean 1.5
    assert mp[0] == pytest.approx(c) and mp[7] == pytest.approx(c)  # unused experts
    assert mp[1] == pytest.approx((2 * a + b + 3 * c) / 6)


def test_routing_stats_limits():
    T, E, k = 64, 8, 1
    # perfectly uniform routing: aux 1, entropy ln E, no imbalance
    p = np.full((T, E), 1.0 / E, np.float32)
    counts = np.full(E, T // E, np.int32)
    out, mp = oracle.routing_stats(p, counts, counts, k)
    assert out[0] == pytest.approx(1.0, rel=1e-6)
    assert out[1] == pytest.approx(math.log(E), rel=1e-6)
    assert out[2] == 0.0 and out[3] == pytest.approx(1.0)
    assert np.allclose(mp, 1.0 / E)
    # everything to expert 0 with certainty: aux E, entropy 0, imbalance E
    p = np.zeros((T, E), np.float32)
    p[:, 0] = 1.0
    routed = np.zeros(E, np.int32)
    routed[0] = T
    kept = routed.copy()
    kept[0] = T // 4
    out, _ = oracle.routing_stats(p, routed, kept, k)
    assert out[0] == pytest.approx(E) and out[1] == 0.0
    assert out[2] == pytest.approx(0.75) and out[3] == pytest.approx(E)
    # no tokens: all zero
    out, _ = oracle.routing_stats(np.zeros((0, E), np.float32), np.zeros(E, np.int32),
                                  np.zeros(E, np.int32), k)
    assert (out == 0).all()


# --------------------------------------------------------------------------
# renormalised top-k gates and the shared expert
# --------------------------------------------------------------------------
def test_renormalised_gates_closed_forms():
    # worked example logits (3 at rank 0, 2 at rank 1, 0 elsewhere): the two
    # renormalised gates are e^3/(e^3+e^2) = 1/(1+e^-1) and 1/(1+e)
    g = np.zeros((6, 8), np.float32)
    for t, (a, b) in enumerate([(1, 2), (2, 1), (1, 3), (2, 4), (3, 5), (4, 6)]):
        g[t, a], g[t, b] = 3.0, 2.0
    _, idx, gate = oracle.softmax_topk(g, 2, renorm=True)
    _, idx0, _ = oracle.softmax_topk(g, 2)
    assert np.array_equal(idx, idx0)  # renormalising changes no choice
    assert np.allclose(gate[:, 0], 1 / (1 + math.exp(-1)), rtol=1e-7)
    assert np.allclose(gate[:, 1], 1 / (1 + math.exp(1)), rtol=1e-7)
    rng = np.random.default_rng(31)
    g = (2 * rng.standard_normal((100, 16))).astype(np.float32)
    # top-1: every gate is exactly one
    _, _, gate1 = oracle.softmax_topk(g, 1, renorm=True)
    assert (gate1 == 1.0).all()
    # k = E: renormalising over every expert changes nothing
    p_all, _, gate_all = oracle.softmax_topk(g, 16, renorm=True)
    _, _, gate_plain = oracle.softmax_topk(g, 16)
    np.testing.assert_allclose(gate_all, gate_plain, rtol=2e-7)
    # a token's k gates sum to one
    _, _, gate4 = oracle.softmax_topk(g, 4, renorm=True)
    np.testing.assert_allclose(gate4.astype(np.float64).sum(axis=1), 1.0, rtol=1e-6)


def test_shared_expert_against_dense_torch():
    torch.manual_seed(41)
    T, d, f = 37, 24, 40
    x = torch.randn(T, d)
    Ws1, Ws3 = torch.randn(f, d) / d**0.5, torch.randn(f, d) / d**0.5
    Ws2 = torch.randn(d, f) / f**0.5
    for act, w3 in ((oracle.SWIGLU, Ws3), (oracle.GELU, None)):
        got = oracle.shared_expert(x, Ws1, w3, Ws2, act)
        xd, a = x.double(), x.double() @ Ws1.double().T
        hh = torch.nn.functional.silu(a) * (xd @ Ws3.double().T) if w3 is not None else \
            torch.nn.functional.gelu(a)
        np.testing.assert_allclose(got, (hh @ Ws2.double().T).numpy(), rtol=1e-10, atol=1e-12)


def test_combine_adds_shared_after_routed_before_residual():
    # one token, one kept assignment with gate 1/2, values chosen so that the
    # three terms are exact: y = (0.5 * 6) + 1.25 + 0.5 = 4.75
    yd = np.array([[6.0]])
    y = oracle.combine(yd, np.array([[0]]), np.array([[0]]), np.array([[0.5]], np.float32),
                       np.array([0, 1]), residual=torch.tensor([[0.5]]), shared=np.array([[1.25]]))
    assert y[0, 0] == 4.75
    # a token whose only assignment was dropped gets shared + residual
    y = oracle.combine(yd, np.array([[0]]), np.array([[-1]]), np.array([[0.5]], np.float32),
                       np.array([0, 0]), residual=torch.tensor([[0.5]]), shared=np.array([[1.25]]))
    assert y[0, 0] == 1.75


# --------------------------------------------------------------------------
# expert-choice routing
# --------------------------------------------------------------------------
def test_expert_choice_against_a_literal_sort():
    rng = np.random.default_rng(61)
    for T, E, k, c in ((40, 8, 2, 1.0), (33, 5, 1, 0.6), (17, 4, 3, 2.0), (9, 3, 1, 0.2)):
        # scores on a coarse grid (negative ones too, and -0) so ties occur
        probs = (rng.integers(-3, 4, size=(T, E)) / 8.0).astype(np.float32)
        probs[rng.random((T, E)) < 0.05] = -0.0
        ec = oracle.expert_choice(probs, c, k)
        C = oracle.capacity(T, k, E, 1, c)[0]
        Cc = min(C, T)
        assert ec.C == Cc and ec.row_token.shape == (E * Cc,)
        for e in range(E):
            want = sorted(range(T), key=lambda t: (-float(probs[t, e]), t))[:Cc]
            assert ec.row_token[e * Cc:(e + 1) * Cc].tolist() == sorted(want)
            for t in range(T):
                row = ec.sel_row[t, e]
                if t in want:
                    assert ec.row_token[row] == t and e * Cc <= row < (e + 1) * Cc
                else:
                    assert row == -1


def test_expert_choice_with_every_token_is_the_dense_soft_mixture():
    # C >= T: every expert takes every token, so the layer is
    # sum_e p_e FFN_e(x), evaluated here densely with torch
    torch.manual_seed(62)
    T, d, E, f = 21, 16, 4, 24
    x = torch.randn(T, d)
    W1, W3 = torch.randn(E, f, d) / d**0.5, torch.randn(E, f, d) / d**0.5
    W2 = torch.randn(E, d, f) / f**0.5
    g = (2 * torch.randn(T, E)).numpy().astype(np.float32)
    probs, _, _ = oracle.softmax_topk(g, 1)
    ec = oracle.expert_choice(g, math.inf, 1)
    assert ec.C == T and (ec.sel_row >= 0).all()
    xd = oracle.dispatch(x, ec.row_token)
    yd = oracle.expert_ffn(xd, ec.expert_offsets, W1, W3, W2, oracle.SWIGLU)
    y = oracle.combine_expert_choice(yd, probs, ec.sel_row)
    xx = x.double()
    a = torch.einsum("td,efd->tef", xx, W1.double())
    u = torch.einsum("td,efd->tef", xx, W3.double())
    ye = torch.einsum("tef,edf->ted", torch.nn.functional.silu(a) * u, W2.double())
    want = torch.einsum("te,ted->td", torch.from_numpy(probs).double(), ye)
    np.testing.assert_allclose(y, want.numpy(), rtol=1e-9, atol=1e-12)


# --------------------------------------------------------------------------
# overflow rerouting to the next-best expert
# --------------------------------------------------------------------------
def _reroute_inputs(g, k):
    probs, idx2, gate2 = oracle.softmax_topk(g, 2 * k)
    return probs, idx2[:, :k], gate2[:, :k], idx2[:, k:], gate2[:, k:]


def test_reroute_worked_example():
    _, choices, _ = _worked_example()
    rows = read_golden("worked_example_reroute.txt")
    kv = {r[0]: r[1:] for r in rows if r[0] not in ("fallback", "rerouted")}
    fallbacks = [tuple(int(v) for v in r[2:4]) for r in rows if r[0] == "fallback"]
    moved = [tuple(int(v) for v in r[1:5]) for r in rows if r[0] == "rerouted"]
    E, k = 8, 2
    g = np.zeros((6, E), np.float32)
    for t, e0, e1 in choices:
        g[t, e0], g[t, e1] = 3.0, 2.0
    probs, idx, gate, fidx, fgate = _reroute_inputs(g, k)
    assert [tuple(r) for r in fidx.tolist()] == fallbacks
    s = oracle.assign_reroute(idx, gate, fidx, fgate, E, 4, 1.0)
    ints = lambda key: [int(v) for v in kv[key]]
    assert s.counts_routed.tolist() == ints("counts_routed")
    assert s.counts_kept.tolist() == ints("counts_kept")
    assert s.expert_offsets.tolist() == ints("expert_offsets")
    assert s.shard_offsets.tolist() == ints("shard_offsets")
    assert s.shard_routed.tolist() == ints("shard_routed")
    assert s.shard_overflow.tolist() == ints("shard_overflow")
    assert s.row_token.tolist() == ints("row_token")
    assert s.dropped == ints("dropped_after")[0] and s.rerouted == len(moved) == 2
    S = math.exp(3) + math.exp(2) + 6
    for t, r, e, pos in moved:
        assert (s.route_idx[t, r], s.slot_pos[t, r]) == (e, pos)
        assert abs(s.route_gate[t, r] - 1 / S) < 1e-8
    # every other assignment keeps its choice, gate and first-pass position
    plain = oracle.assign(idx, E, 4, 1.0)
    for t in range(6):
        for r in range(k):
            if (t, r) not in [(m[0], m[1]) for m in moved]:
                assert s.route_idx[t, r] == idx[t, r] and s.route_gate[t, r] == gate[t, r]
                assert s.slot_pos[t, r] == plain.slot_pos[t, r] >= 0


def _reroute_by_sorting(idx, fidx, E, C):
    """The second pass restated as a sort: every overflowing choice, ordered
    by (rank, token), bids for its fallback; expert e serves the first
    C - kept_first[e] bids it receives."""
    T, k = idx.shape
    # first-pass position by a literal sort of all (expert, rank, token)
    order = sorted(((int(idx[t, r]), r, t) for t in range(T) for r in range(k)))
    pos1, last, n = {}, None, 0
    for e, r, t in order:
        n = n + 1 if e == last else 0
        last = e
        pos1[(t, r)] = n
    kept_first = np.zeros(E, np.int64)
    for (t, r), p in pos1.items():
        kept_first[idx[t, r]] += p < C
    bids = sorted((r, t) for (t, r), p in pos1.items() if p >= C)
    served = {e: [] for e in range(E)}
    target = {}
    for r, t in bids:
        j = sum(pos1[(t, q)] >= C for q in range(r))
        e = int(fidx[t, j])
        target[(t, r)] = e
        served[e].append((t, r))
    slot = {}
    for e, lst in served.items():
        for i, tr in enumerate(lst):
            slot[tr] = kept_first[e] + i if kept_first[e] + i < C else -1
    return pos1, target, slot


@pytest.mark.parametrize("T,E,k,c,skew", [(300, 16, 2, 1.0, 2.0), (257, 8, 1, 0.5, 1.0),
                                          (190, 32, 4, 1.25, 3.0), (64, 4, 2, 0.3, 0.0)])
def test_reroute_against_sorting_and_invariants(T, E, k, c, skew):
    rng = np.random.default_rng(T + E)
    g = (rng.standard_normal((T, E)) + skew * np.log1p(np.arange(E))[None, ::-1]).astype(np.float32)
    probs, idx, gate, fidx, fgate = _reroute_inputs(g, k)
    s = oracle.assign_reroute(idx, gate, fidx, fgate, E, 2 if E % 2 == 0 else 1, c)
    plain = oracle.assign(idx, E, 2 if E % 2 == 0 else 1, c)
    C = s.C
    pos1, target, slot = _reroute_by_sorting(idx, fidx, E, C)
    n_moved = 0
    for t in range(T):
        assert len(set(s.route_idx[t].tolist())) == k  # a token's experts stay distinct
        for r in range(k):
            if pos1[(t, r)] < C:
                assert s.route_idx[t, r] == idx[t, r] and s.slot_pos[t, r] == pos1[(t, r)]
                assert s.route_gate[t, r] == gate[t, r]
            else:
                e = target[(t, r)]
                j = list(fidx[t]).index(e)
                assert s.route_idx[t, r] == e and s.route_gate[t, r] == fgate[t, j] == probs[t, e]
                assert s.slot_pos[t, r] == slot[(t, r)]
                if slot[(t, r)] < 0:
                    assert s.counts_kept[e] == C  # dropped only when the fallback is full
                else:
                    n_moved += 1
    assert s.rerouted == n_moved and s.rerouted + s.dropped == plain.dropped
    assert (s.counts_kept <= C).all() and (s.counts_kept >= plain.counts_kept).all()
    assert np.array_equal(s.counts_routed, plain.counts_routed)
    assert np.array_equal(s.expert_offsets, np.concatenate([[0], np.cumsum(s.counts_kept)]))
    for t in range(T):
        for r in range(k):
            if s.slot_pos[t, r] >= 0:
                assert s.row_token[s.expert_offsets[s.route_idx[t, r]] + s.slot_pos[t, r]] == t
    if skew > 0:
        assert plain.dropped > 0 and s.rerouted > 0  # the cases do exercise the second pass


def test_reroute_without_overflow_is_the_plain_assignment():
    rng = np.random.default_rng(5)
    g = rng.standard_normal((200, 8)).astype(np.float32)
    _, idx, gate, fidx, fgate = _reroute_inputs(g, 2)
    for c in (math.inf, 8.0):
        s = oracle.assign_reroute(idx, gate, fidx, fgate, 8, 4, c)
        p = oracle.assign(idx, 8, 4, c)
        assert p.dropped == 0 and s.rerouted == 0 and s.dropped == 0
        assert np.array_equal(s.route_idx, idx) and np.array_equal(s.route_gate, gate)
        for f in ("slot_pos", "counts_routed", "counts_kept", "expert_offsets", "shard_offsets", "row_token"):
            assert np.array_equal(getattr(s, f), getattr(p, f)), f
