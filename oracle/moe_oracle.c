/*
 * moe_oracle.c -- plain, slow CPU oracle of the capacity-limited top-k
 * mixture-of-experts layer forward.  TEST INFRASTRUCTURE ONLY: it is used by
 * the tests, by the package's smoke check and by the benchmark's CPU-baseline
 * leg.  The CUDA library never links, calls or includes anything here, and
 * this file shares no code, header or table with it.
 *
 * Every function follows one step of the method as the expert-parallelism
 * pages state it, written out by direct loops:
 *
 *   [NG] "Expert Parallelism" notes page (narrativegoldmine.com):
 *        "Components and Architecture" and
 *        "Formal Algorithm: Expert Parallelism Forward Pass".
 *   [TI] "Expert Parallelism" (theinfinity.ai, Systems / Distributed):
 *        the per-device capacity and overflow paragraph and the
 *        6-token / 8-expert / 4-device worked-example caption.
 *   [AS] "Expert Parallelism and the All-to-All Bottleneck"
 *        (ashishsrivastav.com): "The Mechanism of Expert Parallelism",
 *        phases 1-4, and "The All-to-All Communication Pattern".
 *
 * Where the pages are silent the plainest reading is taken; each reading is
 * named at the function that applies it.
 *
 * Precision: router logits in fp32 in one fixed order (the integer top-k
 * decision is taken in the precision of the CUDA path, fp32); everything
 * else (softmax, expert FFN, combine) in fp64.  Build with
 * -ffp-contract=off so that only the explicit fmaf() calls are fused.
 *
 * Parity status per function (what pins it, see the oracle tests):
 *   oracle_capacity        pinned (closed forms of [TI] and the workloads)
 *   oracle_router_logits   pinned (exact small-integer dot products, fp64
 *                          bound, tie cases, a hand-derived rounding case
 *                          that fixes the slice-and-butterfly order)
 *   oracle_softmax_topk    pinned (worked-example closed form, brute force)
 *   oracle_assign          pinned ([TI] worked example, invariants, brute force)
 *   oracle_dispatch        pinned (inverse permutation property)
 *   oracle_expert_ffn      pinned (dense soft-MoE / plain MLP special cases
 *                          against a library matmul)
 *   oracle_combine         pinned (dense all-experts brute force)
 *   oracle_assign_reroute  pinned ([TI] worked example with its two dropped
 *                          assignments rerouted by hand, invariants, no
 *                          overflow = plain assignment)
 *   oracle_routing_stats   pinned (closed forms: uniform, one-hot, hand
 *                          example)
 *   oracle_expert_choice   pinned (brute-force sort, ties, c = infinity)
 *   oracle_combine_expert_choice  pinned (dense brute force when every
 *                          expert takes every token)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_SWIGLU 0
#define ORACLE_GELU 1

/* A bf16 value is the upper 16 bits of the fp32 with the same value. */
static float bf16_bits_to_float(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Element i of a tensor stored as fp32 or bf16, returned exactly as fp32. */
static float elem(const void* p, int dtype, size_t i) {
    if (dtype == ORACLE_BF16) return bf16_bits_to_float(((const uint16_t*)p)[i]);
    return ((const float*)p)[i];
}

/* ------------------------------------------------------------------------ *
 * Capacity.  [TI] capacity paragraph: a device expecting B*k/D tokens
 * provisions C = ceil((B*k/D)*c).  Per expert, as the layer drops per expert,
 * the same rule with E in place of D: C = ceil((T*k/E)*c), evaluated in double
 * in that order.  [NG] "Capacity Factor and Token Dropping": c times the mean
 * load.  An expert can receive at most T assignments (the k choices of a token
 * are distinct), so C is clamped to T; c = +inf means C = T (nothing dropped).
 * C_shard (the per-device figure of [TI]) is clamped to T*k.
 * rows_max = min(E*C, T*k) bounds the kept assignments.
 * ------------------------------------------------------------------------ */
int oracle_capacity(int64_t T, int k, int E, int D, double c,
                    int64_t* C_expert, int64_t* C_shard, int64_t* rows_max) {
    if (T < 0 || k < 1 || E < 1 || D < 1 || !(c > 0.0)) return 1;
    int64_t Tk = T * (int64_t)k;
    int64_t ce, cs;
    if (isinf(c)) {
        ce = T;
        cs = Tk;
    } else {
        double ve = ceil(((double)Tk / (double)E) * c);
        double vs = ceil(((double)Tk / (double)D) * c);
        ce = ve >= (double)T ? T : (int64_t)ve;
        cs = vs >= (double)Tk ? Tk : (int64_t)vs;
    }
    int64_t rm = (int64_t)E * ce;
    if (rm > Tk) rm = Tk;
    *C_expert = ce;
    *C_shard = cs;
    *rows_max = rm;
    return 0;
}

/* ------------------------------------------------------------------------ *
 * Router logits.  [NG] formal algorithm, gate computation: g_t = the routing
 * linear projection of x_t, one logit per expert.  [NG] "Components and
 * Architecture", gating network: an optional per-expert bias on the logits.
 *
 * Fixed summation order (the pages give none; the top-k decision must be
 * reproducible bit for bit).  The hidden index is dealt into 32 slices of
 * runs of 8 consecutive elements: slice j holds i = 256*m + 8*j + q
 * (m = 0, 1, ...; q = 0..7).  Each slice sum is one fp32 fused multiply-add
 * chain over its elements in ascending i, starting from +0.  The 32 slice
 * sums are then combined by a fixed butterfly: for o = 16, 8, 4, 2, 1 every
 * slice j is replaced, all at once, by s[j] + s[j xor o] (fp32 add); after the
 * five rounds every s[j] holds the same value, s[0].  Then g = s[0] + b[e].
 * Wg is [E, d] (nn.Linear out x in).
 * ------------------------------------------------------------------------ */
void oracle_router_logits(int64_t T, int d, int E, int dtype,
                          const void* x, const void* Wg, const float* bias,
                          float* logits /* [T, E] */) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            float s[32];
            for (int j = 0; j < 32; ++j) s[j] = 0.0f;
            for (int i = 0; i < d; ++i) {
                const int j = (i / 8) % 32;
                s[j] = fmaf(elem(x, dtype, (size_t)t * d + i),
                            elem(Wg, dtype, (size_t)e * d + i), s[j]);
            }
            for (int o = 16; o >= 1; o /= 2) {
                float n[32];
                for (int j = 0; j < 32; ++j) n[j] = s[j] + s[j ^ o];
                for (int j = 0; j < 32; ++j) s[j] = n[j];
            }
            float g = s[0];
            if (bias) g = g + bias[e];
            logits[(size_t)t * E + e] = g;
        }
    }
}

/* ------------------------------------------------------------------------ *
 * Softmax, top-k, gates.  [NG] formal algorithm: p_t = softmax(g_t / tau)
 * (tau = 1, the pages fix no value); expert selection e(t) = argmax p_t with
 * gate w_t = p_{t,e(t)}; [NG] "Components and Architecture" and the [AS]
 * routing phase: the top-k experts are selected.
 *
 * Readings: softmax is strictly increasing, so the k largest p are the k
 * largest g; ranking is done on the fp32 logits, largest first, equal logits
 * ranked by the lower expert index.  Rank r = 0 is the largest.  The gate of
 * choice r is the softmax probability of that expert, not renormalised over
 * the k choices.  Softmax in double with the maximum subtracted, rounded to
 * fp32 once.
 *
 * With renorm set (the [NG] "Major Variants" top-2 combination read as a
 * convex combination of the chosen experts): gate r is the softmax over the k
 * chosen logits only, exp(g_r - m) / sum over chosen c of exp(g_c - m), so a
 * token's k gates sum to one.
 * ------------------------------------------------------------------------ */
void oracle_softmax_topk(int64_t T, int E, int k, int renorm, const float* logits,
                         float* probs /* [T, E] or NULL */,
                         int32_t* topk_idx /* [T, k] */,
                         float* topk_gate /* [T, k] */) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const float* g = logits + (size_t)t * E;
        double m = g[0];
        for (int e = 1; e < E; ++e)
            if (g[e] > m) m = g[e];
        double sum = 0.0;
        for (int e = 0; e < E; ++e) sum += exp((double)g[e] - m);
        /* chosen[] marks experts already taken by a higher rank */
        unsigned char chosen[1024];
        for (int e = 0; e < E; ++e) chosen[e] = 0;
        double chosen_sum = 0.0;
        for (int r = 0; r < k; ++r) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (chosen[e]) continue;
                if (best < 0 || g[e] > g[best]) best = e; /* strict: ties keep lower e */
            }
            chosen[best] = 1;
            topk_idx[(size_t)t * k + r] = best;
            chosen_sum += exp((double)g[best] - m);
        }
        const double denom = renorm ? chosen_sum : sum;
        for (int r = 0; r < k; ++r) {
            const int e = topk_idx[(size_t)t * k + r];
            topk_gate[(size_t)t * k + r] = (float)(exp((double)g[e] - m) / denom);
        }
        if (probs)
            for (int e = 0; e < E; ++e)
                probs[(size_t)t * E + e] = (float)(exp((double)g[e] - m) / sum);
    }
}

/* ------------------------------------------------------------------------ *
 * Slot assignment and token dropping.  [NG] "Capacity Factor and Token
 * Dropping": an expert takes at most C assignments, the rest are dropped.
 * [TI] capacity paragraph: per-device overflow max(0, p*B*k - C), where p*B*k
 * is the number of assignments the device receives.
 *
 * Reading (the pages fix no order): assignments are served in the priority
 * (choice rank r, then token index t): every rank-0 choice in token order,
 * then every rank-1 choice, and so on.  pos(t, r) is the number of earlier
 * assignments in that order to the same expert; kept iff pos < C.
 * Experts sit on shards in contiguous blocks of E/D ([AS] all-to-all pattern:
 * 64 experts on 8 GPUs, expert 55 on GPU 6, expert 5 on GPU 0).
 *
 * Outputs: slot_pos (pos or -1 when dropped), per-expert routed and kept
 * counts, expert_offsets (exclusive scan of kept counts, E+1 entries),
 * shard_offsets[s] = expert_offsets[s*E/D] (D+1 entries), per-shard routed
 * count and overflow, row_token[expert_offsets[e] + pos] = t for every kept
 * (t, r), and the total number of dropped assignments.
 * ------------------------------------------------------------------------ */
void oracle_assign(int64_t T, int E, int D, int k, int64_t C, int64_t C_shard,
                   const int32_t* topk_idx, int32_t* slot_pos,
                   int32_t* counts_routed, int32_t* counts_kept,
                   int32_t* expert_offsets, int32_t* shard_offsets,
                   int32_t* shard_routed, int32_t* shard_overflow,
                   int32_t* row_token, int64_t* dropped) {
    int64_t* cnt = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    int64_t ndrop = 0;
    for (int r = 0; r < k; ++r) {
        for (int64_t t = 0; t < T; ++t) {
            int e = topk_idx[(size_t)t * k + r];
            int64_t pos = cnt[e]++;
            if (pos < C) {
                slot_pos[(size_t)t * k + r] = (int32_t)pos;
            } else {
                slot_pos[(size_t)t * k + r] = -1;
                ++ndrop;
            }
        }
    }
    int64_t off = 0;
    for (int e = 0; e < E; ++e) {
        counts_routed[e] = (int32_t)cnt[e];
        counts_kept[e] = (int32_t)(cnt[e] < C ? cnt[e] : C);
        expert_offsets[e] = (int32_t)off;
        off += counts_kept[e];
    }
    expert_offsets[E] = (int32_t)off;
    int per = E / D;
    for (int s = 0; s < D; ++s) {
        int64_t routed = 0;
        for (int e = s * per; e < (s + 1) * per; ++e) routed += cnt[e];
        shard_routed[s] = (int32_t)routed;
        shard_overflow[s] = (int32_t)(routed > C_shard ? routed - C_shard : 0);
        shard_offsets[s] = expert_offsets[s * per];
    }
    shard_offsets[D] = expert_offsets[E];
    for (int64_t t = 0; t < T; ++t)
        for (int r = 0; r < k; ++r) {
            int32_t pos = slot_pos[(size_t)t * k + r];
            if (pos >= 0) row_token[expert_offsets[topk_idx[(size_t)t * k + r]] + pos] = (int32_t)t;
        }
    *dropped = ndrop;
    free(cnt);
}

/* ------------------------------------------------------------------------ *
 * Slot assignment with overflow rerouting.  [NG] "Capacity Factor and Token
 * Dropping" and the load-imbalance list: tokens routed to a full expert are
 * dropped or redirected to a secondary expert, the next-best one; [NG]
 * "Components and Architecture": overflow tokens handled by a fallback
 * routing.
 *
 * Readings (the pages name the fallback only):
 *  - first pass: the plain assignment above on the k choices -- every
 *    first choice keeps the slot it has without rerouting;
 *  - the next-best expert of a token is the next one in its descending-logit
 *    order after its k choices (fallback_idx[t, j] = its rank k + j expert,
 *    fallback_gate[t, j] = that expert's softmax probability); the j-th
 *    overflowing choice of token t (ascending rank) goes to fallback j, so a
 *    token's experts stay distinct;
 *  - rerouted assignments take the capacity the first pass left, in the same
 *    priority order (rank r of the overflowing choice, then token):
 *    pos = kept_first[e] + number of earlier rerouted assignments to e; kept
 *    iff pos < C.  One level only: a rerouted assignment that finds its
 *    fallback full is dropped;
 *  - the assignment then counts for its fallback expert: route_idx[t, r] is
 *    the expert that serves it, route_gate[t, r] its weight (the fallback's
 *    probability when rerouted), slot_pos[t, r] its position or -1.
 * counts_routed and the shard statistics describe the k choices (before
 * capacity, as in the plain assignment); counts_kept, expert_offsets,
 * shard_offsets and row_token describe the rows after rerouting;
 * *rerouted = rerouted assignments that got a slot, *dropped = assignments
 * with no slot at the end.
 * ------------------------------------------------------------------------ */
void oracle_assign_reroute(int64_t T, int E, int D, int k, int64_t C, int64_t C_shard,
                           const int32_t* topk_idx, const float* topk_gate,
                           const int32_t* fallback_idx, const float* fallback_gate,
                           int32_t* route_idx, float* route_gate, int32_t* slot_pos,
                           int32_t* counts_routed, int32_t* counts_kept,
                           int32_t* expert_offsets, int32_t* shard_offsets,
                           int32_t* shard_routed, int32_t* shard_overflow,
                           int32_t* row_token, int64_t* rerouted, int64_t* dropped) {
    int64_t* cnt = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    int64_t* fill = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    int64_t* first_pos = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T * k > 0 ? T * k : 1));
    /* first pass: the k choices in priority order */
    for (int r = 0; r < k; ++r)
        for (int64_t t = 0; t < T; ++t) first_pos[(size_t)t * k + r] = cnt[topk_idx[(size_t)t * k + r]]++;
    for (int e = 0; e < E; ++e) fill[e] = cnt[e] < C ? cnt[e] : C;
    /* second pass: overflowing choices go to their fallback, same order */
    int64_t nre = 0, ndrop = 0;
    for (int r = 0; r < k; ++r) {
        for (int64_t t = 0; t < T; ++t) {
            const size_t i = (size_t)t * k + r;
            if (first_pos[i] < C) {
                route_idx[i] = topk_idx[i];
                route_gate[i] = topk_gate[i];
                slot_pos[i] = (int32_t)first_pos[i];
                continue;
            }
            int j = 0; /* overflowing choices of t ranked before r */
            for (int q = 0; q < r; ++q) j += first_pos[(size_t)t * k + q] >= C;
            const int e = fallback_idx[(size_t)t * k + j];
            route_idx[i] = e;
            route_gate[i] = fallback_gate[(size_t)t * k + j];
            const int64_t pos = fill[e]++;
            if (pos < C) {
                slot_pos[i] = (int32_t)pos;
                ++nre;
            } else {
                slot_pos[i] = -1;
                ++ndrop;
            }
        }
    }
    int64_t off = 0;
    for (int e = 0; e < E; ++e) {
        counts_routed[e] = (int32_t)cnt[e];
        counts_kept[e] = (int32_t)(fill[e] < C ? fill[e] : C);
        expert_offsets[e] = (int32_t)off;
        off += counts_kept[e];
    }
    expert_offsets[E] = (int32_t)off;
    int per = E / D;
    for (int s = 0; s < D; ++s) {
        int64_t routed = 0;
        for (int e = s * per; e < (s + 1) * per; ++e) routed += cnt[e];
        shard_routed[s] = (int32_t)routed;
        shard_overflow[s] = (int32_t)(routed > C_shard ? routed - C_shard : 0);
        shard_offsets[s] = expert_offsets[s * per];
    }
    shard_offsets[D] = expert_offsets[E];
    for (int64_t t = 0; t < T; ++t)
        for (int r = 0; r < k; ++r) {
            const size_t i = (size_t)t * k + r;
            if (slot_pos[i] >= 0) row_token[expert_offsets[route_idx[i]] + slot_pos[i]] = (int32_t)t;
        }
    *rerouted = nre;
    *dropped = ndrop;
    free(first_pos);
    free(fill);
    free(cnt);
}

/* ------------------------------------------------------------------------ *
 * Dispatch (pack).  [AS] phase 2: rows are repacked so that each row holds a
 * token destined for one expert; [NG] dispatch tensor.  Here the pack is a
 * local permutation: xd[row] = x[row_token[row]] for the kept rows, in
 * expert-major order (and so grouped by shard).  A byte copy.
 * ------------------------------------------------------------------------ */
void oracle_dispatch(int64_t rows, int d, int elem_bytes, const void* x,
                     const int32_t* row_token, void* xd) {
    size_t rb = (size_t)d * (size_t)elem_bytes;
    for (int64_t row = 0; row < rows; ++row)
        memcpy((char*)xd + (size_t)row * rb, (const char*)x + (size_t)row_token[row] * rb, rb);
}

/* ------------------------------------------------------------------------ *
 * Expert FFN of one row.  [NG] "Components and Architecture", expert GEMM: a
 * standard transformer MLP per expert; [AS] phase 3.  Forms (no biases,
 * weights nn.Linear out x in):
 *   SwiGLU: a = W1[e] x, u = W3[e] x, h = a * sigmoid(a) * u, y = W2[e] h
 *   GeLU:   a = W1[e] x, h = 0.5 a (1 + erf(a / sqrt 2)),     y = W2[e] h
 * All in double from the stored (fp32 or bf16) values; h is not rounded.
 * ------------------------------------------------------------------------ */
static void ffn_row(int d, int f, int act, int dtype, const void* xrow_base, size_t xrow_off,
                    int e, const void* W1, const void* W3, const void* W2,
                    double* h /* scratch [f] */, double* y /* [d] */) {
    for (int j = 0; j < f; ++j) {
        double a = 0.0, u = 0.0;
        for (int i = 0; i < d; ++i) {
            double xi = elem(xrow_base, dtype, xrow_off + i);
            a += xi * (double)elem(W1, dtype, ((size_t)e * f + j) * d + i);
            if (act == ORACLE_SWIGLU)
                u += xi * (double)elem(W3, dtype, ((size_t)e * f + j) * d + i);
        }
        if (act == ORACLE_SWIGLU)
            h[j] = a / (1.0 + exp(-a)) * u;
        else
            h[j] = 0.5 * a * (1.0 + erf(a / sqrt(2.0)));
    }
    for (int o = 0; o < d; ++o) {
        double s = 0.0;
        for (int j = 0; j < f; ++j) s += h[j] * (double)elem(W2, dtype, ((size_t)e * d + o) * f + j);
        y[o] = s;
    }
}

/* Expert FFN over the packed rows: yd[row] = FFN_e(xd[row]) for every row of
 * expert e, i.e. rows expert_offsets[e] .. expert_offsets[e+1]-1. */
void oracle_expert_ffn(int E, int d, int f, int act, int dtype, const void* xd,
                       const int32_t* expert_offsets, const void* W1, const void* W3,
                       const void* W2, double* yd /* [rows, d] */) {
    for (int e = 0; e < E; ++e) {
        int64_t r0 = expert_offsets[e], r1 = expert_offsets[e + 1];
#pragma omp parallel
        {
            double* h = (double*)malloc(sizeof(double) * (size_t)f);
#pragma omp for schedule(static)
            for (int64_t row = r0; row < r1; ++row)
                ffn_row(d, f, act, dtype, xd, (size_t)row * d, e, W1, W3, W2, h, yd + (size_t)row * d);
            free(h);
        }
    }
}

/* ------------------------------------------------------------------------ *
 * Combine.  [NG] expert combine and formal algorithm: each returned
 * activation is multiplied by its gating weight and a token's k outputs are
 * summed, back in token order ([AS] phase 4); then the residual ([NG]
 * residual addition).  A dropped assignment adds nothing: the token passes
 * through the residual only ([NG] "Capacity Factor and Token Dropping").
 *     y[t] = residual[t] + sum over kept r of gate[t,r] * yd[row(t,r)]
 * residual NULL means no residual term.  A shared expert ([NG] "Major
 * Variants": a dense expert every token goes through, next to the routed
 * ones) adds its output ys[t] after the routed sum and before the residual:
 *     y[t] = residual[t] + (sum over kept r ... + ys[t])
 * shared NULL means no shared expert.
 * ------------------------------------------------------------------------ */
void oracle_combine(int64_t T, int d, int k, int dtype, const int32_t* topk_idx,
                    const int32_t* slot_pos, const float* topk_gate,
                    const int32_t* expert_offsets, const double* yd,
                    const double* shared /* [T, d] or NULL */,
                    const void* residual, double* y /* [T, d] */) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int o = 0; o < d; ++o) {
            double s = 0.0;
            for (int r = 0; r < k; ++r) {
                int32_t pos = slot_pos[(size_t)t * k + r];
                if (pos < 0) continue;
                int64_t row = (int64_t)expert_offsets[topk_idx[(size_t)t * k + r]] + pos;
                s += (double)topk_gate[(size_t)t * k + r] * yd[(size_t)row * d + o];
            }
            if (shared) s += shared[(size_t)t * d + o];
            if (residual) s += (double)elem(residual, dtype, (size_t)t * d + o);
            y[(size_t)t * d + o] = s;
        }
    }
}

/* ------------------------------------------------------------------------ *
 * Layer output of selected tokens, straight from the definition: for each
 * listed token t, y[t] = residual[t] + sum over kept r of
 * gate[t,r] * FFN_{idx[t,r]}(x[t]).  Uses x directly (not the packed rows),
 * so the whole-layer check does not lean on dispatch.  For workloads whose
 * full FFN is too slow on the CPU.
 * ------------------------------------------------------------------------ */
void oracle_token_outputs(int64_t n, const int64_t* tokens, int d, int f, int k, int act,
                          int dtype, const void* x, const int32_t* topk_idx,
                          const int32_t* slot_pos, const float* topk_gate,
                          const void* W1, const void* W3, const void* W2,
                          const void* residual, double* y /* [n, d] */) {
#pragma omp parallel
    {
        double* h = (double*)malloc(sizeof(double) * (size_t)f);
        double* ye = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t q = 0; q < n; ++q) {
            int64_t t = tokens[q];
            double* yo = y + (size_t)q * d;
            for (int o = 0; o < d; ++o) yo[o] = 0.0;
            for (int r = 0; r < k; ++r) {
                if (slot_pos[(size_t)t * k + r] < 0) continue;
                int e = topk_idx[(size_t)t * k + r];
                ffn_row(d, f, act, dtype, x, (size_t)t * d, e, W1, W3, W2, h, ye);
                for (int o = 0; o < d; ++o) yo[o] += (double)topk_gate[(size_t)t * k + r] * ye[o];
            }
            if (residual)
                for (int o = 0; o < d; ++o) yo[o] += (double)elem(residual, dtype, (size_t)t * d + o);
        }
        free(h);
        free(ye);
    }
}

/* ------------------------------------------------------------------------ *
 * Routing statistics.  [NG] "Components and Architecture" and formal
 * algorithm: the auxiliary load-balancing term is the sum over experts of
 * the fraction of tokens sent to the expert times the fraction of router
 * probability it receives; [IS] glossary: the load-balancing loss;
 * "Expert Parallelism" intro page (nhimg.org), practitioner guidance: watch
 * expert utilisation and routing entropy.
 *
 * Readings (the pages give the product form, not the normalisation):
 *   f_e   = routed_e / (T*k), the share of the T*k pre-drop assignments;
 *   P_e   = (1/T) sum_t p[t,e], the mean router probability;
 *   aux   = E * sum_e f_e * P_e (the Switch scaling: 1 for perfectly uniform
 *           routing, E when every token sends everything to one expert);
 *   H     = (1/T) sum_t -sum_e p[t,e] ln p[t,e], with 0 ln 0 = 0 (nats);
 *   drop  = (sum_e routed_e - kept_e) / (T*k);
 *   imbal = max_e routed_e / (T*k/E), the hottest expert's load over the mean.
 * All sums in double; out = {aux, H, drop, imbal}, mean_prob = P (may be
 * NULL).  T = 0 gives zeros.
 * ------------------------------------------------------------------------ */
void oracle_routing_stats(int64_t T, int E, int k, const float* probs /* [T, E] */,
                          const int32_t* counts_routed, const int32_t* counts_kept,
                          double* out /* [4] */, double* mean_prob /* [E] or NULL */) {
    double* P = (double*)calloc((size_t)E, sizeof(double));
    double H = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        double ht = 0.0;
        for (int e = 0; e < E; ++e) {
            const double p = (double)probs[(size_t)t * E + e];
            P[e] += p;
            if (p > 0.0) ht -= p * log(p);
        }
        H += ht;
    }
    double aux = 0.0, routed = 0.0, kept = 0.0, maxr = 0.0;
    const double Tk = (double)T * (double)k;
    for (int e = 0; e < E; ++e) {
        if (T > 0) P[e] /= (double)T;
        const double f = Tk > 0.0 ? (double)counts_routed[e] / Tk : 0.0;
        aux += f * P[e];
        routed += counts_routed[e];
        kept += counts_kept[e];
        if (counts_routed[e] > maxr) maxr = counts_routed[e];
        if (mean_prob) mean_prob[e] = P[e];
    }
    out[0] = (double)E * aux;
    out[1] = T > 0 ? H / (double)T : 0.0;
    out[2] = Tk > 0.0 ? (routed - kept) / Tk : 0.0;
    out[3] = Tk > 0.0 ? maxr / (Tk / (double)E) : 0.0;
    free(P);
}

/* ------------------------------------------------------------------------ *
 * Expert-choice routing.  [NG] "Major Variants": instead of each token
 * choosing its experts, each expert chooses its tokens, which balances the
 * load by construction.
 *
 * Readings (the pages name the variant only): expert e takes the
 * Cc = min(C, T) tokens with the largest router score, the fp32 logit
 * g[t, e] of the routing projection (the integer decision is taken on the
 * same fp32 values the router computes, in its fixed order), equal scores
 * taken in ascending token order (C from the capacity rule, k read as the
 * average number of experts per token); its rows are its tokens in ascending
 * token order, at expert_offsets[e] = e * Cc; the weight of (t, e) is the
 * token's softmax probability probs[t, e]; a token sums the outputs of the
 * experts that took it in ascending expert order (none: 0, plus the
 * residual).
 * Outputs: row_token[e * Cc + j] = j-th token of expert e; sel_row[t*E + e]
 * = its row, or -1 when e did not take t.
 * ------------------------------------------------------------------------ */
void oracle_expert_choice(int64_t T, int E, int64_t C, const float* score /* [T, E] */,
                          int32_t* row_token /* [E * min(C, T)] */,
                          int32_t* sel_row /* [T, E] */) {
    const int64_t Cc = C < T ? C : T;
    for (int64_t i = 0; i < T * (int64_t)E; ++i) sel_row[i] = -1;
#pragma omp parallel
    {
        int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)(T > 0 ? T : 1));
        unsigned char* take = (unsigned char*)malloc((size_t)(T > 0 ? T : 1));
#pragma omp for schedule(static)
        for (int e = 0; e < E; ++e) {
            /* selection sort by (score descending, token ascending), kept
               plain: the first Cc positions are the chosen tokens */
            for (int64_t t = 0; t < T; ++t) {
                order[t] = t;
                take[t] = 0;
            }
            for (int64_t j = 0; j < Cc; ++j) {
                int64_t best = j;
                for (int64_t q = j + 1; q < T; ++q) {
                    const float pb = score[(size_t)order[best] * E + e];
                    const float pq = score[(size_t)order[q] * E + e];
                    if (pq > pb || (pq == pb && order[q] < order[best])) best = q;
                }
                const int64_t tmp = order[j];
                order[j] = order[best];
                order[best] = tmp;
                take[order[j]] = 1;
            }
            int64_t pos = 0;
            for (int64_t t = 0; t < T; ++t) {
                if (!take[t]) continue;
                row_token[(size_t)e * Cc + pos] = (int32_t)t;
                sel_row[(size_t)t * E + e] = (int32_t)(e * Cc + pos);
                ++pos;
            }
        }
        free(order);
        free(take);
    }
}

/* Combine for expert-choice routing: y[t] = sum over experts e that took t,
 * in ascending e, of probs[t,e] * yd[sel_row[t,e]], plus the shared expert's
 * output and the residual (each may be NULL), in double. */
void oracle_combine_expert_choice(int64_t T, int d, int E, int dtype, const float* probs,
                                  const int32_t* sel_row, const double* yd,
                                  const double* shared, const void* residual,
                                  double* y /* [T, d] */) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int o = 0; o < d; ++o) {
            double s = 0.0;
            for (int e = 0; e < E; ++e) {
                const int32_t row = sel_row[(size_t)t * E + e];
                if (row < 0) continue;
                s += (double)probs[(size_t)t * E + e] * yd[(size_t)row * d + o];
            }
            if (shared) s += shared[(size_t)t * d + o];
            if (residual) s += (double)elem(residual, dtype, (size_t)t * d + o);
            y[(size_t)t * d + o] = s;
        }
    }
}
