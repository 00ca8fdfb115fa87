/*
 * moe.h -- C ABI of the single-GPU forward pass of a capacity-limited top-k
 * mixture-of-experts (MoE) layer, hand-written CUDA for B300 (sm_103a).
 *
 * The layer follows the expert-parallelism pages:
 *   "Expert Parallelism" notes page (narrativegoldmine.com), sections
 *     "Components and Architecture" and "Formal Algorithm: Expert
 *     Parallelism Forward Pass" (gate computation, expert selection, token
 *     dispatch, expert computation, expert combine, residual addition);
 *   "Expert Parallelism" (theinfinity.ai, Systems / Distributed), the capacity
 *     paragraph (C = ceil((B*k/D)*c), overflow max(0, p*B*k - C)) and the
 *     6-token / 8-expert / 4-device worked example;
 *   "Expert Parallelism and the All-to-All Bottleneck" (ashishsrivastav.com),
 *     "The Mechanism of Expert Parallelism", phases 1-4, and "The All-to-All
 *     Communication Pattern" (contiguous expert-to-device blocks).
 * The two all-to-all exchanges of the pages become local permutations on one
 * GPU: dispatch packs kept token rows expert-major (so grouped by the D
 * logical shards), combine gathers them back to token order.
 *
 * Conventions shared by every call:
 *  - Problem: T tokens of hidden size d, E experts over D shards (E % D == 0,
 *    shard s holds experts [s*E/D, (s+1)*E/D)), top-k routing, expert FFN
 *    width ffn, capacity factor c (> 0; +INFINITY = no limit).
 *  - Memory: every tensor pointer is a DEVICE pointer owned by the caller.
 *    The library allocates nothing; scratch comes from the caller's workspace
 *    (moe_workspace_size bytes, zero-filled once before its first use).
 *    Pointers must be 16-byte aligned; d and ffn must be multiples of 8.
 *  - Layouts are row-major.  Activations x, xd, yd, y, residual: [rows, d] in
 *    the layer dtype.  Router weight Wg: [E, d] in the layer dtype, bias: [E]
 *    fp32.  Expert weights (nn.Linear out x in): W1, W3: [E, ffn, d];
 *    W2: [E, d, ffn].  topk_idx / slot_pos: [T, k] int32; topk_gate: [T, k]
 *    fp32; probs: [T, E] fp32.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Every call is asynchronous and never synchronises.
 *  - Errors: the return value reports argument validation (nothing is
 *    launched when it fails) and launch errors.  Errors found by a kernel
 *    while running (a bounded wait that gave up) are OR-ed into a status word
 *    in the workspace; moe_device_status() reads and clears it.
 *  - Determinism: every output is a pure function of the inputs; there are
 *    no float atomics, and integer outputs do not depend on scheduling.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage dtype of activations and weights. fp32 accumulation everywhere. */
typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Expert FFN form ("a standard transformer MLP per expert", notes page,
 * "Components and Architecture"):
 *   SWIGLU: h = silu(x W1^T) * (x W3^T), y = h W2^T
 *   GELU:   h = gelu_erf(x W1^T),         y = h W2^T   (W3 unused) */
typedef enum { MOE_ACT_SWIGLU = 0, MOE_ACT_GELU = 1 } moe_act;

typedef struct {
    int64_t T;              /* tokens, >= 0, T*k < 2^31                      */
    int32_t d;              /* hidden size, multiple of 8                     */
    int32_t E;              /* experts, 1..256                                */
    int32_t D;              /* logical shards (devices of the pages), E % D == 0 */
    int32_t k;              /* top-k, 1 <= k <= min(E, 8)                     */
    int32_t ffn;            /* expert FFN width, multiple of 8                */
    double capacity_factor; /* c > 0, +INFINITY = never drop                  */
    int32_t dtype;          /* moe_dtype                                      */
    int32_t act;            /* moe_act                                        */
    int32_t flags;          /* MOE_FLAG_* bits, 0 = none                      */
    int32_t ffn_shared;     /* width of a shared expert (every token goes
                               through it, next to the routed ones); 0 = none,
                               else a multiple of 8                           */
} moe_problem;

/* flags: renormalise a token's k gates to sum to one (the softmax over the k
 * chosen logits) instead of using the plain softmax probabilities. */
#define MOE_FLAG_RENORM 1
/* flags: expert-choice routing -- each expert takes its min(C, T) tokens of
 * highest router logit (ties: lower token first) instead of each token
 * taking its top-k experts; k is read as the average number of experts per
 * token in the capacity rule.  Not combinable with MOE_FLAG_RENORM; needs
 * T <= 49152. */
#define MOE_FLAG_EXPERT_CHOICE 2
/* flags: overflow rerouting -- a choice over its expert's capacity goes to
 * the token's next-best expert instead of being dropped (notes page,
 * "Capacity Factor and Token Dropping": tokens routed to a full expert are
 * dropped or redirected to a secondary expert).  One level: the j-th
 * overflowing choice of a token (ascending rank) goes to its rank k+j expert,
 * rerouted assignments take only the capacity the k choices left, in the
 * same (rank, token) priority, and one that finds its fallback full is
 * dropped.  Needs 2k <= E; not combinable with MOE_FLAG_RENORM or
 * MOE_FLAG_EXPERT_CHOICE.  moe_layer_forward(_shared) reroutes by itself;
 * the step-by-step calls are moe_route_fallback and moe_assign_slots_reroute
 * (moe_assign_slots rejects the flag). */
#define MOE_FLAG_REROUTE 4

enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* a size, pointer, alignment or limit is wrong  */
    MOE_ERR_UNSUPPORTED = 2, /* valid, but outside what this library supports */
    MOE_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required    */
    MOE_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed             */
    MOE_ERR_TIMEOUT = 5,     /* a kernel's bounded wait gave up (device word) */
    MOE_ERR_DEVICE = 6       /* other error recorded by a kernel              */
};

/* Byte offsets of the regions of the layer workspace (all 256-byte aligned).
 * moe_layer_forward leaves every intermediate of the step in its region, so
 * a caller can read routing results and statistics back from the workspace. */
typedef struct {
    size_t status;         /* int32[4]: device error word(s)                 */
    size_t topk_idx;       /* int32[T*k]                                     */
    size_t topk_gate;      /* float[T*k]                                     */
    size_t slot_pos;       /* int32[T*k]                                     */
    size_t counts_routed;  /* int32[E]                                       */
    size_t counts_kept;    /* int32[E]                                       */
    size_t expert_offsets; /* int32[E+1]                                     */
    size_t shard_offsets;  /* int32[D+1]                                     */
    size_t shard_routed;   /* int32[D]                                       */
    size_t shard_overflow; /* int32[D]                                       */
    size_t dropped;        /* int32[1]: dropped assignments                  */
    size_t hist;           /* int32 scratch of the slot assignment           */
    size_t row_token;      /* int32[rows_max]                                */
    size_t xd;             /* dtype[rows_max * d]: packed expert inputs      */
    size_t h;              /* dtype[rows_max * ffn]: expert hidden rows      */
    size_t yd;             /* dtype[rows_max * d]: packed expert outputs     */
    size_t ffn_sync;       /* int32 scratch of the expert FFN (gate/up ->
                              down release counters); every call leaves it
                              zero again                                    */
    size_t stats;          /* uint64[E+1] sums of moe_routing_stats (left zero) */
    size_t hs;             /* dtype[T * ffn_shared]: shared-expert hidden rows */
    size_t ys;             /* dtype[T * d]: shared-expert outputs            */
    size_t shared_sync;    /* int32 scratch of the shared-expert FFN         */
    size_t probs;          /* float[T * E]: router probabilities (expert-choice
                              layer forward only)                           */
    size_t logits;         /* float[T * E]: router logits (expert-choice
                              layer forward only)                           */
    size_t sel_row;        /* int32[T * E]: expert-choice row of (t, e) or -1 */
    size_t fallback_idx;   /* int32[T*k]: next-best experts (rerouting only) */
    size_t fallback_gate;  /* float[T*k]: their probabilities (rerouting only) */
    size_t rerouted;       /* int32[1]: rerouted assignments that got a slot */
    size_t total;          /* = moe_workspace_size                           */
} moe_workspace_layout;

/* Capacity rule.  theinfinity.ai capacity paragraph: a device expecting B*k/D
 * assignments provisions C = ceil((B*k/D)*c); per expert the same rule with E
 * in place of D (notes page, "Capacity Factor and Token Dropping": c times the
 * mean load).  Outputs (host pointers, all required):
 *   *C_expert = min(T, ceil((T*k/E)*c))   (c = inf: T)
 *   *C_shard  = min(T*k, ceil((T*k/D)*c)) (c = inf: T*k), used for the
 *               per-shard overflow max(0, routed_s - C_shard)
 *   *rows_max = min(E*C_expert, T*k), the bound on kept assignments
 *               (expert-choice routing: exactly E*C_expert rows).
 * Host-only; no CUDA call.  Returns MOE_ERR_INVALID_ARG on a bad problem. */
int moe_capacity(const moe_problem* p, int64_t* C_expert, int64_t* C_shard,
                 int64_t* rows_max);

/* Workspace bytes needed by every call of this header for problem *p
 * (host-only).  *bytes receives the size. */
int moe_workspace_size(const moe_problem* p, size_t* bytes);

/* Region offsets inside that workspace (host-only). */
int moe_workspace_layout_of(const moe_problem* p, moe_workspace_layout* out);

/* Router: gate computation and expert selection (notes page, formal
 * algorithm; ashishsrivastav.com phase 1).
 *   g[t,e]   = sum_i x[t,i] * Wg[e,i]  (+ bias[e])   fp32, in one fixed
 *              order: the hidden index is dealt into 32 slices of runs of 8
 *              consecutive elements (slice j holds i = 256*m + 8*j + q,
 *              q = 0..7, m = 0, 1, ...); each slice is one fused multiply-add
 *              chain over its i ascending from +0; the 32 slice sums are
 *              combined by the xor butterfly o = 16, 8, 4, 2, 1 (every slice j
 *              replaced at once by s[j] + s[j ^ o]); then the bias add
 *   probs[t] = softmax(g[t])            (temperature 1)
 *   topk_idx[t, r]  = the expert of rank r (largest logit first; equal logits
 *                     rank the lower expert first)
 *   topk_gate[t, r] = probs[t, topk_idx[t, r]]   (not renormalised), or with
 *                     MOE_FLAG_RENORM the softmax over the k chosen logits
 *                     (a token's k gates sum to one)
 * bias and probs may be NULL.  ws is unused (may be NULL).
 * Without probs, a bf16 layer of up to 128 experts is routed on the tensor
 * cores: the logits come from tcgen05 MMAs, every token whose top-k those
 * logits cannot settle under a stated error bound is re-ranked in the fixed
 * order above, so topk_idx is bit-identical to the fixed order's on every
 * input, and topk_gate agrees with it to within the tensor-core rounding of
 * the logits it uses (well below 1e-5 relative on the tested inputs).  With
 * probs (or fp32, or more experts) every logit is computed in the fixed
 * order. */
int moe_route(const moe_problem* p, const void* x, const void* Wg, const float* bias,
              int32_t* topk_idx, float* topk_gate, float* probs,
              void* ws, size_t ws_bytes, void* stream);

/* Slot assignment and token dropping (notes page, "Capacity Factor and Token
 * Dropping"; theinfinity.ai capacity paragraph).  Assignments are served in
 * the priority (rank r, then token t); pos(t, r) counts the earlier
 * assignments to the same expert; kept iff pos < C_expert.
 *   slot_pos[t, r]    = pos, or -1 when dropped
 *   counts_routed[e]  = assignments to e;  counts_kept[e] = min(routed, C)
 *   expert_offsets    = exclusive scan of counts_kept, E+1 entries
 *   shard_offsets[s]  = expert_offsets[s*E/D], D+1 entries
 *   shard_routed[s]   = sum of counts_routed over the shard's experts
 *   shard_overflow[s] = max(0, shard_routed[s] - C_shard)
 *   row_token[expert_offsets[e] + pos] = t for every kept (t, r); entries at
 *                       and beyond expert_offsets[E] are left unwritten
 *   dropped[0]        = number of dropped assignments (may be NULL)
 * Uses the workspace's hist region and status word. */
int moe_assign_slots(const moe_problem* p, const int32_t* topk_idx, int32_t* slot_pos,
                     int32_t* counts_routed, int32_t* counts_kept, int32_t* expert_offsets,
                     int32_t* shard_offsets, int32_t* shard_routed, int32_t* shard_overflow,
                     int32_t* row_token, int32_t* dropped, void* ws, size_t ws_bytes,
                     void* stream);

/* Dispatch, the pack before the first all-to-all (notes page, token
 * dispatch; ashishsrivastav.com phase 2), done as a local permutation:
 *   xd[row] = x[row_token[row]]  for row < expert_offsets[E]
 * xd has rows_max rows; rows at and beyond expert_offsets[E] are untouched.
 * Bit-exact byte copy. */
int moe_dispatch(const moe_problem* p, const void* x, const int32_t* row_token,
                 const int32_t* expert_offsets, void* xd, void* stream);

/* The same dispatch, walked token by token: for every token t and rank r
 * with slot_pos[t, r] >= 0 (the outputs of moe_assign_slots; topk_idx and
 * slot_pos [T, k] int32),
 *   xd[expert_offsets[topk_idx[t, r]] + slot_pos[t, r]] = x[t]
 * which writes exactly the rows moe_dispatch writes, with the same bytes.
 * Each row of x is read once for all of the token's slots, where the
 * expert-major form reads it once per slot; moe_layer_forward uses this form
 * for k >= 2 when x is larger than half the L2.  A rank whose expert is outside [0, E), whose slot is negative
 * or whose row would reach rows_max stores nothing.  x and xd 16-byte
 * aligned. */
int moe_dispatch_by_token(const moe_problem* p, const void* x, const int32_t* topk_idx,
                          const int32_t* slot_pos, const int32_t* expert_offsets, void* xd,
                          void* stream);

/* Expert computation (notes page, expert GEMM and formal algorithm;
 * ashishsrivastav.com phase 3): for every expert e and every packed row
 * r in [expert_offsets[e], expert_offsets[e+1]):
 *   yd[r] = FFN_e(xd[r])   (form set by p->act; fp32 accumulation, the
 *                           hidden row stored in the layer dtype)
 * bf16 + SwiGLU runs as a grouped GEMM on the tcgen05 tensor cores (TMA-fed,
 * accumulators in tensor memory); other forms on a SIMT kernel.
 * W3 may be NULL for GELU.  Uses the workspace's h region and status word.
 * Rows at and beyond expert_offsets[E] of yd are untouched. */
int moe_expert_ffn(const moe_problem* p, const void* xd, const int32_t* expert_offsets,
                   const void* W1, const void* W3, const void* W2, void* yd,
                   void* ws, size_t ws_bytes, void* stream);

/* Combine (notes page, expert combine and residual addition;
 * ashishsrivastav.com phase 4), back in token order:
 *   y[t] = sum over r with slot_pos[t,r] >= 0, in rank order, of
 *          topk_gate[t,r] * yd[expert_offsets[topk_idx[t,r]] + slot_pos[t,r]]
 *          (+ residual[t])
 * fp32 accumulation, one rounding to the layer dtype; a token whose every
 * assignment was dropped gets 0 (+ residual).  residual may be NULL. */
int moe_combine(const moe_problem* p, const void* yd, const int32_t* topk_idx,
                const int32_t* slot_pos, const int32_t* expert_offsets,
                const float* topk_gate, const void* residual, void* y, void* stream);

/* The whole layer forward: route, assign, dispatch, expert FFN, combine, on
 * one stream, with no host synchronisation.  bias, W3 (GELU) and residual
 * may be NULL.  Intermediates stay in the workspace regions named by
 * moe_workspace_layout_of (probs are not produced).  With MOE_FLAG_REROUTE
 * the topk_idx / topk_gate regions end up holding route_idx / route_gate of
 * moe_assign_slots_reroute. */
int moe_layer_forward(const moe_problem* p, const void* x, const void* Wg, const float* bias,
                      const void* W1, const void* W3, const void* W2, const void* residual,
                      void* y, void* ws, size_t ws_bytes, void* stream);

/* Shared expert (notes page, "Major Variants": an expert every token goes
 * through, next to the routed ones): ys[t] = FFN_shared(x[t]) for every
 * token, the same FFN form as the routed experts (p->act) with width
 * p->ffn_shared (> 0).  Ws1, Ws3: [ffn_shared, d] (Ws3 NULL for GELU);
 * Ws2: [d, ffn_shared]; ys: [T, d] in the layer dtype.  bf16 SwiGLU runs on
 * the same tensor-core FFN kernel as the routed experts (one expert whose
 * rows are x's rows).  Uses the workspace's hs and shared_sync regions. */
int moe_shared_expert_ffn(const moe_problem* p, const void* x, const void* Ws1, const void* Ws3,
                          const void* Ws2, void* ys, void* ws, size_t ws_bytes, void* stream);

/* moe_combine with the shared expert's output added after the routed sum
 * and before the residual (both may be NULL):
 *   y[t] = ((sum over kept r of gate * yd[row]) + shared[t]) + residual[t] */
int moe_combine_shared(const moe_problem* p, const void* yd, const int32_t* topk_idx,
                       const int32_t* slot_pos, const int32_t* expert_offsets,
                       const float* topk_gate, const void* shared, const void* residual,
                       void* y, void* stream);

/* moe_layer_forward with a shared expert (p->ffn_shared > 0; its weights
 * Ws1, Ws3, Ws2 as in moe_shared_expert_ffn): the routed layer, the shared
 * expert over every token, and moe_combine_shared.  With p->ffn_shared == 0
 * it is moe_layer_forward and the shared weights are ignored.
 * moe_layer_forward itself rejects p->ffn_shared != 0.  In the bf16 SwiGLU
 * form the shared expert's FFN launch starts on the SMs that the routed FFN's
 * CTAs leave as they finish (it reads only x and its own weights), and the
 * combine starts only after both have completed. */
int moe_layer_forward_shared(const moe_problem* p, const void* x, const void* Wg, const float* bias,
                             const void* W1, const void* W3, const void* W2, const void* Ws1,
                             const void* Ws3, const void* Ws2, const void* residual, void* y,
                             void* ws, size_t ws_bytes, void* stream);

/* Router for overflow rerouting (p->flags must include MOE_FLAG_REROUTE):
 * moe_route's outputs plus, per token, the next k experts in the same order
 * (descending logit, lower index first on ties) after its k choices:
 *   fallback_idx[t, j]  = the token's rank k+j expert        [T, k] int32
 *   fallback_gate[t, j] = probs[t, fallback_idx[t, j]]      [T, k] fp32
 * probs may be NULL.  No workspace. */
int moe_route_fallback(const moe_problem* p, const void* x, const void* Wg, const float* bias,
                       int32_t* topk_idx, float* topk_gate, int32_t* fallback_idx,
                       float* fallback_gate, float* probs, void* stream);

/* Slot assignment with overflow rerouting (p->flags must include
 * MOE_FLAG_REROUTE).  First pass: the assignment of moe_assign_slots on the
 * k choices.  Second pass: the j-th overflowing choice of token t (ascending
 * rank) moves to fallback j; in (rank, token) priority the moved assignments
 * take positions from the expert's first-pass kept count on, kept iff
 * below C_expert.
 *   route_idx[t, r]   = the expert serving (t, r): its choice, or the
 *                       fallback it moved to                  [T, k] int32
 *   route_gate[t, r]  = that expert's gate (topk_gate, or fallback_gate)
 *   slot_pos[t, r]    = its position at route_idx, or -1 when it has none
 *   counts_routed     = first-pass assignments per expert (as moe_assign_slots)
 *   counts_kept       = rows per expert after rerouting (<= C_expert)
 *   expert_offsets, shard_offsets, row_token: of the rows after rerouting
 *   shard_routed, shard_overflow: of the k choices (as moe_assign_slots)
 *   dropped[0]  = assignments with no slot at the end      (may be NULL)
 *   rerouted[0] = moved assignments that got a slot         (may be NULL)
 * route_idx / route_gate may be the same buffers as topk_idx / topk_gate
 * (updated in place).  moe_combine takes route_idx, slot_pos, route_gate.
 * Uses the workspace's hist region and status word. */
int moe_assign_slots_reroute(const moe_problem* p, const int32_t* topk_idx, const float* topk_gate,
                             const int32_t* fallback_idx, const float* fallback_gate,
                             int32_t* route_idx, float* route_gate, int32_t* slot_pos,
                             int32_t* counts_routed, int32_t* counts_kept, int32_t* expert_offsets,
                             int32_t* shard_offsets, int32_t* shard_routed, int32_t* shard_overflow,
                             int32_t* row_token, int32_t* dropped, int32_t* rerouted, void* ws,
                             size_t ws_bytes, void* stream);

/* Router logits and probabilities without the top-k: logits [T, E] fp32 in
 * the router's fixed order (bias included, as moe_route computes them),
 * probs [T, E] the softmax (may be NULL).  For expert-choice routing. */
int moe_router_logits(const moe_problem* p, const void* x, const void* Wg, const float* bias,
                      float* logits, float* probs, void* stream);

/* Expert-choice routing, the selection (notes page, "Major Variants": each
 * expert chooses its tokens).  From the router logits [T, E] of
 * moe_router_logits and C = C_expert of moe_capacity (C <= T):
 *   expert e takes the C tokens with the largest logits[t, e], equal values
 *   in ascending token order (the choice is taken on the router's own fp32
 *   values, so it is exact);
 *   row_token[e*C + j]  = its j-th token in ascending token order  [E*C]
 *   expert_offsets[e]   = e*C                                       [E+1]
 *   sel_row[t*E + e]    = the row of (t, e), or -1 if e did not take t  [T*E]
 * Exact (integer radix select and scans).  Needs p->flags to include
 * MOE_FLAG_EXPERT_CHOICE.  No workspace. */
int moe_expert_choice_assign(const moe_problem* p, const float* logits, int32_t* row_token,
                             int32_t* expert_offsets, int32_t* sel_row, void* stream);

/* Combine for expert-choice routing:
 *   y[t] = ((sum over e with sel_row[t,e] >= 0, ascending e, of
 *            probs[t,e] * yd[sel_row[t,e]]) + shared[t]) + residual[t]
 * fp32 accumulation, one rounding; shared and residual may be NULL. */
int moe_combine_expert_choice(const moe_problem* p, const void* yd, const float* probs,
                              const int32_t* sel_row, const void* shared, const void* residual,
                              void* y, void* stream);

/* Slot assignment without a workspace, for callers that cannot allocate
 * device memory (an operator inside a host framework that owns every device
 * allocation and passes only input and output buffers, or a latency-critical
 * path that must avoid cudaMalloc's implicit synchronisation).  The pages have
 * no counterpart of this entry point; it computes exactly what
 * moe_assign_slots computes, with the same arguments minus the workspace.
 * Its scratch (histograms, completion ticket, status word) is one file-scope
 * __device__ array of 4 MiB + 256 B that every GPU loading the library holds
 * until the process exits.  Limits and rules:
 *   - accepted only if E * k * ceil(T / 32) <= 1048576; larger problems
 *     return MOE_ERR_WORKSPACE and launch nothing;
 *   - the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, once per device, that device current); make that
 *     first call before any stream capture.  The driver places the array on a
 *     device when it loads the library's module there, which under CUDA's
 *     lazy module loading is that first call: a caller that needs every later
 *     call free of that one-time placement makes one warm-up call per device;
 *   - all calls share the array and each starts by clearing its completion
 *     ticket: calls whose work overlaps on the GPU (other streams, other host
 *     threads) race and must be serialised by the caller;
 *   - an expert id outside [0, E) counts as no assignment (as in
 *     moe_assign_slots) and sets the array's status word, which calls do not
 *     clear; moe_assign_slots_static_status() reads and clears it;
 *   - no cudaMalloc, cudaFree or other allocating call is made. */
int moe_assign_slots_static(const moe_problem* p, const int32_t* topk_idx, int32_t* slot_pos,
                            int32_t* counts_routed, int32_t* counts_kept, int32_t* expert_offsets,
                            int32_t* shard_offsets, int32_t* shard_routed, int32_t* shard_overflow,
                            int32_t* row_token, int32_t* dropped, void* stream);

/* The device status of moe_assign_slots_static on the current device, the
 * counterpart of moe_device_status for that workspace-free entry point (the
 * pages have no counterpart of it either): synchronises `stream`, reads the
 * status word of the static scratch array (errors OR-ed in by every call
 * since the last read), clears it and returns MOE_OK, MOE_ERR_DEVICE (an
 * expert id outside [0, E) was seen) or MOE_ERR_TIMEOUT (or MOE_ERR_CUDA if a
 * CUDA call failed).  Allocates nothing; the word is copied to a host stack
 * variable. */
int moe_assign_slots_static_status(void* stream);

/* Indices of the moe_routing_stats outputs. */
enum {
    MOE_STAT_AUX = 0,       /* load-balancing term E * sum_e f_e * P_e       */
    MOE_STAT_ENTROPY = 1,   /* mean routing entropy, nats                    */
    MOE_STAT_DROP = 2,      /* dropped assignments / (T*k)                   */
    MOE_STAT_IMBALANCE = 3, /* max_e routed_e / (T*k/E)                      */
    MOE_NUM_STATS = 4
};

/* Routing statistics as device outputs (notes page, "Components and
 * Architecture" and the formal algorithm's auxiliary load-balancing term:
 * the share of tokens an expert receives times the share of router
 * probability it receives, summed over experts; glossary page: the
 * load-balancing loss; intro page, practitioner guidance: expert utilisation
 * and routing entropy).  From the router probabilities of moe_route and the
 * counts of moe_assign_slots:
 *   f_e = counts_routed[e] / (T*k)   P_e = (1/T) sum_t probs[t,e]
 *   stats[MOE_STAT_AUX]       = E * sum_e f_e * P_e   (1 = perfectly uniform)
 *   stats[MOE_STAT_ENTROPY]   = (1/T) sum_t -sum_e p ln p  (0 ln 0 = 0)
 *   stats[MOE_STAT_DROP]      = sum_e (counts_routed - counts_kept) / (T*k)
 *   stats[MOE_STAT_IMBALANCE] = max_e counts_routed[e] / (T*k/E)
 *   mean_prob[e]              = P_e                   (may be NULL)
 * probs: [T, E] fp32, counts: [E] int32, stats: float[MOE_NUM_STATS], all
 * device pointers.  Deterministic: the sums over tokens are 64-bit
 * fixed-point integers (units of 2^-36), the final combination one fixed-order
 * fp32 pass.  Needs T <= 2^25 (else MOE_ERR_UNSUPPORTED).  Uses the
 * workspace's stats region (left zero) and a ticket in its status region;
 * T = 0 gives zeros. */
int moe_routing_stats(const moe_problem* p, const float* probs, const int32_t* counts_routed,
                      const int32_t* counts_kept, float* stats, float* mean_prob,
                      void* ws, size_t ws_bytes, void* stream);

/* Page-locked host memory for layer inputs and outputs (cudaHostAlloc,
 * portable to every device).  Copies between it and the device run at the
 * link's full rate; on the measured B300 hosts a copy from it was about five
 * times faster than one from memory pinned by other means.  *ptr = NULL for
 * bytes == 0.  Free with moe_host_free (NULL is a no-op). */
int moe_host_alloc(size_t bytes, void** ptr);
int moe_host_free(void* ptr);

/* Device staging bytes moe_layer_forward_host needs for problem *p: two input
 * and two output buffers of T*d elements (each 256-byte aligned). */
int moe_host_staging_size(const moe_problem* p, size_t* bytes);

/* The layer forward from host buffers, n_steps times: step i copies x_host[i]
 * ([T, d], host memory -- page-locked, e.g. from moe_host_alloc, for the
 * copies to be asynchronous) to the device, runs moe_layer_forward on it
 * (no residual, no shared expert: p->ffn_shared must be 0) and copies the
 * result to y_host[i].  Step i's input copy, step i-1's layer and step i-2's
 * output copy overlap: the copies run on two copy streams the library keeps
 * per device, the layers on `stream` one after another (never concurrently:
 * the expert FFN kernel's CTAs wait on one another and assume the GPU to
 * themselves), ordered by events; `staging` (device, moe_host_staging_size
 * bytes) holds two input and two output buffers.  Asynchronous: the copies
 * start after the work already queued on `stream`, and `stream` reaches the
 * end of the call's work only after the last output copy.  The library's copy
 * streams are shared by all calls on a device, so calls must not overlap
 * from several host threads.  A failure returns at once, leaving the steps
 * queued so far in flight. */
int moe_layer_forward_host(const moe_problem* p, int64_t n_steps, const void* const* x_host,
                           const void* Wg, const float* bias, const void* W1, const void* W3,
                           const void* W2, void* const* y_host, void* staging, size_t staging_bytes,
                           void* ws, size_t ws_bytes, void* stream);

/* Number of kernels one moe_layer_forward(_shared) launches for problem *p
 * (host-only): router and slot assignment (2 when the slot histogram
 * E*k*ceil(T/32) is small enough for the fused slot-and-pack kernel, else 3
 * with dispatch; expert choice 3, rerouting 4), the expert FFN (1 launch on
 * the bf16 SwiGLU tensor-core path, else 2; twice with a shared expert) and
 * combine.  0 for T == 0. */
int moe_layer_launch_count(const moe_problem* p, int* launches);

/* Synchronises `stream`, reads the workspace's device status word, clears it
 * and returns MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE (or MOE_ERR_CUDA if
 * the synchronisation itself failed). */
int moe_device_status(void* ws, void* stream);

/* Static English text of a status code. */
const char* moe_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
