// api.cu -- the extern "C" boundary declared in include/moe.h: argument
// validation, the capacity rule, workspace layout, and the launch sequence of
// the layer forward.  No allocation, no host synchronisation (except in
// moe_device_status, whose job it is).
#include <algorithm>
#include <cmath>
#include <mutex>

#include "assign_scan.cuh"

namespace moe {
namespace {

inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }
inline size_t esize(int dtype) { return dtype == MOE_BF16 ? 2 : 4; }
inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Capacity rule (theinfinity.ai capacity paragraph, per expert with E in
// place of D): C = min(T, ceil((T*k/E)*c)); C_shard = min(T*k, ceil((T*k/D)*c)).
int capacity(const moe_problem* p, int64_t* C, int64_t* Cs, int64_t* rows_max) {
    const int64_t Tk = p->T * (int64_t)p->k;
    const double c = p->capacity_factor;
    if (std::isinf(c)) {
        *C = p->T;
        *Cs = Tk;
    } else {
        const double ve = std::ceil(((double)Tk / (double)p->E) * c);
        const double vs = std::ceil(((double)Tk / (double)p->D) * c);
        *C = ve >= (double)p->T ? p->T : (int64_t)ve;
        *Cs = vs >= (double)Tk ? Tk : (int64_t)vs;
    }
    *rows_max = (p->flags & MOE_FLAG_EXPERT_CHOICE) ? (int64_t)p->E * *C : std::min<int64_t>((int64_t)p->E * *C, Tk);
    return MOE_OK;
}

int validate(const moe_problem* p) {
    if (!p) return MOE_ERR_INVALID_ARG;
    if (p->T < 0 || p->d < 8 || p->d % 8 || p->ffn < 8 || p->ffn % 8) return MOE_ERR_INVALID_ARG;
    if (p->E < 1 || p->D < 1 || p->E % p->D) return MOE_ERR_INVALID_ARG;
    if (p->k < 1 || p->k > p->E) return MOE_ERR_INVALID_ARG;
    if (!(p->capacity_factor > 0.0)) return MOE_ERR_INVALID_ARG;  // also rejects NaN
    if (p->dtype != MOE_F32 && p->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (p->act != MOE_ACT_SWIGLU && p->act != MOE_ACT_GELU) return MOE_ERR_INVALID_ARG;
    if (p->flags & ~(MOE_FLAG_RENORM | MOE_FLAG_EXPERT_CHOICE | MOE_FLAG_REROUTE)) return MOE_ERR_INVALID_ARG;
    if ((p->flags & MOE_FLAG_RENORM) && (p->flags & MOE_FLAG_EXPERT_CHOICE)) return MOE_ERR_INVALID_ARG;
    // rerouting: plain probabilities as gates, top-k routing, k fallbacks per token
    if ((p->flags & MOE_FLAG_REROUTE) && (p->flags & (MOE_FLAG_RENORM | MOE_FLAG_EXPERT_CHOICE)))
        return MOE_ERR_INVALID_ARG;
    if ((p->flags & MOE_FLAG_REROUTE) && 2 * p->k > p->E) return MOE_ERR_INVALID_ARG;
    if (p->ffn_shared < 0 || p->ffn_shared % 8) return MOE_ERR_INVALID_ARG;
    if (p->E > 256 || p->k > 8) return MOE_ERR_UNSUPPORTED;
    if (p->T * (int64_t)p->k >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)p->d * p->ffn >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)p->d * p->ffn_shared >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
    // expert choice keeps an expert's probability column in shared memory
    if ((p->flags & MOE_FLAG_EXPERT_CHOICE) && p->T > 49152) return MOE_ERR_UNSUPPORTED;
    if ((p->flags & MOE_FLAG_EXPERT_CHOICE) && p->T * (int64_t)p->E >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

}  // namespace

int to_problem(const moe_problem* mp, Problem* p) {
    int rc = validate(mp);
    if (rc != MOE_OK) return rc;
    p->T = mp->T;
    p->d = mp->d;
    p->E = mp->E;
    p->D = mp->D;
    p->k = mp->k;
    p->ffn = mp->ffn;
    p->dtype = mp->dtype;
    p->act = mp->act;
    p->flags = mp->flags;
    p->ffn_shared = mp->ffn_shared;
    capacity(mp, &p->C, &p->C_shard, &p->rows_max);
    p->nblk = ceil_div(p->T, kAssignBlock);
    return MOE_OK;
}

namespace {

// The shared expert as a problem of its own: one expert whose rows are all T
// tokens in order, width ffn_shared.
Problem shared_problem(const Problem& p) {
    Problem s = p;
    s.E = 1;
    s.D = 1;
    s.k = 1;
    s.ffn = p.ffn_shared;
    s.C = p.T;
    s.C_shard = p.T;
    s.rows_max = p.T;
    return s;
}

void layout(const Problem& p, moe_workspace_layout* L) {
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align256(o + std::max<size_t>(bytes, 1));
        return at;
    };
    const size_t Tk = (size_t)p.T * p.k, eb = esize(p.dtype), rm = (size_t)p.rows_max;
    L->status = take(4 * sizeof(int32_t));
    L->topk_idx = take(Tk * 4);
    L->topk_gate = take(Tk * 4);
    L->slot_pos = take(Tk * 4);
    L->counts_routed = take((size_t)p.E * 4);
    L->counts_kept = take((size_t)p.E * 4);
    L->expert_offsets = take((size_t)(p.E + 1) * 4);
    L->shard_offsets = take((size_t)(p.D + 1) * 4);
    L->shard_routed = take((size_t)p.D * 4);
    L->shard_overflow = take((size_t)p.D * 4);
    L->dropped = take(4);
    L->hist = take((size_t)p.E * p.k * (size_t)p.nblk * 4);
    L->row_token = take(rm * 4);
    L->xd = take(rm * p.d * eb);
    L->h = take(rm * p.ffn * eb);
    L->yd = take(rm * p.d * eb);
    L->ffn_sync = take(ffn_sync_ints(p) * sizeof(int32_t));
    L->stats = take((size_t)(p.E + 1) * sizeof(unsigned long long));
    const size_t Ts = p.ffn_shared > 0 ? (size_t)p.T : 0;
    L->hs = take(Ts * p.ffn_shared * eb);
    L->ys = take(Ts * p.d * eb);
    L->shared_sync = take(p.ffn_shared > 0 ? ffn_sync_ints(shared_problem(p)) * sizeof(int32_t) : 0);
    const size_t TE = (p.flags & MOE_FLAG_EXPERT_CHOICE) ? (size_t)p.T * p.E : 0;
    L->probs = take(TE * sizeof(float));
    L->logits = take(TE * sizeof(float));
    L->sel_row = take(TE * sizeof(int32_t));
    const size_t Tkr = (p.flags & MOE_FLAG_REROUTE) ? Tk : 0;
    L->fallback_idx = take(Tkr * 4);
    L->fallback_gate = take(Tkr * 4);
    L->rerouted = take(4);
    L->total = o;
}

int check_ws(const Problem& p, void* ws, size_t ws_bytes, moe_workspace_layout* L) {
    layout(p, L);
    if (!ws || ws_bytes < L->total || !aligned16(ws)) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// L2 bytes of the device, queried once per process (a function-local static,
// thread-safe; every device the library drives is the same part)
int64_t l2_bytes() {
    static const int64_t n = []() -> int64_t {
        int dev = 0, v = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess || v <= 0) v = 126 << 20;
        return v;
    }();
    return n;
}

// The shared expert's FFN over all T tokens (rows of x in order) into ys;
// `order`: FfnOrder bits of its tensor-core launch.
int run_shared_expert(const Problem& p, const moe_workspace_layout& L, char* w, const void* x, const void* Ws1,
                      const void* Ws3, const void* Ws2, void* ys, cudaStream_t s, int order = 0) {
    const Problem sp = shared_problem(p);
    void* hs = w + L.hs;
    int* status = (int*)(w + L.status);
    cudaError_t e;
    if (p.dtype == MOE_BF16 && p.act == MOE_ACT_SWIGLU) {
        e = launch_ffn_tc(sp, x, nullptr, Ws1, Ws3, Ws2, hs, ys, status, (int*)(w + L.shared_sync), s, order);
        if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
    } else {
        e = launch_ffn_simt(sp, x, nullptr, Ws1, Ws3, Ws2, hs, ys, s);
    }
    return cuda_rc(e);
}

int layer_forward(const moe_problem* mp, const void* x, const void* Wg, const float* bias, const void* W1,
                  const void* W3, const void* W2, const void* Ws1, const void* Ws3, const void* Ws2,
                  const void* residual, void* y, void* ws, size_t ws_bytes, void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (!x || !Wg || !W1 || !W2 || !y || (p.act == MOE_ACT_SWIGLU && !W3)) return MOE_ERR_INVALID_ARG;
    const bool has_shared = p.ffn_shared > 0;
    if (has_shared && (!Ws1 || !Ws2 || (p.act == MOE_ACT_SWIGLU && !Ws3))) return MOE_ERR_INVALID_ARG;
    if (has_shared && (!aligned16(Ws1) || !aligned16(Ws2) || (Ws3 && !aligned16(Ws3))))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(Wg) || !aligned16(W1) || !aligned16(W2) || (W3 && !aligned16(W3)) ||
        !aligned16(y) || (residual && !aligned16(residual)))
        return MOE_ERR_INVALID_ARG;
    moe_workspace_layout L;
    rc = check_ws(p, ws, ws_bytes, &L);
    if (rc != MOE_OK) return rc;
    if (p.T == 0) return MOE_OK;
    char* w = (char*)ws;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t* idx = (int32_t*)(w + L.topk_idx);
    float* gate = (float*)(w + L.topk_gate);
    int32_t* slot = (int32_t*)(w + L.slot_pos);
    int32_t* off = (int32_t*)(w + L.expert_offsets);
    int32_t* row_token = (int32_t*)(w + L.row_token);
    int* status = (int*)(w + L.status);
    void *xd = w + L.xd, *h = w + L.h, *yd = w + L.yd;

    int32_t* hist = (int32_t*)(w + L.hist);
    const bool ec = (p.flags & MOE_FLAG_EXPERT_CHOICE) != 0;
    float* probs = (float*)(w + L.probs);
    float* logits = (float*)(w + L.logits);
    int32_t* sel_row = (int32_t*)(w + L.sel_row);
    cudaError_t e;
    bool packed = false;  // slot assignment and dispatch done by one kernel
    if (ec) {
        // expert choice: router logits and probabilities, then each expert
        // takes its tokens by logit
        e = launch_route(p, x, Wg, bias, nullptr, nullptr, probs, s, logits, nullptr, nullptr, status);
        if (e == cudaSuccess) e = launch_ec_select(p, logits, row_token, off, sel_row, s);
    } else {
        // router + count pass (status[1] is the count pass's completion ticket), then the rank pass
        const AssignScan scan{hist, (int32_t*)(w + L.counts_routed), (int32_t*)(w + L.counts_kept), off,
                              (int32_t*)(w + L.shard_offsets), (int32_t*)(w + L.shard_routed),
                              (int32_t*)(w + L.shard_overflow), (int32_t*)(w + L.dropped),
                              (unsigned*)(status + 1), p.E, p.D, p.k, p.nblk, p.C, p.C_shard};
        if (p.flags & MOE_FLAG_REROUTE) {
            // the choices and their fallbacks, then the reroute and place passes
            // (final experts and gates overwrite idx and gate in place)
            int32_t* fb_idx = (int32_t*)(w + L.fallback_idx);
            float* fb_gate = (float*)(w + L.fallback_gate);
            e = launch_route_count(p, x, Wg, bias, idx, gate, scan, s, fb_idx, fb_gate, status);
            AssignScan second = scan;
            second.second = true;
            second.rerouted = (int32_t*)(w + L.rerouted);
            if (e == cudaSuccess)
                e = launch_reroute(p, idx, gate, fb_idx, fb_gate, idx, gate, slot, second, row_token, status, s);
        } else if (assign_pack_fits(p)) {
            // small histogram: the router only counts; one kernel scans, places and packs
            AssignScan deferred = scan;
            deferred.defer = true;
            e = launch_route_count(p, x, Wg, bias, idx, gate, deferred, s, nullptr, nullptr, status);
            if (e == cudaSuccess) e = launch_assign_pack(p, x, idx, scan, slot, row_token, xd, status, s);
            packed = true;
        } else {
            e = launch_route_count(p, x, Wg, bias, idx, gate, scan, s, nullptr, nullptr, status);
            if (e == cudaSuccess) e = launch_rank(p, idx, hist, off, slot, row_token, status, s);
        }
    }
    // With k >= 2 and an x larger than half the L2, the token-major form: it
    // reads each token's row once for all its slots, where the expert-major
    // gather reads it once per slot, a whole expert segment apart (the 8x7B
    // shape: 166 -> 135 us).  When x fits in L2 those second reads hit there
    // and the gather, one warp per kept row rather than per token, is as fast
    // or faster (the 64-expert layer: 10.5 against 11.3 us).  Expert choice
    // has no token-major slots.
    const bool by_token = !ec && p.k >= 2 && (int64_t)p.T * p.d * (int64_t)esize(p.dtype) > l2_bytes() / 2;
    if (e == cudaSuccess && !packed)
        e = by_token ? launch_scatter(p, x, idx, slot, off, xd, s) : launch_dispatch(p, x, row_token, off, xd, s);
    // With a shared expert (tensor-core form) the routed FFN lets the shared
    // expert's FFN launch as its CTAs run out of tiles, and the shared FFN --
    // which reads only x and its weights and writes only its own hs, ys and
    // counters -- waits for the routed one at its end: its CTAs fill the SMs
    // of the routed launch's tail, and the combine still starts after both.
    const bool overlap_shared = has_shared && p.dtype == MOE_BF16 && p.act == MOE_ACT_SWIGLU && p.rows_max > 0;
    if (e == cudaSuccess) {
        if (p.dtype == MOE_BF16 && p.act == MOE_ACT_SWIGLU) {
            e = launch_ffn_tc(p, xd, off, W1, W3, W2, h, yd, status, (int*)(w + L.ffn_sync), s,
                              overlap_shared ? kFfnReleaseNext : 0);
            if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
        } else {
            e = launch_ffn_simt(p, xd, off, W1, W3, W2, h, yd, s);
        }
    }
    void* ys = has_shared ? (void*)(w + L.ys) : nullptr;
    if (e == cudaSuccess && has_shared) {
        const int rc2 = run_shared_expert(p, L, w, x, Ws1, Ws3, Ws2, ys, s, overlap_shared ? kFfnWaitAtEnd : 0);
        if (rc2 != MOE_OK) return rc2;
    }
    if (e == cudaSuccess)
        e = ec ? launch_ec_combine(p, yd, probs, sel_row, ys, residual, y, s)
               : launch_combine(p, yd, idx, slot, off, gate, residual, y, s, ys);
    return cuda_rc(e);
}

// ---- host pipeline: the copy streams and events of moe_layer_forward_host,
// made once per device and kept for the life of the process
struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, in_done[2] = {}, comp_done[2] = {}, out_done[2] = {};
    bool ready = false;
};
constexpr int kMaxDevices = 64;
HostPipe g_pipes[kMaxDevices];
std::mutex g_pipe_mu;

int host_pipe(HostPipe** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe& hp = g_pipes[dev];
    if (!hp.ready) {
        bool ok = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; ok && i < 2; ++i)
            ok = cudaEventCreateWithFlags(&hp.in_done[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&hp.comp_done[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&hp.out_done[i], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) return MOE_ERR_CUDA;
        hp.ready = true;
    }
    *out = &hp;
    return MOE_OK;
}

size_t host_staging_bytes(const Problem& p) { return 4 * align256((size_t)p.T * p.d * esize(p.dtype)); }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_capacity(const moe_problem* p, int64_t* C_expert, int64_t* C_shard, int64_t* rows_max) {
    if (!C_expert || !C_shard || !rows_max) return MOE_ERR_INVALID_ARG;
    int rc = validate(p);
    if (rc != MOE_OK) return rc;
    return capacity(p, C_expert, C_shard, rows_max);
}

int moe_workspace_size(const moe_problem* mp, size_t* bytes) {
    if (!bytes) return MOE_ERR_INVALID_ARG;
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    moe_workspace_layout L;
    layout(p, &L);
    *bytes = L.total;
    return MOE_OK;
}

int moe_workspace_layout_of(const moe_problem* mp, moe_workspace_layout* out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    layout(p, out);
    return MOE_OK;
}

int moe_route(const moe_problem* mp, const void* x, const void* Wg, const float* bias, int32_t* topk_idx,
              float* topk_gate, float* probs, void* ws, size_t ws_bytes, void* stream) {
    (void)ws;
    (void)ws_bytes;
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (p.T == 0) return MOE_OK;
    if (!x || !Wg || !topk_idx || !topk_gate || !aligned16(x) || !aligned16(Wg)) return MOE_ERR_INVALID_ARG;
    return cuda_rc(launch_route(p, x, Wg, bias, topk_idx, topk_gate, probs, (cudaStream_t)stream));
}

int moe_assign_slots(const moe_problem* mp, const int32_t* topk_idx, int32_t* slot_pos, int32_t* counts_routed,
                     int32_t* counts_kept, int32_t* expert_offsets, int32_t* shard_offsets,
                     int32_t* shard_routed, int32_t* shard_overflow, int32_t* row_token, int32_t* dropped,
                     void* ws, size_t ws_bytes, void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (p.flags & MOE_FLAG_REROUTE) return MOE_ERR_INVALID_ARG;  // see moe_assign_slots_reroute
    if ((p.T > 0 && (!topk_idx || !slot_pos || !row_token)) || !counts_routed || !counts_kept ||
        !expert_offsets || !shard_offsets || !shard_routed || !shard_overflow)
        return MOE_ERR_INVALID_ARG;
    moe_workspace_layout L;
    rc = check_ws(p, ws, ws_bytes, &L);
    if (rc != MOE_OK) return rc;
    int* status = (int*)((char*)ws + L.status);
    return cuda_rc(launch_assign(p, topk_idx, slot_pos, counts_routed, counts_kept, expert_offsets, shard_offsets,
                                 shard_routed, shard_overflow, row_token, dropped,
                                 (int32_t*)((char*)ws + L.hist), status, (cudaStream_t)stream));
}

int moe_route_fallback(const moe_problem* mp, const void* x, const void* Wg, const float* bias, int32_t* topk_idx,
                       float* topk_gate, int32_t* fallback_idx, float* fallback_gate, float* probs, void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (!(p.flags & MOE_FLAG_REROUTE)) return MOE_ERR_INVALID_ARG;
    if (p.T == 0) return MOE_OK;
    if (!x || !Wg || !topk_idx || !topk_gate || !fallback_idx || !fallback_gate || !aligned16(x) ||
        !aligned16(Wg))
        return MOE_ERR_INVALID_ARG;
    return cuda_rc(launch_route(p, x, Wg, bias, topk_idx, topk_gate, probs, (cudaStream_t)stream, nullptr,
                                fallback_idx, fallback_gate));
}

int moe_assign_slots_reroute(const moe_problem* mp, const int32_t* topk_idx, const float* topk_gate,
                             const int32_t* fallback_idx, const float* fallback_gate, int32_t* route_idx,
                             float* route_gate, int32_t* slot_pos, int32_t* counts_routed, int32_t* counts_kept,
                             int32_t* expert_offsets, int32_t* shard_offsets, int32_t* shard_routed,
                             int32_t* shard_overflow, int32_t* row_token, int32_t* dropped, int32_t* rerouted,
                             void* ws, size_t ws_bytes, void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (!(p.flags & MOE_FLAG_REROUTE)) return MOE_ERR_INVALID_ARG;
    if ((p.T > 0 && (!topk_idx || !topk_gate || !fallback_idx || !fallback_gate || !route_idx || !route_gate ||
                     !slot_pos || !row_token)) ||
        !counts_routed || !counts_kept || !expert_offsets || !shard_offsets || !shard_routed || !shard_overflow)
        return MOE_ERR_INVALID_ARG;
    moe_workspace_layout L;
    rc = check_ws(p, ws, ws_bytes, &L);
    if (rc != MOE_OK) return rc;
    char* w = (char*)ws;
    int* status = (int*)(w + L.status);
    int32_t* hist = (int32_t*)(w + L.hist);
    cudaStream_t s = (cudaStream_t)stream;
    // first pass: count and scan of the k choices (no rank pass); T = 0 stops here with zero counts
    const AssignScan first{hist, counts_routed, counts_kept, expert_offsets, shard_offsets, shard_routed,
                           shard_overflow, dropped, (unsigned*)(status + 1), p.E, p.D, p.k, p.nblk, p.C,
                           p.C_shard};
    cudaError_t e = launch_count(p, topk_idx, first, status, s);
    if (e != cudaSuccess || p.nblk == 0) {
        if (e == cudaSuccess && rerouted) e = cudaMemsetAsync(rerouted, 0, sizeof(int32_t), s);
        return cuda_rc(e);
    }
    AssignScan second = first;
    second.second = true;
    second.rerouted = rerouted;
    return cuda_rc(launch_reroute(p, topk_idx, topk_gate, fallback_idx, fallback_gate, route_idx, route_gate,
                                  slot_pos, second, row_token, status, s));
}

int moe_dispatch(const moe_problem* mp, const void* x, const int32_t* row_token, const int32_t* expert_offsets,
                 void* xd, void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (p.rows_max == 0) return MOE_OK;
    if (!x || !row_token || !expert_offsets || !xd || !aligned16(x) || !aligned16(xd)) return MOE_ERR_INVALID_ARG;
    return cuda_rc(launch_dispatch(p, x, row_token, expert_offsets, xd, (cudaStream_t)stream));
}

int moe_dispatch_by_token(const moe_problem* mp, const void* x, const int32_t* topk_idx, const int32_t* slot_pos,
                          const int32_t* expert_offsets, void* xd, void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (p.rows_max == 0 || p.T == 0) return MOE_OK;
    if (!x || !topk_idx || !slot_pos || !expert_offsets || !xd || !aligned16(x) || !aligned16(xd))
        return MOE_ERR_INVALID_ARG;
    return cuda_rc(launch_scatter(p, x, topk_idx, slot_pos, expert_offsets, xd, (cudaStream_t)stream));
}

int moe_expert_ffn(const moe_problem* mp, const void* xd, const int32_t* expert_offsets, const void* W1,
                   const void* W3, const void* W2, void* yd, void* ws, size_t ws_bytes, void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (!expert_offsets || !W1 || !W2 || !xd || !yd) return MOE_ERR_INVALID_ARG;
    if (p.act == MOE_ACT_SWIGLU && !W3) return MOE_ERR_INVALID_ARG;
    if (!aligned16(xd) || !aligned16(yd) || !aligned16(W1) || !aligned16(W2) || (W3 && !aligned16(W3)))
        return MOE_ERR_INVALID_ARG;
    moe_workspace_layout L;
    rc = check_ws(p, ws, ws_bytes, &L);
    if (rc != MOE_OK) return rc;
    if (p.rows_max == 0) return MOE_OK;
    void* h = (char*)ws + L.h;
    int* status = (int*)((char*)ws + L.status);
    cudaStream_t s = (cudaStream_t)stream;
    if (p.dtype == MOE_BF16 && p.act == MOE_ACT_SWIGLU) {
        cudaError_t e = launch_ffn_tc(p, xd, expert_offsets, W1, W3, W2, h, yd, status,
                                      (int*)((char*)ws + L.ffn_sync), s);
        if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
        return cuda_rc(e);
    }
    return cuda_rc(launch_ffn_simt(p, xd, expert_offsets, W1, W3, W2, h, yd, s));
}

int moe_combine(const moe_problem* mp, const void* yd, const int32_t* topk_idx, const int32_t* slot_pos,
                const int32_t* expert_offsets, const float* topk_gate, const void* residual, void* y,
                void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (p.T == 0) return MOE_OK;
    if (!yd || !topk_idx || !slot_pos || !expert_offsets || !topk_gate || !y || !aligned16(yd) ||
        !aligned16(y) || (residual && !aligned16(residual)))
        return MOE_ERR_INVALID_ARG;
    return cuda_rc(launch_combine(p, yd, topk_idx, slot_pos, expert_offsets, topk_gate, residual, y,
                                  (cudaStream_t)stream));
}

int moe_layer_forward(const moe_problem* mp, const void* x, const void* Wg, const float* bias, const void* W1,
                      const void* W3, const void* W2, const void* residual, void* y, void* ws, size_t ws_bytes,
                      void* stream) {
    if (mp && mp->ffn_shared != 0) return MOE_ERR_INVALID_ARG;  // needs moe_layer_forward_shared
    return layer_forward(mp, x, Wg, bias, W1, W3, W2, nullptr, nullptr, nullptr, residual, y, ws, ws_bytes,
                         stream);
}

int moe_layer_forward_shared(const moe_problem* mp, const void* x, const void* Wg, const float* bias,
                             const void* W1, const void* W3, const void* W2, const void* Ws1, const void* Ws3,
                             const void* Ws2, const void* residual, void* y, void* ws, size_t ws_bytes,
                             void* stream) {
    return layer_forward(mp, x, Wg, bias, W1, W3, W2, Ws1, Ws3, Ws2, residual, y, ws, ws_bytes, stream);
}

int moe_shared_expert_ffn(const moe_problem* mp, const void* x, const void* Ws1, const void* Ws3,
                          const void* Ws2, void* ys, void* ws, size_t ws_bytes, void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (p.ffn_shared <= 0) return MOE_ERR_INVALID_ARG;
    if (!x || !Ws1 || !Ws2 || !ys || (p.act == MOE_ACT_SWIGLU && !Ws3)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(Ws1) || !aligned16(Ws2) || (Ws3 && !aligned16(Ws3)) || !aligned16(ys))
        return MOE_ERR_INVALID_ARG;
    moe_workspace_layout L;
    rc = check_ws(p, ws, ws_bytes, &L);
    if (rc != MOE_OK) return rc;
    if (p.T == 0) return MOE_OK;
    return run_shared_expert(p, L, (char*)ws, x, Ws1, Ws3, Ws2, ys, (cudaStream_t)stream);
}

int moe_combine_shared(const moe_problem* mp, const void* yd, const int32_t* topk_idx, const int32_t* slot_pos,
                       const int32_t* expert_offsets, const float* topk_gate, const void* shared,
                       const void* residual, void* y, void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (p.T == 0) return MOE_OK;
    if (!yd || !topk_idx || !slot_pos || !expert_offsets || !topk_gate || !y || !aligned16(yd) ||
        !aligned16(y) || (residual && !aligned16(residual)) || (shared && !aligned16(shared)))
        return MOE_ERR_INVALID_ARG;
    return cuda_rc(launch_combine(p, yd, topk_idx, slot_pos, expert_offsets, topk_gate, residual, y,
                                  (cudaStream_t)stream, shared));
}

int moe_router_logits(const moe_problem* mp, const void* x, const void* Wg, const float* bias, float* logits,
                      float* probs, void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (p.T == 0) return MOE_OK;
    if (!x || !Wg || !logits || !aligned16(x) || !aligned16(Wg)) return MOE_ERR_INVALID_ARG;
    return cuda_rc(launch_route(p, x, Wg, bias, nullptr, nullptr, probs, (cudaStream_t)stream, logits));
}

int moe_expert_choice_assign(const moe_problem* mp, const float* logits, int32_t* row_token,
                             int32_t* expert_offsets, int32_t* sel_row, void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (!(p.flags & MOE_FLAG_EXPERT_CHOICE)) return MOE_ERR_INVALID_ARG;
    if (!expert_offsets || (p.T > 0 && (!logits || !row_token || !sel_row))) return MOE_ERR_INVALID_ARG;
    return cuda_rc(launch_ec_select(p, logits, row_token, expert_offsets, sel_row, (cudaStream_t)stream));
}

int moe_combine_expert_choice(const moe_problem* mp, const void* yd, const float* probs, const int32_t* sel_row,
                              const void* shared, const void* residual, void* y, void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (!(p.flags & MOE_FLAG_EXPERT_CHOICE)) return MOE_ERR_INVALID_ARG;
    if (p.T == 0) return MOE_OK;
    if (!yd || !probs || !sel_row || !y || !aligned16(yd) || !aligned16(y) || (shared && !aligned16(shared)) ||
        (residual && !aligned16(residual)))
        return MOE_ERR_INVALID_ARG;
    return cuda_rc(launch_ec_combine(p, yd, probs, sel_row, shared, residual, y, (cudaStream_t)stream));
}

int moe_routing_stats(const moe_problem* mp, const float* probs, const int32_t* counts_routed,
                      const int32_t* counts_kept, float* stats, float* mean_prob, void* ws, size_t ws_bytes,
                      void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if ((p.T > 0 && !probs) || !counts_routed || !counts_kept || !stats) return MOE_ERR_INVALID_ARG;
    if (p.T > ((int64_t)1 << 25)) return MOE_ERR_UNSUPPORTED;  // the 64-bit fixed-point sums
    moe_workspace_layout L;
    rc = check_ws(p, ws, ws_bytes, &L);
    if (rc != MOE_OK) return rc;
    char* w = (char*)ws;
    // status[2] is the statistics kernel's completion ticket
    return cuda_rc(launch_routing_stats(p, probs, counts_routed, counts_kept, stats, mean_prob,
                                        (unsigned long long*)(w + L.stats), (unsigned*)(w + L.status) + 2,
                                        (cudaStream_t)stream));
}

int moe_host_alloc(size_t bytes, void** ptr) {
    if (!ptr) return MOE_ERR_INVALID_ARG;
    *ptr = nullptr;
    if (bytes == 0) return MOE_OK;
    return cudaHostAlloc(ptr, bytes, cudaHostAllocPortable) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_host_free(void* ptr) {
    if (!ptr) return MOE_OK;
    return cudaFreeHost(ptr) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_host_staging_size(const moe_problem* mp, size_t* bytes) {
    if (!bytes) return MOE_ERR_INVALID_ARG;
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    *bytes = host_staging_bytes(p);
    return MOE_OK;
}

int moe_layer_forward_host(const moe_problem* mp, int64_t n_steps, const void* const* x_host, const void* Wg,
                           const float* bias, const void* W1, const void* W3, const void* W2,
                           void* const* y_host, void* staging, size_t staging_bytes, void* ws, size_t ws_bytes,
                           void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (p.ffn_shared != 0 || n_steps < 0) return MOE_ERR_INVALID_ARG;
    if (n_steps == 0 || p.T == 0) return MOE_OK;
    if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
    for (int64_t i = 0; i < n_steps; ++i)
        if (!x_host[i] || !y_host[i]) return MOE_ERR_INVALID_ARG;
    const size_t xb = (size_t)p.T * p.d * esize(p.dtype), slot = align256(xb);
    if (!staging || staging_bytes < host_staging_bytes(p) || !aligned16(staging)) return MOE_ERR_WORKSPACE;
    moe_workspace_layout L;
    rc = check_ws(p, ws, ws_bytes, &L);
    if (rc != MOE_OK) return rc;
    HostPipe* hp = nullptr;
    rc = host_pipe(&hp);
    if (rc != MOE_OK) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    char* st = (char*)staging;
    void* xs[2] = {st, st + slot};
    void* ys[2] = {st + 2 * slot, st + 3 * slot};
    auto ck = [](cudaError_t e) { return e == cudaSuccess; };
    // the copies start after the work already queued on `stream`
    if (!ck(cudaEventRecord(hp->start, s)) || !ck(cudaStreamWaitEvent(hp->in, hp->start, 0)) ||
        !ck(cudaStreamWaitEvent(hp->out, hp->start, 0)))
        return MOE_ERR_CUDA;
    for (int64_t i = 0; i < n_steps; ++i) {
        const int b = (int)(i & 1);
        // x buffer b is free once step i-2's layer has read it
        if (i >= 2 && !ck(cudaStreamWaitEvent(hp->in, hp->comp_done[b], 0))) return MOE_ERR_CUDA;
        if (!ck(cudaMemcpyAsync(xs[b], x_host[i], xb, cudaMemcpyHostToDevice, hp->in)) ||
            !ck(cudaEventRecord(hp->in_done[b], hp->in)) || !ck(cudaStreamWaitEvent(s, hp->in_done[b], 0)))
            return MOE_ERR_CUDA;
        // y buffer b is free once step i-2's output copy has read it
        if (i >= 2 && !ck(cudaStreamWaitEvent(s, hp->out_done[b], 0))) return MOE_ERR_CUDA;
        rc = layer_forward(mp, xs[b], Wg, bias, W1, W3, W2, nullptr, nullptr, nullptr, nullptr, ys[b], ws, ws_bytes,
                           stream);
        if (rc != MOE_OK) return rc;
        if (!ck(cudaEventRecord(hp->comp_done[b], s)) || !ck(cudaStreamWaitEvent(hp->out, hp->comp_done[b], 0)) ||
            !ck(cudaMemcpyAsync(y_host[i], ys[b], xb, cudaMemcpyDeviceToHost, hp->out)) ||
            !ck(cudaEventRecord(hp->out_done[b], hp->out)))
            return MOE_ERR_CUDA;
    }
    // `stream` completes only after every output copy
    for (int b = 0; b < 2 && b < n_steps; ++b)
        if (!ck(cudaStreamWaitEvent(s, hp->out_done[b], 0))) return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_layer_launch_count(const moe_problem* mp, int* launches) {
    if (!launches) return MOE_ERR_INVALID_ARG;
    Problem p;
    int rc = to_problem(mp, &p);
    if (rc != MOE_OK) return rc;
    if (p.T == 0) {
        *launches = 0;
        return MOE_OK;
    }
    // the branches of layer_forward: routing and slots, dispatch, FFN(s), combine
    const int ffn = (p.dtype == MOE_BF16 && p.act == MOE_ACT_SWIGLU) ? 1 : 2;
    int n;
    if (p.flags & MOE_FLAG_EXPERT_CHOICE) n = 2 + 1;        // router, selection; dispatch
    else if (p.flags & MOE_FLAG_REROUTE) n = 3 + 1;         // router, reroute, place; dispatch
    else if (assign_pack_fits(p)) n = 2;                    // router, slot-and-pack
    else n = 2 + 1;                                         // router, rank; dispatch
    n += ffn + (p.ffn_shared > 0 ? ffn : 0) + 1;            // routed (+ shared) FFN, combine
    *launches = n;
    return MOE_OK;
}

int moe_device_status(void* ws, void* stream) {
    if (!ws) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    int word = 0;
    // the status word is the first region of every layout
    if (cudaMemcpy(&word, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpy(ws, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (word & kDevTimeout) return MOE_ERR_TIMEOUT;
    if (word) return MOE_ERR_DEVICE;
    return MOE_OK;
}

const char* moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "valid problem outside what this library supports";
        case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "a kernel's bounded wait timed out";
        case MOE_ERR_DEVICE: return "a kernel recorded an error (bad index)";
        default: return "unknown status";
    }
}

}  // extern "C"
