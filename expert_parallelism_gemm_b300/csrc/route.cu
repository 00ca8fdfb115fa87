// route.cu -- router: logits, softmax, top-k and gates.
//
// "Expert Parallelism" notes page (narrativegoldmine.com), "Formal
// Algorithm: Expert Parallelism Forward Pass": gate computation (logits of the
// routing projection, p = softmax(g / tau), tau = 1) and expert selection
// (gate weight = probability of the chosen expert); "Components and
// Architecture": top-k selection and an optional per-expert logit bias.
//
// Logit order (fixed so that the top-k decision is reproducible bit for bit):
// the hidden index is dealt into 32 slices of runs of 8 consecutive elements,
// slice j = { i = 256 m + 8 j + q : q = 0..7 }; each slice sum is one fp32
// fused multiply-add chain in ascending i from +0; the 32 slice sums are
// combined by the xor butterfly o = 16, 8, 4, 2, 1 (every slice j replaced by
// s[j] + s[j ^ o] at once), which leaves the same value in every slice; then
// the bias is added.
//
// That order maps onto a warp: lane j owns slice j.  A CTA handles one
// assignment block of 32 tokens with 8 warps; warp w owns tokens 4w..4w+3
// and, in pass p, experts RE*p..RE*p+RE-1 (RE = 8, or 16 for 9..64 experts) --
// 4*RE (token, expert) pairs, so each lane keeps 4*RE slice sums and every
// 16-byte shared-memory load feeds 8*RE (x row) or 32 (Wg row) multiply-adds
// per lane.  The hidden dimension is walked in
// chunks of 256 elements (8 per lane) through an S-stage ring of TMA tile
// copies: per chunk one thread issues two 2-D box loads (the CTA's 32 x rows
// and the pass's RE Wg rows, in their storage type, zero-filled past T, E and
// d -- a zero element adds an exact zero product) that complete on the
// stage's "full" mbarrier; each warp, done with a chunk, arrives on the
// stage's "empty" mbarrier, and only the issuing thread waits on that before
// refilling the stage (no CTA-wide barrier per chunk).  Every wait is bounded
// in time; on expiry the kernel records MOE_ERR_TIMEOUT's device bit and
// stops computing.
// After the last chunk of a pass the warp reduces its pairs with the
// butterfly in reduce-scatter form: in round o a lane keeps the half of its
// pairs selected by bit o of its lane index and adds the partner's copy of
// that half, which is the butterfly's own sum s[j] + s[j ^ o] for those pairs;
// after five rounds lane j holds pairs (4*RE/32) j .. (4*RE/32) j + 4*RE/32 - 1.
// Passes repeat for every group of RE experts, re-reading x from L2.
//
// Softmax and top-k run from a shared-memory logit table: one thread per token
// for up to 32 experts, one warp per token above that.  The gate of choice r
// is its softmax probability, or -- when renormalising -- exp(g_r - m) over
// the sum of the k chosen exp(g - m), added in rank order.  For overflow
// rerouting the same selection continues for k more ranks: the token's next
// k experts (its fallbacks) and their softmax probabilities.
//
// Inside the layer forward the router also starts the slot assignment: a CTA
// holds exactly one assignment block of kAssignBlock tokens, so it counts its
// tokens' rank-r choices per expert (one warp match per rank), writes that
// block's histogram entries, and the last CTA to finish scans them
// (assign_scan.cuh) -- or, when the histogram is small, leaves the scan to the
// fused slot-and-pack kernel (assign_pack.cu).  The standalone router call
// leaves all of this out.
#include <math_constants.h>

#include "assign_scan.cuh"

namespace moe {
namespace {

constexpr int kRT = 4;                       // tokens per warp tile
constexpr int kRouteThreads = 256;           // 8 warps x 4 tokens = 32 tokens
constexpr int kTok = 32;                     // tokens per CTA
constexpr int kKC = 256;                     // hidden elements per chunk (32 lanes x 8)
static_assert(kTok == kAssignBlock, "one CTA per assignment block");
static_assert(kRouteThreads / 32 * kRT == kTok, "warp tiles cover the CTA's tokens");

constexpr uint64_t kRouteTimeoutNs = 2000000000ull;  // 2 s: far above any legitimate wait

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t route_timer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Wait for the phase of `parity`.  Gives up (false) when *abort is raised or
// after kRouteTimeoutNs, then raising *abort and recording the timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = route_timer();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (route_timer() - t0 > kRouteTimeoutNs) {
            *abort = 1;
            if (status) atomicOr(status, kDevTimeout);
            return false;
        }
    }
    return true;
}
// 2-D box of `map` at (c0 = column, c1 = row) into shared memory at dst.
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        ::"r"(dst), "l"((uint64_t)map), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

// 8 consecutive fp32 elements of a shared-memory row (the fp32 router; the
// bf16 one feeds its packed halves to fma8_bf16 instead).
__device__ __forceinline__ void load8(const uint8_t* p, float (&v)[8], float*) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 16);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
}

// acc = fma(x[j], w[j], acc) for the 8 bf16 elements j = 0..7 of a 16-byte
// vector pair, in ascending j (element 2i is the low half of word i).  The
// mixed-precision FMA takes the bf16 halves as they are: widening bf16 to fp32
// is exact, so each step rounds exactly as fmaf on the widened values does,
// and no unpacking instructions are spent.
__device__ __forceinline__ void fma8_bf16(float& acc, const uint4& x, const uint4& w) {
    asm("{\n"
        " .reg .b16 x0, x1, x2, x3, x4, x5, x6, x7, w0, w1, w2, w3, w4, w5, w6, w7;\n"
        " mov.b32 {x0, x1}, %1;\n mov.b32 {x2, x3}, %2;\n mov.b32 {x4, x5}, %3;\n mov.b32 {x6, x7}, %4;\n"
        " mov.b32 {w0, w1}, %5;\n mov.b32 {w2, w3}, %6;\n mov.b32 {w4, w5}, %7;\n mov.b32 {w6, w7}, %8;\n"
        " fma.rn.f32.bf16 %0, x0, w0, %0;\n fma.rn.f32.bf16 %0, x1, w1, %0;\n"
        " fma.rn.f32.bf16 %0, x2, w2, %0;\n fma.rn.f32.bf16 %0, x3, w3, %0;\n"
        " fma.rn.f32.bf16 %0, x4, w4, %0;\n fma.rn.f32.bf16 %0, x5, w5, %0;\n"
        " fma.rn.f32.bf16 %0, x6, w6, %0;\n fma.rn.f32.bf16 %0, x7, w7, %0;\n"
        "}"
        : "+f"(acc)
        : "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w), "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w));
}

// One reduce-scatter round of the butterfly over offset O: of the N values
// a[0..N), keep the half chosen by bit O of the lane and add the partner's.
template <int O, int N, int M>
__device__ __forceinline__ void rs_round(float (&a)[M], int lane) {
    const bool hi = (lane & O) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const float send = hi ? a[i] : a[i + N / 2];
        const float keep = hi ? a[i + N / 2] : a[i];
        a[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
    }
}

// Gates of one token's k choices (chosen[r] = logit of choice r, m = the
// token's largest logit, inv = 1 / sum over all experts of exp(g - m)).
__device__ __forceinline__ void write_gates(float* gate, const float (&chosen)[8], int k, float m, float inv,
                                            int renorm) {
    if (!renorm) {
        for (int r = 0; r < k; ++r) gate[r] = expf(chosen[r] - m) * inv;
        return;
    }
    float den = 0.0f;
    for (int r = 0; r < k; ++r) den += expf(chosen[r] - m);
    for (int r = 0; r < k; ++r) gate[r] = expf(chosen[r] - m) / den;
}

// ring stages: 4 for bf16 (3 for fp32, whose chunks are twice the bytes);
// at up to 8 experts 3, where 62 KB of shared memory and 80 registers a thread
// leave room for three CTAs per SM (five stages, the earlier choice, left
// two), and for bf16 rows longer than 1024 elements 2, with four CTAs per SM
// (64 registers).  Measured with identical indices: the 8x7B-shape router
// (d = 4096) 86 us with five stages, 80 with three, 76 with two; the one at
// T = 4096, d = 1024, 11.0 us with three or five, 12.4 with two.
template <typename T>
__host__ __device__ constexpr int route_stages() {
    return sizeof(T) == 2 ? 4 : 3;
}
template <typename T>
constexpr int route_stages_small_e() {
    return 3;
}
constexpr int kRouteStagesLongRows = 2;  // bf16, up to 8 experts, d > 1024

// experts per pass: 8, or 16 above 8 experts
template <int RE>
size_t route_smem_bytes(int elem_bytes, int stages, int E, int k) {
    const int epad = (E + RE - 1) / RE * RE;
    return 128 + (size_t)stages * (kTok + RE) * kKC * elem_bytes + (size_t)kTok * (epad + 1) * sizeof(float) +
           (size_t)k * E * sizeof(int);
}

template <typename T, int RE, int S>
__global__ void __launch_bounds__(kRouteThreads, S == 2 ? 4 : 2)
route_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw, int64_t T_, int d,
             int E, int k, const float* __restrict__ bias, int32_t* __restrict__ topk_idx,
             float* __restrict__ topk_gate, float* __restrict__ probs, float* __restrict__ logits,
             int32_t* __restrict__ fb_idx, float* __restrict__ fb_gate, const int renorm, int* status,
             const AssignScan scan) {
    constexpr int RP = kKC * (int)sizeof(T);         // ring row pitch, bytes
    constexpr int kStageRows = kTok + RE;            // x rows, then the pass's Wg rows
    constexpr uint32_t kStageBytes = (uint32_t)kStageRows * RP;
    constexpr int NP = kRT * RE;                     // (token, expert) pairs per warp
    constexpr int PL = NP / 32;                      // pairs per lane after the butterfly

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * S];    // per stage: copies landed ("full"), warps done ("empty")
    __shared__ int s_abort;
    const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(smem_raw);
    uint8_t* ring = smem_raw + ((128u - (raw_s & 127u)) & 127u);  // [S][kStageRows][RP], TMA-aligned
    const int npass = (E + RE - 1) / RE;
    const int LGP = npass * RE + 1;
    float* lg = reinterpret_cast<float*>(ring + (size_t)S * kStageRows * RP);  // [kTok][LGP]
    int* cnt = reinterpret_cast<int*>(lg + kTok * LGP);                         // [k][E]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t t0 = (int64_t)blockIdx.x * kTok;
    const int nchunks = (d + kKC - 1) / kKC;
    const int nq = npass * nchunks;
    const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
    const uint32_t bar_s = (uint32_t)__cvta_generic_to_shared(bars);
    const uint32_t empty_s = bar_s + 8u * S;
    volatile int* abort_flag = &s_abort;
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(bar_s + 8u * i, 1);
            mbar_init(empty_s + 8u * i, kRouteThreads / 32);
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    dep_wait();

    // thread 0 loads flattened chunk q = (pass, chunk) into ring slot q % S:
    // the CTA's x rows and the pass's Wg rows, one box each
    int issued = 0;
    auto issue = [&](int q) {
        if (q < nq) {
            const int pass = q / nchunks, c = q - pass * nchunks;
            const uint32_t slot = ring_s + (uint32_t)(q % S) * kStageBytes;
            const uint32_t bar = bar_s + 8u * (uint32_t)(q % S);
            mbar_expect_tx(bar, kStageBytes);
            tma_box(slot, &tmx, bar, c * kKC, (int)t0);
            tma_box(slot + (uint32_t)(kTok * RP), &tmw, bar, c * kKC, pass * RE);
            issued = q + 1;
        }
    };

    float acc[NP];  // slice sums of pair p = rt * RE + re
#pragma unroll
    for (int p = 0; p < NP; ++p) acc[p] = 0.0f;

    if (tid == 0)
        for (int q = 0; q < S - 1; ++q) issue(q);
    for (int q = 0; q < nq; ++q) {
        // thread 0 refills the stage of chunk q-1 with chunk q+S-1 once every
        // warp is done with chunk q-1 (stage S-1 is still unused at q = 0)
        if (tid == 0 && q + S - 1 < nq) {
            if (q == 0 || mbar_wait_bounded(empty_s + 8u * (uint32_t)((q - 1) % S),
                                            (uint32_t)(((q - 1) / S) & 1), abort_flag, status))
                issue(q + S - 1);
        }
        // the warp leaves together (its lanes meet again in shuffles) if any
        // lane's wait gave up
        const bool landed =
            mbar_wait_bounded(bar_s + 8u * (uint32_t)(q % S), (uint32_t)((q / S) & 1), abort_flag, status);
        if (!__all_sync(0xffffffffu, landed)) break;
        const uint8_t* base = ring + (size_t)(q % S) * kStageRows * RP + lane * 8 * (int)sizeof(T);
        if constexpr (sizeof(T) == 2) {
            uint4 xq[kRT];
#pragma unroll
            for (int rt = 0; rt < kRT; ++rt)
                xq[rt] = *reinterpret_cast<const uint4*>(base + (size_t)(kRT * warp + rt) * RP);
#pragma unroll
            for (int re = 0; re < RE; ++re) {
                const uint4 wq = *reinterpret_cast<const uint4*>(base + (size_t)(kTok + re) * RP);
#pragma unroll
                for (int rt = 0; rt < kRT; ++rt) fma8_bf16(acc[rt * RE + re], xq[rt], wq);
            }
        } else {
            float xv[kRT][8];
#pragma unroll
            for (int rt = 0; rt < kRT; ++rt) load8(base + (size_t)(kRT * warp + rt) * RP, xv[rt], (T*)nullptr);
#pragma unroll
            for (int re = 0; re < RE; ++re) {
                float wv[8];
                load8(base + (size_t)(kTok + re) * RP, wv, (T*)nullptr);
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int rt = 0; rt < kRT; ++rt)
                        acc[rt * RE + re] = fmaf(xv[rt][j], wv[j], acc[rt * RE + re]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_s + 8u * (uint32_t)(q % S));  // this warp is done with the stage
        const int pass = q / nchunks;
        if (q - pass * nchunks == nchunks - 1) {
            // end of a pass: butterfly in reduce-scatter form, lane j gets
            // pairs PL*j .. PL*j + PL - 1
            rs_round<16, NP>(acc, lane);
            rs_round<8, NP / 2>(acc, lane);
            rs_round<4, NP / 4>(acc, lane);
            rs_round<2, NP / 8>(acc, lane);
            rs_round<1, NP / 16>(acc, lane);
#pragma unroll
            for (int i = 0; i < PL; ++i) {
                const int pr = PL * lane + i;
                const int tl = kRT * warp + pr / RE;
                const int e = pass * RE + pr % RE;
                if (e < E) {
                    const float g = bias ? acc[i] + bias[e] : acc[i];
                    lg[tl * LGP + e] = g;
                    if (logits && t0 + tl < T_) logits[(size_t)(t0 + tl) * E + e] = g;
                }
            }
#pragma unroll
            for (int p = 0; p < NP; ++p) acc[p] = 0.0f;
        }
    }
    __syncthreads();
    if (s_abort) {
        // a wait gave up: thread 0 waits (bounded) for the copies that may
        // still be in flight -- the last S-1 it issued, each in its own stage
        // -- and the rest runs on zero logits so that every index stays in
        // range (the status word reports the error)
        if (tid == 0) {
            int quiet = 0;
            for (int c = issued - (S - 1) > 0 ? issued - (S - 1) : 0; c < issued; ++c)
                if (!mbar_wait_bounded(bar_s + 8u * (uint32_t)(c % S), (uint32_t)((c / S) & 1), &quiet, status))
                    break;
        }
        for (int i = tid; i < kTok * LGP; i += kRouteThreads) lg[i] = 0.0f;
    }
    if (scan.hist)
        for (int i = tid; i < k * E; i += kRouteThreads) cnt[i] = 0;
    __syncthreads();
    const bool count = scan.hist != nullptr;
    const int kr = fb_idx ? 2 * k : k;  // ranks selected: the choices, then the fallbacks

    if (E <= 32) {
        // softmax + top-k: one thread per token, warp 0 (rows of tokens past T
        // hold bias-only logits and write nothing); a rank's per-expert counts
        // for the block come from one warp match, stored by each group's
        // first lane (no shared-memory atomics)
        if (tid < kTok) {
            const int64_t t = t0 + tid;
            const bool valid = t < T_;
            const float* gl = lg + tid * LGP;
            float m = -CUDART_INF_F;
            for (int e = 0; e < E; ++e) m = fmaxf(m, gl[e]);
            float s = 0.0f;
            for (int e = 0; e < E; ++e) s += expf(gl[e] - m);
            const float inv = 1.0f / s;
            if (probs && valid)
                for (int e = 0; e < E; ++e) probs[(size_t)t * E + e] = expf(gl[e] - m) * inv;
            uint32_t taken = 0;
            float chosen[8];
            for (int r = 0; r < kr; ++r) {
                int be = -1;
                float bv = -CUDART_INF_F;
                for (int e = 0; e < E; ++e) {
                    // ascending e with a strict '>' keeps the lower index on ties
                    if (!(taken >> e & 1u) && (be < 0 || gl[e] > bv)) {
                        bv = gl[e];
                        be = e;
                    }
                }
                taken |= 1u << be;
                if (r >= k) {
                    if (valid) {
                        fb_idx[(size_t)t * k + r - k] = be;
                        if (fb_gate) fb_gate[(size_t)t * k + r - k] = expf(bv - m) * inv;
                    }
                    continue;
                }
                chosen[r] = bv;
                if (valid && topk_idx) topk_idx[(size_t)t * k + r] = be;
                if (count) {
                    const int key = valid ? be : -1;
                    const uint32_t same = __match_any_sync(0xffffffffu, key);
                    if (valid && tid == __ffs(same) - 1) cnt[r * E + be] = __popc(same);
                }
            }
            if (valid && topk_gate) write_gates(topk_gate + (size_t)t * k, chosen, k, m, inv, renorm);
        }
    } else {
        // softmax + top-k: one warp per token, lane holds experts lane + 32 q
        constexpr int kMaxPerLane = 256 / 32;
        for (int tt = warp; tt < kTok; tt += kRouteThreads / 32) {
            const int64_t t = t0 + tt;
            if (t >= T_) break;
            float gv[kMaxPerLane];
            float m = -CUDART_INF_F;
#pragma unroll
            for (int q = 0; q < kMaxPerLane; ++q) {
                const int e = lane + 32 * q;
                gv[q] = e < E ? lg[tt * LGP + e] : -CUDART_INF_F;
                m = fmaxf(m, gv[q]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            float s = 0.0f;
#pragma unroll
            for (int q = 0; q < kMaxPerLane; ++q)
                if (lane + 32 * q < E) s += expf(gv[q] - m);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            const float inv = 1.0f / s;
            if (probs) {
#pragma unroll
                for (int q = 0; q < kMaxPerLane; ++q) {
                    const int e = lane + 32 * q;
                    if (e < E) probs[(size_t)t * E + e] = expf(gv[q] - m) * inv;
                }
            }
            uint32_t taken = 0;
            float chosen[8];
            for (int r = 0; r < kr; ++r) {
                float bv = -CUDART_INF_F;
                int be = 0x7fffffff;
#pragma unroll
                for (int q = 0; q < kMaxPerLane; ++q) {
                    const int e = lane + 32 * q;
                    if (e < E && !(taken >> q & 1u) && (gv[q] > bv || be == 0x7fffffff)) {
                        // within a lane e grows with q, so '>' keeps the lower index on ties
                        bv = gv[q];
                        be = e;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                    if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) {
                        bv = ov;
                        be = oe;
                    }
                }
                if ((be & 31) == lane) taken |= 1u << (be >> 5);
                if (r >= k) {
                    if (lane == 0) {
                        fb_idx[(size_t)t * k + r - k] = be;
                        if (fb_gate) fb_gate[(size_t)t * k + r - k] = expf(bv - m) * inv;
                    }
                    continue;
                }
                chosen[r] = bv;
                if (lane == 0) {
                    if (topk_idx) topk_idx[(size_t)t * k + r] = be;
                    if (count) atomicAdd(&cnt[r * E + be], 1);
                }
            }
            if (lane == 0 && topk_gate) write_gates(topk_gate + (size_t)t * k, chosen, k, m, inv, renorm);
        }
    }
    if (count) {
        __syncthreads();
        const int64_t b = blockIdx.x;  // this CTA's assignment block
        for (int i = tid; i < k * E; i += kRouteThreads) {
            const int e = i / k, r = i % k;
            scan.hist[((size_t)e * k + r) * scan.nblk + b] = cnt[r * E + e];
        }
        // histogram reads kept ahead of the scan: two for bf16, none for fp32
        // (whose 16-expert instance would spill under the 128-register cap)
        if (!scan.defer) finish_assign_scan<sizeof(T) == 2 ? 2 : 0>(scan);
    }
}

template <typename T, int RE, int S>
cudaError_t launch_route_re(const Problem& p, const void* x, const void* Wg, const float* bias,
                            int32_t* topk_idx, float* topk_gate, float* probs, float* logits,
                            int32_t* fb_idx, float* fb_gate, int* status, const AssignScan& scan, cudaStream_t s) {
    CUtensorMap tmx, tmw;
    if (!encode_row_tiles(&tmx, x, p.dtype, (uint64_t)p.T, (uint64_t)p.d, kKC, kTok) ||
        !encode_row_tiles(&tmw, Wg, p.dtype, (uint64_t)p.E, (uint64_t)p.d, kKC, RE))
        return cudaErrorInvalidValue;
    const size_t smem = route_smem_bytes<RE>((int)sizeof(T), S, p.E, p.k);
    auto kern = route_kernel<T, RE, S>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const unsigned grid = (unsigned)ceil_div(p.T, kTok);
    return launch_k(kern, dim3(grid), dim3(kRouteThreads), smem, s, tmx, tmw, p.T, p.d, p.E, p.k, bias, topk_idx,
                    topk_gate, probs, logits, fb_idx, fb_gate, (int)(p.flags & MOE_FLAG_RENORM), status, scan);
}

// 16 experts per pass for 9..64 experts (measured faster at 64), 8 otherwise
// (measured faster at 8 and 128); the deeper ring for up to 8 experts
template <typename T>
cudaError_t launch_route_t(const Problem& p, const void* x, const void* Wg, const float* bias,
                           int32_t* topk_idx, float* topk_gate, float* probs, float* logits,
                           int32_t* fb_idx, float* fb_gate, int* status, const AssignScan& scan,
                           cudaStream_t s) {
    if constexpr (sizeof(T) == 2) {
        if (p.E <= 8 && p.d > 1024)
            return launch_route_re<T, 8, kRouteStagesLongRows>(p, x, Wg, bias, topk_idx, topk_gate, probs, logits,
                                                               fb_idx, fb_gate, status, scan, s);
    }
    if (p.E <= 8)
        return launch_route_re<T, 8, route_stages_small_e<T>()>(p, x, Wg, bias, topk_idx, topk_gate, probs, logits,
                                                                fb_idx, fb_gate, status, scan, s);
    if (p.E <= 64)
        return launch_route_re<T, 16, route_stages<T>()>(p, x, Wg, bias, topk_idx, topk_gate, probs, logits,
                                                         fb_idx, fb_gate, status, scan, s);
    return launch_route_re<T, 8, route_stages<T>()>(p, x, Wg, bias, topk_idx, topk_gate, probs, logits, fb_idx,
                                                    fb_gate, status, scan, s);
}

}  // namespace

cudaError_t launch_route(const Problem& p, const void* x, const void* Wg, const float* bias,
                         int32_t* topk_idx, float* topk_gate, float* probs, cudaStream_t s, float* logits,
                         int32_t* fallback_idx, float* fallback_gate, int* status) {
    if (p.T == 0) return cudaSuccess;
    AssignScan none{};
    // the tensor-core router when only indices and gates are asked for
    if (route_tc_eligible(p) && !probs && !logits && !fallback_idx)
        return launch_route_tc(p, x, Wg, bias, topk_idx, topk_gate, none, status, s);
    if (p.dtype == MOE_BF16)
        return launch_route_t<__nv_bfloat16>(p, x, Wg, bias, topk_idx, topk_gate, probs, logits, fallback_idx,
                                             fallback_gate, status, none, s);
    return launch_route_t<float>(p, x, Wg, bias, topk_idx, topk_gate, probs, logits, fallback_idx, fallback_gate,
                                 status, none, s);
}

cudaError_t launch_route_count(const Problem& p, const void* x, const void* Wg, const float* bias,
                               int32_t* topk_idx, float* topk_gate, const AssignScan& scan,
                               cudaStream_t s, int32_t* fallback_idx, float* fallback_gate, int* status) {
    if (p.T == 0) return cudaErrorInvalidValue;  // callers handle T = 0 without a launch
    if (route_tc_eligible(p) && !fallback_idx)
        return launch_route_tc(p, x, Wg, bias, topk_idx, topk_gate, scan, status, s);
    if (p.dtype == MOE_BF16)
        return launch_route_t<__nv_bfloat16>(p, x, Wg, bias, topk_idx, topk_gate, nullptr, nullptr, fallback_idx,
                                             fallback_gate, status, scan, s);
    return launch_route_t<float>(p, x, Wg, bias, topk_idx, topk_gate, nullptr, nullptr, fallback_idx,
                                 fallback_gate, status, scan, s);
}

}  // namespace moe
