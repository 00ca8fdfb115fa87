// route_tc.cu -- the bf16 router on the tensor cores, with a top-k that is
// exact in the router's fixed logit order.
//
// "Expert Parallelism" notes page (narrativegoldmine.com), "Formal Algorithm:
// Expert Parallelism Forward Pass": gate computation (logits of the routing
// projection, p = softmax(g), temperature 1) and expert selection (gate
// weight = probability of the chosen expert); "Components and Architecture":
// top-k selection, optional per-expert logit bias.
//
// The top-k decision is defined on the logits in one fixed fp32 order (32
// slices of runs of 8 consecutive hidden elements, one fused multiply-add
// chain each, combined by an xor butterfly; route.cu).  Computing every logit
// that way costs T*E*d scalar multiply-adds, which bounds the SIMT router by
// instruction issue far above its memory time once E reaches 64.  Here the
// logits are first computed on the tensor cores, g^ = x Wg^T in bf16 with
// fp32 accumulation, and the fixed order is used only where it can change
// the answer:
//
//  1. GEMM.  A persistent launch, one CTA per SM, walks tiles of 128 tokens.
//     Per 64-element hidden chunk one thread issues two TMA loads (128-byte
//     swizzle) into one stage: the chunk of the E Wg rows (E padded to a
//     multiple of 16, rows past E zero-filled), and after it the chunk of the
//     tile's 128 x rows.  Per K = 16 step two tcgen05.mma (M = 128): x times
//     the Wg rows into the logit accumulator of the current K group, and x
//     times x into the Gram accumulator, whose diagonal is ||x_t||^2 at no
//     extra memory traffic.  The hidden dimension is split into nc groups of
//     consecutive stages, each accumulated in its own tensor-memory columns
//     (as many as the 384 columns after the Gram block hold), and the
//     epilogue adds the nc partial logits in ascending group order in fp32.
//     A shorter accumulation per group is what keeps the error bound tight.
//
//  2. Error bound.  Under the accumulation model stated below,
//     |g^[t,e] + b[e] - g[t,e]| <= theta_t with
//       theta_t = c_d * ||x_t|| * max_e ||Wg_e|| + 2^-22 * max_e |g^[t,e] + b[e]|,
//     where g is the fixed-order logit and c_d covers the tensor-core
//     accumulation (each MMA step of a group adds at most
//     kHwUlp * (|accumulator| + sum |products|) of error -- 32 fp32 ulps of the
//     magnitude, several times more than a truncating adder of 16 aligned
//     products loses -- and a group has 4 * stages-per-group steps), the nc - 1
//     fp32 additions of the groups, and the fixed order's own rounding (one
//     unit roundoff per multiply-add of a slice chain and per butterfly
//     level), each bounded through sum_i |x_i w_i| <= ||x|| ||w||
//     (Cauchy-Schwarz).
//
//  3. Candidates.  Let v_k be the k-th largest g^ + b of the token.  Every
//     expert with g^ + b < v_k - 2 theta is beaten, in exact fixed-order
//     values, by each of the k experts at or above v_k, so the true top-k lies
//     in U = { e : g^ + b >= v_k - 2 theta }.  When the gaps between the
//     token's k+1 largest g^ are all above 2 theta the order of g^ is the
//     order of g: the token is certain and takes the k largest g^ as they are.
//     Otherwise the warp recomputes the logits of U in the fixed order (lane
//     j = slice j, the row read back from L2, four 256-element blocks of loads
//     in flight), exactly as the SIMT router computes them, and ranks them:
//     largest first, equal values to the lower expert.  Indices are therefore
//     those of the fixed order, bit for bit, on every input.
//
//  4. Gates.  Softmax with the shift m = max g^ + b: the denominator adds
//     exp(g - m) of the recomputed experts and exp(g^ + b - m) of the others
//     (in ascending expert order); a certain token's gates come from g^.  A
//     gate's relative error is thus the tensor-core error of the logits it
//     uses, weighted by their probabilities.  RENORM gates use the chosen
//     logits only.
//
// In the layer forward the epilogue also writes the slot assignment's block
// histogram (one warp = 32 tokens = one assignment block), and the last CTA
// scans it (assign_scan.cuh), or the slot-and-pack kernel does.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 tensor-memory
// allocation and MMA issue, warps 2-9 the epilogue, two per tensor-memory lane
// quarter (warp w reads lanes 32 * (w % 4) ..): the pair splits the quarter's
// accumulator columns between them, meets on a shared-memory barrier, and then
// each ranks 16 of the quarter's 32 tokens.  One accumulator set per CTA: the
// stage ring (up to 10 stages) keeps loading the next tile while the epilogue
// runs.  Every mbarrier wait is
// bounded; on expiry the kernel records MOE_ERR_TIMEOUT's device bit, stops,
// drains its own copies and MMAs (bounded), frees tensor memory and returns.
#include <math_constants.h>

#include "assign_scan.cuh"

namespace moe {
namespace {

constexpr int kTM = 128;            // tokens per tile (MMA M)
constexpr int kBK = 64;             // hidden elements per stage (one 128-byte swizzle row of bf16)
constexpr int kUK = 16;             // K per MMA instruction
constexpr int kRtThreads = 320;
constexpr int kEpiWarps = 8;       // two per tensor-memory lane quarter
constexpr int kTmemCols = 512;
// tensor-memory columns: x x^T at 0, the Wg Gram block at 128 (first tile
// only), then the nc groups of partial logits (n_pad columns each)
constexpr int kGramXCol = 0;
constexpr int kGramWCol = 128;
constexpr int kLogitCol0 = 256;
constexpr int kMaxGroups = 16;
constexpr int kLogitPitch = kTM + 1;  // floats per expert row of the epilogue's logit table
constexpr int kEPerLane = 4;          // experts per lane when a warp walks one token (E <= 128)
constexpr int kTokPar = 4;            // tokens a warp ranks side by side
constexpr int kMaxStages = 10;
constexpr int kStageBudget = 200 * 1024;      // shared memory for the stage ring and the logit table
constexpr uint64_t kTcTimeoutNs = 2000000000ull;  // 2 s: far above any legitimate wait
// tensor-core accumulation model: error per MMA step <= kHwUlp * magnitude
constexpr double kHwUlp = 1.0 / (1 << 18);

struct __align__(8) RtShared {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t gfull[kMaxGroups];  // a group's partial logits (and, with the last, the Gram blocks) are done
    uint64_t tempty;
    uint64_t wdone;   // the epilogue warps' max ||Wg_e||^2 are in
    uint64_t drain;
    uint64_t pair[4];  // the two epilogue warps of a lane quarter: table complete, then ranks stored
    uint32_t tmem_base;
    int abort_flag;
    float wmax_sq;   // max_e ||Wg_e||^2 (bit pattern max, values >= 0)
    float bias[256]; // the router bias (zero without one)
    int sel[kTM * 8];  // the tile's chosen experts, token-major, k per token
};

struct RtArgs {
    int64_t T;
    int d, E, k, n_pad;   // n_pad = E rounded up to 16
    int stages;           // ring stages
    int spc, nc;          // hidden stages per accumulation group; groups
    int renorm;
    float c_d;            // theta_t = c_d * ||x_t|| * max ||Wg_e|| + 2^-22 max |g^|
    float gram_scale;     // upper-bound factor for the Gram diagonal
    const __nv_bfloat16* x;
    const __nv_bfloat16* Wg;
    const float* bias;
    int32_t* topk_idx;
    float* topk_gate;
    int* status;
};

// ---------------------------------------------------------------- PTX ----
__device__ __forceinline__ uint32_t s_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool bar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase of `parity`; false when another role raised the abort
// flag or after kTcTimeoutNs (then raising it and recording the timeout).
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
    if (bar_try(bar, parity)) return true;
    const uint64_t t0 = gtimer();
    for (;;) {
        if (bar_try(bar, parity)) return true;
        if (*abort_flag) return false;
        if (gtimer() - t0 > kTcTimeoutNs) {
            *abort_flag = 1;
            if (status) atomicOr(status, kDevTimeout);
            return false;
        }
    }
}
// Bounded wait on the way out; ignores the abort flag.
__device__ __forceinline__ void bar_drain(uint32_t bar, uint32_t parity, int* status) {
    const uint64_t t0 = gtimer();
    while (!bar_try(bar, parity)) {
        if (gtimer() - t0 > kTcTimeoutNs) {
            if (status) atomicOr(status, kDevTimeout);
            return;
        }
    }
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        ::"r"(dst), "l"((uint64_t)map), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// K-major operand, 128-byte swizzle, 8-row groups 1024 B apart, version 1.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, K-major.
__host__ __device__ constexpr uint32_t idesc_m128(int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void mma_1sm(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit_1sm(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// 16 columns of this warp's 32 tensor-memory lanes into v; complete only
// after tmem_wait_ld()
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
        " [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// acc = fma(x[j], w[j], acc), j = 0..7 ascending, on the bf16 halves of two
// 16-byte vectors (the mixed-precision FMA rounds exactly as fmaf on the
// widened values); the fixed order's chain step.
__device__ __forceinline__ void fma8(float& acc, const uint4& x, const uint4& w) {
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
__device__ __forceinline__ uint4 ldg16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Fixed-order logits of token row xr against NB Wg rows (nb of them used;
// the whole warp, lane j owns slice j).  Four 256-element blocks of loads are
// issued before their multiply-adds, which run in ascending element order.
// Every lane returns the same values.
template <int NB>
__device__ __forceinline__ void fixed_order_logits(const __nv_bfloat16* xr, const __nv_bfloat16* Wg, int d,
                                                   const int (&e)[NB], int nb, int lane, float (&out)[NB]) {
    float s[NB];
#pragma unroll
    for (int i = 0; i < NB; ++i) s[i] = 0.0f;
    int base = 8 * lane;
    for (; base + 768 < d; base += 1024) {
        uint4 xv[4], wv[NB][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) xv[u] = ldg16(xr + base + 256 * u);
#pragma unroll
        for (int i = 0; i < NB; ++i)
#pragma unroll
            for (int u = 0; u < 4; ++u)
                wv[i][u] = i < nb ? ldg16(Wg + (size_t)e[i] * d + base + 256 * u) : xv[u];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int i = 0; i < NB; ++i) fma8(s[i], xv[u], wv[i][u]);
    }
    for (; base < d; base += 256) {
        const uint4 xv = ldg16(xr + base);
#pragma unroll
        for (int i = 0; i < NB; ++i)
            if (i < nb) fma8(s[i], xv, ldg16(Wg + (size_t)e[i] * d + base));
    }
#pragma unroll
    for (int i = 0; i < NB; ++i) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s[i] = s[i] + __shfl_xor_sync(0xffffffffu, s[i], o);
        out[i] = s[i];
    }
}

// Order-preserving 32-bit image of a float (larger value, larger unsigned
// bits; -0 must have been turned into +0 first) and its inverse.
__device__ __forceinline__ uint32_t order_bits(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float from_order_bits(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// (v, e) ranks before entry p of a list sorted by value descending, index
// ascending on ties (an entry with index -1 is empty).
__device__ __forceinline__ bool ranks_before(float v, int e, float lvp, int lep) {
    return lep < 0 || v > lvp || (v == lvp && e < lep);
}
// Insert (v, e) into such a list, keeping its first n entries (n <= L;
// entries at n and beyond are not touched).  Unrolled so the list stays in
// registers: entry p takes entry p-1 when (v, e) ranks before that one, else
// (v, e) itself when it ranks before entry p; a value that ranks after entry
// n-1 changes nothing.
template <int L>
__device__ __forceinline__ void list_insert(float (&lv)[L], int (&le)[L], int n, float v, int e) {
#pragma unroll
    for (int p = L - 1; p >= 0; --p) {
        if (p < n) {
            if (p > 0 && ranks_before(v, e, lv[p - 1], le[p - 1])) {
                lv[p] = lv[p - 1];
                le[p] = le[p - 1];
            } else if (ranks_before(v, e, lv[p], le[p])) {
                lv[p] = v;
                le[p] = e;
            }
        }
    }
}

// KM: largest k this instance serves
template <int KM>
__global__ void __launch_bounds__(kRtThreads, 1)
route_tc_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw, const RtArgs a,
                const AssignScan scan) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = s_u32(smem_raw);
    uint8_t* ring = smem_raw + ((1024 - (raw & 1023)) & 1023);
    const int S = a.stages;
    const int NP = a.n_pad;
    const uint32_t stage_bytes = (uint32_t)(NP + kTM) * 128u;
    RtShared& sh = *reinterpret_cast<RtShared*>(ring + (size_t)S * stage_bytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = (int)((a.T + kTM - 1) / kTM);
    const int nchunks = (a.d + kBK - 1) / kBK;
    const int nc = a.nc, spc = a.spc;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            bar_init(s_u32(&sh.full[s]), 1);
            bar_init(s_u32(&sh.empty[s]), 1);
        }
        for (int j = 0; j < nc; ++j) bar_init(s_u32(&sh.gfull[j]), 1);
        bar_init(s_u32(&sh.tempty), kEpiWarps);
        bar_init(s_u32(&sh.wdone), kEpiWarps);
        for (int j = 0; j < 4; ++j) bar_init(s_u32(&sh.pair[j]), 2);
        bar_init(s_u32(&sh.drain), 1);
        sh.abort_flag = 0;
        sh.wmax_sq = 0.0f;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s_u32(&sh.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_before();
    __syncthreads();
    tc_after();
    dep_wait();  // global memory only from here on
    const uint32_t tmem_base = sh.tmem_base;
    volatile int* abort_flag = &sh.abort_flag;
    int* status = a.status;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer --
        int stage = 0;
        uint32_t phase = 0;
        // stages with a copy issued, and the phase parity of their last one
        // (bit masks: an array indexed by the stage would live in local memory)
        uint32_t issued = 0, issued_par = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            for (int c = 0; c < nchunks; ++c) {
                if (!bar_wait(s_u32(&sh.empty[stage]), phase ^ 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
                const uint32_t sb = s_u32(ring + (size_t)stage * stage_bytes);
                const uint32_t fb = s_u32(&sh.full[stage]);
                bar_expect_tx(fb, stage_bytes);
                tma_2d(sb, &tmw, fb, c * kBK, 0);                                // Wg rows (zero past E)
                tma_2d(sb + (uint32_t)NP * 128u, &tmx, fb, c * kBK, tile * kTM);  // x rows (zero past T)
                issued |= 1u << stage;
                issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // copies in flight land before the CTA leaves
        for (int s = 0; s < S; ++s)
            if ((issued >> s) & 1u) bar_drain(s_u32(&sh.full[s]), (issued_par >> s) & 1u, status);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------- MMA issuer --
        int stage = 0;
        uint32_t phase = 0, tphase = 0;
        bool first = true;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            if (!bar_wait(s_u32(&sh.tempty), tphase ^ 1u, abort_flag, status)) break;
            tc_after();
            bool ok = true;
            for (int c = 0; c < nchunks; ++c) {
                if (!bar_wait(s_u32(&sh.full[stage]), phase, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_after();
                const uint32_t sb = s_u32(ring + (size_t)stage * stage_bytes);
                const uint32_t sa = sb + (uint32_t)NP * 128u;
                const int grp = c / spc;  // accumulation group of this stage
                const uint32_t d_logit = tmem_base + (uint32_t)(kLogitCol0 + grp * NP);
#pragma unroll
                for (int kk = 0; kk < kBK / kUK; ++kk) {
                    const uint64_t ad = desc_sw128(sa + kk * 32);
                    mma_1sm(d_logit, ad, desc_sw128(sb + kk * 32), idesc_m128(NP), ((c - grp * spc) | kk) != 0);
                    mma_1sm(tmem_base + kGramXCol, ad, ad, idesc_m128(kTM), (c | kk) != 0);
                    if (first) {
                        // the stage's first 128 rows (the Wg rows, then x rows)
                        // against themselves: ||Wg_e||^2 on the diagonal
                        const uint64_t wd = desc_sw128(sb + kk * 32);
                        mma_1sm(tmem_base + kGramWCol, wd, wd, idesc_m128(kTM), (c | kk) != 0);
                    }
                }
                mma_commit_1sm(s_u32(&sh.empty[stage]));
                if (c - grp * spc == spc - 1 || c == nchunks - 1) mma_commit_1sm(s_u32(&sh.gfull[grp]));
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            first = false;
            tphase ^= 1u;
        }
        mma_commit_1sm(s_u32(&sh.drain));
        bar_drain(s_u32(&sh.drain), 0, status);
    } else if (warp >= 2) {
        // --------------------------------------------------- epilogue --
        const int q = warp & 3;          // tensor-memory lane quarter of this warp
        const int half = (warp - 2) >> 2;  // which of the quarter's two warps
        const bool own = (lane >> 4) == half;  // this lane's token is ranked by this warp
        const uint32_t pair_bar = s_u32(&sh.pair[q]);
        const int E = a.E, k = a.k, d = a.d;
        for (int e = threadIdx.x - 64; e < E; e += 32 * kEpiWarps) sh.bias[e] = a.bias ? a.bias[e] : 0.0f;
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
        const float* bias = sh.bias;  // zero without a router bias
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        // logit table [n_pad][kLogitPitch]: expert-major, one column per token of
        // the tile (the pitch keeps both a thread's row walk and a warp's
        // expert walk free of bank conflicts)
        float* gt = reinterpret_cast<float*>(ring + (size_t)S * stage_bytes + sizeof(RtShared));
        const int row = q * 32 + lane;  // this thread's token within the tile
        float wmax = 0.0f;
        uint32_t tphase = 0;
        bool first = true;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            const int64_t t = (int64_t)tile * kTM + row;
            const bool valid = t < a.T;
            const int64_t blk = ((int64_t)tile * kTM + q * 32) / kAssignBlock;  // assignment block of this warp

            // the groups' partial logits, added into the table in ascending
            // group order as each group's MMAs complete (while later groups
            // still stream in); the pair's two warps take alternate 32-column
            // blocks of the accumulator
            bool ok = true;
            for (int j = 0; j < nc && ok; ++j) {
                ok = __all_sync(0xffffffffu, bar_wait(s_u32(&sh.gfull[j]), tphase, abort_flag, status));
                if (!ok) break;
                tc_after();
                const uint32_t tg = tmem_base + lanes + (uint32_t)(kLogitCol0 + j * NP);
                for (int c0 = 32 * half; c0 < NP; c0 += 64) {
                    float v0[16], v1[16];
                    tmem_ld16_nowait(tg + c0, v0);
                    if (c0 + 16 < NP) tmem_ld16_nowait(tg + c0 + 16, v1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float* p0 = gt + (c0 + i) * kLogitPitch + row;
                        *p0 = j ? *p0 + v0[i] : v0[i];
                    }
                    if (c0 + 16 < NP) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float* p1 = gt + (c0 + 16 + i) * kLogitPitch + row;
                            *p1 = j ? *p1 + v1[i] : v1[i];
                        }
                    }
                }
            }
            if (!ok) break;
            // Gram diagonals: ||x_t||^2 (column row of the x block) and, on the
            // CTA's first tile, ||Wg_e||^2 (lane e of the Wg block)
            float xsq, wsq = 0.0f;
            {
                float g0[16], g1[16], w0[16], w1[16];
                tmem_ld16_nowait(tmem_base + lanes + kGramXCol + q * 32, g0);
                tmem_ld16_nowait(tmem_base + lanes + kGramXCol + q * 32 + 16, g1);
                if (first) {
                    tmem_ld16_nowait(tmem_base + lanes + kGramWCol + q * 32, w0);
                    tmem_ld16_nowait(tmem_base + lanes + kGramWCol + q * 32 + 16, w1);
                }
                tmem_wait_ld();
                xsq = 0.0f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    xsq = lane == i ? g0[i] : xsq;
                    xsq = lane == i + 16 ? g1[i] : xsq;
                    if (first) {
                        wsq = lane == i ? w0[i] : wsq;
                        wsq = lane == i + 16 ? w1[i] : wsq;
                    }
                }
            }
            // everything needed is in registers and shared memory: the
            // accumulators are free for the next tile
            tc_before();
            __syncwarp();
            if (lane == 0) {
                bar_arrive(s_u32(&sh.tempty));
                bar_arrive(pair_bar);  // this warp's columns of the table are in
            }
            if (first) {
                // max_e ||Wg_e||^2 (rows past E hold x rows: excluded); the four
                // warps' maxima meet on an mbarrier (a bounded wait, so a warp
                // that gave up earlier cannot leave the others stuck)
                float wm = row < E ? fmaxf(wsq, 0.0f) : 0.0f;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
                if (lane == 0) {
                    atomicMax(reinterpret_cast<int*>(&sh.wmax_sq), __float_as_int(wm));
                    bar_arrive(s_u32(&sh.wdone));
                }
                if (!__all_sync(0xffffffffu, bar_wait(s_u32(&sh.wdone), 0, abort_flag, status))) break;
                wmax = sqrtf(*reinterpret_cast<volatile float*>(&sh.wmax_sq) * a.gram_scale) * (1.0f + 1e-6f);
                first = false;
            }
            // the other warp's columns (two phases of the pair barrier per
            // tile: 0 = table complete, 1 = ranks stored)
            if (!__all_sync(0xffffffffu, bar_wait(pair_bar, 0, abort_flag, status))) break;

            // the warp's 16 tokens, four at a time, lane = expert (expert
            // lane + 32 i): per token the k+1 largest g^ + b by repeated argmax
            // (a warp max of order-preserving bits, then the lowest expert
            // holding it), max |g^ + b|, and the softmax denominator over every
            // expert (an xor-butterfly sum of exp(g^ + b - m), m = the largest);
            // the token's own lane keeps the results
            const int K1 = k < E ? k + 1 : k;
            float lv[KM + 1];
            int le[KM + 1];
#pragma unroll
            for (int i = 0; i <= KM; ++i) {
                lv[i] = -CUDART_INF_F;
                le[i] = -1;
            }
            float maxabs = 0.0f, s_all = 0.0f;
            // Each step below is written for kTokPar tokens side by side, so
            // that their warp reductions are independent neighbours in the
            // instruction stream and overlap (one token's chain alone is a
            // row of dependent reductions).
            for (int j0 = 16 * half; j0 < 16 * half + 16; j0 += kTokPar) {
                float v[kTokPar][kEPerLane];
#pragma unroll
                for (int u = 0; u < kTokPar; ++u)
#pragma unroll
                    for (int i = 0; i < kEPerLane; ++i) {
                        const int e = lane + 32 * i;
                        // + 0.0f turns -0 into +0, so order-preserving bits tie as the values do
                        v[u][i] = e < E ? gt[e * kLogitPitch + q * 32 + j0 + u] + bias[e] + 0.0f : -CUDART_INF_F;
                    }
                float la[kTokPar];
#pragma unroll
                for (int u = 0; u < kTokPar; ++u) {
                    la[u] = 0.0f;
#pragma unroll
                    for (int i = 0; i < kEPerLane; ++i)
                        if (lane + 32 * i < E) la[u] = fmaxf(la[u], fabsf(v[u][i]));
                }
#pragma unroll
                for (int u = 0; u < kTokPar; ++u)
                    la[u] = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(la[u])));
                float top[kTokPar];
#pragma unroll
                for (int r = 0; r <= KM; ++r) {
                    if (r < K1) {
                        // each token: this lane's largest remaining value (lower
                        // expert first), then the warp's largest and the lowest
                        // expert holding it
                        uint32_t ob[kTokPar], om[kTokPar];
                        int bi[kTokPar], be[kTokPar];
#pragma unroll
                        for (int u = 0; u < kTokPar; ++u) {
                            float bv = -CUDART_INF_F;
                            bi[u] = 0;
#pragma unroll
                            for (int i = 0; i < kEPerLane; ++i)
                                if (v[u][i] > bv) {
                                    bv = v[u][i];
                                    bi[u] = i;
                                }
                            ob[u] = order_bits(bv);
                        }
#pragma unroll
                        for (int u = 0; u < kTokPar; ++u) om[u] = __reduce_max_sync(0xffffffffu, ob[u]);
#pragma unroll
                        for (int u = 0; u < kTokPar; ++u)
                            be[u] = (int)__reduce_min_sync(0xffffffffu,
                                                           ob[u] == om[u] ? (uint32_t)(lane + 32 * bi[u]) : 0xffffffffu);
#pragma unroll
                        for (int u = 0; u < kTokPar; ++u) {
                            const float val = from_order_bits(om[u]);
                            // a select per entry: a store to v[u][be >> 5] would
                            // put the token's values in local memory
#pragma unroll
                            for (int i = 0; i < kEPerLane; ++i)
                                v[u][i] = be[u] == lane + 32 * i ? -CUDART_INF_F : v[u][i];
                            if (r == 0) top[u] = val;
                            if (lane == j0 + u) {
                                lv[r] = val;
                                le[r] = be[u];
                            }
                        }
                    }
                }
                // the denominators (the removed entries are restored from the
                // table), then one xor butterfly for all of them
                float sum[kTokPar];
#pragma unroll
                for (int u = 0; u < kTokPar; ++u) {
                    sum[u] = 0.0f;
#pragma unroll
                    for (int i = 0; i < kEPerLane; ++i) {
                        const int e = lane + 32 * i;
                        if (e < E) sum[u] += __expf(gt[e * kLogitPitch + q * 32 + j0 + u] + bias[e] - top[u]);
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int u = 0; u < kTokPar; ++u) sum[u] += __shfl_xor_sync(0xffffffffu, sum[u], o);
#pragma unroll
                for (int u = 0; u < kTokPar; ++u)
                    if (lane == j0 + u) {
                        maxabs = la[u];
                        s_all = sum[u];
                    }
            }
            const float m = lv[0];  // the largest g^ + b: the softmax shift
            const float xn = sqrtf(fmaxf(xsq, 0.0f) * a.gram_scale) * (1.0f + 1e-6f);
            const float theta2 = 2.0f * (a.c_d * xn * wmax + 2.4e-7f * maxabs);
            // certain: the k+1 largest g^ are more than 2 theta apart; vk = the
            // k-th (the least of the k largest: the list is in descending order,
            // and a minimum keeps the list out of local memory where lv[k - 1]
            // would not)
            bool certain = true;
            float vk = lv[0];
#pragma unroll
            for (int r = 0; r < KM; ++r) {
                if (r + 1 < K1) certain = certain && (lv[r] - lv[r + 1] > theta2);
                if (r < k) vk = fminf(vk, lv[r]);
            }
            const bool redo = own && valid && !certain;
            // an uncertain token's candidates U: every expert within 2 theta of
            // its k-th largest
            const float band = vk - theta2;

            // a certain token keeps its k largest g^; an uncertain one ranks
            // the fixed-order logits of U, recomputed one token at a time
            // across the warp (its candidates found by a ballot over the
            // table), and swaps their terms of the denominator for
            // exp(g - m) of the recomputed values
            float rv[KM];
            int re[KM];
#pragma unroll
            for (int i = 0; i < KM; ++i) {
                rv[i] = redo ? -CUDART_INF_F : lv[i];
                re[i] = redo ? -1 : le[i];
            }
            float s_exact = 0.0f;
            const uint32_t redo_warp = __ballot_sync(0xffffffffu, redo);
            for (uint32_t todo = redo_warp; todo; todo &= todo - 1) {
                const int j = __ffs(todo) - 1;
                const float band_j = __shfl_sync(0xffffffffu, band, j);
                const __nv_bfloat16* xr = a.x + (size_t)((int64_t)tile * kTM + q * 32 + j) * d;
                for (int c0 = 0; c0 < E; c0 += 32) {
                    const int ec = c0 + lane;
                    const float gc = ec < E ? gt[ec * kLogitPitch + q * 32 + j] + bias[ec] : -CUDART_INF_F;
                    uint32_t bits = __ballot_sync(0xffffffffu, gc >= band_j);
                    while (bits) {
                        int e2[2] = {0, 0};
                        int nb = 0;
#pragma unroll
                        for (int z = 0; z < 2; ++z)
                            if (bits) {
                                e2[z] = c0 + __ffs(bits) - 1;
                                bits &= bits - 1;
                                nb = z + 1;
                            }
                        float g2[2];
                        fixed_order_logits<2>(xr, a.Wg, d, e2, nb, lane, g2);
                        if (lane == j) {
#pragma unroll
                            for (int z = 0; z < 2; ++z)
                                if (z < nb) {
                                    const float g = g2[z] + bias[e2[z]];
                                    list_insert(rv, re, k, g, e2[z]);
                                    const float gh = gt[e2[z] * kLogitPitch + row] + bias[e2[z]];
                                    s_exact += __expf(g - m) - __expf(gh - m);
                                }
                        }
                    }
                }
            }

            if (own && valid) {
                const float inv = 1.0f / (s_all + s_exact);
                float den = 0.0f;
#pragma unroll
                for (int r = 0; r < KM; ++r)
                    if (a.renorm && r < k) den += expf(rv[r] - m);
#pragma unroll
                for (int r = 0; r < KM; ++r)
                    if (r < k) {
                        a.topk_idx[(size_t)t * k + r] = re[r];
                        a.topk_gate[(size_t)t * k + r] = a.renorm ? expf(rv[r] - m) / den : expf(rv[r] - m) * inv;
                    }
            }
            if (own) {
#pragma unroll
                for (int r = 0; r < KM; ++r)
                    if (r < k) sh.sel[row * KM + r] = valid ? re[r] : -1;
            }
            // both warps' ranks are stored, and both are done with the table
            // (the next tile rewrites it only after this point)
            __syncwarp();
            if (lane == 0) bar_arrive(pair_bar);
            if (!__all_sync(0xffffffffu, bar_wait(pair_bar, 1, abort_flag, status))) break;
            if (half == 0 && scan.hist && blk < scan.nblk) {
                // the quarter's 32 tokens are one assignment block: its
                // per-(expert, rank) counts (zero for experts it does not choose)
                for (int i = lane; i < E * k; i += 32) scan.hist[(size_t)i * scan.nblk + blk] = 0;
                __syncwarp();
#pragma unroll
                for (int r = 0; r < KM; ++r)
                    if (r < k) {
                        const int key = valid ? sh.sel[row * KM + r] : -1;
                        const uint32_t same = __match_any_sync(0xffffffffu, key);
                        if (valid && lane == __ffs(same) - 1)
                            scan.hist[((size_t)key * k + r) * scan.nblk + blk] = __popc(same);
                    }
            }
            __syncwarp();
            tphase ^= 1u;
        }
    }
    tc_before();
    __syncthreads();
    if (warp == 1) {
        tc_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
    if (scan.hist && !scan.defer) finish_assign_scan(scan);
}

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
    static const EncodeFn fn = []() -> EncodeFn {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return (EncodeFn)ptr;
        return nullptr;
    }();
    return fn;
}

// bf16 row-major [rows, cols], box [box_rows, 64], 128-byte swizzle, zero fill
bool map_sw128(EncodeFn enc, CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static const int n = []() {
        int dev = 0, v = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        return v;
    }();
    return n;
}

}  // namespace

// Up to 16 experts the fixed-order SIMT router is faster (its E multiply-adds
// per loaded element cost less than this kernel's Gram products and per-tile
// epilogue; measured at 8 experts, one call at full clock, L2 flushed, with
// identical indices: 11.5 against 26.7 us at T = 4096, d = 1024, and 86
// against 115 us at T = 32768, d = 4096); above 128 the per-token logit table
// no longer fits next to the stage ring.
bool route_tc_eligible(const Problem& p) { return p.dtype == MOE_BF16 && p.T > 0 && p.E > 16 && p.E <= 128; }

cudaError_t launch_route_tc(const Problem& p, const void* x, const void* Wg, const float* bias, int32_t* topk_idx,
                            float* topk_gate, const AssignScan& scan, int* status, cudaStream_t s) {
    EncodeFn enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    RtArgs a{};
    a.T = p.T;
    a.d = p.d;
    a.E = p.E;
    a.k = p.k;
    a.n_pad = (p.E + 15) / 16 * 16;
    const int stage_bytes = (a.n_pad + kTM) * 128;
    // the table holds n_pad rows: the group sums write every accumulator
    // column, the padding ones included (never read back)
    const int table_bytes = a.n_pad * kLogitPitch * (int)sizeof(float);
    a.stages = std::min(kMaxStages, (kStageBudget - table_bytes) / stage_bytes);
    a.renorm = (p.flags & MOE_FLAG_RENORM) != 0;
    // accumulation groups: as many as the columns after the Gram block hold
    const int nstages = (int)ceil_div(p.d, kBK);
    const int nc_max = std::min(kMaxGroups, (kTmemCols - kLogitCol0) / a.n_pad);
    a.spc = (int)ceil_div(nstages, nc_max);
    a.nc = (int)ceil_div(nstages, a.spc);
    // c_d: the tensor-core steps of one group (4 per stage) at 2 kHwUlp each
    // (accumulator and products), plus one unit roundoff for each addition of
    // the groups, each multiply-add of the fixed order's slice chain (8 per
    // 256 elements) and each of its five butterfly levels
    const double steps = 4.0 * a.spc;
    const double adds = (double)(a.nc - 1) + 8.0 * (double)((p.d + 255) / 256) + 5.0;
    a.c_d = (float)((2.0 * steps * kHwUlp + adds * std::ldexp(1.0, -24)) * 1.01);
    // an upper-bound factor for the two Gram diagonals (sums of squares over
    // all 4 * nstages MMA steps, so the same model bounds their error)
    const double gram_steps = 4.0 * nstages;
    a.gram_scale = (float)(1.0 + 2.0 * gram_steps * kHwUlp + 1e-6);
    a.x = (const __nv_bfloat16*)x;
    a.Wg = (const __nv_bfloat16*)Wg;
    a.bias = bias;
    a.topk_idx = topk_idx;
    a.topk_gate = topk_gate;
    a.status = status;
    CUtensorMap mx, mw;
    if (!map_sw128(enc, &mx, x, (uint64_t)p.T, (uint64_t)p.d, kTM) ||
        !map_sw128(enc, &mw, Wg, (uint64_t)p.E, (uint64_t)p.d, (uint32_t)a.n_pad))
        return cudaErrorInvalidValue;
    const size_t smem = 1024 + (size_t)a.stages * stage_bytes + sizeof(RtShared) + (size_t)table_bytes;
    const int ntiles = (int)ceil_div(p.T, kTM);
    const unsigned grid = (unsigned)std::min(ntiles, sm_count());
    auto run = [&](auto kern) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        return launch_k(kern, dim3(grid), dim3(kRtThreads), smem, s, mx, mw, a, scan);
    };
    // instances: k <= 2 or <= 8
    if (p.k <= 2) return run(route_tc_kernel<2>);
    return run(route_tc_kernel<8>);
}

}  // namespace moe
