// stats.cu -- routing statistics: the load-balancing term, routing entropy,
// dropped fraction and load imbalance, as device outputs.
//
// "Expert Parallelism" notes page (narrativegoldmine.com), "Components and
// Architecture" and the formal algorithm's last step: an auxiliary
// load-balancing term, the sum over experts of the share of tokens an expert
// receives times the share of router probability it receives.  "Expert
// Parallelism" glossary (inferensys.com): the load-balancing loss.
// "Expert Parallelism" intro page (nhimg.org), practitioner guidance:
// monitor expert utilisation and routing entropy.
//
//   f_e   = counts_routed[e] / (T*k)          (pre-drop assignments)
//   P_e   = mean over tokens of probs[t, e]
//   aux   = E * sum_e f_e * P_e
//   H     = mean over tokens of -sum_e p ln p (0 ln 0 = 0), in nats
//   drop  = (sum_e routed_e - kept_e) / (T*k)
//   imbal = max_e routed_e / (T*k / E)
//
// One kernel, deterministic without fp64.  Sums are kept in 64-bit fixed
// point (units of 2^-36): each probability p (and each -p ln p, formed in fp32
// with logf) is scaled by 2^36 -- exact -- and rounded to an integer (exact
// for p >= 2^-13, else within 2^-37), and integer sums do not depend on their
// order; T <= 2^25 keeps every sum below 2^64.  So CTA b reduces tokens [b*tb, (b+1)*tb) with its threads as
// R = floor(256 / E) token lanes of E experts (thread r*E + e reads probs[t, e]
// for t = first + r, first + r + R, ...; consecutive threads read consecutive
// floats), adds its lanes per expert in shared memory, and adds the E + 1
// results into global accumulators with integer atomics.  The last CTA to
// finish (integer ticket) takes the sums (atomic exchange with zero, which
// leaves them ready for the next call) and forms the statistics in fp32 with
// one warp in a fixed order.  B300's fp64 units are far too slow for this:
// an fp64 version spent over 20 us in its final additions.
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRun = 16;                 // loads issued together per thread
constexpr float kFix = 68719476736.0f;  // 2^36

__device__ __forceinline__ unsigned long long to_fixed(float v) { return __float2ull_rn(v * kFix); }

__global__ void __launch_bounds__(kThreads)
stats_kernel(int64_t T, int E, int k, int64_t tb, const float* __restrict__ probs,
             const int32_t* __restrict__ counts_routed, const int32_t* __restrict__ counts_kept,
             unsigned long long* __restrict__ acc, unsigned* ticket, float* __restrict__ out,
             float* __restrict__ mean_prob) {
    dep_wait();
    __shared__ unsigned long long sP[256];
    __shared__ unsigned long long sH;
    __shared__ float sTerm[256];
    __shared__ bool s_last;
    const int tid = threadIdx.x, lane = tid & 31;
    const int R = kThreads / E;  // token lanes (E <= kThreads)
    const int64_t t0 = (int64_t)blockIdx.x * tb;
    const int64_t t1 = min(T, t0 + tb);
    if (tid < E) sP[tid] = 0ull;
    if (tid == 0) sH = 0ull;
    __syncthreads();

    unsigned long long P = 0ull, H = 0ull;
    if (tid < R * E) {
        const int r = tid / E, e = tid - r * E;
        const float* col = probs + e;
        for (int64_t t = t0 + r; t < t1; t += (int64_t)kRun * R) {
            float v[kRun];
#pragma unroll
            for (int j = 0; j < kRun; ++j) {
                const int64_t tj = t + (int64_t)j * R;
                v[j] = tj < t1 ? col[(size_t)tj * E] : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < kRun; ++j) {
                P += to_fixed(v[j]);
                if (v[j] > 0.0f) H += to_fixed(-v[j] * logf(v[j]));
            }
        }
        atomicAdd(&sP[e], P);
    }
    // entropy: every thread's share, warp sums first
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) H += __shfl_xor_sync(0xffffffffu, H, o);
    if (lane == 0) atomicAdd(&sH, H);
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) atomicAdd(acc + e, sP[e]);
    if (tid == 0) atomicAdd(acc + E, sH);
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // last CTA: take the sums (leaving zeros), means in fp32
    const float invT = T > 0 ? 1.0f / (float)T : 0.0f;
    const float Tk = (float)T * (float)k;
    for (int e = tid; e < E; e += kThreads) {
        const float mp = (float)atomicExch(acc + e, 0ull) * (1.0f / kFix) * invT;
        if (mean_prob) mean_prob[e] = mp;
        sTerm[e] = Tk > 0.0f ? (float)counts_routed[e] / Tk * mp : 0.0f;
    }
    __syncthreads();
    if (tid < 32) {
        // fixed order: lane l takes experts l, l + 32, ..., then a xor tree
        float aux = 0.0f;
        long long routed = 0, kept = 0;
        int maxr = 0;
        for (int e = lane; e < E; e += 32) {
            aux += sTerm[e];
            const int cr = counts_routed[e];
            routed += cr;
            kept += counts_kept[e];
            maxr = max(maxr, cr);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            aux += __shfl_xor_sync(0xffffffffu, aux, o);
            routed += __shfl_xor_sync(0xffffffffu, routed, o);
            kept += __shfl_xor_sync(0xffffffffu, kept, o);
            maxr = max(maxr, __shfl_xor_sync(0xffffffffu, maxr, o));
        }
        if (lane == 0) {
            const float Hsum = (float)atomicExch(acc + E, 0ull) * (1.0f / kFix);
            out[MOE_STAT_AUX] = (float)E * aux;
            out[MOE_STAT_ENTROPY] = Hsum * invT;
            out[MOE_STAT_DROP] = Tk > 0.0f ? (float)(routed - kept) / Tk : 0.0f;
            out[MOE_STAT_IMBALANCE] = Tk > 0.0f ? (float)maxr / (Tk / (float)E) : 0.0f;
            *ticket = 0u;  // ready for the next call
        }
    }
}

}  // namespace

int64_t stats_blocks(int64_t T) { return T <= 0 ? 1 : std::min<int64_t>(kStatBlocks, ceil_div(T, 64)); }

cudaError_t launch_routing_stats(const Problem& p, const float* probs, const int32_t* counts_routed,
                                 const int32_t* counts_kept, float* stats, float* mean_prob,
                                 unsigned long long* acc, unsigned* ticket, cudaStream_t s) {
    const int64_t nb = stats_blocks(p.T);
    const int64_t tb = p.T <= 0 ? 0 : ceil_div(p.T, nb);
    return launch_k(stats_kernel, dim3((unsigned)nb), dim3(kThreads), 0, s, p.T, p.E, p.k, tb, probs,
                    counts_routed, counts_kept, acc, ticket, stats, mean_prob);
}

}  // namespace moe
