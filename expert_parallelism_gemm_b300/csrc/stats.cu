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
// One kernel, deterministic: CTA b reduces tokens [b*tb, (b+1)*tb) -- warp w
// takes every 8th token, lane l the experts l, l+32, ... -- in fp64, the
// eight warps combined in warp order, and writes E+1 partial sums; the last
// CTA to finish (integer ticket) adds the at most kStatBlocks partials in
// block order and writes the statistics.  Each -p ln p term is formed in
// fp32 (logf) and accumulated in fp64.
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kStatWarps = kThreads / 32;
constexpr int kMaxPerLane = 256 / 32;  // experts per lane (E <= 256)

__global__ void __launch_bounds__(kThreads)
stats_kernel(int64_t T, int E, int k, int64_t tb, const float* __restrict__ probs,
             const int32_t* __restrict__ counts_routed, const int32_t* __restrict__ counts_kept,
             double* __restrict__ partials, unsigned* ticket, float* __restrict__ out,
             float* __restrict__ mean_prob) {
    dep_wait();
    dep_release();
    __shared__ double sP[kStatWarps][256];
    __shared__ double sH[kStatWarps];
    __shared__ bool s_last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t0 = (int64_t)blockIdx.x * tb;
    const int64_t t1 = min(T, t0 + tb);

    double pa[kMaxPerLane];
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q) pa[q] = 0.0;
    double h = 0.0;
    // tokens in batches of four per warp: the loads of a batch are issued
    // before any is consumed; the sums still run in token order
    constexpr int kBatch = 4;
    for (int64_t tb0 = t0 + warp; tb0 < t1; tb0 += kBatch * kStatWarps) {
        float v[kBatch][kMaxPerLane];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int64_t t = tb0 + (int64_t)j * kStatWarps;
#pragma unroll
            for (int q = 0; q < kMaxPerLane; ++q) {
                const int e = lane + 32 * q;
                v[j][q] = (t < t1 && e < E) ? probs[(size_t)t * E + e] : 0.0f;
            }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
#pragma unroll
            for (int q = 0; q < kMaxPerLane; ++q) {
                const float p = v[j][q];
                pa[q] += (double)p;
                if (p > 0.0f) h -= (double)(p * logf(p));
            }
    }
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q) {
        const int e = lane + 32 * q;
        if (e < E) sP[warp][e] = pa[q];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) h += __shfl_xor_sync(0xffffffffu, h, o);
    if (lane == 0) sH[warp] = h;
    __syncthreads();
    double* mine = partials + (size_t)blockIdx.x * (E + 1);
    for (int e = threadIdx.x; e <= E; e += kThreads) {
        double s = 0.0;
        for (int w = 0; w < kStatWarps; ++w) s += e < E ? sP[w][e] : sH[w];
        mine[e] = s;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // last CTA: block partials in block order
    const int nb = gridDim.x;
    for (int e = threadIdx.x; e <= E; e += kThreads) {
        double s = 0.0;
        for (int b0 = 0; b0 < nb; b0 += 16) {
            double v[16];  // loads issued together, added in block order
#pragma unroll
            for (int j = 0; j < 16; ++j)
                v[j] = b0 + j < nb ? __ldcg(partials + (size_t)(b0 + j) * (E + 1) + e) : 0.0;
#pragma unroll
            for (int j = 0; j < 16; ++j) s += v[j];
        }
        if (e < E) sP[0][e] = T > 0 ? s / (double)T : 0.0;
        else sH[0] = T > 0 ? s / (double)T : 0.0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const double Tk = (double)T * (double)k;
        double aux = 0.0, routed = 0.0, kept = 0.0, maxr = 0.0;
        for (int e = 0; e < E; ++e) {
            const double f = Tk > 0.0 ? (double)counts_routed[e] / Tk : 0.0;
            aux += f * sP[0][e];
            routed += counts_routed[e];
            kept += counts_kept[e];
            maxr = fmax(maxr, (double)counts_routed[e]);
        }
        out[MOE_STAT_AUX] = (float)((double)E * aux);
        out[MOE_STAT_ENTROPY] = (float)sH[0];
        out[MOE_STAT_DROP] = (float)(Tk > 0.0 ? (routed - kept) / Tk : 0.0);
        out[MOE_STAT_IMBALANCE] = (float)(Tk > 0.0 ? maxr / (Tk / (double)E) : 0.0);
        *ticket = 0u;  // ready for the next call
    }
    if (mean_prob)
        for (int e = threadIdx.x; e < E; e += kThreads) mean_prob[e] = (float)sP[0][e];
}

}  // namespace

int64_t stats_blocks(int64_t T) { return T <= 0 ? 1 : std::min<int64_t>(kStatBlocks, ceil_div(T, 64)); }

cudaError_t launch_routing_stats(const Problem& p, const float* probs, const int32_t* counts_routed,
                                 const int32_t* counts_kept, float* stats, float* mean_prob,
                                 double* partials, unsigned* ticket, cudaStream_t s) {
    const int64_t nb = stats_blocks(p.T);
    const int64_t tb = p.T <= 0 ? 0 : ceil_div(p.T, nb);
    return launch_k(stats_kernel, dim3((unsigned)nb), dim3(kThreads), 0, s, p.T, p.E, p.k, tb, probs,
                    counts_routed, counts_kept, partials, ticket, stats, mean_prob);
}

}  // namespace moe
