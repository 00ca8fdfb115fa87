// route.cu -- router: logits, softmax, top-k and gates.
//
// "Expert Parallelism" notes page (narrativegoldmine.com), "Formal
// Algorithm: Expert Parallelism Forward Pass": gate computation (logits of the
// routing projection, p = softmax(g / tau), tau = 1) and expert selection
// (gate weight = probability of the chosen expert); "Components and
// Architecture": top-k selection and an optional per-expert logit bias.
//
// Each logit is one fp32 fused multiply-add chain over the hidden index in
// ascending order, starting from +0, followed by the bias add.  That order is
// what makes the top-k decision reproducible bit for bit; any thread may own
// a (token, expert) pair as long as it keeps the chain's order.
//
// Layout: one CTA of 256 threads handles 32 tokens and every expert.  Thread
// (tg = tid % 32, eg = tid / 32) owns token tg and experts eg, eg+8, ...  The
// hidden dimension is walked in chunks of 64: x[32 x 64] and Wg[E x 64] are
// staged to shared memory as fp32 (x rows padded so that the 32 lanes' 16-byte
// reads of 32 different rows hit distinct banks; Wg rows are read by all 32
// lanes of a warp at once, a broadcast).  Then one warp per token computes the
// softmax and the top-k by warp-wide (value, index) reductions.
#include "common.cuh"

#include <math_constants.h>

namespace moe {
namespace {

constexpr int kTokPerCta = 32;
constexpr int kChunk = 64;
constexpr int kXPitch = kChunk + 4;  // floats

template <typename T, int NE>
__global__ void __launch_bounds__(kThreads)
route_kernel(int64_t T_, int d, int E, int k, const T* __restrict__ x,
             const T* __restrict__ Wg, const float* __restrict__ bias,
             int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate,
             float* __restrict__ probs) {
    constexpr int VE = vec_elems<T>();           // elements per 16-byte vector
    constexpr int kVecPerRow = kChunk / VE;      // vectors per chunk row
    const int Epad = NE * 8;
    extern __shared__ __align__(16) float smem[];
    float* xs = smem;                                   // [32][kXPitch]
    float* wsm = xs + kTokPerCta * kXPitch;             // [Epad][kChunk]
    float* lg = wsm + Epad * kChunk;                    // [32][Epad + 1]
    const int lgp = Epad + 1;

    const int tid = threadIdx.x;
    const int tg = tid & 31, eg = tid >> 5;
    const int64_t t0 = (int64_t)blockIdx.x * kTokPerCta;

    float acc[NE];
#pragma unroll
    for (int j = 0; j < NE; ++j) acc[j] = 0.0f;

    for (int k0 = 0; k0 < d; k0 += kChunk) {
        const int n = min(kChunk, d - k0);  // multiple of VE
        // stage x chunk: 32 rows x kVecPerRow vectors
        for (int v = tid; v < kTokPerCta * kVecPerRow; v += kThreads) {
            const int r = v / kVecPerRow, c = (v % kVecPerRow) * VE;
            float vals[8];
            if (t0 + r < T_ && c < n) {
                Vec16 q = ld_nc_v16(x + (size_t)(t0 + r) * d + k0 + c);
                unpack(q, vals, (T*)nullptr);
            } else {
#pragma unroll
                for (int j = 0; j < VE; ++j) vals[j] = 0.0f;
            }
#pragma unroll
            for (int j = 0; j < VE; ++j) xs[r * kXPitch + c + j] = vals[j];
        }
        // stage Wg chunk: Epad rows
        for (int v = tid; v < Epad * kVecPerRow; v += kThreads) {
            const int e = v / kVecPerRow, c = (v % kVecPerRow) * VE;
            float vals[8];
            if (e < E && c < n) {
                Vec16 q = ld_nc_v16(Wg + (size_t)e * d + k0 + c);
                unpack(q, vals, (T*)nullptr);
            } else {
#pragma unroll
                for (int j = 0; j < VE; ++j) vals[j] = 0.0f;
            }
#pragma unroll
            for (int j = 0; j < VE; ++j) wsm[e * kChunk + c + j] = vals[j];
        }
        __syncthreads();
        const float* xr = xs + tg * kXPitch;
        for (int i = 0; i < n; i += 4) {
            const float4 xv = *reinterpret_cast<const float4*>(xr + i);
#pragma unroll
            for (int j = 0; j < NE; ++j) {
                const float4 wv = *reinterpret_cast<const float4*>(wsm + (eg + 8 * j) * kChunk + i);
                acc[j] = fmaf(xv.x, wv.x, acc[j]);
                acc[j] = fmaf(xv.y, wv.y, acc[j]);
                acc[j] = fmaf(xv.z, wv.z, acc[j]);
                acc[j] = fmaf(xv.w, wv.w, acc[j]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < NE; ++j) {
        const int e = eg + 8 * j;
        if (e < E) lg[tg * lgp + e] = bias ? acc[j] + bias[e] : acc[j];
    }
    __syncthreads();

    // softmax + top-k: warp w handles tokens w, w+8, w+16, w+24
    const int lane = tid & 31, warp = tid >> 5;
    constexpr int kMaxPerLane = (NE * 8 + 31) / 32;
    for (int tt = warp; tt < kTokPerCta; tt += kThreads / 32) {
        const int64_t t = t0 + tt;
        if (t >= T_) break;
        float g[kMaxPerLane];
        float m = -CUDART_INF_F;
#pragma unroll
        for (int q = 0; q < kMaxPerLane; ++q) {
            const int e = lane + 32 * q;
            g[q] = e < E ? lg[tt * lgp + e] : -CUDART_INF_F;
            m = fmaxf(m, g[q]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float s = 0.0f;
#pragma unroll
        for (int q = 0; q < kMaxPerLane; ++q)
            if (lane + 32 * q < E) s += expf(g[q] - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        const float inv = 1.0f / s;
        if (probs) {
#pragma unroll
            for (int q = 0; q < kMaxPerLane; ++q) {
                const int e = lane + 32 * q;
                if (e < E) probs[(size_t)t * E + e] = expf(g[q] - m) * inv;
            }
        }
        uint32_t taken = 0;
        for (int r = 0; r < k; ++r) {
            float bv = -CUDART_INF_F;
            int be = 0x7fffffff;
#pragma unroll
            for (int q = 0; q < kMaxPerLane; ++q) {
                const int e = lane + 32 * q;
                if (e < E && !(taken >> q & 1u) && (g[q] > bv || be == 0x7fffffff)) {
                    // within a lane e grows with q, so '>' keeps the lower index on ties
                    bv = g[q];
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
            if (lane == 0) {
                topk_idx[(size_t)t * k + r] = be;
                topk_gate[(size_t)t * k + r] = expf(bv - m) * inv;
            }
        }
    }
}

template <typename T, int NE>
cudaError_t launch_route_t(const Problem& p, const void* x, const void* Wg, const float* bias,
                           int32_t* topk_idx, float* topk_gate, float* probs, cudaStream_t s) {
    const int Epad = NE * 8;
    const size_t smem =
        sizeof(float) * ((size_t)kTokPerCta * kXPitch + (size_t)Epad * kChunk + 32 * (Epad + 1));
    auto kern = route_kernel<T, NE>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const unsigned grid = (unsigned)ceil_div(p.T, kTokPerCta);
    kern<<<grid, kThreads, smem, s>>>(p.T, p.d, p.E, p.k, (const T*)x, (const T*)Wg, bias, topk_idx,
                                     topk_gate, probs);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_ne(const Problem& p, const void* x, const void* Wg, const float* bias,
                        int32_t* topk_idx, float* topk_gate, float* probs, cudaStream_t s) {
    const int ne = (p.E + 7) / 8;
    if (ne <= 1) return launch_route_t<T, 1>(p, x, Wg, bias, topk_idx, topk_gate, probs, s);
    if (ne <= 2) return launch_route_t<T, 2>(p, x, Wg, bias, topk_idx, topk_gate, probs, s);
    if (ne <= 4) return launch_route_t<T, 4>(p, x, Wg, bias, topk_idx, topk_gate, probs, s);
    if (ne <= 8) return launch_route_t<T, 8>(p, x, Wg, bias, topk_idx, topk_gate, probs, s);
    if (ne <= 16) return launch_route_t<T, 16>(p, x, Wg, bias, topk_idx, topk_gate, probs, s);
    return launch_route_t<T, 32>(p, x, Wg, bias, topk_idx, topk_gate, probs, s);
}

}  // namespace

cudaError_t launch_route(const Problem& p, const void* x, const void* Wg, const float* bias,
                         int32_t* topk_idx, float* topk_gate, float* probs, cudaStream_t s) {
    if (p.T == 0) return cudaSuccess;
    if (p.dtype == MOE_BF16)
        return dispatch_ne<__nv_bfloat16>(p, x, Wg, bias, topk_idx, topk_gate, probs, s);
    return dispatch_ne<float>(p, x, Wg, bias, topk_idx, topk_gate, probs, s);
}

}  // namespace moe
