// ec.cu -- expert-choice routing: each expert takes its tokens.
//
// "Expert Parallelism" notes page (narrativegoldmine.com), "Major Variants":
// expert-choice routing lets every expert pick the tokens it processes, which
// balances the load by construction.
//
// Expert e takes the Cc = min(C, T) tokens with the largest router score,
// the fp32 logit g[t, e] (the same values the router computes, so the choice
// is exact); equal scores are taken in ascending token order.  Its rows are
// its tokens in ascending token order, from row e * Cc.  A token's output is
// the sum, in ascending expert order, of probs[t, e] (its softmax
// probability) times the outputs of the experts that took it (plus a shared
// expert and the residual when given).
//
// Selection: one CTA per expert holds the expert's logit column in shared
// memory as 32-bit keys that order like the floats (sign bit flipped for
// non-negative values, all bits flipped for negative ones, -0 read as +0) and
// finds the Cc-th largest key K by an 8-bit radix select
// (four histogram passes, most significant digit first, integer shared-memory
// counts; one warp scans the 256 bins to find each digit).  A token is taken if its key is above K, or equal to K and among
// the first (Cc - number above K) equal keys in token order; rows follow from
// a block-wide scan of the taken flags in token order.  Integer work only, so
// the selection is exact and does not depend on scheduling.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kEcThreads = 1024;

// Exclusive scan of one int per thread over the CTA; returns the thread's
// prefix and writes the total to *total.  sh: 33 ints of shared memory
// (32 warp prefixes, then the total).
__device__ int ec_block_scan(int v, int* sh, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    __syncthreads();
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < nw ? sh[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        sh[lane] = wi - w;
        if (lane == 31) sh[32] = wi;  // nw <= 32, so lane 31 holds the total
    }
    __syncthreads();
    const int res = sh[warp] + incl - v;
    *total = sh[32];
    __syncthreads();
    return res;
}

// Unsigned key with the order of the float value (finite inputs; -0 == +0).
__device__ __forceinline__ uint32_t order_key(float v) {
    uint32_t b = __float_as_uint(v);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(kEcThreads)
ec_select_kernel(int64_t T, int E, int64_t Cc, const float* __restrict__ logits, int32_t* __restrict__ row_token,
                 int32_t* __restrict__ sel_row, int32_t* __restrict__ expert_offsets) {
    dep_wait();
    extern __shared__ uint32_t keys[];  // [T]
    __shared__ int hist[256];
    __shared__ int scan_sh[33];
    __shared__ uint32_t s_prefix;
    __shared__ int s_want;
    const int e = blockIdx.x;
    const int tid = threadIdx.x;
    for (int64_t t = tid; t < T; t += kEcThreads) keys[t] = order_key(logits[(size_t)t * E + e]);
    if (tid == 0) {
        expert_offsets[e] = (int32_t)((int64_t)e * Cc);
        if (e == E - 1) expert_offsets[E] = (int32_t)((int64_t)E * Cc);
        s_prefix = 0u;
        s_want = (int)Cc;
    }
    __syncthreads();
    const bool all = Cc >= T;
    if (!all) {
        // radix select of the Cc-th largest key, most significant digit first
        uint32_t mask = 0u;
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int b = tid; b < 256; b += kEcThreads) hist[b] = 0;
            __syncthreads();
            const uint32_t prefix = s_prefix;
            for (int64_t t = tid; t < T; t += kEcThreads) {
                const uint32_t kk = keys[t];
                if ((kk & mask) == prefix) atomicAdd(&hist[(kk >> shift) & 255u], 1);
            }
            __syncthreads();
            if (tid < 32) {
                // the digit holding the want-th largest key: lane l takes the
                // bins 255 - 8l .. 248 - 8l (descending), a warp scan gives the
                // count of keys in the bins above them, and the one bin where
                // the running count first reaches want is the digit
                const int want = s_want;
                int loc = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) loc += hist[255 - 8 * tid - j];
                __syncwarp();  // every lane has read s_want before one lane rewrites it
                int incl = loc;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int n = __shfl_up_sync(0xffffffffu, incl, o);
                    if (tid >= o) incl += n;
                }
                int cum = incl - loc;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int h = hist[255 - 8 * tid - j];
                    if (cum < want && cum + h >= want) {
                        s_prefix = prefix | ((uint32_t)(255 - 8 * tid - j) << shift);
                        s_want = want - cum;  // keys equal to the digit prefix still to take
                    }
                    cum += h;
                }
            }
            mask |= 255u << shift;
            __syncthreads();
        }
    }
    const uint32_t K = s_prefix;
    const int take_eq = s_want;  // among keys == K, the first take_eq in token order
    // each thread owns a contiguous run of tokens, so scans follow token order
    const int64_t per = (T + kEcThreads - 1) / kEcThreads;
    const int64_t r0 = min(T, (int64_t)tid * per), r1 = min(T, r0 + per);
    int n_eq = 0;
    if (!all)
        for (int64_t t = r0; t < r1; ++t) n_eq += keys[t] == K;
    int tot;
    int eq_before = ec_block_scan(n_eq, scan_sh, &tot);
    int n_take = 0;
    {
        int eq = eq_before;
        for (int64_t t = r0; t < r1; ++t) {
            const uint32_t kk = keys[t];
            const bool take = all || kk > K || (kk == K && eq++ < take_eq);
            n_take += take;
        }
    }
    int pos = ec_block_scan(n_take, scan_sh, &tot);
    int eq = eq_before;
    for (int64_t t = r0; t < r1; ++t) {
        const uint32_t kk = keys[t];
        const bool take = all || kk > K || (kk == K && eq++ < take_eq);
        int32_t row = -1;
        if (take) {
            row = (int32_t)((int64_t)e * Cc + pos);
            row_token[row] = (int32_t)t;
            ++pos;
        }
        sel_row[(size_t)t * E + e] = row;
    }
}

// CB vector columns per lane per pass over the token's experts
template <typename T, int CB>
__global__ void __launch_bounds__(kThreads)
ec_combine_kernel(int64_t Tn, int64_t rows_max, int E, int d, const T* __restrict__ yd,
                  const float* __restrict__ probs, const int32_t* __restrict__ sel_row,
                  const T* __restrict__ shared, const T* __restrict__ residual, T* __restrict__ y) {
    dep_wait();
    constexpr int VE = vec_elems<T>();
    const int nv = d / VE;
    const int lane = threadIdx.x & 31;
    constexpr int kWarps = kThreads / 32;
    for (int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t < Tn;
         t += (int64_t)gridDim.x * kWarps) {
        // the column loop is warp-uniform (ballots and shuffles below need
        // every lane); each lane checks its own columns against nv
        for (int vb = 0; vb < nv; vb += 32 * CB) {
            const int v0 = vb + lane;
            float acc[CB][8];
#pragma unroll
            for (int c = 0; c < CB; ++c)
#pragma unroll
                for (int j = 0; j < VE; ++j) acc[c][j] = 0.0f;
            // experts that took t, in ascending order: groups of 32 by ballot
            for (int e0 = 0; e0 < E; e0 += 32) {
                const int e = e0 + lane;
                int32_t row = e < E ? sel_row[(size_t)t * E + e] : -1;
                if (row >= rows_max) row = -1;  // inconsistent input: contributes nothing
                const float gate = row >= 0 ? probs[(size_t)t * E + e] : 0.0f;
                uint32_t bits = __ballot_sync(0xffffffffu, row >= 0);
                while (bits) {
                    const int src = __ffs(bits) - 1;
                    bits &= bits - 1;
                    const int64_t r = __shfl_sync(0xffffffffu, row, src);
                    const float g = __shfl_sync(0xffffffffu, gate, src);
                    Vec16 q[CB];
#pragma unroll
                    for (int c = 0; c < CB; ++c)
                        if (v0 + 32 * c < nv) q[c] = ld_nc_v16(yd + (size_t)r * d + (v0 + 32 * c) * VE);
#pragma unroll
                    for (int c = 0; c < CB; ++c) {
                        if (v0 + 32 * c >= nv) continue;
                        float vals[8];
                        unpack(q[c], vals, (T*)nullptr);
#pragma unroll
                        for (int j = 0; j < VE; ++j) acc[c][j] = fmaf(g, vals[j], acc[c][j]);
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < CB; ++c) {
                const int v = v0 + 32 * c;
                if (v >= nv) continue;
                if (shared) {
                    float sv[8];
                    unpack(ld_nc_v16(shared + (size_t)t * d + v * VE), sv, (T*)nullptr);
#pragma unroll
                    for (int j = 0; j < VE; ++j) acc[c][j] += sv[j];
                }
                if (residual) {
                    float rv[8];
                    unpack(ld_nc_v16(residual + (size_t)t * d + v * VE), rv, (T*)nullptr);
#pragma unroll
                    for (int j = 0; j < VE; ++j) acc[c][j] += rv[j];
                }
                st_v16(y + (size_t)t * d + v * VE, pack(acc[c], (T*)nullptr));
            }
        }
    }
}

inline unsigned ec_grid(int64_t items) {
    const int64_t g = ceil_div(items, kThreads / 32);
    return (unsigned)(g < 1 ? 1 : (g > 148 * 32 ? 148 * 32 : g));
}

}  // namespace

size_t ec_select_smem(int64_t T) { return (size_t)T * sizeof(uint32_t); }

cudaError_t launch_ec_select(const Problem& p, const float* logits, int32_t* row_token, int32_t* expert_offsets,
                             int32_t* sel_row, cudaStream_t s) {
    const size_t smem = ec_select_smem(p.T);
    cudaError_t err =
        cudaFuncSetAttribute(ec_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    return launch_k(ec_select_kernel, dim3((unsigned)p.E), dim3(kEcThreads), smem, s, p.T, p.E, p.C, logits,
                    row_token, sel_row, expert_offsets);
}

cudaError_t launch_ec_combine(const Problem& p, const void* yd, const float* probs, const int32_t* sel_row,
                              const void* shared, const void* residual, void* y, cudaStream_t s) {
    if (p.T == 0) return cudaSuccess;
    const unsigned g = ec_grid(p.T);
    if (p.dtype == MOE_BF16)
        return launch_k(ec_combine_kernel<__nv_bfloat16, 4>, dim3(g), dim3(kThreads), 0, s, p.T, p.rows_max, p.E,
                        p.d, (const __nv_bfloat16*)yd, probs, sel_row, (const __nv_bfloat16*)shared,
                        (const __nv_bfloat16*)residual, (__nv_bfloat16*)y);
    return launch_k(ec_combine_kernel<float, 4>, dim3(g), dim3(kThreads), 0, s, p.T, p.rows_max, p.E, p.d,
                    (const float*)yd, probs, sel_row, (const float*)shared, (const float*)residual, (float*)y);
}

}  // namespace moe
