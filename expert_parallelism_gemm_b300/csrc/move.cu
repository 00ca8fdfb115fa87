// move.cu -- dispatch (pack) and combine, the two permutations that stand in
// for the pages' two all-to-all exchanges on one GPU.
//
// Dispatch: "Expert Parallelism and the All-to-All Bottleneck"
// (ashishsrivastav.com), phase 2: rows are repacked so each row holds a token
// destined for one expert; "Expert Parallelism" notes page
// (narrativegoldmine.com), token dispatch tensor.  xd[row] = x[row_token[row]].
//
// Combine: same blog, phase 4 (results reassembled in token order); notes
// page, expert combine (gate-weighted sum of a token's k outputs) and residual
// addition.  One fixed order per token: fp32 fused multiply-adds over the
// ranks in ascending order from +0, then the residual, then one rounding.
//
// Both are HBM-bound copies: one warp per row or token, each lane moving 16
// bytes per step, so a warp touches 512 contiguous bytes per instruction.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = kThreads / 32;

template <typename T>
__global__ void __launch_bounds__(kThreads)
dispatch_kernel(int64_t Tn, int64_t rows_max, int E, int d, const T* __restrict__ x,
                const int32_t* __restrict__ row_token, const int32_t* __restrict__ expert_offsets,
                T* __restrict__ xd) {
    constexpr int VE = vec_elems<T>();
    // rows past rows_max do not exist in xd; a token id outside [0, T) is skipped
    const int64_t rows = min((int64_t)expert_offsets[E], rows_max);
    const int nv = d / VE;
    const int lane = threadIdx.x & 31;
    for (int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); row < rows;
         row += (int64_t)gridDim.x * kWarps) {
        const int64_t t = row_token[row];
        if (t < 0 || t >= Tn) continue;
        const T* src = x + (size_t)t * d;
        T* dst = xd + (size_t)row * d;
        for (int v = lane; v < nv; v += 32) st_v16(dst + v * VE, ld_nc_v16(src + v * VE));
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
combine_kernel(int64_t Tn, int64_t rows_max, int E, int d, int k, const T* __restrict__ yd, const int32_t* __restrict__ topk_idx,
               const int32_t* __restrict__ slot_pos, const int32_t* __restrict__ expert_offsets,
               const float* __restrict__ topk_gate, const T* __restrict__ residual, T* __restrict__ y) {
    constexpr int VE = vec_elems<T>();
    const int nv = d / VE;
    const int lane = threadIdx.x & 31;
    for (int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t < Tn;
         t += (int64_t)gridDim.x * kWarps) {
        // lane r < k fetches assignment r; broadcast below
        int64_t my_row = -1;
        float my_gate = 0.0f;
        if (lane < k) {
            const int pos = slot_pos[(size_t)t * k + lane];
            const int e = topk_idx[(size_t)t * k + lane];
            if (pos >= 0 && e >= 0 && e < E) {
                my_row = (int64_t)expert_offsets[e] + pos;
                my_gate = topk_gate[(size_t)t * k + lane];
                if (my_row >= rows_max) my_row = -1;  // inconsistent input: contributes nothing
            }
        }
        for (int v = lane; v - lane < nv; v += 32) {
            float acc[VE];
#pragma unroll
            for (int j = 0; j < VE; ++j) acc[j] = 0.0f;
            for (int r = 0; r < k; ++r) {
                const int64_t row = __shfl_sync(0xffffffffu, my_row, r);
                const float g = __shfl_sync(0xffffffffu, my_gate, r);
                if (row < 0 || v >= nv) continue;
                float vals[8];
                unpack(ld_nc_v16(yd + (size_t)row * d + v * VE), vals, (T*)nullptr);
#pragma unroll
                for (int j = 0; j < VE; ++j) acc[j] = fmaf(g, vals[j], acc[j]);
            }
            if (v >= nv) continue;
            if (residual) {
                float rv[8];
                unpack(ld_nc_v16(residual + (size_t)t * d + v * VE), rv, (T*)nullptr);
#pragma unroll
                for (int j = 0; j < VE; ++j) acc[j] += rv[j];
            }
            st_v16(y + (size_t)t * d + v * VE, pack(acc, (T*)nullptr));
        }
    }
}

inline unsigned grid_for(int64_t items) {
    const int64_t g = ceil_div(items, kWarps);
    return (unsigned)(g < 1 ? 1 : (g > 148 * 32 ? 148 * 32 : g));
}

}  // namespace

cudaError_t launch_dispatch(const Problem& p, const void* x, const int32_t* row_token,
                            const int32_t* expert_offsets, void* xd, cudaStream_t s) {
    if (p.rows_max == 0) return cudaSuccess;
    const unsigned g = grid_for(p.rows_max);
    if (p.dtype == MOE_BF16)
        dispatch_kernel<__nv_bfloat16><<<g, kThreads, 0, s>>>(
            p.T, p.rows_max, p.E, p.d, (const __nv_bfloat16*)x, row_token, expert_offsets,
            (__nv_bfloat16*)xd);
    else
        dispatch_kernel<float><<<g, kThreads, 0, s>>>(p.T, p.rows_max, p.E, p.d, (const float*)x,
                                                      row_token, expert_offsets, (float*)xd);
    return cudaGetLastError();
}

cudaError_t launch_combine(const Problem& p, const void* yd, const int32_t* topk_idx,
                           const int32_t* slot_pos, const int32_t* expert_offsets,
                           const float* topk_gate, const void* residual, void* y, cudaStream_t s) {
    if (p.T == 0) return cudaSuccess;
    const unsigned g = grid_for(p.T);
    if (p.dtype == MOE_BF16)
        combine_kernel<__nv_bfloat16><<<g, kThreads, 0, s>>>(
            p.T, p.rows_max, p.E, p.d, p.k, (const __nv_bfloat16*)yd, topk_idx, slot_pos, expert_offsets, topk_gate,
            (const __nv_bfloat16*)residual, (__nv_bfloat16*)y);
    else
        combine_kernel<float><<<g, kThreads, 0, s>>>(p.T, p.rows_max, p.E, p.d, p.k, (const float*)yd, topk_idx,
                                                     slot_pos, expert_offsets, topk_gate,
                                                     (const float*)residual, (float*)y);
    return cudaGetLastError();
}

}  // namespace moe
