// move.cu -- dispatch (pack) and combine, the two permutations that stand in
// for the pages' two all-to-all exchanges on one GPU.
//
// Dispatch: "Expert Parallelism and the All-to-All Bottleneck"
// (ashishsrivastav.com), phase 2: rows are repacked so each row holds a token
// destined for one expert; "Expert Parallelism" notes page
// (narrativegoldmine.com), token dispatch tensor.  xd[row] = x[row_token[row]],
// walked expert-major (a gather through row_token) or token-major (each
// token's row stored to its k slots).
//
// Combine: same blog, phase 4 (results reassembled in token order); notes
// page, expert combine (gate-weighted sum of a token's k outputs) and residual
// addition.  One fixed order per token: fp32 fused multiply-adds over the
// ranks in ascending order from +0, then the shared expert's output (notes
// page, "Major Variants": a dense expert every token goes through), then the
// residual, then one rounding.
//
// Both are HBM-bound copies: one warp per row or token, each lane moving 16
// bytes per access, so a warp touches 512 contiguous bytes per instruction.
// Each lane issues a batch of loads (4 vectors for dispatch; for combine, the
// k source rows of 2 vector columns, 1 for k > 2, plus the shared expert's
// output and the residual) before it consumes any, so several loads per lane
// are in flight.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = kThreads / 32;

template <typename T>
__global__ void __launch_bounds__(kThreads)
dispatch_kernel(int64_t Tn, int64_t rows_max, int E, int d, const T* __restrict__ x,
                const int32_t* __restrict__ row_token, const int32_t* __restrict__ expert_offsets,
                T* __restrict__ xd) {
    dep_wait();
    constexpr int VE = vec_elems<T>();
    constexpr int B = 4;  // 16-byte loads in flight per lane before the stores
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
        for (int v0 = lane; v0 < nv; v0 += 32 * B) {
            Vec16 q[B];
#pragma unroll
            for (int j = 0; j < B; ++j)
                if (v0 + 32 * j < nv) q[j] = ld_nc_v16(src + (v0 + 32 * j) * VE);
#pragma unroll
            for (int j = 0; j < B; ++j)
                if (v0 + 32 * j < nv) st_v16(dst + (v0 + 32 * j) * VE, q[j]);
        }
    }
}

// Token-major form of the same permutation: one warp per token reads its x
// row once and stores it to each of its kept slots, row expert_offsets[e] +
// slot_pos[t, r] (the row the gather form finds through row_token).  With k
// ranks a token's row is needed k times; the gather form reads it once per
// slot, and those reads lie a whole expert segment apart, too far for L2 on
// the large layers (the Mixtral 8x7B shape moved 1.07 GB for 805 MB of
// algorithmic bytes).  Lanes r < k fetch rank r's destination; an invalid
// expert, a dropped rank (slot -1) or a row past rows_max stores nothing.
template <typename T>
__global__ void __launch_bounds__(kThreads)
scatter_kernel(int64_t Tn, int64_t rows_max, int E, int d, int k, const T* __restrict__ x,
               const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ slot_pos,
               const int32_t* __restrict__ expert_offsets, T* __restrict__ xd) {
    dep_wait();
    constexpr int VE = vec_elems<T>();
    constexpr int B = 4;  // 16-byte loads in flight per lane before the stores
    const int nv = d / VE;
    const int lane = threadIdx.x & 31;
    for (int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t < Tn;
         t += (int64_t)gridDim.x * kWarps) {
        int64_t row = -1;
        if (lane < k) {
            const int e = topk_idx[t * k + lane];
            const int pos = slot_pos[t * k + lane];
            if (e >= 0 && e < E && pos >= 0) {
                const int64_t r = (int64_t)expert_offsets[e] + pos;
                if (r < rows_max) row = r;
            }
        }
        const unsigned kept = __ballot_sync(0xffffffffu, row >= 0);
        if (!kept) continue;
        const T* src = x + (size_t)t * d;
        for (int v0 = lane; v0 < nv; v0 += 32 * B) {
            Vec16 q[B];
#pragma unroll
            for (int j = 0; j < B; ++j)
                if (v0 + 32 * j < nv) q[j] = ld_nc_v16(src + (v0 + 32 * j) * VE);
            for (unsigned m = kept; m; m &= m - 1) {
                const int r = __ffs(m) - 1;
                const int64_t dst_row = __shfl_sync(0xffffffffu, row, r);
                T* dst = xd + (size_t)dst_row * d;
#pragma unroll
                for (int j = 0; j < B; ++j)
                    if (v0 + 32 * j < nv) st_v16(dst + (v0 + 32 * j) * VE, q[j]);
            }
        }
    }
}

// CB vector columns per lane per step, each gathering up to KM ranks, so all
// of a step's loads are issued before the first multiply-add.  CB * KM is
// kept at 4 or 8 vectors: more would hold the kernel to two CTAs per SM by
// its registers, and a warp's one token per pass leaves it latency-bound.
template <typename T, int CB, int KM>
__global__ void __launch_bounds__(kThreads)
combine_kernel(int64_t Tn, int64_t rows_max, int E, int d, int k, const T* __restrict__ yd,
               const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ slot_pos,
               const int32_t* __restrict__ expert_offsets, const float* __restrict__ topk_gate,
               const T* __restrict__ shared, const T* __restrict__ residual, T* __restrict__ y) {
    dep_wait();
    constexpr int VE = vec_elems<T>();  // KM: ranks this instantiation handles (k <= KM)
    const int nv = d / VE;
    const int lane = threadIdx.x & 31;
    for (int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t < Tn;
         t += (int64_t)gridDim.x * kWarps) {
        // lane r < k fetches assignment r; every lane then holds all k
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
        int64_t rows[KM];
        float gates[KM];
#pragma unroll
        for (int r = 0; r < KM; ++r) {
            rows[r] = __shfl_sync(0xffffffffu, my_row, r);
            gates[r] = __shfl_sync(0xffffffffu, my_gate, r);
            if (r >= k) rows[r] = -1;
        }
        for (int v0 = lane; v0 < nv; v0 += 32 * CB) {
            Vec16 q[CB][KM];
            Vec16 rq[CB], sq[CB];
#pragma unroll
            for (int c = 0; c < CB; ++c) {
                const int v = v0 + 32 * c;
#pragma unroll
                for (int r = 0; r < KM; ++r)
                    if (rows[r] >= 0 && v < nv) q[c][r] = ld_nc_v16(yd + (size_t)rows[r] * d + v * VE);
                if (shared && v < nv) sq[c] = ld_nc_v16(shared + (size_t)t * d + v * VE);
                if (residual && v < nv) rq[c] = ld_nc_v16(residual + (size_t)t * d + v * VE);
            }
#pragma unroll
            for (int c = 0; c < CB; ++c) {
                const int v = v0 + 32 * c;
                if (v >= nv) continue;
                float acc[VE];
#pragma unroll
                for (int j = 0; j < VE; ++j) acc[j] = 0.0f;
#pragma unroll
                for (int r = 0; r < KM; ++r) {
                    if (rows[r] < 0) continue;
                    float vals[8];
                    unpack(q[c][r], vals, (T*)nullptr);
#pragma unroll
                    for (int j = 0; j < VE; ++j) acc[j] = fmaf(gates[r], vals[j], acc[j]);
                }
                if (shared) {
                    float sv[8];
                    unpack(sq[c], sv, (T*)nullptr);
#pragma unroll
                    for (int j = 0; j < VE; ++j) acc[j] += sv[j];
                }
                if (residual) {
                    float rv[8];
                    unpack(rq[c], rv, (T*)nullptr);
#pragma unroll
                    for (int j = 0; j < VE; ++j) acc[j] += rv[j];
                }
                st_v16(y + (size_t)t * d + v * VE, pack(acc, (T*)nullptr));
            }
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
        return launch_k(dispatch_kernel<__nv_bfloat16>, dim3(g), dim3(kThreads), 0, s, p.T, p.rows_max, p.E,
                        p.d, (const __nv_bfloat16*)x, row_token, expert_offsets, (__nv_bfloat16*)xd);
    return launch_k(dispatch_kernel<float>, dim3(g), dim3(kThreads), 0, s, p.T, p.rows_max, p.E, p.d,
                    (const float*)x, row_token, expert_offsets, (float*)xd);
}

cudaError_t launch_scatter(const Problem& p, const void* x, const int32_t* topk_idx, const int32_t* slot_pos,
                           const int32_t* expert_offsets, void* xd, cudaStream_t s) {
    if (p.rows_max == 0 || p.T == 0) return cudaSuccess;
    const unsigned g = grid_for(p.T);
    if (p.dtype == MOE_BF16)
        return launch_k(scatter_kernel<__nv_bfloat16>, dim3(g), dim3(kThreads), 0, s, p.T, p.rows_max, p.E, p.d,
                        p.k, (const __nv_bfloat16*)x, topk_idx, slot_pos, expert_offsets, (__nv_bfloat16*)xd);
    return launch_k(scatter_kernel<float>, dim3(g), dim3(kThreads), 0, s, p.T, p.rows_max, p.E, p.d, p.k,
                    (const float*)x, topk_idx, slot_pos, expert_offsets, (float*)xd);
}

template <typename T>
cudaError_t launch_combine_t(const Problem& p, unsigned g, const void* yd, const int32_t* topk_idx,
                             const int32_t* slot_pos, const int32_t* expert_offsets, const float* topk_gate,
                             const void* shared, const void* residual, void* y, cudaStream_t s) {
    const T* ydt = (const T*)yd;
    const T* st = (const T*)shared;
    const T* rt = (const T*)residual;
    T* yt = (T*)y;
    auto kern = p.k <= 2 ? combine_kernel<T, 2, 2> : p.k <= 4 ? combine_kernel<T, 1, 4> : combine_kernel<T, 1, 8>;
    return launch_k(kern, dim3(g), dim3(kThreads), 0, s, p.T, p.rows_max, p.E, p.d, p.k, ydt, topk_idx,
                    slot_pos, expert_offsets, topk_gate, st, rt, yt);
}

cudaError_t launch_combine(const Problem& p, const void* yd, const int32_t* topk_idx,
                           const int32_t* slot_pos, const int32_t* expert_offsets,
                           const float* topk_gate, const void* residual, void* y, cudaStream_t s,
                           const void* shared) {
    if (p.T == 0) return cudaSuccess;
    const unsigned g = grid_for(p.T);
    if (p.dtype == MOE_BF16)
        return launch_combine_t<__nv_bfloat16>(p, g, yd, topk_idx, slot_pos, expert_offsets, topk_gate,
                                               shared, residual, y, s);
    return launch_combine_t<float>(p, g, yd, topk_idx, slot_pos, expert_offsets, topk_gate, shared, residual,
                                   y, s);
}

}  // namespace moe
