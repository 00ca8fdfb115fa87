// ffn_simt.cu -- expert FFN on CUDA cores, for the forms the tensor-core
// path does not take (fp32 storage, or the GeLU form).
//
// "Expert Parallelism" notes page (narrativegoldmine.com), "Components and
// Architecture", expert GEMM: a standard transformer MLP per expert; formal
// algorithm, expert computation on the tokens each expert received.
//   SwiGLU: h = silu(x W1^T) * (x W3^T);  GeLU: h = 0.5 a (1 + erf(a/sqrt2))
//   y = h W2^T
// Grouped over experts: CTA (m-tile, n-tile, expert) computes a 64 x 64 tile
// of expert e's rows [expert_offsets[e], expert_offsets[e+1]).  The grid's
// m extent is the capacity bound, so no count is read back to the host.
// fp32 accumulation; h is stored in the layer dtype.
#include "common.cuh"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;
enum Mode { kSwiGLU = 0, kGeLU = 1, kPlain = 2 };

template <typename T, int MODE>
__global__ void __launch_bounds__(kThreads)
ffn_simt_kernel(int N, int K, int64_t rows_max, const T* __restrict__ A,
                const int32_t* __restrict__ expert_offsets, const T* __restrict__ B,
                const T* __restrict__ B3, T* __restrict__ out) {
    dep_wait();
    const int e = blockIdx.z;
    // no offsets: one expert whose rows are 0..rows_max-1 (the shared expert)
    const int64_t o0 = expert_offsets ? (int64_t)expert_offsets[e] : 0;
    const int64_t o1 = expert_offsets ? (int64_t)expert_offsets[e + 1] : rows_max;
    const int64_t r0 = o0 + (int64_t)blockIdx.x * BM;
    // rows never reach past rows_max, whatever the offsets say
    const int64_t r1 = min(o1, rows_max);
    if (r0 < 0) return;
    if (r0 >= r1) return;
    const int n0 = blockIdx.y * BN;
    const T* Be = B + (size_t)e * N * K;
    const T* B3e = MODE == kSwiGLU ? B3 + (size_t)e * N * K : nullptr;

    __shared__ float As[BK][BM + 1];
    __shared__ float Bs[BK][BN + 1];
    __shared__ float B3s[MODE == kSwiGLU ? BK : 1][BN + 1];

    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;  // 16 x 16 threads, 4 x 4 each
    float acc[4][4] = {};
    float acc3[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += BK) {
        for (int i = threadIdx.x; i < BM * BK; i += kThreads) {
            const int m = i / BK, kk = i % BK;
            const int64_t row = r0 + m;
            As[kk][m] = (row < r1 && k0 + kk < K) ? Elem<T>::to_f(A[(size_t)row * K + k0 + kk]) : 0.0f;
            const int n = n0 + m;  // BN == BM
            const bool okb = n < N && k0 + kk < K;
            Bs[kk][m] = okb ? Elem<T>::to_f(Be[(size_t)n * K + k0 + kk]) : 0.0f;
            if (MODE == kSwiGLU) B3s[kk][m] = okb ? Elem<T>::to_f(B3e[(size_t)n * K + k0 + kk]) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[4], b[4], b3[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = As[kk][ty * 4 + i];
                b[i] = Bs[kk][tx * 4 + i];
                if (MODE == kSwiGLU) b3[i] = B3s[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                    if (MODE == kSwiGLU) acc3[i][j] = fmaf(a[i], b3[j], acc3[i][j]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t row = r0 + ty * 4 + i;
        if (row >= r1) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= N) continue;
            float v = acc[i][j];
            if (MODE == kSwiGLU) v = v / (1.0f + expf(-v)) * acc3[i][j];
            if (MODE == kGeLU) v = 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
            out[(size_t)row * N + n] = Elem<T>::from_f(v);
        }
    }
}

template <typename T>
cudaError_t launch_t(const Problem& p, const void* xd, const int32_t* off, const void* W1,
                     const void* W3, const void* W2, void* h, void* yd, cudaStream_t s) {
    const unsigned mt = (unsigned)ceil_div(p.C, BM);
    const dim3 g1(mt, (unsigned)ceil_div(p.ffn, BN), (unsigned)p.E);
    cudaError_t err;
    if (p.act == MOE_ACT_SWIGLU)
        err = launch_k(ffn_simt_kernel<T, kSwiGLU>, g1, dim3(kThreads), 0, s, p.ffn, p.d, p.rows_max,
                       (const T*)xd, off, (const T*)W1, (const T*)W3, (T*)h);
    else
        err = launch_k(ffn_simt_kernel<T, kGeLU>, g1, dim3(kThreads), 0, s, p.ffn, p.d, p.rows_max,
                       (const T*)xd, off, (const T*)W1, (const T*)nullptr, (T*)h);
    if (err != cudaSuccess) return err;
    const dim3 g2(mt, (unsigned)ceil_div(p.d, BN), (unsigned)p.E);
    return launch_k(ffn_simt_kernel<T, kPlain>, g2, dim3(kThreads), 0, s, p.d, p.ffn, p.rows_max, (const T*)h,
                    off, (const T*)W2, (const T*)nullptr, (T*)yd);
}

}  // namespace

cudaError_t launch_ffn_simt(const Problem& p, const void* xd, const int32_t* expert_offsets,
                            const void* W1, const void* W3, const void* W2, void* h, void* yd,
                            cudaStream_t s) {
    if (p.C == 0) return cudaSuccess;
    if (p.dtype == MOE_BF16)
        return launch_t<__nv_bfloat16>(p, xd, expert_offsets, W1, W3, W2, h, yd, s);
    return launch_t<float>(p, xd, expert_offsets, W1, W3, W2, h, yd, s);
}

}  // namespace moe
