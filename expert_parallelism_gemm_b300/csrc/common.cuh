// common.cuh -- small shared pieces of the CUDA library: element types,
// vector loads, device status bits and the internal launcher declarations.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

// Bits OR-ed into the workspace status word by kernels.
constexpr int kDevTimeout = 1;   // a bounded mbarrier wait gave up
constexpr int kDevBadIndex = 2;  // an index read from memory was out of range

constexpr int kThreads = 256;
constexpr int kAssignBlock = 32;  // tokens per slot-assignment block (one warp)
constexpr int kStatBlocks = 64;   // most CTAs (and partial sums) of the routing-statistics kernel

struct Problem {
    int64_t T;
    int d, E, D, k, ffn;
    int dtype, act;
    int flags, ffn_shared;
    int64_t C, C_shard, rows_max;
    int64_t nblk;  // ceil(T / kAssignBlock)
};

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Validates the caller's problem (MOE_OK or the status to return) and fills
// *p with it plus the derived capacity, row bound and block count; every
// entry point starts here (api.cu).
int to_problem(const moe_problem* mp, Problem* p);

// fp32 <-> storage type
template <typename T>
struct Elem;
template <>
struct Elem<float> {
    static __device__ __forceinline__ float to_f(float v) { return v; }
    static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <>
struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// 16 bytes of a row, as 4 x 32-bit words.
struct alignas(16) Vec16 {
    uint32_t w[4];
};

__device__ __forceinline__ Vec16 ld_nc_v16(const void* p) {
    Vec16 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
    return v;
}
__device__ __forceinline__ Vec16 ld_v16(const void* p) {
    Vec16 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
    return v;
}
__device__ __forceinline__ void st_v16(void* p, const Vec16& v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]),
                 "r"(v.w[2]), "r"(v.w[3])
                 : "memory");
}

// Unpack 16 bytes into fp32 values: 8 for bf16, 4 for fp32.
__device__ __forceinline__ void unpack(const Vec16& v, float* out, __nv_bfloat16*) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        out[2 * j] = __uint_as_float(v.w[j] << 16);
        out[2 * j + 1] = __uint_as_float(v.w[j] & 0xffff0000u);
    }
}
__device__ __forceinline__ void unpack(const Vec16& v, float* out, float*) {
#pragma unroll
    for (int j = 0; j < 4; ++j) out[j] = __uint_as_float(v.w[j]);
}
// Pack fp32 values (round to nearest even for bf16).
__device__ __forceinline__ Vec16 pack(const float* in, __nv_bfloat16*) {
    Vec16 v;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        __nv_bfloat162 b = __floats2bfloat162_rn(in[2 * j], in[2 * j + 1]);
        v.w[j] = *reinterpret_cast<uint32_t*>(&b);
    }
    return v;
}
__device__ __forceinline__ Vec16 pack(const float* in, float*) {
    Vec16 v;
#pragma unroll
    for (int j = 0; j < 4; ++j) v.w[j] = __float_as_uint(in[j]);
    return v;
}

template <typename T>
__host__ __device__ constexpr int vec_elems() {
    return 16 / (int)sizeof(T);
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// launch_k() (programmatic stream serialisation) and calls dep_wait() -- which
// returns once all earlier work on the stream has completed and is visible --
// before its first global-memory access; only setup that touches no global
// memory (shared-memory barriers, tensor-memory allocation) comes before it.
// No kernel triggers its dependents early (griddepcontrol.launch_dependents):
// with the trigger at each kernel's start the layer measured the same with a
// cold L2 and 2% slower back to back (the next kernel's CTAs sat resident
// beside the running one), so dependents launch as each kernel completes.
__device__ __forceinline__ void dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---- launchers (each returns cudaGetLastError() of its launches) ----------
// logits (optional): the fp32 router logits [T, E], bias included
// status (optional): the workspace's status word, for a copy that never lands
cudaError_t launch_route(const Problem& p, const void* x, const void* Wg, const float* bias,
                         int32_t* topk_idx, float* topk_gate, float* probs, cudaStream_t s,
                         float* logits = nullptr, int32_t* fallback_idx = nullptr,
                         float* fallback_gate = nullptr, int* status = nullptr);

// router plus the count pass of the slot assignment (hist and scan outputs in
// `scan`, defined in assign_scan.cuh); T must be > 0
struct AssignScan;
// fallback_idx / fallback_gate (optional, [T, k]): the token's next k experts
// after its choices (ranks k .. 2k-1) and their probabilities
cudaError_t launch_route_count(const Problem& p, const void* x, const void* Wg, const float* bias,
                               int32_t* topk_idx, float* topk_gate, const AssignScan& scan,
                               cudaStream_t s, int32_t* fallback_idx = nullptr,
                               float* fallback_gate = nullptr, int* status = nullptr);

// bf16 router on the tensor cores (route_tc.cu): top-k indices identical to
// the fixed-order router's, gates within the tensor-core error of the
// experts it does not recompute; no probabilities, logits or fallbacks.
// scan.hist null: no slot-assignment count pass.  cudaErrorNotSupported when
// the tensor-map encoder is unavailable.
bool route_tc_eligible(const Problem& p);
cudaError_t launch_route_tc(const Problem& p, const void* x, const void* Wg, const float* bias, int32_t* topk_idx,
                            float* topk_gate, const AssignScan& scan, int* status, cudaStream_t s);

cudaError_t launch_assign(const Problem& p, const int32_t* topk_idx, int32_t* slot_pos,
                          int32_t* counts_routed, int32_t* counts_kept, int32_t* expert_offsets,
                          int32_t* shard_offsets, int32_t* shard_routed, int32_t* shard_overflow,
                          int32_t* row_token, int32_t* dropped, int32_t* hist, int* status,
                          cudaStream_t s);

// count pass alone (histogram, then the last CTA's scan into a's outputs)
cudaError_t launch_count(const Problem& p, const int32_t* topk_idx, const AssignScan& a, int* status,
                         cudaStream_t s);

// overflow rerouting after a count pass of the k choices (hist holds their
// scanned prefixes): the reroute pass (with the second scan, `second` =
// the same scan outputs with .second set) and the place pass.  route_idx /
// route_gate may alias topk_idx / topk_gate.
cudaError_t launch_reroute(const Problem& p, const int32_t* topk_idx, const float* topk_gate,
                           const int32_t* fallback_idx, const float* fallback_gate, int32_t* route_idx,
                           float* route_gate, int32_t* slot_pos, const AssignScan& second, int32_t* row_token,
                           int* status, cudaStream_t s);

// slot positions, scan outputs and the pack in one kernel, after a router
// launch that wrote the histogram with scan.defer set; for problems where
// assign_pack_fits() holds
bool assign_pack_fits(const Problem& p);
cudaError_t launch_assign_pack(const Problem& p, const void* x, const int32_t* topk_idx, const AssignScan& a,
                               int32_t* slot_pos, int32_t* row_token, void* xd, int* status, cudaStream_t s);

// rank pass alone (the histogram already holds the scanned prefixes)
cudaError_t launch_rank(const Problem& p, const int32_t* topk_idx, const int32_t* hist,
                        const int32_t* expert_offsets, int32_t* slot_pos, int32_t* row_token, int* status,
                        cudaStream_t s);

cudaError_t launch_dispatch(const Problem& p, const void* x, const int32_t* row_token,
                            const int32_t* expert_offsets, void* xd, cudaStream_t s);
// the same permutation token-major: each token's x row read once, stored to
// each of its kept slots (expert_offsets[e] + slot_pos)
cudaError_t launch_scatter(const Problem& p, const void* x, const int32_t* topk_idx, const int32_t* slot_pos,
                           const int32_t* expert_offsets, void* xd, cudaStream_t s);

// shared: optional shared-expert output [T, d], added after the routed sum
cudaError_t launch_combine(const Problem& p, const void* yd, const int32_t* topk_idx,
                           const int32_t* slot_pos, const int32_t* expert_offsets,
                           const float* topk_gate, const void* residual, void* y, cudaStream_t s,
                           const void* shared = nullptr);

// routing statistics: `acc` holds E+1 64-bit fixed-point sums and `ticket`
// one int, both zero before the launch and left zero
int64_t stats_blocks(int64_t T);
cudaError_t launch_routing_stats(const Problem& p, const float* probs, const int32_t* counts_routed,
                                 const int32_t* counts_kept, float* stats, float* mean_prob,
                                 unsigned long long* acc, unsigned* ticket, cudaStream_t s);

// expert-choice routing (ec.cu)
cudaError_t launch_ec_select(const Problem& p, const float* logits, int32_t* row_token, int32_t* expert_offsets,
                             int32_t* sel_row, cudaStream_t s);
cudaError_t launch_ec_combine(const Problem& p, const void* yd, const float* probs, const int32_t* sel_row,
                              const void* shared, const void* residual, void* y, cudaStream_t s);

cudaError_t launch_ffn_simt(const Problem& p, const void* xd, const int32_t* expert_offsets,
                            const void* W1, const void* W3, const void* W2, void* h, void* yd,
                            cudaStream_t s);

// Tensor map of a row-major [rows, cols] matrix (bf16 or fp32) for unswizzled
// TMA tile loads of box_rows x box_cols; out-of-range elements read as zero.
// False when the encoder is unavailable or rejects the arguments.
bool encode_row_tiles(CUtensorMap* m, const void* base, int dtype, uint64_t rows, uint64_t cols, uint32_t box_cols,
                      uint32_t box_rows);

// tcgen05 grouped GEMM path (bf16 + SwiGLU). Returns cudaErrorNotSupported
// when the tensor-map encoder cannot be obtained.
// `sync` is the workspace's ffn_sync region (ffn_sync_ints(p) ints, zero
// before the first launch; each launch leaves it zero again).
// `order` (FfnOrder bits) relaxes the launch's ordering against its neighbours
// on the stream:
//  - kFfnReleaseNext: every CTA lets the next kernel launch once it has issued
//    its last tile's loads (griddepcontrol.launch_dependents), so that kernel's
//    CTAs take the SMs this launch's CTAs leave while its last tiles finish;
//  - kFfnWaitAtEnd: the launch waits for the previous kernel at its end instead
//    of its start.  Only for a launch that reads nothing the kernels before it
//    in the stream write or still read, and that follows a kernel all of whose
//    CTAs wait for their own predecessor before they let it launch (every
//    kernel of this library): then all earlier kernels but that one are done,
//    and the wait at the end keeps the kernel after this one from starting
//    before that one completes.
enum FfnOrder : int { kFfnReleaseNext = 1, kFfnWaitAtEnd = 2 };
cudaError_t launch_ffn_tc(const Problem& p, const void* xd, const int32_t* expert_offsets,
                          const void* W1, const void* W3, const void* W2, void* h, void* yd,
                          int* status, int* sync, cudaStream_t s, int order = 0);
size_t ffn_sync_ints(const Problem& p);

}  // namespace moe
