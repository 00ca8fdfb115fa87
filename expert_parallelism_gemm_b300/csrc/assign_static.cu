// assign_static.cu -- moe_assign_slots_static: the slot assignment for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand this library a workspace: a
// plugin or custom operator inside a host framework that owns every device
// allocation and passes an operator only its input and output buffers, or a
// latency-critical path that must not take cudaMalloc's implicit device
// synchronisation.  For them this entry point keeps the assignment's scratch
// (the per-block expert histograms, plus the completion ticket and status
// words) in one file-scope __device__ array instead of a caller workspace.
//
// Limits and rules, stated in include/moe.h as well:
//  - the array holds kStaticHistInts histogram entries, so a problem is
//    accepted only if E * k * ceil(T / 32) <= kStaticHistInts; every GPU
//    that loads the library keeps the array (4 MiB + 256 B) until exit;
//  - the first call on a device looks up the array's device address with
//    cudaGetSymbolAddress (once per device, with that device current); make
//    that first call before any stream capture;
//  - every call shares the one array: calls whose kernels overlap on the
//    GPU (different streams, or several host threads) race;
//  - each call clears the completion ticket and the spare words after it
//    (cudaMemsetAsync, no allocation); the histogram needs no clearing;
//  - errors the kernels find (an expert id outside [0, E)) are OR-ed into the
//    array's status word, which no call clears: it accumulates until
//    moe_assign_slots_static_status() reads and clears it, as
//    moe_device_status() does for a workspace;
//  - the array is placed on a device when the library's module is loaded
//    there, which under CUDA's lazy module loading is the first call on that
//    device; a caller that needs every later call free of that one-time
//    placement makes one warm-up call per device first.
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr int64_t kStaticWords = 64;              // status [0], ticket [1], spare; 256 B
constexpr int64_t kStaticHistInts = 1ll << 20;    // 4 MiB of histogram entries
constexpr int kMaxDevices = 64;

__device__ __align__(256) int32_t g_assign_scratch[kStaticWords + kStaticHistInts];

// Device address of g_assign_scratch per device ordinal (the host-side name
// of the array is only a stand-in and must never be passed to a kernel).
int32_t* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

cudaError_t scratch_for_current_device(int32_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_assign_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = (int32_t*)ptr;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_assign_slots_static(const moe_problem* mp, const int32_t* topk_idx, int32_t* slot_pos,
                                       int32_t* counts_routed, int32_t* counts_kept,
                                       int32_t* expert_offsets, int32_t* shard_offsets,
                                       int32_t* shard_routed, int32_t* shard_overflow, int32_t* row_token,
                                       int32_t* dropped, void* stream) {
    Problem p;
    int rc = to_problem(mp, &p);  // the same validation and derived sizes as moe_assign_slots
    if (rc != MOE_OK) return rc;
    if (p.flags & MOE_FLAG_REROUTE) return MOE_ERR_INVALID_ARG;  // rerouting has its own entry point
    if ((p.T > 0 && (!topk_idx || !slot_pos || !row_token)) || !counts_routed || !counts_kept ||
        !expert_offsets || !shard_offsets || !shard_routed || !shard_overflow)
        return MOE_ERR_INVALID_ARG;
    if ((int64_t)p.E * p.k * p.nblk > kStaticHistInts) return MOE_ERR_WORKSPACE;  // beyond the static array
    int32_t* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    // the ticket and spare words; the status word [0] keeps earlier errors
    if (cudaMemsetAsync(scratch + 1, 0, (kStaticWords - 1) * sizeof(int32_t), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    cudaError_t e = launch_assign(p, topk_idx, slot_pos, counts_routed, counts_kept, expert_offsets,
                                  shard_offsets, shard_routed, shard_overflow, row_token, dropped,
                                  scratch + kStaticWords, (int*)scratch, s);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_assign_slots_static_status(void* stream) {
    int32_t* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    int32_t word = 0;
    if (cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (word != 0) {
        const int32_t zero = 0;
        if (cudaMemcpy(scratch, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (word & kDevTimeout) return MOE_ERR_TIMEOUT;
    return word ? MOE_ERR_DEVICE : MOE_OK;
}
