// assign.cu -- slot assignment and token dropping.
//
// "Expert Parallelism" notes page (narrativegoldmine.com), "Capacity Factor
// and Token Dropping": an expert processes at most C assignments per forward
// pass, the rest are dropped.  "Expert Parallelism" (theinfinity.ai), capacity
// paragraph: per-device capacity C = ceil((B*k/D)*c) and overflow
// max(0, p*B*k - C).  "Expert Parallelism and the All-to-All Bottleneck"
// (ashishsrivastav.com), "The All-to-All Communication Pattern": experts sit
// on devices in contiguous blocks (64 experts on 8 GPUs, expert 55 on GPU 6).
//
// Priority: every rank-0 choice in token order, then every rank-1 choice, ...
// pos(t, r) = number of earlier assignments (in that order) to the same
// expert; kept iff pos < C.  Computed in three integer passes, so the result
// does not depend on scheduling:
//   1. count: one warp per (rank r, block b of 32 tokens) writes the block's
//      per-expert histogram hist[e][r][b] (warp match on the expert id);
//   2. scan:  one CTA per expert turns hist[e][*][*] into its exclusive prefix
//      in (r, b) order and writes the routed / kept counts; the last CTA to
//      finish (integer atomic ticket) writes expert and shard offsets, shard
//      statistics and the dropped total;
//   3. rank:  one warp per (r, b): pos = prefix + number of lower lanes with
//      the same expert; writes slot_pos and row_token.
#include "common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Expert of assignment (t, r), or -1 for a token past T.  An id outside
// [0, E) is recorded in the status word and treated as no assignment.
__device__ __forceinline__ int load_expert(const int32_t* idx, int64_t t, int r, int64_t T, int k,
                                           int E, int* status) {
    if (t >= T) return -1;
    int e = idx[(size_t)t * k + r];
    if (e < 0 || e >= E) {
        atomicOr(status, kDevBadIndex);
        return -1;
    }
    return e;
}

__global__ void __launch_bounds__(kThreads)
count_kernel(int64_t T, int E, int k, int64_t nblk, const int32_t* __restrict__ idx,
             int32_t* __restrict__ hist, int* status) {
    const int lane = threadIdx.x & 31;
    const int64_t b = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int r = blockIdx.y;
    if (b >= nblk) return;
    const int e = load_expert(idx, b * kAssignBlock + lane, r, T, k, E, status);
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    for (int z = lane; z < E; z += 32) hist[((size_t)z * k + r) * nblk + b] = 0;
    __syncwarp();
    if (e >= 0 && lane == __ffs(same) - 1) hist[((size_t)e * k + r) * nblk + b] = __popc(same);
}

// Block-wide exclusive scan of one int per thread; returns the prefix and
// writes the block total to *total.
__device__ int block_exclusive_scan(int v, int* sh /* [32] */, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
        int w = lane < kThreads / 32 ? sh[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        if (lane < kThreads / 32) sh[lane] = wi - w;
        if (lane == kThreads / 32 - 1) sh[31] = wi;
    }
    __syncthreads();
    const int res = sh[warp] + incl - v;
    *total = sh[31];
    return res;
}

__global__ void __launch_bounds__(kThreads)
scan_kernel(int E, int D, int k, int64_t nblk, int64_t C, int64_t C_shard, int32_t* __restrict__ hist,
            int32_t* __restrict__ counts_routed, int32_t* __restrict__ counts_kept,
            int32_t* __restrict__ expert_offsets, int32_t* __restrict__ shard_offsets,
            int32_t* __restrict__ shard_routed, int32_t* __restrict__ shard_overflow,
            int32_t* __restrict__ dropped, unsigned* ticket) {
    __shared__ int sh[32];
    __shared__ bool last;
    const int e = blockIdx.x;
    const int64_t L = (int64_t)k * nblk;
    int32_t* h = hist + (size_t)e * L;
    int running = 0;
    for (int64_t base = 0; base < L; base += kThreads) {
        const int64_t i = base + threadIdx.x;
        const int v = i < L ? h[i] : 0;
        int tot;
        const int ex = block_exclusive_scan(v, sh, &tot);
        if (i < L) h[i] = running + ex;
        running += tot;
    }
    if (threadIdx.x == 0) {
        counts_routed[e] = running;
        counts_kept[e] = (int)min((int64_t)running, C);
        __threadfence();
        last = atomicAdd(ticket, 1u) == (unsigned)(gridDim.x - 1);
    }
    __syncthreads();
    if (!last) return;
    // last CTA: offsets and statistics over all experts (E <= 256 = threads)
    __threadfence();
    const int tid = threadIdx.x;
    const int routed = tid < E ? ((volatile int32_t*)counts_routed)[tid] : 0;
    const int kept = tid < E ? ((volatile int32_t*)counts_kept)[tid] : 0;
    __shared__ int off_s[257];
    __shared__ int routed_s[256];
    int total_kept;
    const int ex = block_exclusive_scan(kept, sh, &total_kept);
    if (tid < E) {
        off_s[tid] = ex;
        routed_s[tid] = routed;
        expert_offsets[tid] = ex;
    }
    int total_drop;
    block_exclusive_scan(routed - kept, sh, &total_drop);
    if (tid == 0) {
        off_s[E] = total_kept;
        expert_offsets[E] = total_kept;
        if (dropped) dropped[0] = total_drop;
        *ticket = 0u;  // ready for the next call on this workspace
    }
    __syncthreads();
    const int per = E / D;
    if (tid < D) {
        int64_t rs = 0;
        for (int q = tid * per; q < (tid + 1) * per; ++q) rs += routed_s[q];
        shard_routed[tid] = (int32_t)rs;
        shard_overflow[tid] = (int32_t)(rs > C_shard ? rs - C_shard : 0);
        shard_offsets[tid] = off_s[tid * per];
    }
    if (tid == 0) shard_offsets[D] = total_kept;
}

__global__ void __launch_bounds__(kThreads)
rank_kernel(int64_t T, int E, int k, int64_t nblk, int64_t C, const int32_t* __restrict__ idx,
            const int32_t* __restrict__ hist, const int32_t* __restrict__ expert_offsets,
            int32_t* __restrict__ slot_pos, int32_t* __restrict__ row_token, int* status) {
    const int lane = threadIdx.x & 31;
    const int64_t b = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int r = blockIdx.y;
    if (b >= nblk) return;
    const int64_t t = b * kAssignBlock + lane;
    const int e = load_expert(idx, t, r, T, k, E, status);
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    if (t >= T) return;
    if (e < 0) {
        slot_pos[(size_t)t * k + r] = -1;
        return;
    }
    const int64_t pos = (int64_t)hist[((size_t)e * k + r) * nblk + b] + __popc(same & lanemask_lt());
    const bool kept = pos < C;
    slot_pos[(size_t)t * k + r] = kept ? (int32_t)pos : -1;
    if (kept) row_token[expert_offsets[e] + pos] = (int32_t)t;
}

}  // namespace

cudaError_t launch_assign(const Problem& p, const int32_t* topk_idx, int32_t* slot_pos,
                          int32_t* counts_routed, int32_t* counts_kept, int32_t* expert_offsets,
                          int32_t* shard_offsets, int32_t* shard_routed, int32_t* shard_overflow,
                          int32_t* row_token, int32_t* dropped, int32_t* hist, int* status,
                          cudaStream_t s) {
    const dim3 grid((unsigned)ceil_div(p.nblk, kThreads / 32), (unsigned)p.k);
    if (p.nblk > 0)
        count_kernel<<<grid, kThreads, 0, s>>>(p.T, p.E, p.k, p.nblk, topk_idx, hist, status);
    // status[1] is the scan's completion ticket
    scan_kernel<<<p.E, kThreads, 0, s>>>(p.E, p.D, p.k, p.nblk, p.C, p.C_shard, hist, counts_routed,
                                         counts_kept, expert_offsets, shard_offsets, shard_routed,
                                         shard_overflow, dropped, (unsigned*)(status + 1));
    if (p.nblk > 0)
        rank_kernel<<<grid, kThreads, 0, s>>>(p.T, p.E, p.k, p.nblk, p.C, topk_idx, hist,
                                              expert_offsets, slot_pos, row_token, status);
    return cudaGetLastError();
}

}  // namespace moe
