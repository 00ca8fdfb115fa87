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
// expert; kept iff pos < C.  Computed in two integer passes, so the result
// does not depend on scheduling:
//   1. count: one warp per (rank r, block b of 32 tokens) writes the block's
//      per-expert histogram hist[e][r][b] (warp match on the expert id); the
//      last CTA to finish (integer atomic ticket) scans every expert's
//      histogram into exclusive prefixes in (r, b) order and writes counts,
//      expert and shard offsets, shard statistics and the dropped total
//      (assign_scan.cuh).  The layer forward's router writes the histogram
//      and runs the same scan itself, so it skips this kernel (and on small
//      histograms leaves scan, positions and pack to assign_pack.cu);
//   2. rank:  one warp per (r, b): pos = prefix + number of lower lanes with
//      the same expert; writes slot_pos and row_token.
//
// Overflow rerouting ("Expert Parallelism" notes page, "Capacity Factor and
// Token Dropping": a choice over capacity may be redirected to a secondary
// expert, the next-best one).  After the count pass of the k choices:
//   2'. reroute: one warp per block b, lane = token, ranks in ascending order:
//       the first-pass position as in the rank pass; a choice with pos < C
//       keeps its expert, gate and position; the j-th overflowing choice of a
//       token takes its fallback j (the token's rank k + j expert and that
//       expert's probability) and is marked pending.  The warp then writes
//       the block's histogram of pending assignments per (expert, rank) in
//       place of the first-pass one, and the last CTA scans it with every
//       expert's prefixes starting from its first-pass kept count (second
//       pass of assign_scan.cuh), which fixes the final counts and offsets;
//   3'. place: one warp per (r, b): a pending assignment's position is its
//       prefix + number of lower lanes pending for the same expert, kept iff
//       below C; every kept assignment writes its row_token entry at the
//       final offsets.
// Rerouted assignments therefore take only the capacity the first pass left,
// in the same (rank, token) priority, one level deep.
#include <algorithm>

#include "assign_scan.cuh"

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
count_kernel(int64_t T, int E, int k, int64_t nblk, const int32_t* __restrict__ idx, AssignScan a,
             int* status) {
    dep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t b = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int r = blockIdx.y;
    if (b < nblk) {
        const int e = load_expert(idx, b * kAssignBlock + lane, r, T, k, E, status);
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        for (int z = lane; z < E; z += 32) a.hist[((size_t)z * k + r) * nblk + b] = 0;
        __syncwarp();
        if (e >= 0 && lane == __ffs(same) - 1) a.hist[((size_t)e * k + r) * nblk + b] = __popc(same);
    }
    finish_assign_scan(a);
}

__global__ void __launch_bounds__(kThreads)
rank_kernel(int64_t T, int E, int k, int64_t nblk, int64_t C, const int32_t* __restrict__ idx,
            const int32_t* __restrict__ hist, const int32_t* __restrict__ expert_offsets,
            int32_t* __restrict__ slot_pos, int32_t* __restrict__ row_token, int* status) {
    dep_wait();
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

constexpr int32_t kPending = -2;  // slot_pos of a rerouted assignment between reroute and place

__global__ void __launch_bounds__(kThreads)
reroute_kernel(int64_t T, int E, int k, int64_t nblk, int64_t C, const int32_t* idx, const float* gate,
               const int32_t* __restrict__ fb_idx, const float* __restrict__ fb_gate, int32_t* route_idx,
               float* route_gate, int32_t* __restrict__ slot_pos, AssignScan a, int* status) {
    dep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t b = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (b < nblk) {
        const int64_t t = b * kAssignBlock + lane;
        // first-pass positions, read before the histogram is reused
        int e1[8], pos1[8];
        for (int r = 0; r < k; ++r) {
            const int e = load_expert(idx, t, r, T, k, E, status);
            const uint32_t same = __match_any_sync(0xffffffffu, e);
            e1[r] = e;
            pos1[r] = e >= 0 ? a.hist[((size_t)e * k + r) * nblk + b] + __popc(same & lanemask_lt()) : -1;
        }
        __syncwarp();
        for (int i = lane; i < E * k; i += 32) a.hist[(size_t)i * nblk + b] = 0;
        __syncwarp();
        int j = 0;  // overflowing choices of this token so far
        for (int r = 0; r < k; ++r) {
            int key = -1;
            if (t < T) {
                const size_t i = (size_t)t * k + r;
                const float g = gate[i];  // read before route_gate, which may alias gate, is written
                if (e1[r] < 0) {
                    route_idx[i] = -1;
                    route_gate[i] = 0.0f;
                    slot_pos[i] = -1;
                } else if (pos1[r] < C) {
                    route_idx[i] = e1[r];
                    route_gate[i] = g;
                    slot_pos[i] = pos1[r];
                } else {
                    const size_t fi = (size_t)t * k + j++;
                    const int e2 = fb_idx[fi];
                    if (e2 < 0 || e2 >= E) {
                        atomicOr(status, kDevBadIndex);
                        route_idx[i] = -1;
                        route_gate[i] = 0.0f;
                        slot_pos[i] = -1;
                    } else {
                        route_idx[i] = e2;
                        route_gate[i] = fb_gate[fi];
                        slot_pos[i] = kPending;
                        key = e2;
                    }
                }
            }
            const uint32_t same = __match_any_sync(0xffffffffu, key);
            if (key >= 0 && lane == __ffs(same) - 1) a.hist[((size_t)key * k + r) * nblk + b] = __popc(same);
        }
    }
    finish_assign_scan(a);
}

__global__ void __launch_bounds__(kThreads)
place_kernel(int64_t T, int k, int64_t nblk, int64_t C, int64_t rows_max, const int32_t* __restrict__ route_idx,
             const int32_t* __restrict__ hist, const int32_t* __restrict__ expert_offsets,
             int32_t* __restrict__ slot_pos, int32_t* __restrict__ row_token, int* status) {
    dep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t b = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int r = blockIdx.y;
    if (b >= nblk) return;
    const int64_t t = b * kAssignBlock + lane;
    const size_t i = (size_t)t * k + r;
    const int sp = t < T ? slot_pos[i] : -1;
    const int e = sp == kPending || sp >= 0 ? route_idx[i] : -1;
    const uint32_t same = __match_any_sync(0xffffffffu, sp == kPending ? e : -1);
    if (e < 0) return;
    int64_t pos = sp;
    if (sp == kPending) {
        pos = (int64_t)hist[((size_t)e * k + r) * nblk + b] + __popc(same & lanemask_lt());
        if (pos >= C) {
            slot_pos[i] = -1;
            return;
        }
        slot_pos[i] = (int32_t)pos;
    }
    const int64_t row = expert_offsets[e] + pos;
    if (row < rows_max) row_token[row] = (int32_t)t;
    else atomicOr(status, kDevBadIndex);
}

}  // namespace

cudaError_t launch_reroute(const Problem& p, const int32_t* topk_idx, const float* topk_gate,
                           const int32_t* fallback_idx, const float* fallback_gate, int32_t* route_idx,
                           float* route_gate, int32_t* slot_pos, const AssignScan& second, int32_t* row_token,
                           int* status, cudaStream_t s) {
    if (p.nblk == 0) return cudaSuccess;
    const dim3 grid((unsigned)ceil_div(p.nblk, kThreads / 32));
    cudaError_t e = launch_k(reroute_kernel, grid, dim3(kThreads), 0, s, p.T, p.E, p.k, p.nblk, p.C, topk_idx,
                             topk_gate, fallback_idx, fallback_gate, route_idx, route_gate, slot_pos, second,
                             status);
    if (e != cudaSuccess) return e;
    return launch_k(place_kernel, dim3(grid.x, (unsigned)p.k), dim3(kThreads), 0, s, p.T, p.k, p.nblk, p.C,
                    p.rows_max, (const int32_t*)route_idx, (const int32_t*)second.hist,
                    (const int32_t*)second.expert_offsets, slot_pos, row_token, status);
}

cudaError_t launch_count(const Problem& p, const int32_t* topk_idx, const AssignScan& a, int* status,
                         cudaStream_t s) {
    // at least one CTA, so that T = 0 still writes zero counts and offsets
    const dim3 grid((unsigned)std::max<int64_t>(1, ceil_div(p.nblk, kThreads / 32)), (unsigned)p.k);
    return launch_k(count_kernel, grid, dim3(kThreads), 0, s, p.T, p.E, p.k, p.nblk, topk_idx, a, status);
}

cudaError_t launch_assign(const Problem& p, const int32_t* topk_idx, int32_t* slot_pos,
                          int32_t* counts_routed, int32_t* counts_kept, int32_t* expert_offsets,
                          int32_t* shard_offsets, int32_t* shard_routed, int32_t* shard_overflow,
                          int32_t* row_token, int32_t* dropped, int32_t* hist, int* status,
                          cudaStream_t s) {
    // status[1] is the count pass's completion ticket
    const AssignScan a{hist, counts_routed, counts_kept, expert_offsets, shard_offsets, shard_routed,
                       shard_overflow, dropped, (unsigned*)(status + 1), p.E, p.D, p.k, p.nblk, p.C,
                       p.C_shard};
    cudaError_t e = launch_count(p, topk_idx, a, status, s);
    if (e != cudaSuccess || p.nblk == 0) return e;
    return launch_rank(p, topk_idx, hist, expert_offsets, slot_pos, row_token, status, s);
}

cudaError_t launch_rank(const Problem& p, const int32_t* topk_idx, const int32_t* hist,
                        const int32_t* expert_offsets, int32_t* slot_pos, int32_t* row_token, int* status,
                        cudaStream_t s) {
    if (p.nblk == 0) return cudaSuccess;
    const dim3 grid((unsigned)ceil_div(p.nblk, kThreads / 32), (unsigned)p.k);
    return launch_k(rank_kernel, grid, dim3(kThreads), 0, s, p.T, p.E, p.k, p.nblk, p.C, topk_idx, hist,
                    expert_offsets, slot_pos, row_token, status);
}

}  // namespace moe
