// assign_pack.cu -- slot positions and the pack in one kernel, for the layer
// forward when the slot-assignment histogram is small.
//
// "Expert Parallelism" notes page (narrativegoldmine.com), "Capacity Factor
// and Token Dropping" (at most C assignments per expert, the rest dropped) and
// token dispatch; "Expert Parallelism and the All-to-All Bottleneck"
// (ashishsrivastav.com), phase 2 (rows repacked so each holds a token bound
// for one expert); "Expert Parallelism" (theinfinity.ai), capacity paragraph
// (per-device overflow).
//
// The router has written the per-block histogram hist[e][r][b] (rank-r choices
// of expert e among block b's 32 tokens).  CTA (b, r) of this kernel:
//   1. loads the whole histogram into shared memory and turns it into
//      exclusive prefixes in (r, b) order per expert, one warp per expert --
//      the same priority and integer arithmetic as the last-CTA scan of the
//      other path, done redundantly by every CTA (a few KB each) so that no
//      CTA waits for another;
//   2. derives kept counts and expert offsets (CTA (0, 0) also writes the
//      counts, offsets, shard statistics and dropped total);
//   3. warp 0 places the block's 32 rank-r assignments: pos = prefix + number
//      of lower lanes with the same expert, kept iff pos < C;
//   4. all eight warps copy the block's kept token rows to xd, four rows per
//      warp, 16-byte vectors with several loads in flight per lane.
// Results equal those of the count + scan + rank + dispatch passes bit for bit.
#include <algorithm>

#include "assign_scan.cuh"

namespace moe {
namespace {

__device__ __forceinline__ uint32_t lane_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
assign_pack_kernel(int64_t Tn, int d, const T* __restrict__ x, const int32_t* __restrict__ idx,
                   const AssignScan a, int32_t* __restrict__ slot_pos, int32_t* __restrict__ row_token,
                   T* __restrict__ xd, int64_t rows_max, int* status) {
    extern __shared__ int sh[];  // [E * k * nblk] prefixes, then offsets [E + 1], routed [E]
    __shared__ int s_row[kAssignBlock];  // row of each lane's assignment, or -1
    dep_wait();
    const int E = a.E, k = a.k;
    const int64_t nblk = a.nblk;
    const int64_t L = (int64_t)k * nblk, n = (int64_t)E * L;
    int* s_off = sh + n;
    int* s_routed = s_off + E + 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kWarpsHere = kThreads / 32;

    for (int64_t i = tid; i < n; i += kThreads) sh[i] = __ldcg(a.hist + i);
    __syncthreads();
    // 1. per expert: exclusive prefixes in (r, b) order, 256 entries a round
    //    held as 8 rows of 32 (entry 32 j + lane in v[j]: conflict-free in
    //    shared memory), each row scanned across the lanes, the rows' totals
    //    added in row order
    for (int e = warp; e < E; e += kWarpsHere) {
        int* h = sh + (int64_t)e * L;
        int running = 0;
        for (int64_t base = 0; base < L; base += 256) {
            const int64_t i0 = base + lane;
            int v[8], incl[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v[j] = i0 + 32 * j < L ? h[i0 + 32 * j] : 0;
                incl[j] = v[j];
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int m = __shfl_up_sync(0xffffffffu, incl[j], o);
                    if (lane >= o) incl[j] += m;
                }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (i0 + 32 * j < L) h[i0 + 32 * j] = running + incl[j] - v[j];
                running += __shfl_sync(0xffffffffu, incl[j], 31);
            }
        }
        if (lane == 0) s_routed[e] = running;
    }
    __syncthreads();
    // 2. kept counts and expert offsets (E <= 256: up to 8 experts a lane)
    if (warp == 0) {
        const int per = (E + 31) / 32;
        int loc = 0, drop = 0;
        for (int j = 0; j < per; ++j) {
            const int e = lane * per + j;
            if (e < E) {
                const int kept = (int)min((int64_t)s_routed[e], a.C);
                loc += kept;
                drop += s_routed[e] - kept;
            }
        }
        int incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int m = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += m;
            drop += __shfl_xor_sync(0xffffffffu, drop, o);
        }
        int run = incl - loc;
        for (int j = 0; j < per; ++j) {
            const int e = lane * per + j;
            if (e < E) {
                s_off[e] = run;
                run += (int)min((int64_t)s_routed[e], a.C);
            }
        }
        if (lane == 31) s_off[E] = incl;
        if (lane == 0 && blockIdx.x == 0 && blockIdx.y == 0 && a.dropped) a.dropped[0] = drop;
    }
    __syncthreads();
    if (blockIdx.x == 0 && blockIdx.y == 0) {
        for (int e = tid; e < E; e += kThreads) {
            a.counts_routed[e] = s_routed[e];
            a.counts_kept[e] = (int)min((int64_t)s_routed[e], a.C);
        }
        for (int e = tid; e <= E; e += kThreads) a.expert_offsets[e] = s_off[e];
        const int per = E / a.D;
        for (int s = tid; s < a.D; s += kThreads) {
            int64_t rs = 0;
            for (int q = s * per; q < (s + 1) * per; ++q) rs += s_routed[q];
            a.shard_routed[s] = (int32_t)rs;
            a.shard_overflow[s] = (int32_t)(rs > a.C_shard ? rs - a.C_shard : 0);
            a.shard_offsets[s] = s_off[s * per];
        }
        if (tid == 0) a.shard_offsets[a.D] = s_off[E];
    }
    // 3. this CTA's block b and rank r
    const int64_t b = blockIdx.x;
    const int r = blockIdx.y;
    if (warp == 0) {
        const int64_t t = b * kAssignBlock + lane;
        int e = -1;
        if (t < Tn) {
            e = idx[(size_t)t * k + r];
            if (e < 0 || e >= E) {
                atomicOr(status, kDevBadIndex);
                e = -1;
            }
        }
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        int row = -1;
        if (t < Tn) {
            int32_t sp = -1;
            if (e >= 0) {
                const int64_t pos = (int64_t)sh[((int64_t)e * k + r) * nblk + b] + __popc(same & lane_lt());
                if (pos < a.C) {
                    sp = (int32_t)pos;
                    const int64_t rr = (int64_t)s_off[e] + pos;
                    if (rr < rows_max) {
                        row = (int)rr;
                        row_token[rr] = (int32_t)t;
                    } else {
                        atomicOr(status, kDevBadIndex);
                    }
                }
            }
            slot_pos[(size_t)t * k + r] = sp;
        }
        s_row[lane] = row;
    }
    __syncthreads();
    // 4. copy the block's kept rows: warp w takes lanes w, w + 8, w + 16, w + 24
    constexpr int VE = vec_elems<T>();
    const int nv = d / VE;
    for (int i = warp; i < kAssignBlock; i += kWarpsHere) {
        const int row = s_row[i];
        if (row < 0) continue;
        const T* src = x + (size_t)(b * kAssignBlock + i) * d;
        T* dst = xd + (size_t)row * d;
        for (int v0 = lane; v0 < nv; v0 += 32 * 4) {
            Vec16 q[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (v0 + 32 * j < nv) q[j] = ld_nc_v16(src + (v0 + 32 * j) * VE);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (v0 + 32 * j < nv) st_v16(dst + (v0 + 32 * j) * VE, q[j]);
        }
    }
}

}  // namespace

bool assign_pack_fits(const Problem& p) {
    const int64_t n = (int64_t)p.E * p.k * p.nblk;
    // shared-memory copy of the histogram, and its redundant reads by every
    // CTA kept to a few MB of L2 traffic
    return p.nblk > 0 && n <= 16384 && n * 4 * p.nblk * p.k <= ((int64_t)32 << 20);
}

cudaError_t launch_assign_pack(const Problem& p, const void* x, const int32_t* topk_idx, const AssignScan& a,
                               int32_t* slot_pos, int32_t* row_token, void* xd, int* status, cudaStream_t s) {
    const size_t smem = ((size_t)p.E * p.k * p.nblk + 2 * (size_t)p.E + 1) * sizeof(int);
    const dim3 grid((unsigned)p.nblk, (unsigned)p.k);
    if (p.dtype == MOE_BF16) {
        auto kern = assign_pack_kernel<__nv_bfloat16>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        return launch_k(kern, grid, dim3(kThreads), smem, s, p.T, p.d, (const __nv_bfloat16*)x, topk_idx, a,
                        slot_pos, row_token, (__nv_bfloat16*)xd, p.rows_max, status);
    }
    auto kern = assign_pack_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(kern, grid, dim3(kThreads), smem, s, p.T, p.d, (const float*)x, topk_idx, a, slot_pos,
                    row_token, (float*)xd, p.rows_max, status);
}

}  // namespace moe
