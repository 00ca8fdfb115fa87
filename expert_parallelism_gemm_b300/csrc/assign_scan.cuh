// assign_scan.cuh -- the second half of the slot-assignment count pass, run by
// whichever CTA of a counting kernel finishes last.
//
// "Expert Parallelism" notes page (narrativegoldmine.com), "Capacity Factor
// and Token Dropping": an expert keeps at most C assignments; "Expert
// Parallelism" (theinfinity.ai), capacity paragraph: per-device overflow
// max(0, p*B*k - C_shard), with p*B*k the assignments routed to the device;
// "Expert Parallelism and the All-to-All Bottleneck" (ashishsrivastav.com):
// experts sit on devices in contiguous blocks.
//
// The counting kernels (the standalone count kernel and the router's fused
// tail) write hist[e][r][b] = number of rank-r choices of expert e among the
// tokens of block b (kAssignBlock tokens), then call finish_assign_scan().
// Every CTA bumps an integer ticket; the last one turns hist into exclusive
// prefixes in (r, b) order per expert -- the priority order rank first, then
// token -- and writes the routed and kept counts, expert and shard offsets,
// shard statistics and the dropped total.  Integer arithmetic only, so the
// result does not depend on which CTA finishes last.
//
// Second pass of overflow rerouting (`second` set): hist holds the counts of
// the rerouted assignments; each expert's prefixes start from its first-pass
// kept count (read from counts_kept), kept becomes min(first-pass kept +
// rerouted, C), counts_routed is left as the first pass wrote it, and
// `rerouted` receives the number of rerouted assignments that found room.
#pragma once

#include "common.cuh"

namespace moe {

struct AssignScan {
    int32_t* hist;  // [E][k][nblk]; counts in, exclusive prefixes out
    int32_t* counts_routed;
    int32_t* counts_kept;
    int32_t* expert_offsets;
    int32_t* shard_offsets;
    int32_t* shard_routed;
    int32_t* shard_overflow;
    int32_t* dropped;  // may be null
    unsigned* ticket;  // zero before the launch; reset to zero by the last CTA
    int E, D, k;
    int64_t nblk, C, C_shard;
    int32_t* rerouted = nullptr;  // second pass only; may be null
    bool second = false;
    bool defer = false;  // the router writes the histogram only; a later kernel scans it
};

// Call from every thread of every CTA after the CTA's hist entries are
// written (no thread may have returned early).  Works for any block size
// that is a multiple of 32.
// kScanDepth: histogram chunks each warp reads ahead of the one it scans
// (registers: 8 per chunk per thread; 0 reads each chunk just before its scan).
template <int kScanDepth = 4>
__device__ __forceinline__ void finish_assign_scan(const AssignScan& a) {
    __shared__ bool s_last;
    __shared__ int s_routed[256];
    __shared__ int s_kept_off[257];
    __shared__ int s_moved[256];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        s_last = atomicAdd(a.ticket, 1u) == gridDim.x * gridDim.y * gridDim.z - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int64_t L = (int64_t)a.k * a.nblk;
    // one warp per expert: exclusive scan of its k * nblk counts, in place,
    // 256 entries per chunk held as 8 rows of 32 (entry 32 j + lane of the
    // chunk in v[j]), so every load and store of a warp covers 128
    // contiguous bytes.  Each row is scanned across the lanes, two rows at a
    // time packed in the halves of one word: an entry counts the tokens of
    // one 32-token block, so a row's prefixes stay below 2^16.  The rows'
    // totals are then added in row order.  A warp's chunks, expert after
    // expert, are read kScanDepth ahead of the one being scanned.  Every
    // entry is read before it is overwritten: chunk c is loaded while chunk
    // c - kScanDepth is scanned, and stored only when its own turn comes.
    static_assert(kAssignBlock * 32 < (1 << 16), "row prefixes must fit 16 bits");
    const int nch = L > 0 ? (int)((L + 255) / 256) : 1;  // chunks per expert (an empty one still reports)
    const int ncw = (warp < a.E ? (a.E - 1 - warp) / nwarps + 1 : 0) * nch;  // chunks of this warp
    // the next chunk to read: its expert and index within the expert
    int ld_e = warp, ld_ch = 0, ld_c = 0;
    auto load_next = [&](int (&v)[8]) {
        if (ld_c < ncw) {
            const int64_t i0 = (int64_t)ld_ch * 256 + lane;
            const int32_t* h = a.hist + (size_t)ld_e * L;
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = i0 + 32 * j < L ? __ldcg(h + i0 + 32 * j) : 0;
            ++ld_c;
            if (++ld_ch == nch) {
                ld_ch = 0;
                ld_e += nwarps;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = 0;
        }
    };
    int buf[kScanDepth + 1][8];
#pragma unroll
    for (int q = 0; q < kScanDepth; ++q) load_next(buf[q]);
    int running = 0, first_kept = 0;
    int e = warp, ch = 0;  // the chunk being scanned
    for (int c = 0; c < ncw; ++c) {
        load_next(buf[kScanDepth]);
        int32_t* h = a.hist + (size_t)e * L;
        if (ch == 0) {
            first_kept = a.second ? __ldcg(a.counts_kept + e) : 0;
            running = first_kept;
        }
        const int64_t i0 = (int64_t)ch * 256 + lane;
        uint32_t pk[4];  // rows j and j + 4
#pragma unroll
        for (int j = 0; j < 4; ++j) pk[j] = (uint32_t)buf[0][j] | ((uint32_t)buf[0][j + 4] << 16);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t n = __shfl_up_sync(0xffffffffu, pk[j], o);
                if (lane >= o) pk[j] += n;
            }
        uint32_t tot[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) tot[j] = __shfl_sync(0xffffffffu, pk[j], 31);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int incl = (int)(j < 4 ? pk[j] & 0xffffu : pk[j - 4] >> 16);
            if (i0 + 32 * j < L) h[i0 + 32 * j] = running + incl - buf[0][j];
            running += (int)(j < 4 ? tot[j] & 0xffffu : tot[j - 4] >> 16);
        }
#pragma unroll
        for (int q = 0; q < kScanDepth; ++q)
#pragma unroll
            for (int j = 0; j < 8; ++j) buf[q][j] = buf[q + 1][j];
        if (ch == nch - 1 && lane == 0) {
            const int kept = (int)min((int64_t)running, a.C);
            const int routed = a.second ? __ldcg(a.counts_routed + e) : running;
            s_routed[e] = routed;
            s_kept_off[e] = kept;
            s_moved[e] = kept - first_kept;
            if (!a.second) a.counts_routed[e] = routed;
            a.counts_kept[e] = kept;
        }
        if (++ch == nch) {
            ch = 0;
            e += nwarps;
        }
    }
    __syncthreads();
    if (warp == 0) {
        // expert offsets: exclusive scan of the kept counts (E <= 256)
        const int per = (a.E + 31) / 32;
        int loc_kept = 0, loc_drop = 0, loc_moved = 0;
        for (int j = 0; j < per; ++j) {
            const int e = lane * per + j;
            if (e < a.E) {
                loc_kept += s_kept_off[e];
                loc_drop += s_routed[e] - s_kept_off[e];
                loc_moved += s_moved[e];
            }
        }
        int incl = loc_kept, drop = loc_drop, moved = loc_moved;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
            drop += __shfl_xor_sync(0xffffffffu, drop, o);
            moved += __shfl_xor_sync(0xffffffffu, moved, o);
        }
        int run = incl - loc_kept;
        for (int j = 0; j < per; ++j) {
            const int e = lane * per + j;
            if (e < a.E) {
                const int kept = s_kept_off[e];
                s_kept_off[e] = run;
                a.expert_offsets[e] = run;
                run += kept;
            }
        }
        if (lane == 31) {
            s_kept_off[a.E] = incl;
            a.expert_offsets[a.E] = incl;
        }
        if (lane == 0) {
            if (a.dropped) a.dropped[0] = drop;
            if (a.second && a.rerouted) a.rerouted[0] = moved;
            *a.ticket = 0u;  // ready for the next call on this scratch
        }
    }
    __syncthreads();
    const int per = a.E / a.D;
    for (int s = threadIdx.x; s < a.D; s += blockDim.x) {
        int64_t rs = 0;
        for (int q = s * per; q < (s + 1) * per; ++q) rs += s_routed[q];
        a.shard_routed[s] = (int32_t)rs;
        a.shard_overflow[s] = (int32_t)(rs > a.C_shard ? rs - a.C_shard : 0);
        a.shard_offsets[s] = s_kept_off[s * per];
    }
    if (threadIdx.x == 0) a.shard_offsets[a.D] = s_kept_off[a.E];
}

}  // namespace moe
