// ffn_tc.cu -- expert FFN as a grouped bf16 GEMM on the 5th-generation
// tensor cores (tcgen05), fed by TMA, accumulating in tensor memory (TMEM).
//
// "Expert Parallelism" notes page (narrativegoldmine.com), "Components and
// Architecture", expert GEMM: the expert's feed-forward network, a standard
// transformer MLP; formal algorithm, expert computation proportional to the
// tokens each expert received.  "Expert Parallelism and the All-to-All
// Bottleneck" (ashishsrivastav.com), phase 3: each device multiplies only the
// tokens assigned to its local experts.
//
// One persistent launch over the packed, expert-major rows computes both
//   gate/up: h[r, :] = silu(xd[r] W1[e]^T) * (xd[r] W3[e]^T)   (SwiGLU fused
//            into the epilogue: one 128 x 256 accumulator tile holds 128
//            gate columns and the 128 matching up columns)
//   down:    yd[r, :] = h[r] W2[e]^T
// from one tile list: each expert's gate/up tiles, then -- once `lag` more
// tiles have been placed -- its down tiles (the launcher sets `lag` past the
// end of the list, so every down tile follows the last gate/up tile).  A down
// tile reads h rows of one (expert, m-tile pair); its producer waits (bounded,
// acquire) until the four epilogue warps of both CTAs of every gate/up tile
// of that pair have stored their rows and released a counter, then issues its
// TMA loads after a proxy fence.  With the slack the wait is rarely taken, and
// there is no tail between the two GEMMs.  The last CTA to leave zeroes the
// counters for the next launch.
// Ragged expert sizes stay on the device: each CTA reads expert_offsets,
// counts the m-tiles of every expert and walks the tile list persistently.
//
// CTAs run in clusters of two on neighbouring SMs and compute 256 x 256
// tiles together with the 2-SM form of the tensor-core MMA
// (tcgen05.mma.cta_group::2, M = 256): CTA rank r holds the 128 A rows of
// m-tile 2*mp + r and one 128-row half of the 256-row weight tile, and each
// CTA's tensor memory receives its own 128 accumulator rows.  Per k-step an SM
// therefore takes in 32 KB of operands instead of the 48 KB a one-SM
// 128 x 256 tile needs, which is what bounds this kernel, and six stages fit.
// A cluster walks the list of pair tiles (expert, n-tile, m-tile pair) with
// stride = number of clusters.  An m-tile with no rows (odd count) still takes
// part in its pair's loads and MMAs and stores nothing.
//
// When the capacity keeps every expert within one 128-row tile (C <= 128, as
// in layers of many small experts), or within two while the mean load per
// expert fits one, most pair tiles would be half padding; the kernel then
// runs in its one-CTA form instead: no clusters, 128 x 256 tiles with the
// one-SM MMA (tcgen05.mma.cta_group::1, M = 128), each CTA loading its A tile
// and the whole 256-row weight tile (4 stages of 48 KB), release counters per
// (expert, m-tile).  Everything else is shared.
//
// Per CTA (one per SM, 192 threads):
//   warp 0   TMA producer: its A tile [128 x 64] and its B half [128 x 64]
//            per stage (128-byte swizzle, 6 stages of 32 KB); both CTAs'
//            copies complete on the leader CTA's "full" barrier;
//   warp 1   tensor-memory allocation (512 columns = two 128 x 256 fp32
//            accumulators, allocated by both CTAs together) and, in the
//            leader CTA on one lane, the MMA issuer: M=256, N=256, K=16, bf16
//            in, fp32 accumulate; each commit arrives on the barriers of both
//            CTAs (stage free / tile done);
//   warps 2-5 epilogue: tcgen05.ld of this CTA's accumulator rows (warp w
//            reads TMEM lanes 32*(w%4)..+31), activation, bf16 round, staged
//            through shared memory and stored as 128-byte row segments, only
//            the rows that belong to the tile's expert; then both
//            CTAs' epilogue warps release the accumulator on the leader's
//            barrier.
// Every mbarrier wait is bounded in time; on expiry the kernel records
// kDevTimeout in the status word, stops issuing work, waits (bounded) for its
// own copies and MMAs in flight, frees its TMEM and returns.
#include <cuda.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int BM = 128;       // rows per tile (MMA M)
constexpr int BN = 256;       // MMA N (gate/up: 128 + 128 columns)
constexpr int BK = 64;        // K per stage (one 128-byte swizzle atom of bf16)
constexpr int UK = 16;        // K per MMA instruction
constexpr int kMaxStages = 6;
constexpr int kTcThreads = 192;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int TMEM_COLS = 512;
constexpr int kMaxE = 256;
// The kernel runs in one of two forms, CL = CTAs per cluster:
//  CL = 2: pairs of CTAs compute 256-row tiles with the 2-SM MMA; each CTA
//          loads its 128 A rows and half of the 256-row weight tile;
//  CL = 1: single CTAs compute 128-row tiles (M = 128) and load the whole
//          weight tile; used when the capacity keeps every expert within one
//          128-row tile, where a pair tile would be at least half padding.
// stage = own A tile + own share of the weight tile
template <int CL>
__host__ __device__ constexpr int stage_bytes() { return A_BYTES + B_BYTES / CL; }
template <int CL>
__host__ __device__ constexpr int num_stages() { return CL == 2 ? 6 : 4; }
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s: far above any legitimate wait

// shared-memory map after the 1024-aligned stage area
struct __align__(8) TcShared {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int nseg;
    int total_tiles;
    int offs[kMaxE + 1];
    int seg_start[2 * kMaxE + 1];  // first tile of each segment, then the total
    int seg_info[2 * kMaxE];       // kind << 16 | expert (kind 0 gate/up, 1 down)
    int queue[kMaxE];              // experts whose down segments are not placed yet
    int queue_end[kMaxE];          // tile position where each one's gate/up segment ends
};
// Epilogue staging: each epilogue warp writes 64 output columns of its 32
// rows into a padded shared buffer, then stores them four 128-byte row
// segments per instruction (instead of 32 scattered 16-byte pieces).
constexpr int kStgCols = 64;
constexpr int kStgPitch = kStgCols * 2 + 16;  // bytes; rows 16 B apart in bank space
constexpr int kStgWarpBytes = 32 * kStgPitch;
template <int CL>
__host__ __device__ constexpr size_t stg_offset() {
    return (size_t)num_stages<CL>() * stage_bytes<CL>() + ((sizeof(TcShared) + 127) / 128) * 128;
}
template <int CL>
__host__ __device__ constexpr size_t smem_bytes() { return 1024 + stg_offset<CL>() + 4 * kStgWarpBytes; }
static_assert(smem_bytes<2>() <= 227 * 1024 && smem_bytes<1>() <= 227 * 1024, "shared memory");

struct FfnArgs {
    int E, d, ffn, rows_max;
    int n1, k1;    // gate/up: n-tiles of 128 output columns per expert, k-blocks over d
    int n2, k2;    // down: n-tiles of 256 output columns per expert, k-blocks over ffn
    int mp_cap;    // bound on tile units (m-tile pairs, or m-tiles when CL = 1) per expert
    int lag;       // tiles placed between an expert's last gate/up tile and its down tiles
    const int32_t* expert_offsets;  // null: one expert whose rows are 0..rows_max-1
    __nv_bfloat16* h;
    __nv_bfloat16* yd;
    int* status;
    // [0] exit ticket; [1 + e * mp_cap + mp] epilogue-warp releases of the
    // gate/up tiles of (expert e, unit mp); [1 + E * mp_cap] tiles whose
    // loads have all been issued (the progress window).  Zero at launch; the
    // last CTA to leave zeroes it again.
    int* sync;
    int order;  // FfnOrder bits
};

// ---------------------------------------------------------------- PTX ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase of `parity` to complete.  Gives up when another role has
// raised the abort flag or after kTimeoutNs (then raises it and records the
// timeout).  Returns true when the phase completed.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kTimeoutNs) {
            *abort_flag = 1;
            atomicOr(status, kDevTimeout);
            return false;
        }
    }
}
// Drain wait used on the way out: bounded, ignores the abort flag.
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity, int* status) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kTimeoutNs) {
            atomicOr(status, kDevTimeout);
            return;
        }
    }
}
// A tile into this CTA's shared memory, completing its bytes on `bar`, a
// barrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                                 int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"((uint64_t)map), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}
// A tile into this CTA's shared memory, completing on this CTA's barrier.
__device__ __forceinline__ void tma_load_2d_own(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        ::"r"(dst), "l"((uint64_t)map), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}
// shared::cluster address of the same shared variable in CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of both CTAs of the cluster meets here.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle,
// 8-row groups 1024 bytes apart (stride byte offset), leading byte offset
// unused for swizzled K-major (set to 16 B), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// 2-SM MMA, issued by the leader CTA: A rows and B columns come half from
// each CTA of the pair (same shared-memory offsets), D rows land in each CTA's
// own tensor memory.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// One-SM MMA (M = 128): A, B and D all in this CTA.
__device__ __forceinline__ void mma_bf16_one(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit_one(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_local(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Arrive on the barrier at offset `bar` of this CTA once the MMAs issued so
// far complete.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// The same, on the barrier at offset `bar` in every CTA of `mask`.
__device__ __forceinline__ void mma_commit_mc(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(mask)
        : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
        " [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b);
}

// Tile units of an expert with `rows` rows: m-tile pairs (CL = 2) or m-tiles.
template <int CL>
__host__ __device__ __forceinline__ int tile_units(int rows) {
    const int mte = (rows + BM - 1) / BM;
    return CL == 2 ? (mte + 1) / 2 : mte;
}

// Tile -> (kind, expert, m-tile of this CTA, n-tile, unit).  Segment s covers
// the tiles [seg_start[s], seg_start[s+1]) of one kind and expert.  Within a
// segment the units are taken in groups: a group runs through all its
// n-tiles, unit fastest, before the next group starts, so the tiles in flight
// share a weight tile and read the A rows of one group only.  Down tiles use
// smaller groups (their A rows, h, are ffn / d times longer).  Measured on the
// Mixtral 8x7B shape with the progress window: DRAM reads per launch 27.2 GB
// with 16 / 16, 19.9 GB with 16 / 8, 20.1 GB with 16 / 4, 23.1 GB with 8 / 8.
// A unit is an m-tile pair (CL = 2: rank r of the cluster takes m-tile
// 2 * pair + r) or one m-tile (CL = 1).
constexpr int kGroupUnits = 16;     // gate/up segments
constexpr int kGroupUnitsDown = 8;  // down segments
// A remainder of at most this many units joins the group before it instead of
// forming a group of its own, which would stream all of the expert's weights
// once more for a few rows (an expert of 33 units, as on the Mixtral 8x7B shape
// where each expert keeps about 8192 rows: groups 16 + 17 instead of 16 + 16 + 1;
// one launch there read 16.6 GB from DRAM instead of 17.8 GB, in the same time).
constexpr int kMergeUnits = 7;
constexpr int kMergeUnitsDown = 2;
template <int CL>
__device__ __forceinline__ void tile_coords(int tile, const TcShared& S, int n1, int n2, int rank, int& kind,
                                            int& e, int& mt, int& nt, int& mp) {
    int lo = 0, hi = S.nseg - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (S.seg_start[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    kind = S.seg_info[lo] >> 16;
    e = S.seg_info[lo] & 0xffff;
    const int local = tile - S.seg_start[lo];
    const int mpe = tile_units<CL>(S.offs[e + 1] - S.offs[e]);
    const int n = kind == 0 ? n1 : n2;
    const int G = kind == 0 ? kGroupUnits : kGroupUnitsDown;
    int full = mpe / G;  // complete groups
    const int rem = mpe - full * G;
    if (full > 0 && rem > 0 && rem <= (kind == 0 ? kMergeUnits : kMergeUnitsDown)) --full;
    if (local < full * G * n) {
        const int g = local / (G * n), r = local - g * G * n;
        nt = r / G;
        mp = g * G + (r - nt * G);
    } else {
        const int gs = mpe - full * G;  // the last group: the remainder, alone or merged
        const int r = local - full * G * n;
        nt = r / gs;
        mp = full * G + (r - nt * gs);
    }
    mt = CL * mp + rank;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

template <int CL>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_ffn_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
              const __grid_constant__ CUtensorMap tmB3, const __grid_constant__ CUtensorMap tmA2,
              const __grid_constant__ CUtensorMap tmB2, const FfnArgs args) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* stages = smem_raw + ((1024 - (raw & 1023)) & 1023);
    constexpr int STAGES = num_stages<CL>();
    constexpr int STAGE_BYTES = stage_bytes<CL>();
    TcShared& S = *reinterpret_cast<TcShared*>(stages + (size_t)STAGES * STAGE_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = args.E;
    const int rank = CL == 2 ? (int)cluster_rank() : 0;
    const int cluster = blockIdx.x / CL, nclusters = gridDim.x / CL;
    constexpr uint16_t kPairMask = (1u << CL) - 1;
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&S.full[s]), 1);   // leader: its expect_tx; both CTAs' bytes
            mbar_init(smem_u32(&S.empty[s]), 1);  // the leader's MMA commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&S.tfull[b]), 1);
            mbar_init(smem_u32(&S.tempty[b]), 4 * CL);  // leader: epilogue warps of every CTA of the cluster
        }
        mbar_init(smem_u32(&S.drain), 1);
        S.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        if constexpr (CL == 2) {
            // one warp of each CTA of the pair allocates together
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(&S.tmem_base)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(&S.tmem_base)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    // global memory only from here on (earlier kernels on the stream are done,
    // or, with kFfnWaitAtEnd, write and read nothing this launch touches)
    if (!(args.order & kFfnWaitAtEnd)) dep_wait();
    if (warp == 0) {
        // expert offsets; they must be non-decreasing within [0, rows_max],
        // otherwise the kernel records kDevBadIndex and computes nothing
        bool bad = false;
        // no offsets: one expert over all rows_max rows (the shared expert)
        const int32_t* eo = args.expert_offsets;
        for (int e = lane; e <= E; e += 32) {
            const int o = eo ? eo[e] : (e == 0 ? 0 : args.rows_max);
            S.offs[e] = o;
            bad |= o < 0 || o > args.rows_max || (eo && e > 0 && o < eo[e - 1]);
        }
        bad = __any_sync(0xffffffffu, bad);
        __syncwarp();
        if (lane == 0) {
            if (bad && blockIdx.x == 0) atomicOr(args.status, kDevBadIndex);
            // tile list: gate/up segments in expert order; an expert's down
            // segment follows once `lag` further tiles have been placed after
            // its gate/up segment (or at the end)
            int pos = 0, nseg = 0, qh = 0, qt = 0;
            auto pairs = [&](int e) { return tile_units<CL>(S.offs[e + 1] - S.offs[e]); };
            auto place_down = [&](int e) {
                S.seg_start[nseg] = pos;
                S.seg_info[nseg++] = (1 << 16) | e;
                pos += pairs(e) * args.n2;
            };
            for (int e = 0; e < E && !bad; ++e) {
                const int mpe = pairs(e);
                if (mpe == 0) continue;
                S.seg_start[nseg] = pos;
                S.seg_info[nseg++] = e;
                pos += mpe * args.n1;
                S.queue[qt] = e;
                S.queue_end[qt++] = pos;
                while (qh < qt && pos - S.queue_end[qh] >= args.lag) place_down(S.queue[qh++]);
            }
            while (qh < qt) place_down(S.queue[qh++]);
            S.seg_start[nseg] = pos;
            S.nseg = nseg;
            S.total_tiles = pos;
        }
    }
    tc_fence_before();
    __syncthreads();
    // both CTAs' barriers are initialised before either signals the other
    if constexpr (CL == 2) cluster_sync();
    tc_fence_after();

    const int total_tiles = S.total_tiles;
    const uint32_t tmem_base = S.tmem_base;
    volatile int* abort_flag = &S.abort_flag;
    int* status = args.status;
    const int n1 = args.n1, n2 = args.n2;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer --
        int stage = 0;
        uint32_t phase = 0;
        int issued_parity[STAGES];
        for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
        // Progress window: a cluster starts tile t only once t - nclusters
        // tiles have had all their loads issued, so the clusters stay within
        // one tile of each other and the tiles in flight share their A rows
        // and weight tiles in L2.  (Left alone they drift apart: on the
        // Mixtral 8x7B shape by about 20 tiles over the gate/up phase, and the
        // operands in flight then far exceed L2.  With the window and groups
        // of 16 units one launch there read 27 GB from DRAM instead of 49 GB
        // and ran 8% faster.)  The slowest cluster never waits: when it is
        // at its k-th tile, t = cluster + k * nclusters, every cluster has
        // issued at least k tiles, so the count is at least k * nclusters >
        // t - nclusters.  A narrower window could leave it waiting.
        // Short launches (under 32 tiles per cluster) cannot drift far, and
        // layers whose experts hold at most a few tile units (capacity under 8
        // units) have little A to share; both run without the window (the
        // Mixtral-style layer, 16 tiles per cluster: 133 -> 131 us; the
        // 128-expert layers at capacity 160-256 rows lost 2% with it).
        int* const progress = args.sync + 1 + (size_t)args.E * args.mp_cap;
        const int window = total_tiles >= 32 * nclusters && args.mp_cap >= 8 ? nclusters : total_tiles;
        for (int tile = cluster; tile < total_tiles && !*abort_flag; tile += nclusters) {
            if (leader && tile >= window && ld_acquire(progress) < tile - window) {
                const uint64_t t0 = globaltimer();
                while (ld_acquire(progress) < tile - window) {
                    if (*abort_flag) break;
                    if (globaltimer() - t0 > kTimeoutNs) {
                        *abort_flag = 1;
                        atomicOr(status, kDevTimeout);
                        break;
                    }
                }
                if (*abort_flag) break;
            }
            int kind, e, mt, nt, mp;
            tile_coords<CL>(tile, S, n1, n2, rank, kind, e, mt, nt, mp);
            const int a_row = S.offs[e] + mt * BM;
            const CUtensorMap* amap;
            const CUtensorMap* bmap;
            int b_row, k_blocks;
            // second weight half (CL = 1 loads both halves itself)
            const CUtensorMap* bmap2 = nullptr;
            int b_row2 = 0;
            if (kind == 0) {
                // gate/up: rank 0 loads the W1 (gate) rows, rank 1 the W3 (up) rows
                // (one CTA: W1 rows, then W3 rows)
                amap = &tmA1;
                bmap = rank == 1 ? &tmB3 : &tmB1;
                b_row = e * args.ffn + nt * (BN / 2);
                bmap2 = &tmB3;
                b_row2 = b_row;
                k_blocks = args.k1;
            } else {
                // down: rank r loads rows 128 r .. 128 r + 127 of the 256-row W2 tile
                // (one CTA: both)
                amap = &tmA2;
                bmap = &tmB2;
                b_row = e * args.d + nt * BN + rank * (BN / 2);
                bmap2 = &tmB2;
                b_row2 = b_row + BN / 2;
                k_blocks = args.k2;
                // its A rows are h rows of (e, mp): wait until every gate/up
                // tile of them has been stored (four epilogue warps per CTA)
                const int* cnt = args.sync + 1 + (size_t)e * args.mp_cap + mp;
                const int target = 4 * CL * n1;
                if (ld_acquire(cnt) < target) {
                    const uint64_t t0 = globaltimer();
                    while (ld_acquire(cnt) < target) {
                        if (*abort_flag) break;
                        if (globaltimer() - t0 > kTimeoutNs) {
                            *abort_flag = 1;
                            atomicOr(status, kDevTimeout);
                            break;
                        }
                    }
                }
                if (*abort_flag) break;
                // the stores were made through the generic proxy; TMA reads
                // through the async proxy
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            bool ok = true;
            for (int kb = 0; kb < k_blocks; ++kb) {
                if (!wait_phase(smem_u32(&S.empty[stage]), phase ^ 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
                const uint32_t sa = smem_u32(stages + (size_t)stage * STAGE_BYTES);
                if constexpr (CL == 2) {
                    // the leader's full barrier counts both CTAs' bytes of the stage
                    const uint32_t fb = map_to_rank(smem_u32(&S.full[stage]), 0);
                    if (leader) mbar_arrive_expect_tx(smem_u32(&S.full[stage]), CL * STAGE_BYTES);
                    tma_load_2d_pair(sa, amap, fb, kb * BK, a_row);
                    tma_load_2d_pair(sa + A_BYTES, bmap, fb, kb * BK, b_row);
                } else {
                    const uint32_t fb = smem_u32(&S.full[stage]);
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    tma_load_2d_own(sa, amap, fb, kb * BK, a_row);
                    tma_load_2d_own(sa + A_BYTES, bmap, fb, kb * BK, b_row);
                    tma_load_2d_own(sa + A_BYTES + B_BYTES / 2, bmap2, fb, kb * BK, b_row2);
                }
                issued_parity[stage] = (int)phase;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (leader) atomicAdd(progress, 1);
        }
        // this CTA starts no further tile: the next kernel may take the SMs
        // that the CTAs which are done leave (the first trigger of a CTA counts)
        if (args.order & kFfnReleaseNext) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        // copies still in flight must land before the CTA leaves: the leader
        // sees them on its full barriers; the other CTA once the leader's MMA
        // has released the stage they filled
        for (int s = 0; s < STAGES; ++s)
            if (issued_parity[s] >= 0)
                drain_phase(smem_u32(leader ? &S.full[s] : &S.empty[s]), (uint32_t)issued_parity[s], status);
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------------------------- MMA issuer --
        constexpr uint32_t idesc = idesc_bf16(CL * BM, BN);
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = cluster; tile < total_tiles; tile += nclusters) {
            int kind, e, mt, nt, mp;
            tile_coords<CL>(tile, S, n1, n2, rank, kind, e, mt, nt, mp);
            const int k_blocks = kind == 0 ? args.k1 : args.k2;
            if (!wait_phase(smem_u32(&S.tempty[acc]), acc_phase ^ 1u, abort_flag, status)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            bool ok = true;
            for (int kb = 0; kb < k_blocks; ++kb) {
                if (!wait_phase(smem_u32(&S.full[stage]), phase, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = smem_u32(stages + (size_t)stage * STAGE_BYTES);
                const uint32_t sb = sa + A_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / UK; ++kk) {
                    if constexpr (CL == 2)
                        mma_bf16_pair(d_tmem, sw128_desc(sa + kk * UK * 2), sw128_desc(sb + kk * UK * 2), idesc,
                                      (kb | kk) != 0);
                    else
                        mma_bf16_one(d_tmem, sw128_desc(sa + kk * UK * 2), sw128_desc(sb + kk * UK * 2), idesc,
                                     (kb | kk) != 0);
                }
                if constexpr (CL == 2) mma_commit_mc(smem_u32(&S.empty[stage]), kPairMask);
                else mma_commit_one(smem_u32(&S.empty[stage]));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if constexpr (CL == 2) mma_commit_mc(smem_u32(&S.tfull[acc]), kPairMask);
            else mma_commit_one(smem_u32(&S.tfull[acc]));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        // every MMA this thread issued has completed once `drain` flips
        if constexpr (CL == 2) mma_commit(smem_u32(&S.drain));
        else mma_commit_one(smem_u32(&S.drain));
        drain_phase(smem_u32(&S.drain), 0, status);
    } else if (warp >= 2) {
        // --------------------------------------------------- epilogue --
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = cluster; tile < total_tiles; tile += nclusters) {
            int kind, e, mt, nt, mp;
            tile_coords<CL>(tile, S, n1, n2, rank, kind, e, mt, nt, mp);
            // every lane polls; the warp goes on only if all saw the tile done
            // (tcgen05.ld below needs the whole warp), so an abort that races
            // the phase cannot split it
            if (!__all_sync(0xffffffffu, wait_phase(smem_u32(&S.tfull[acc]), acc_phase, abort_flag, status)))
                break;
            tc_fence_after();
            const int rows_e = S.offs[e + 1] - S.offs[e];
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            uint8_t* stg = stages + stg_offset<CL>() + (size_t)q * kStgWarpBytes;
            const int n_out = kind == 0 ? args.ffn : args.d;
            const int ncols = kind == 0 ? BN / 2 : BN;  // output columns of this tile
            const int col0 = nt * ncols;
            __nv_bfloat16* obase =
                (kind == 0 ? args.h : args.yd) + (size_t)(S.offs[e] + mt * BM + q * 32) * n_out;
            const int rows_left = rows_e - (mt * BM + q * 32);  // this warp's rows [0, rows_left) are stored
#pragma unroll 1
            for (int part = 0; part < ncols; part += kStgCols) {
#pragma unroll 1
                for (int c = 0; c < kStgCols; c += 16) {
                    uint32_t pk[8];
                    if (kind == 0) {
                        // SwiGLU: accumulator columns 0-127 are gate, 128-255 up
                        uint32_t g[16], u[16];
                        tmem_ld16(taddr + part + c, g);
                        tmem_ld16(taddr + BN / 2 + part + c, u);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float h2[2];
#pragma unroll
                            for (int z = 0; z < 2; ++z) {
                                const float a = __uint_as_float(g[2 * j + z]);
                                const float b = __uint_as_float(u[2 * j + z]);
                                h2[z] = __fdividef(a, 1.0f + __expf(-a)) * b;
                            }
                            pk[j] = pack_bf16x2(h2[0], h2[1]);
                        }
                    } else {
                        uint32_t a[16];
                        tmem_ld16(taddr + part + c, a);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            pk[j] = pack_bf16x2(__uint_as_float(a[2 * j]), __uint_as_float(a[2 * j + 1]));
                    }
                    uint32_t* srow = reinterpret_cast<uint32_t*>(stg + lane * kStgPitch + c * 2);
                    *reinterpret_cast<uint4*>(srow) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    *reinterpret_cast<uint4*>(srow + 4) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
                __syncwarp();
                // four rows of 128 B per instruction; rows past the expert and
                // columns past n_out are not stored
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = 4 * i + (lane >> 3), ch = lane & 7;
                    const int col = col0 + part + ch * 8;
                    if (r < rows_left && col < n_out) {
                        const uint4 v = *reinterpret_cast<const uint4*>(stg + r * kStgPitch + ch * 16);
                        st_v16(obase + (size_t)r * n_out + col, Vec16{{v.x, v.y, v.z, v.w}});
                    }
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CL == 2) mbar_arrive_cluster(map_to_rank(smem_u32(&S.tempty[acc]), 0));
                else mbar_arrive_local(smem_u32(&S.tempty[acc]));
            }
            if (kind == 0) {
                // release this warp's h rows to the down tiles that read them:
                // the warp barrier orders every lane's stores before lane 0's
                // release-add (gpu scope), whose release covers them, so the
                // consumer's acquire of the counter sees all 32 lanes' rows
                __syncwarp();
                if (lane == 0)
                    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(
                                     args.sync + 1 + (size_t)e * args.mp_cap + mp),
                                 "r"(1)
                                 : "memory");
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }
    tc_fence_before();
    __syncthreads();
    // no CTA leaves (or frees tensor memory) while its peer may still read
    // its operands, write its accumulators or arrive on its barriers
    if constexpr (CL == 2) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (CL == 2)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                         "r"(TMEM_COLS)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                         "r"(TMEM_COLS)
                         : "memory");
    }
    // not done before the kernel this launch did not wait for at its start
    if (args.order & kFfnWaitAtEnd) dep_wait();
    // the last CTA out zeroes the release counters for the next launch
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(args.sync, 1) == (int)gridDim.x - 1) {
            __threadfence();
            const int n = 2 + E * args.mp_cap;  // the counters and the progress window
            for (int i = 1; i < n; ++i) args.sync[i] = 0;
            __threadfence();
            args.sync[0] = 0;
        }
    }
}

// ------------------------------------------------------------- host ------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

// Looked up once per process (a function-local static: thread-safe).
EncodeTiledFn get_encoder() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return (EncodeTiledFn)ptr;
        return nullptr;
    }();
    return fn;
}

// 2-D bf16 map over a row-major [rows, cols] matrix, box [box_rows, 64], 128 B swizzle.
bool make_map(EncodeTiledFn enc, CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
              uint32_t box_rows) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool encode_row_tiles(CUtensorMap* m, const void* base, int dtype, uint64_t rows, uint64_t cols, uint32_t box_cols,
                      uint32_t box_rows) {
    EncodeTiledFn enc = get_encoder();
    if (!enc) return false;
    const uint64_t eb = dtype == MOE_BF16 ? 2 : 4;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * eb};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, dtype == MOE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
               const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// Both queries below run once per process (function-local statics, so
// thread-safe); every device the library drives is the same part.
int num_sms() {
    static const int n = []() {
        int dev = 0, v = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        return v;
    }();
    return n;
}

// Launch of form CL (clusters of CL CTAs) with programmatic dependent launch.
template <int CL, typename... KArgs, typename... Args>
cudaError_t launch_form(void (*kern)(KArgs...), unsigned clusters, cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(clusters * CL);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem_bytes<CL>();
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CL;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CL == 2 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Clusters of form CL that can be resident at once (one CTA per SM).
template <int CL>
int max_clusters() {
    static const int n = []() {
        int c = 0;
        if constexpr (CL == 2) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(num_sms() / CL * CL));
            cfg.blockDim = dim3(kTcThreads);
            cfg.dynamicSmemBytes = smem_bytes<CL>();
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = CL;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&c, tc_ffn_kernel<CL>, &cfg) != cudaSuccess || c <= 0)
                c = num_sms() / CL;
        } else {
            int per_sm = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_ffn_kernel<CL>, kTcThreads,
                                                              smem_bytes<CL>()) != cudaSuccess ||
                per_sm <= 0)
                per_sm = 1;
            c = per_sm * num_sms();
        }
        return c;
    }();
    return n;
}

template <int CL>
cudaError_t launch_ffn_form(const Problem& p, const CUtensorMap& mA1, const CUtensorMap& mB1, const CUtensorMap& mB3,
                            const CUtensorMap& mA2, const CUtensorMap& mB2, FfnArgs a, cudaStream_t s) {
    // per device, so set on every launch (a cheap host call)
    cudaError_t e1 =
        cudaFuncSetAttribute(tc_ffn_kernel<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<CL>());
    if (e1 != cudaSuccess) return e1;
    // upper bound of tile units over all experts: sum_e units(n_e) with
    // m-tiles mt_e = ceil(n_e / BM), n_e <= C, sum_e mt_e <= ceil(rows_max / BM) + E
    const int64_t mt_cap = ceil_div(p.C, BM);
    const int64_t unit_cap = CL == 2 ? ceil_div(mt_cap, 2) : mt_cap;
    const int64_t mt_total = ceil_div(p.rows_max, BM) + (int64_t)p.E;
    const int64_t unit_bound =
        std::min<int64_t>((int64_t)p.E * unit_cap, CL == 2 ? ceil_div(mt_total + (int64_t)p.E, 2) : mt_total);
    a.mp_cap = (int)unit_cap;
    // all clusters must be resident at once (down tiles wait on gate/up tiles
    // of other clusters), so never more than the occupancy allows
    const unsigned clusters =
        (unsigned)std::max<int64_t>(1, std::min<int64_t>(max_clusters<CL>(), unit_bound * (a.n1 + a.n2)));
    return launch_form<CL>(tc_ffn_kernel<CL>, clusters, s, mA1, mB1, mB3, mA2, mB2, a);
}

}  // namespace

size_t ffn_sync_ints(const Problem& p) {
    // the exit ticket, one counter per (expert, tile unit) -- m-tile pairs, or
    // m-tiles for the one-CTA form; sized for m-tiles, the larger count, so
    // that either form fits -- and the progress window
    return 2 + (size_t)p.E * (size_t)ceil_div(p.C, BM);
}

cudaError_t launch_ffn_tc(const Problem& p, const void* xd, const int32_t* expert_offsets,
                          const void* W1, const void* W3, const void* W2, void* h, void* yd,
                          int* status, int* sync, cudaStream_t s, int order) {
    if (p.rows_max == 0) return cudaSuccess;
    EncodeTiledFn enc = get_encoder();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap mA1, mB1, mB3, mA2, mB2;
    const uint64_t rows = (uint64_t)p.rows_max, E = (uint64_t)p.E;
    if (!make_map(enc, &mA1, xd, rows, p.d, BM) || !make_map(enc, &mB1, W1, E * p.ffn, p.d, BN / 2) ||
        !make_map(enc, &mB3, W3, E * p.ffn, p.d, BN / 2) || !make_map(enc, &mA2, h, rows, p.ffn, BM) ||
        !make_map(enc, &mB2, W2, E * p.d, p.ffn, BN / 2))
        return cudaErrorInvalidValue;
    FfnArgs a{};
    a.E = p.E;
    a.d = p.d;
    a.ffn = p.ffn;
    a.rows_max = (int)p.rows_max;
    a.n1 = (int)ceil_div(p.ffn, BN / 2);
    a.k1 = (int)ceil_div(p.d, BK);
    a.n2 = (int)ceil_div(p.d, BN);
    a.k2 = (int)ceil_div(p.ffn, BK);
    a.expert_offsets = expert_offsets;
    a.h = (__nv_bfloat16*)h;
    a.yd = (__nv_bfloat16*)yd;
    a.status = status;
    a.sync = sync;
    a.order = order;
    // Down tiles are several times longer than gate/up tiles (K = ffn vs d), so
    // they all go after the last gate/up tile: every cluster then ends on one
    // or two of them instead of a few clusters finishing the last expert's.
    a.lag = 1 << 30;
    // one-CTA tiles when the capacity keeps every expert within one 128-row
    // tile (a pair tile would be at least half padding), or within two while
    // the mean load per expert fits one (most pair tiles would be half
    // padding; measured at 128 experts, capacity 160 and 256 rows: 650 ->
    // 631 us, while a Zipf-skewed 64-expert layer with a mean of 256 rows
    // per expert ran 4% slower in this form); pairs otherwise
    const bool thin = p.C <= BM || (p.C <= 2 * BM && p.T * p.k <= (int64_t)p.E * BM);
    if (thin) return launch_ffn_form<1>(p, mA1, mB1, mB3, mA2, mB2, a, s);
    return launch_ffn_form<2>(p, mA1, mB1, mB3, mA2, mB2, a, s);
}

}  // namespace moe
