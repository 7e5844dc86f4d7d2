// K1: tcgen05 tree-verify MLA-absorb attention for bf16 inputs (fp32 accumulate).
//
// What it computes is the definition of page "The Verify-Attn Kernel: A Single File
// Write ..." (section "The Design Journey: From Concept to CUDA"): per row (b,i,h)
// the scores s_j = scale * (q_nope . c_kv[j] + q_pe . k_pe[j]) over the visible keys
// (shared prefix, tree ancestors, self), a softmax over them, and the latent output
// sum_j p_j c_kv[j] with its log-sum-exp. The long-context tiling the pages plan
// (online softmax over key blocks, page "The Verify-Attn Kernel ...", section
// "Design Decisions and Trade-Offs") is how the key loop runs here.
//
// GB300 design (differs from the pages' SIMT block-per-(b,h,i) kernel):
//  * All heads x tree queries of one sequence form the M dimension: a work unit is
//    128 consecutive query rows of one sequence and a range of 128-key blocks.
//    Every head shares the latent cache, so S = Q K^T and O = P V are dense
//    contractions on the 5th-generation tensor cores.
//  * A unit runs on a 2-CTA cluster split by role, because one SM cannot hold
//    Q (128 x 576 bf16), the 128 x 512 fp32 output accumulator and the scores:
//      - rank 0, the S-CTA: Q_nope lives in tensor memory as the MMA A operand
//        (256 columns), Q_pe in shared memory; per key block it computes
//        S[128 x 128] into one of two TMEM score buffers (256 columns), runs the
//        online softmax (one thread per row), and writes P (bf16) straight into
//        the O-CTA's shared memory over DSMEM;
//      - rank 1, the O-CTA: the whole fp32 O[128 x 512] accumulator occupies its
//        512 TMEM columns; per block it issues O += P V (N = 256, two halves) with
//        V = c_kv tiles fetched by TMA, and rescales rows of O in TMEM on the rare
//        occasions the running maximum grows past the threshold below.
//  * Key blocks are aligned to END at kv_len, so no row at or beyond
//    prefix_len + T is ever fetched; the leading block may start before row 0,
//    where TMA fills zeros and the mask removes the keys. Only blocks holding tree
//    keys (or those leading zeros) evaluate the mask, from packed ancestor bits.
//  * Online softmax in base 2 with a lazy maximum: the running max m used for
//    exp2(x - m) is only raised when a block's max exceeds it by more than 8, so
//    p <= 256 and O is rescaled only then (exact either way: o = O / l).
//  * Every wait is bounded; on a lost arrival the kernel records a status in the
//    caller's error word, drains its own in-flight copies and MMAs, frees TMEM and
//    returns (no trap, no hang).
#include "kdt_internal.cuh"
#include "tc_ptx.cuh"

#include <math.h>
#include <string.h>

// Optional per-block stage timestamps for pipeline analysis. Compiled out unless a
// tracing build defines the hook before including this file.
#ifndef KDT_TC_TRACE
#define KDT_TC_TRACE(event, block) ((void)0)
#endif

namespace kdt {
namespace {

using namespace tc;

// Trace events (rank 0 = S-CTA, rank 1 = O-CTA).
enum TraceEvent {
    kEvSMmaStart = 0,    // S MMA thread: score buffer free, starts issuing block
    kEvSMmaIssued,       // S MMA thread: all chunks of the block issued
    kEvSoftmaxIn,        // softmax warp 4: scores of the block in TMEM
    kEvSoftmaxLoaded,    // softmax warp 4: scores loaded, buffer released
    kEvSoftmaxSlot,      // softmax warp 4: P slot free in the O-CTA
    kEvSoftmaxSent,      // softmax warp 4: P written and published
    kEvCorrIn,           // correction warp 4: P of the block arrived
    kEvOMmaStart,        // O MMA thread: block checked, starts issuing P.V
    kEvOMmaIssued,       // O MMA thread: P.V of the block issued
    kNumTraceEvents
};

constexpr int kRows = 128;             // query rows per unit (MMA M)
constexpr int kKeys = 128;             // keys per block (S MMA N, P.V K)
constexpr int kThreads = 384;          // 12 warps
constexpr int kChunkBytes = kKeys * 128;          // [128 keys x 64 dims] bf16, 128B-swizzled: 16 KB
// TMA throughput per SM grows with the bytes of one request (fixed cost per box),
// so key tiles travel as 32 KB requests (two 64-dim sub-tiles) and value halves as
// 64 KB requests (four sub-tiles), from a 4-D view of the cache.
constexpr int kSlotBytes = 2 * kChunkBytes;       // S-CTA ring slot: 128 keys x 128 dims
constexpr int kSlotsPerBlock = 5;                 // 4 latent slots + 1 rope slot (half used)
constexpr int kNK = 4;                            // S-CTA key ring slots (128 KB)
constexpr int kPBytes = kRows * kKeys * 2;        // P tile: 32 KB (two 128B-swizzled halves)
constexpr int kNP = 2;                            // P slots in the O-CTA
constexpr int kVHalfBytes = 4 * kChunkBytes;      // V for 256 latent columns: 64 KB
constexpr int kNV = 2;                            // V half slots in the O-CTA
constexpr uint64_t kWaitLimit = 200000000ull;     // ns a wait may poll before giving up
constexpr float kRescaleThreshold = 8.0f;         // log2 units

// Shared-memory layout (same offsets in both CTAs of the cluster; roles use
// different parts). All tiles 1024-byte aligned for the 128B swizzle.
constexpr int kOffQpe = 0;                                  // S: Q_pe tile 16 KB
constexpr int kOffKRing = kOffQpe + kChunkBytes;            // S: 4 x 32 KB
constexpr int kOffPStage = kOffKRing + kNK * kSlotBytes;    // S: 2 x 32 KB staging of P
constexpr int kOffAStage = kOffPStage + kNP * kPBytes;      // S: [kNP][128] alpha staging
constexpr int kOffRowMax = kOffAStage + kNP * kRows * 4;    // S: [2 blocks][2 halves][128] partial maxima
constexpr int kOffLSum = kOffRowMax + 2 * 2 * kRows * 4;    // S: [128] partial row sums
constexpr int kOffP = 0;                                    // O: 2 x 32 KB
constexpr int kOffV = kOffP + kNP * kPBytes;                // O: 2 x 64 KB
constexpr int kOffAlpha = kOffV + kNV * kVHalfBytes;        // O: [kNP][128] floats
constexpr int kOffStats = kOffAlpha + kNP * kRows * 4;      // O: [128] x (m, l)
constexpr int kSEnd = kOffLSum + kRows * 4;
constexpr int kOEnd = kOffStats + kRows * 8;
constexpr uint32_t kPTx = kPBytes + kRows * 4;              // bytes landing in a P slot per block
constexpr int kTileBytes = kSEnd > kOEnd ? kSEnd : kOEnd;
constexpr int kSmemBytes = kTileBytes + 1024;               // + alignment slack

struct Barriers {
    // S-CTA
    uint64_t kfull[kNK], kempty[kNK];
    uint64_t sfull[2], sempty[2];
    uint64_t qpe_full, q_ready;
    uint64_t pempty[kNP];          // arrived by the O-CTA's MMA commits (multicast)
    // O-CTA
    uint64_t pfull[kNP];           // arrived remotely by the S-CTA softmax warps
    uint64_t vfull[kNV], vempty[kNV];
    // Per-block handshake between the correction warps and the MMA thread. Each pair
    // strictly alternates (request -> response), so every parity wait is exact.
    uint64_t corr_done;            // correction warps -> MMA: block j checked (need_rescale set)
    uint64_t ack;                  // MMA -> correction warps: flag of block j read
    uint64_t o_ready;              // MMA -> correction warps: all P.V before block j complete
    uint64_t rescaled;             // correction warps -> MMA: rows of O rescaled
    uint64_t stats_full;
    uint64_t sync_bar;             // MMA thread's own completion probe (mid-stream)
    uint64_t drain;                // completion probe for this CTA's own MMAs before TMEM is freed
    int need_rescale;
    uint32_t tmem_base;
    int abort_flag;
};

struct TcParams {
    int B, T, H, W;
    int rows_seq;          // T*H
    int row_tiles;         // ceil(rows_seq / 128)
    int num_splits, blocks_per_split;
    int64_t rows_total;
    const __nv_bfloat16 *q_nope;
    const int32_t *prefix_len;
    const uint32_t *vis;
    float scale_log2;
    float *out, *lse, *part_o, *part_lse;
    int32_t *err;
    int tail_tiles, tail_splits;   // tail splitting (see VerifyParams); 0 = off
};

__device__ __forceinline__ bool aborted(const Barriers &bar) {
    return *reinterpret_cast<const volatile int *>(&bar.abort_flag) != 0;
}

// Wait until every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void drain_mmas(Barriers &bar) {
    mma_commit(&bar.drain);
    mbar_wait(&bar.drain, 0, kWaitLimit);
}

// Order this thread's DSMEM stores (generic proxy) before a later release-arrive
// by another lane, and make them visible to the peer's tensor-core reads.
__device__ __forceinline__ void publish_remote_stores() {
    asm volatile("fence.proxy.async;" ::: "memory");
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
}

__device__ __forceinline__ void set_abort(Barriers &bar, int32_t *err, int code) {
    bar.abort_flag = 1;
    if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ bool wait_or_abort(Barriers &bar, uint64_t *b, uint32_t parity, int32_t *err,
                                              int code) {
    if (*reinterpret_cast<volatile int *>(&bar.abort_flag)) return false;
    if (mbar_wait(b, parity, kWaitLimit)) return true;
    set_abort(bar, err, code);
    return false;
}

__device__ __forceinline__ bool wait_cluster_or_abort(Barriers &bar, uint64_t *b, uint32_t parity, int32_t *err,
                                                      int code) {
    if (*reinterpret_cast<volatile int *>(&bar.abort_flag)) return false;
    if (mbar_wait_cluster(b, parity, kWaitLimit)) return true;
    set_abort(bar, err, code);
    return false;
}

// Warp-uniform waits: every lane polls, and the warp proceeds only if all lanes saw
// the phase complete, so warp-collective tcgen05 loads/stores after a wait are never
// reached by part of a warp.
__device__ __forceinline__ bool warp_wait(Barriers &bar, uint64_t *b, uint32_t parity, int32_t *err, int code) {
    return __all_sync(0xffffffffu, wait_or_abort(bar, b, parity, err, code));
}

__device__ __forceinline__ bool warp_wait_cluster(Barriers &bar, uint64_t *b, uint32_t parity, int32_t *err,
                                                  int code) {
    return __all_sync(0xffffffffu, wait_cluster_or_abort(bar, b, parity, err, code));
}

// Copy `bytes` (multiple of 16) from this CTA's shared memory to the same-layout
// buffer in CTA `rank`, completing as transaction bytes on that CTA's barrier.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_local, const void *src, uint32_t bytes,
                                                  uint64_t *bar_local, uint32_t rank) {
    uint32_t dst, mbar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(dst) : "r"(dst_local), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(mbar) : "r"(smem_u32(bar_local)), "r"(rank));
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "r"(smem_u32(src)), "r"(bytes), "r"(mbar)
                 : "memory");
}

// Named barrier over `count` threads that also ORs a per-thread flag across them.
template <int kId, int kCount>
__device__ __forceinline__ bool barrier_or(bool flag) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pin, pout;\n\t"
        "setp.ne.u32 pin, %1, 0;\n\t"
        "bar.red.or.pred pout, %2, %3, pin;\n\t"
        "selp.u32 %0, 1, 0, pout;\n\t}"
        : "=r"(r)
        : "r"(flag ? 1u : 0u), "n"(kId), "n"(kCount)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// TMEM-address helpers: lane field in bits [31:16].
__device__ __forceinline__ uint32_t tmem_lane_addr(uint32_t base, int warp, uint32_t col) {
    return base + ((uint32_t)(32 * (warp & 3)) << 16) + col;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    verify_tc_kernel(const __grid_constant__ CUtensorMap map_ckv2, const __grid_constant__ CUtensorMap map_ckv4,
                     const __grid_constant__ CUtensorMap map_kpe, const __grid_constant__ CUtensorMap map_qpe,
                     const TcParams p) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ Barriers bar;
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~static_cast<uintptr_t>(1023));
    const uint32_t rank = cluster_ctarank();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- unit -> (b, row tile, key range) ------------------------------------------
    // Uniform mode: unit = (tile, split) with num_splits key ranges per tile. Tail mode
    // (tail_splits > 0, num_splits == 1): tiles before the last tail_tiles are whole
    // units; each of the last tail_tiles tiles is cut into tail_splits key ranges so the
    // final wave of clusters is as full as the others.
    const int unit = blockIdx.x >> 1;
    const int tiles = p.B * p.row_tiles;
    const int first_tail = tiles - p.tail_tiles;
    int tile, split, nsplit;
    if (p.tail_splits > 0) {
        if (unit < first_tail) {
            tile = unit;
            split = 0;
            nsplit = 1;
        } else {
            tile = first_tail + (unit - first_tail) / p.tail_splits;
            split = (unit - first_tail) % p.tail_splits;
            nsplit = p.tail_splits;
        }
    } else {
        tile = unit / p.num_splits;
        split = unit % p.num_splits;
        nsplit = p.num_splits;
    }
    const int rt = tile % p.row_tiles;
    const int b = tile / p.row_tiles;
    const int P = p.prefix_len[b];
    const int kv_len = P + p.T;
    const int nblk = (kv_len + kKeys - 1) / kKeys;
    const int bps = p.tail_splits > 0 ? (nblk + nsplit - 1) / nsplit : p.blocks_per_split;
    const int kb0 = split * bps;
    const int kb1 = min(nblk, kb0 + bps);
    const int nb = kb1 > kb0 ? kb1 - kb0 : 0;       // blocks of this unit (0: empty split)
    const int key_base = kv_len - nblk * kKeys;     // first key of block 0 (<= 0)
    const int r0 = rt * kRows;

    // ---- set-up: barriers, TMEM ------------------------------------------------------
    if (threadIdx.x == 0) {
        for (int i = 0; i < kNK; ++i) { mbar_init(&bar.kfull[i], 1); mbar_init(&bar.kempty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&bar.sfull[i], 1); mbar_init(&bar.sempty[i], 8); }
        mbar_init(&bar.qpe_full, 1);
        mbar_init(&bar.q_ready, 8);
        for (int i = 0; i < kNP; ++i) { mbar_init(&bar.pempty[i], 1); mbar_init(&bar.pfull[i], 1); }
        for (int i = 0; i < kNV; ++i) { mbar_init(&bar.vfull[i], 1); mbar_init(&bar.vempty[i], 1); }
        mbar_init(&bar.corr_done, 1);
        mbar_init(&bar.ack, 1);
        mbar_init(&bar.o_ready, 1);
        mbar_init(&bar.rescaled, 1);
        mbar_init(&bar.sync_bar, 1);
        bar.need_rescale = 0;
        mbar_init(&bar.stats_full, 4);
        mbar_init(&bar.drain, 1);
        bar.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&bar.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();            // peer barriers initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem = bar.tmem_base;

    if (rank == 0) {
        // =============================== S-CTA ===============================
        unsigned char *qpe_tile = smem + kOffQpe;
        unsigned char *kring = smem + kOffKRing;
        const uint32_t tmem_q = tmem;                 // Q_nope: columns [0, 256)
        const uint32_t tmem_s0 = tmem + 256;          // score buffers at 256 and 384
        if (warp == 0) {
            // ---------------- TMA producer: Q_pe once, then key chunks ----------------
            if (elect_one() && nb > 0) {
                tma_prefetch_desc(&map_ckv2);
                tma_prefetch_desc(&map_kpe);
                mbar_arrive_expect_tx(&bar.qpe_full, kChunkBytes);
                tma_load_2d(qpe_tile, &map_qpe, &bar.qpe_full, 0, (int)((int64_t)b * p.rows_seq + r0));
                int slot = 0;
                uint32_t phase = 0;
                int issued = 0;
                for (int j = 0; j < nb && !aborted(bar); ++j) {
                    const int key0 = key_base + (kb0 + j) * kKeys;
                    for (int c = 0; c < kSlotsPerBlock; ++c) {
                        if (issued >= kNK && !wait_or_abort(bar, &bar.kempty[slot], phase ^ 1, p.err, -2)) break;
                        if (c < 4) {      // latent dims [128c, 128c + 128): two sub-tiles in one request
                            mbar_arrive_expect_tx(&bar.kfull[slot], kSlotBytes);
                            tma_load_4d(kring + slot * kSlotBytes, &map_ckv2, &bar.kfull[slot], 0, key0, 2 * c, b);
                        } else {          // rope dims
                            mbar_arrive_expect_tx(&bar.kfull[slot], kChunkBytes);
                            tma_load_3d(kring + slot * kSlotBytes, &map_kpe, &bar.kfull[slot], 0, key0, b);
                        }
                        ++issued;
                        if (++slot == kNK) { slot = 0; phase ^= 1; }
                    }
                }
                // drain: every issued chunk must land before this CTA may exit
                const int outstanding = issued < kNK ? issued : kNK;
                int s = slot;
                uint32_t ph = phase;
                for (int k = 0; k < outstanding; ++k) {
                    if (--s < 0) { s = kNK - 1; ph ^= 1; }
                    mbar_wait(&bar.kfull[s], ph, kWaitLimit);
                }
            }
        } else if (warp == 1) {
            // ---------------- MMA issuer: S = Q K^T ---------------------------------------
            if (elect_one() && nb > 0) {
                const uint32_t idesc = idesc_bf16_f32(kRows, kKeys, 0, 0);
                bool ok = wait_or_abort(bar, &bar.q_ready, 0, p.err, -3) &&
                          wait_or_abort(bar, &bar.qpe_full, 0, p.err, -3);
                tc_fence_after();
                int slot = 0;
                uint32_t phase = 0;
                for (int j = 0; j < nb && ok; ++j) {
                    const int buf = j & 1;
                    if (j >= 2 && !(ok = wait_or_abort(bar, &bar.sempty[buf], ((j >> 1) - 1) & 1, p.err, -4))) break;
                    tc_fence_after();
                    KDT_TC_TRACE(kEvSMmaStart, j);
                    const uint32_t d = tmem_s0 + buf * kKeys;
                    for (int c = 0; c < kSlotsPerBlock; ++c) {
                        if (!(ok = wait_or_abort(bar, &bar.kfull[slot], phase, p.err, -5))) break;
                        tc_fence_after();
                        const uint32_t kaddr = smem_u32(kring + slot * kSlotBytes);
                        if (c < 4) {
                            for (int t = 0; t < 2; ++t)            // sub-tile t: dims 128c + 64t .. +64
                                for (int kk = 0; kk < 4; ++kk) {
                                    const uint64_t bdesc = sdesc_sw128(kaddr + t * kChunkBytes + kk * 32, 16, 1024);
                                    mma_ts(d, tmem_q + 64 * c + 32 * t + 8 * kk, bdesc, idesc,
                                           (c > 0 || t > 0 || kk > 0) ? 1u : 0u);
                                }
                        } else {
                            for (int kk = 0; kk < 4; ++kk)
                                mma_ss(d, sdesc_sw128(smem_u32(qpe_tile) + kk * 32, 16, 1024),
                                       sdesc_sw128(kaddr + kk * 32, 16, 1024), idesc, 1u);
                        }
                        mma_commit(&bar.kempty[slot]);
                        if (++slot == kNK) { slot = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    mma_commit(&bar.sfull[buf]);
                    KDT_TC_TRACE(kEvSMmaIssued, j);
                }
                drain_mmas(bar);
            }
        } else if (warp >= 4) {
            // ---------------- Q_nope -> TMEM, then softmax ---------------------------------
            // Eight warps: warp w serves the 32 rows of TMEM lane quadrant (w % 4); warps 4-7
            // take keys 0..63 of each block, warps 8-11 keys 64..127.
            const int half = (warp - 4) >> 2;
            const int row = 32 * (warp & 3) + lane;
            const int R = r0 + row;
            const bool row_valid = R < p.rows_seq;
            {
                const uint4 *src = reinterpret_cast<const uint4 *>(p.q_nope + ((int64_t)b * p.rows_seq + R) * kDc);
                for (int c8 = 4 * half; c8 < 4 * half + 4; ++c8) {     // 4 x 32 columns = 256 bf16
                    uint32_t w[32];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint4 v = row_valid ? __ldg(src + c8 * 8 + q) : make_uint4(0u, 0u, 0u, 0u);
                        w[4 * q] = v.x; w[4 * q + 1] = v.y; w[4 * q + 2] = v.z; w[4 * q + 3] = v.w;
                    }
                    tmem_st32(tmem_lane_addr(tmem_q, warp, c8 * 32), w);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.q_ready);
            }
            const int qi = min(R, p.rows_seq - 1) / p.H;
            const uint32_t *visrow = p.vis + ((int64_t)b * p.T + qi) * p.W;
            float *rowmax_s = reinterpret_cast<float *>(smem + kOffRowMax);
            float *lsum_s = reinterpret_cast<float *>(smem + kOffLSum);
            float m_run = -INFINITY;                               // log2 units, same in both halves
            float l_run = 0.f;                                     // this half's share of the row sum
            bool ok = true;
            bool fail = false;
            for (int j = 0; j < nb; ++j) {
                // No warp leaves this loop on its own: every iteration meets the other seven
                // at the named barrier, which ORs their failures.
                const int buf = j & 1;
                const int ps = j % kNP;
                ok = ok && warp_wait(bar, &bar.sfull[buf], (j >> 1) & 1, p.err, -6);
                float x[64];
                float mx = -INFINITY;
                if (ok) {
                    tc_fence_after();
                    if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvSoftmaxIn, j);
                    uint32_t r0v[32], r1v[32];
                    const uint32_t sbase = tmem_s0 + buf * kKeys + 64 * half;
                    tmem_ld32(tmem_lane_addr(sbase, warp, 0), r0v);
                    tmem_ld32(tmem_lane_addr(sbase, warp, 32), r1v);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        x[q] = __uint_as_float(r0v[q]) * p.scale_log2;
                        x[32 + q] = __uint_as_float(r1v[q]) * p.scale_log2;
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar.sempty[buf]);  // score buffer may be overwritten
                    if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvSoftmaxLoaded, j);
                    const int key0 = key_base + (kb0 + j) * kKeys + 64 * half;
                    if (key0 < 0 || key0 + 64 > P) {               // leading pad or tree keys: mask
#pragma unroll
                        for (int c = 0; c < 64; ++c) {
                            const int key = key0 + c;
                            bool vis = key >= 0;
                            if (vis && key >= P) {
                                const int t = key - P;
                                vis = (__ldg(visrow + (t >> 5)) >> (t & 31)) & 1u;
                            }
                            if (!vis) x[c] = -INFINITY;
                        }
                    }
#pragma unroll
                    for (int c = 0; c < 64; ++c) mx = fmaxf(mx, x[c]);
                    rowmax_s[(buf * 2 + half) * kRows + row] = mx;
                }
                if (barrier_or<2, 256>(!ok)) {
                    fail = true;
                    break;
                }
                mx = fmaxf(mx, rowmax_s[(buf * 2 + (half ^ 1)) * kRows + row]);
                float alpha = 1.f;
                if (mx > m_run + kRescaleThreshold || (m_run == -INFINITY && mx > -INFINITY)) {
                    alpha = (m_run == -INFINITY) ? 1.f : fast_exp2(m_run - mx);
                    m_run = mx;
                    l_run *= alpha;
                }
                // the peer's P slot and this CTA's staging slot ps are free once P.V of
                // block j - kNP is done
                ok = j < kNP || warp_wait_cluster(bar, &bar.pempty[ps], ((j / kNP) - 1) & 1, p.err, -7);
                if (!ok) continue;                                 // caught at the next barrier
                if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvSoftmaxSlot, j);
                // staging slot ps: its previous copy (block j - kNP) landed before P.V of that
                // block could run, which the pempty wait above has seen
                unsigned char *stage = smem + kOffPStage + ps * kPBytes + half * (kPBytes / 2);
                float lsum = 0.f;
                const bool live = m_run > -INFINITY;
#pragma unroll
                for (int u = 0; u < 8; ++u) {                      // 8 chunks of 8 keys
                    uint32_t w[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float e0 = live ? fast_exp2(x[u * 8 + 2 * q] - m_run) : 0.f;
                        const float e1 = live ? fast_exp2(x[u * 8 + 2 * q + 1] - m_run) : 0.f;
                        lsum += e0 + e1;
                        w[q] = pack_bf16x2(e0, e1);
                    }
                    *reinterpret_cast<uint4 *>(stage + row * 128 + ((u ^ (row & 7)) << 4)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
                l_run += lsum;
                float *astage = reinterpret_cast<float *>(smem + kOffAStage + ps * kRows * 4);
                if (half == 0) astage[row] = alpha;
                fence_proxy_async_smem();                          // staging visible to the copy engine
                __syncwarp();
                if (lane == 0) {
                    const uint32_t rows_off = (uint32_t)(32 * (warp & 3)) * 128;
                    bulk_copy_to_peer(smem_u32(smem + kOffP + ps * kPBytes + half * (kPBytes / 2) + rows_off),
                                      stage + rows_off, 32 * 128, &bar.pfull[ps], 1);
                    if (half == 0) {
                        const uint32_t a_off = (uint32_t)(32 * (warp & 3)) * 4;
                        bulk_copy_to_peer(smem_u32(smem + kOffAlpha + ps * kRows * 4 + a_off),
                                          reinterpret_cast<unsigned char *>(astage) + a_off, 32 * 4, &bar.pfull[ps], 1);
                    }
                }
                if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvSoftmaxSent, j);
            }
            // The peer's MMA commits free a P slot by arriving on pempty here; the arrivals
            // for the last kNP blocks are consumed before this CTA may leave, so none can
            // land in the shared memory of a CTA that later runs on this SM.
            if (!fail && ok && warp == 4) {
                for (int ps = 0; ps < kNP && ps < nb; ++ps) {
                    const int j_last = ps + ((nb - 1 - ps) / kNP) * kNP;
                    ok = warp_wait_cluster(bar, &bar.pempty[ps], (j_last / kNP) & 1, p.err, -18) && ok;
                }
            }
            // final statistics for the O-CTA epilogue: (m, l) with l summed over both halves
            if (half == 1) lsum_s[row] = l_run;
            fail = barrier_or<2, 256>(fail || !ok) || fail;
            if (!fail && half == 0 && nb > 0) {
                const uint32_t dst = map_to_rank(smem + kOffStats + row * 8, 1);
                st_cluster_f32(dst, m_run);
                st_cluster_f32(dst + 4, l_run + lsum_s[row]);
                publish_remote_stores();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(&bar.stats_full, 1);
            }
        }
    } else {
        // =============================== O-CTA ===============================
        unsigned char *pbase = smem + kOffP;
        unsigned char *vbase = smem + kOffV;
        const float *alpha_s = reinterpret_cast<const float *>(smem + kOffAlpha);
        const float2 *stats_s = reinterpret_cast<const float2 *>(smem + kOffStats);
        if (warp == 0) {
            // ---------------- TMA producer: V halves -----------------------------------------
            if (elect_one() && nb > 0) {
                tma_prefetch_desc(&map_ckv4);
                int slot = 0;
                uint32_t phase = 0;
                int issued = 0;
                for (int j = 0; j < nb && !aborted(bar); ++j) {
                    const int key0 = key_base + (kb0 + j) * kKeys;
                    for (int h = 0; h < 2; ++h) {
                        if (issued >= kNV && !wait_or_abort(bar, &bar.vempty[slot], phase ^ 1, p.err, -8)) break;
                        mbar_arrive_expect_tx(&bar.vfull[slot], kVHalfBytes);
                        // latent dims [256h, 256h + 256): four sub-tiles in one request
                        tma_load_4d(vbase + slot * kVHalfBytes, &map_ckv4, &bar.vfull[slot], 0, key0, 4 * h, b);
                        ++issued;
                        if (++slot == kNV) { slot = 0; phase ^= 1; }
                    }
                }
                const int outstanding = issued < kNV ? issued : kNV;
                int s = slot;
                uint32_t ph = phase;
                for (int k = 0; k < outstanding; ++k) {
                    if (--s < 0) { s = kNV - 1; ph ^= 1; }
                    mbar_wait(&bar.vfull[s], ph, kWaitLimit);
                }
            }
        } else if (warp == 1) {
            // ---------------- MMA issuer: O += P V --------------------------------------------
            if (elect_one() && nb > 0) {
                const uint32_t idesc = idesc_bf16_f32(kRows, 256, 0, 1);
                int slot = 0;
                uint32_t phase = 0;
                uint32_t rs_phase = 0, sync_phase = 0;
                bool ok = true;
                for (int j = 0; j < nb && ok; ++j) {
                    const int ps = j % kNP;
                    if (!(ok = wait_or_abort(bar, &bar.corr_done, j & 1, p.err, -9))) break;
                    KDT_TC_TRACE(kEvOMmaStart, j);
                    const int need = *reinterpret_cast<volatile int *>(&bar.need_rescale);
                    mbar_arrive(&bar.ack);
                    if (need) {
                        // let every P.V issued so far finish, hand O to the correction warps,
                        // and wait until they have rescaled it
                        mma_commit(&bar.sync_bar);
                        if (!(ok = wait_or_abort(bar, &bar.sync_bar, sync_phase, p.err, -15))) break;
                        sync_phase ^= 1;
                        tc_fence_before();
                        mbar_arrive(&bar.o_ready);
                        if (!(ok = wait_or_abort(bar, &bar.rescaled, rs_phase, p.err, -16))) break;
                        rs_phase ^= 1;
                    }
                    tc_fence_after();
                    const uint32_t paddr = smem_u32(pbase + ps * kPBytes);
                    for (int h = 0; h < 2; ++h) {
                        if (!(ok = wait_or_abort(bar, &bar.vfull[slot], phase, p.err, -10))) break;
                        tc_fence_after();
                        const uint32_t vaddr = smem_u32(vbase + slot * kVHalfBytes);
                        for (int kk = 0; kk < kKeys / 16; ++kk) {
                            const uint64_t adesc = sdesc_sw128(paddr + (kk >> 2) * (kPBytes / 2) + (kk & 3) * 32, 16, 1024);
                            const uint64_t bdesc = sdesc_sw128(vaddr + kk * 2048, kChunkBytes, 1024);
                            mma_ss(tmem + 256 * h, adesc, bdesc, idesc, (j > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(&bar.vempty[slot]);
                        if (++slot == kNV) { slot = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    KDT_TC_TRACE(kEvOMmaIssued, j);
                    // release the P slot in the S-CTA once this block's P.V has read it
                    asm volatile(
                        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], "
                        "%1;" ::"r"(smem_u32(&bar.pempty[ps])),
                        "h"((uint16_t)1)
                        : "memory");
                }
                drain_mmas(bar);
            }
        } else if (warp >= 4 && warp < 8) {
            // ---------------- correction (rare rescale) and epilogue -------------------------
            // Warps 4-7 only (one per TMEM lane quadrant): named barrier 1 counts 128 threads.
            const int row = 32 * (warp & 3) + lane;
            bool ok = true;
            uint32_t rs_phase = 0;
            for (int j = 0; j < nb; ++j) {
                // Every correction warp reaches the named barriers below each block, whatever
                // happened, so a timeout in one warp cannot strand the others there; the
                // decision to stop is the barrier's OR-reduction of the warps' failures.
                const int ps = j % kNP;
                if (threadIdx.x == 128) mbar_arrive_expect_tx(&bar.pfull[ps], kPTx);   // P + alpha of block j
                ok = ok && warp_wait_cluster(bar, &bar.pfull[ps], (j / kNP) & 1, p.err, -11);
                if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvCorrIn, j);
                const float a = ok ? alpha_s[ps * kRows + row] : 1.f;
                const bool mine = ok && j > 0 && __any_sync(0xffffffffu, a != 1.f);
                uint32_t fail_any, need_any;
                asm volatile(
                    "{\n\t.reg .pred pin, pout;\n\t"
                    "setp.ne.u32 pin, %1, 0;\n\t"
                    "bar.red.or.pred pout, 1, 128, pin;\n\t"
                    "selp.u32 %0, 1, 0, pout;\n\t}"
                    : "=r"(fail_any)
                    : "r"(ok ? 0u : 1u)
                    : "memory");
                asm volatile(
                    "{\n\t.reg .pred pin, pout;\n\t"
                    "setp.ne.u32 pin, %1, 0;\n\t"
                    "bar.red.or.pred pout, 1, 128, pin;\n\t"
                    "selp.u32 %0, 1, 0, pout;\n\t}"
                    : "=r"(need_any)
                    : "r"(mine ? 1u : 0u)
                    : "memory");
                if (fail_any) {
                    ok = false;
                    break;
                }
                if (threadIdx.x == 128) {
                    bar.need_rescale = need_any ? 1 : 0;
                    mbar_arrive(&bar.corr_done);          // release: need_rescale visible to the MMA thread
                }
                if (need_any) {
                    // O is handed over once every P.V before block j has completed
                    ok = warp_wait(bar, &bar.o_ready, rs_phase, p.err, -12);
                    tc_fence_after();
                    if (ok) {               // whole warp; rows that need no rescale multiply by 1
                        for (int c = 0; c < 512 / 32; ++c) {
                            uint32_t r[32];
                            const uint32_t addr = tmem_lane_addr(tmem, warp, c * 32);
                            tmem_ld32(addr, r);
                            tmem_wait_ld();
#pragma unroll
                            for (int q = 0; q < 32; ++q) r[q] = __float_as_uint(__uint_as_float(r[q]) * a);
                            tmem_st32(addr, r);
                        }
                        tmem_wait_st();
                    }
                    tc_fence_before();
                    asm volatile(
                        "{\n\t.reg .pred pin, pout;\n\t"
                        "setp.ne.u32 pin, %1, 0;\n\t"
                        "bar.red.or.pred pout, 1, 128, pin;\n\t"
                        "selp.u32 %0, 1, 0, pout;\n\t}"
                        : "=r"(fail_any)
                        : "r"(ok ? 0u : 1u)
                        : "memory");
                    if (fail_any) {
                        ok = false;
                        break;
                    }
                    if (threadIdx.x == 128) mbar_arrive(&bar.rescaled);
                    rs_phase ^= 1;
                }
                // the MMA thread has read this block's flag before the next one is written
                ok = warp_wait(bar, &bar.ack, j & 1, p.err, -17);
            }
            // epilogue
            const int R = r0 + row;
            const int64_t grow = (int64_t)b * p.rows_seq + R;
            float *orow, *lrow;
            if (nsplit == 1) {
                orow = p.out + grow * kDc;
                lrow = p.lse ? p.lse + grow : nullptr;
            } else if (p.tail_splits > 0) {                  // compact tail partials
                const int64_t nrows = (int64_t)p.tail_tiles * kRows;
                const int64_t k = (int64_t)(tile - first_tail) * kRows + row;
                orow = p.part_o + ((int64_t)split * nrows + k) * kDc;
                lrow = p.part_lse + (int64_t)split * nrows + k;
            } else {
                orow = p.part_o + ((int64_t)split * p.rows_total + grow) * kDc;
                lrow = p.part_lse + (int64_t)split * p.rows_total + grow;
            }
            if (nb == 0) {
                if (R < p.rows_seq) {
                    for (int c = 0; c < kDc; c += 4) *reinterpret_cast<float4 *>(orow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (lrow) *lrow = -INFINITY;
                }
            } else if (ok && warp_wait(bar, &bar.drain, 0, p.err, -13) &&
                       warp_wait_cluster(bar, &bar.stats_full, 0, p.err, -14)) {
                tc_fence_after();
                const float2 st = stats_s[row];
                const float inv = st.y > 0.f ? 1.f / st.y : 0.f;
                for (int c = 0; c < 512 / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tmem_lane_addr(tmem, warp, c * 32), r);
                    tmem_wait_ld();
                    if (R < p.rows_seq) {
#pragma unroll
                        for (int q = 0; q < 32; q += 4)
                            *reinterpret_cast<float4 *>(orow + c * 32 + q) =
                                make_float4(__uint_as_float(r[q]) * inv, __uint_as_float(r[q + 1]) * inv,
                                            __uint_as_float(r[q + 2]) * inv, __uint_as_float(r[q + 3]) * inv);
                    }
                }
                if (R < p.rows_seq && lrow) *lrow = st.y > 0.f ? 0.6931471805599453f * (st.x + log2f(st.y)) : -INFINITY;
            }
        }
    }

    // ---- teardown ------------------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (aborted(bar)) {
        // Error path only: copies the peer issued before it noticed may still be in
        // flight; give them time to land (they take microseconds) before either CTA
        // of the cluster can leave.
        const uint64_t t0 = global_ns();
        do {
            __nanosleep(1000);
        } while (global_ns() - t0 < 200000ull);
    }
    cluster_sync();            // no CTA leaves while its peer may still touch its shared memory
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

bool make_map(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
              const cuuint32_t *box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint32_t es[4] = {1, 1, 1, 1};
    memset(m, 0, sizeof(*m));
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int tc_rows_per_unit() { return kRows; }
int tc_keys_per_block() { return kKeys; }

cudaError_t launch_verify_tc(const VerifyParams &vp, cudaStream_t s) {
    CUtensorMap map_ckv2, map_ckv4, map_kpe, map_qpe;
    const cuuint64_t L = (cuuint64_t)vp.L;
    {
        // c_kv viewed as [B][8 dim-blocks][L keys][64]: a box of (64, 128 keys, n blocks)
        // lands as n consecutive [128 x 64] 128B-swizzled sub-tiles.
        cuuint64_t dims[4] = {64, L, (cuuint64_t)(kDc / 64), (cuuint64_t)vp.B};
        cuuint64_t strides[3] = {(cuuint64_t)kDc * 2, 128, L * kDc * 2};
        cuuint32_t box2[4] = {64, kKeys, 2, 1};
        cuuint32_t box4[4] = {64, kKeys, 4, 1};
        if (!make_map(&map_ckv2, vp.c_kv, 4, dims, strides, box2)) return cudaErrorInvalidValue;
        if (!make_map(&map_ckv4, vp.c_kv, 4, dims, strides, box4)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[3] = {(cuuint64_t)kDr, L, (cuuint64_t)vp.B};
        cuuint64_t strides[2] = {(cuuint64_t)kDr * 2, L * kDr * 2};
        cuuint32_t box[3] = {64, kKeys, 1};
        if (!make_map(&map_kpe, vp.k_pe, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)kDr, (cuuint64_t)vp.rows_total};
        cuuint64_t strides[1] = {(cuuint64_t)kDr * 2};
        cuuint32_t box[2] = {64, kRows};
        if (!make_map(&map_qpe, vp.q_pe, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    TcParams p;
    p.B = vp.B;
    p.T = vp.T;
    p.H = vp.H;
    p.W = vp.W;
    p.rows_seq = vp.T * vp.H;
    p.row_tiles = (p.rows_seq + kRows - 1) / kRows;
    p.num_splits = vp.num_splits;
    p.blocks_per_split = vp.blocks_per_split;
    p.rows_total = vp.rows_total;
    p.q_nope = static_cast<const __nv_bfloat16 *>(vp.q_nope);
    p.prefix_len = vp.prefix_len;
    p.vis = vp.vis;
    p.scale_log2 = vp.scale_log2;
    p.out = vp.out;
    p.lse = vp.lse;
    p.part_o = vp.part_o;
    p.part_lse = vp.part_lse;
    p.err = vp.err;
    p.tail_tiles = vp.tail_tiles;
    p.tail_splits = vp.tail_splits;
    const int64_t tiles = (int64_t)p.B * p.row_tiles;
    const int64_t units = p.tail_splits > 0 ? tiles - p.tail_tiles + (int64_t)p.tail_tiles * p.tail_splits
                                            : tiles * p.num_splits;
    cudaError_t e = cudaFuncSetAttribute(verify_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    verify_tc_kernel<<<(unsigned)(2 * units), kThreads, kSmemBytes, s>>>(map_ckv2, map_ckv4, map_kpe, map_qpe, p);
    return cudaGetLastError();
}

}  // namespace kdt
