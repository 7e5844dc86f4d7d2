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
//    256 consecutive query rows (two 128-row tiles) of one sequence and a range of
//    128-key blocks. Every head shares the latent cache, so S = Q K^T and O = P V are
//    dense contractions on the 5th-generation tensor cores.
//  * A unit runs on a 4-CTA cluster of two CTA pairs, each pair one M = 256 MMA
//    (tcgen05 .cta_group::2): the S pair (ranks 0, 1) computes scores and the
//    softmax, the O pair (ranks 2, 3) accumulates the output; S-CTA k hands its
//    128 rows of P to O-CTA 2 + k. In a pair each CTA loads only HALF of the B
//    operand (S pair: 64 of a block's 128 keys; O pair: 128 of 256 latent columns),
//    and the MMA reads both halves, so every SM fetches and stores half the cache
//    bytes a single-CTA MMA of the same rows would. Roles are split because one SM
//    cannot hold Q (128 x 576 bf16), the 128 x 512 fp32 output accumulator and the
//    scores:
//      - an S-CTA: its Q_nope rows live in tensor memory as the MMA A operand
//        (256 columns), Q_pe in shared memory; per key block the pair computes
//        S[256 x 128] into one of two TMEM score buffers (256 columns), each CTA
//        runs the online softmax of its rows (one thread per row) and copies P
//        (bf16) and the block's rescale factors into its O-CTA's shared memory with
//        ONE bulk copy (the copy engine's cost is per request, not per byte);
//      - an O-CTA: the fp32 O[128 x 512] accumulator of its rows occupies its 512
//        TMEM columns; per block the pair issues O += P V (N = 256, two halves) and
//        rescales rows of O in TMEM on the rare occasions the running maximum
//        grows past the threshold below.
//  * Key blocks are aligned to END at kv_len, so no row at or beyond
//    prefix_len + T is ever fetched; the leading block may start before row 0,
//    where TMA fills zeros and the mask removes the keys. Only blocks holding tree
//    keys (or those leading zeros) evaluate the mask, from packed ancestor bits.
//  * Online softmax in base 2 with a lazy maximum: the running max m used for
//    exp2(x - m) is only raised when a block's max exceeds it by more than 20, so
//    p <= 2^20 and O is rescaled only then (exact either way: o = O / l). P is
//    rounded to bf16, whose exponent range is fp32's, so the bound only keeps l and
//    O (fp32) far from overflow; a smaller one rescales often on caches with
//    outlier keys (a few times larger than the rest), and every rescale drains the
//    P.V pipe.
//  * Every wait is bounded; on a lost arrival the kernel records a status in the
//    caller's error word, drains its own in-flight copies and MMAs, frees TMEM and
//    returns (no trap, no hang).
#include "kdt_internal.cuh"
#include "tc_ptx.cuh"

#include <atomic>
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

// Trace events (ranks 0-1 = S-CTAs, ranks 2-3 = O-CTAs).
enum TraceEvent {
    kEvSMmaStart = 0,    // S MMA thread: score buffer free, starts issuing block
    kEvSMmaIssued,       // S MMA thread: all chunks of the block issued
    kEvSoftmaxIn,        // softmax warp 4: scores of the block in TMEM
    kEvSoftmaxLoaded,    // softmax warp 4: scores loaded, buffer released
    kEvSoftmaxSlot,      // softmax warp 4: P slot free in the O-CTA
    kEvSoftmaxSent,      // softmax: P of the block staged and its copy issued
    kEvCorrIn,           // correction warp 4: P of the block arrived
    kEvOMmaStart,        // O MMA thread: block checked, starts issuing P.V
    kEvOMmaIssued,       // O MMA thread: P.V of the block issued
    kEvKIssue,           // S producer: key chunk u requested (index = chunk use)
    kEvKFull,            // S MMA thread: key chunk u landed in both CTAs
    kEvSoftmaxLd,        // softmax warp 4: scores in registers
    kEvVIssue,           // O producer: value chunk u requested
    kEvVFull,            // O MMA thread: value chunk u landed in both CTAs
    kEvKEmpty,           // S producer: the pair's MMAs finished reading key chunk u
    kEvKIssued,          // S MMA thread: the MMAs of key chunk u are issued
    kEvRFull,            // S MMA thread: rope chunk of block j landed
    kEvSoftmaxMax,       // softmax warp 4: row maxima of both halves agreed
    kEvSoftmaxStaged,    // softmax warp 4: its rows of P staged
    kEvQReady,           // softmax warp 4: Q_nope of item i in TMEM (index = item)
    kEvStatsSent,        // softmax warp 4: statistics of item i sent
    kEvOFree,            // O MMA thread: O of item i - 1 read out, item i may start
    kEvEpiIn,            // epilogue warp 4: P.V and statistics of item i complete
    kEvEpiOut,           // epilogue warp 4: O of item i written
    kEvQpeIssued,        // S producer: Q_pe of item i requested
    kEvItemEnd0,         // softmax warp 4: item i's blocks done, at the statistics barrier
    kEvItemEnd1,         // softmax warp 8: the same
    kEvItemBar,          // softmax warp 4: statistics barrier passed
    kNumTraceEvents
};

constexpr int kRows = 128;             // query rows per CTA (the pair's MMA has M = 256)
constexpr int kKeys = 128;             // keys per block (S MMA N, P.V K)
constexpr int kHalfKeys = kKeys / 2;   // keys of a block held by one S-CTA
constexpr int kThreads = 384;          // 12 warps
constexpr int kQPrefetchBlocks = 6;               // blocks before an item's end that warm L2 with the next Q
constexpr uint32_t kQPrefetchChunk = 32768;       // bytes per L2 prefetch request
constexpr int kKvPrefetchBlocks = 4;              // key blocks the L2 prefetch runs ahead of the loads
// Operand tiles are [rows x 64 bf16] with 128-byte rows, 128B-swizzled.
constexpr int kKSub = kHalfKeys * 128;            // S-CTA key sub-tile [64 keys x 64 dims]: 8 KB
constexpr int kVSub = kKeys * 128;                // O-CTA value sub-tile [128 keys x 64 dims]: 16 KB
// Tiles travel as 32 KB requests from 4-D views of the cache (few, large requests:
// the copy engine's cost is per request).
constexpr int kKSubPerChunk = 4;                  // 64-dim sub-tiles per latent key chunk
constexpr int kKChunks = 8 / kKSubPerChunk;       // latent key chunks per block
constexpr int kKSlotBytes = kKSubPerChunk * kKSub;   // S latent ring slot: 64 keys x 256 latent dims
constexpr int kNK = 3;                            // S-CTA latent key ring slots (96 KB, 1.5 blocks)
constexpr int kNR = 4;                            // S-CTA rope key ring slots of kKSub (32 KB, four blocks)
constexpr int kQpeBytes = kRows * 128;            // Q_pe tile of one S-CTA: 16 KB
constexpr int kPBytes = kRows * kKeys * 2;        // P tile of one CTA: 32 KB (two 128B-swizzled halves)
// A P slot holds the tile followed by the block's rescale factors, so one bulk copy
// per block carries both.
constexpr int kPSlotBytes = kPBytes + 1024;       // 32 KB P + alpha[128] (+ pad to 1 KB alignment)
constexpr uint32_t kPTx = kPBytes + kRows * 4;    // bytes copied into a P slot per block
constexpr int kNS = 2;                            // S-CTA staging slots (free once the copy landed)
constexpr int kNP = 4;                            // O-CTA P slots (free once P.V of the block ran)
constexpr int kVSubPerChunk = 2;                  // 64-dim sub-tiles per value chunk of one O-CTA
constexpr int kVChunks = 4 / kVSubPerChunk;       // value chunks per block (an O-CTA's 256 latent dims)
constexpr int kVSlotBytes = kVSubPerChunk * kVSub;   // O ring slot: 128 keys x 128 latent dims
constexpr int kNV = 2;                            // O-CTA value ring slots (64 KB)
constexpr uint32_t kCmdDone = 0xffffffffu;        // correction command: no more rescales
constexpr uint64_t kWaitLimit = 200000000ull;     // ns a wait may poll before giving up (default)
constexpr float kRescaleThreshold = 20.0f;        // log2 units
constexpr int kMaxClusters = 48;                  // partial states then fit the no-alloc scratch
constexpr int kSeqTable = 64;                     // sequences whose block counts a CTA keeps in shared memory
// O-CTA correction/epilogue warps: kEpiWarps / 4 per TMEM lane quadrant, each taking an
// equal share of the 512 columns; each warp transposes [32 rows x kEpiCols] at a time.
// Eight warps (twice the stores in flight while O drains) measured no faster than four.
constexpr int kEpiWarps = 4;
constexpr int kEpiGroupCols = 512 * 4 / kEpiWarps;   // TMEM columns of one warp
constexpr int kEpiCols = 16;

// Shared-memory layout (same offsets in every CTA of the cluster; roles use
// different parts). All tiles 1024-byte aligned for the 128B swizzle.
constexpr int kOffQpe = 0;                                  // S: Q_pe tile 16 KB
constexpr int kOffKRing = kOffQpe + kQpeBytes;              // S: 3 x 32 KB latent keys
constexpr int kOffRRing = kOffKRing + kNK * kKSlotBytes;   // S: 4 x 8 KB rope keys
constexpr int kOffPStage = kOffRRing + kNR * kKSub;         // S: 2 x 33 KB staging of P + alpha
constexpr int kOffRowMax = kOffPStage + kNS * kPSlotBytes;  // S: [2 blocks][2 halves][128] partial maxima
constexpr int kOffLSum = kOffRowMax + 2 * 2 * kRows * 4;    // S: [128] partial row sums
constexpr int kOffP = 0;                                    // O: 4 x 33 KB P + alpha
constexpr int kOffV = kOffP + kNP * kPSlotBytes;            // O: 2 x 32 KB values
constexpr int kOffStats = kOffV + kNV * kVSlotBytes;        // O: [2 items][128] x (m, l)
constexpr int kOffEpi = kOffStats + 2 * kRows * 8;          // O: epilogue transpose, [32 rows][kEpiCols fp32] a warp
constexpr int kSEnd = kOffLSum + kRows * 4;
constexpr int kOEnd = kOffEpi + kEpiWarps * 32 * kEpiCols * 4;
constexpr int kTileBytes = kSEnd > kOEnd ? kSEnd : kOEnd;
constexpr int kSmemBytes = kTileBytes + 1024;               // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// Barriers (same layout in every CTA). "leader" = the even CTA of a pair, which
// issues the pair's MMAs; barriers the MMA thread waits on live in the leader.
struct Barriers {
    // S pair
    uint64_t kfull[kNK];           // leader: both halves of a latent key chunk landed (tx of both CTAs)
    uint64_t kempty[kNK];          // each S-CTA: its half of the chunk was read (MMA commit)
    uint64_t rfull[kNR];           // leader: both halves of a rope key chunk landed
    uint64_t rempty[kNR];          // each S-CTA: its rope chunk was read
    uint64_t sfull[2];             // each S-CTA: scores of a block are in its TMEM
    uint64_t sempty[2];            // leader: both CTAs' softmax warps have read the buffer (16 arrivals)
    uint64_t qpe_full;             // leader: both Q_pe tiles of the item landed
    uint64_t qpe_empty;            // each S-CTA: the item's last rope MMAs read its Q_pe tile
    uint64_t q_ready;              // leader: both CTAs' Q_nope stored in TMEM (16 arrivals)
    uint64_t pempty[kNP];          // each S-CTA: O-CTA P slot free again (O pair's MMA commit)
    uint64_t sfree[kNS];           // each S-CTA: the copy out of a staging slot has landed
    uint64_t staged[kNS][2];       // each S-CTA: the four warps of a half have staged their rows
    // O pair
    uint64_t pfull[kNP];           // each O-CTA: P + alpha of a block landed from its S-CTA
    uint64_t pready[kNP];          // leader: P slot filled in both O-CTAs, their rescale flags written
    uint64_t vfull[kNV];           // leader: both halves of a value chunk landed
    uint64_t vempty[kNV];          // each O-CTA: its half of the chunk was read
    // Rare rescale hand-over: the MMA thread lets its P.V drain, then sends `go` with a
    // command (P slot whose alphas to apply, or kCmdDone at the end) to each O-CTA whose
    // rows need it, and waits for `rescaled` (one arrival per O-CTA).
    uint64_t go;                   // each O-CTA: a command is in `cmd`
    uint64_t rescaled;             // leader: rows of O rescaled (or no rescale needed) per O-CTA
    uint64_t stats_full[2];        // each O-CTA: an item's (m, l) of its rows from its S-CTA (by item parity)
    uint64_t stats_empty[2];       // each S-CTA: the O-CTA epilogue has read that buffer
    uint64_t o_done;               // each O-CTA: every P.V of the item has completed
    uint64_t o_free;               // O leader: both O-CTAs' epilogues have read O (one arrival a warp)
    uint64_t sync_bar;             // leader: MMA thread's own completion probe (mid-stream)
    uint64_t drain;                // completion of all MMAs of the pair before TMEM is read or freed
    uint32_t need[2][kNP];         // leader: per-CTA "some row of O needs a rescale" per P slot
    uint32_t cmd;                  // each O-CTA: correction command
    int kseen[2];                  // S leader: latest latent chunk use each MMA issuer saw land
    int work_wleft;                      // this cluster's whole units (see the decomposition below)
    int work_u0, work_kb0, work_left;    // its tail range
    int work_count;                      // its key blocks
    uint32_t tmem_base;
    int abort_flag;
    uint64_t wait_ns;              // how long a wait may poll before the kernel gives up
    int64_t sched_B[kMaxClusters + 1];   // tail cut points of all clusters (cluster_schedule)
    int nb_tab[kSeqTable];               // key blocks of each sequence, when B <= kSeqTable
};

struct TcParams {
    int B, T, H, W;
    int rows_seq;          // T*H
    int row_tiles;         // ceil(rows_seq / 128)
    int64_t rows_total;
    const __nv_bfloat16 *q_nope;
    int64_t q_stride;              // elements between consecutive query rows of q_nope
    const int32_t *prefix_len;
    const uint32_t *vis;
    float scale_log2;
    float *out, *lse;
    float *part_o, *part_lse;      // [2 * clusters][256] partial states of units cut by the work split
    int32_t *err;
    int pairs_per_seq;             // work units (two row tiles each) per sequence
    uint64_t wait_ns;              // wait limit (kWaitLimit unless a test shortens it)
    int fault;                     // test hook: 1 = withhold the first item's Q-ready arrivals
    int64_t *sched;                // [R, kov, cut points B[0..C]] for the merge pass, or NULL
};

// ---- work decomposition ----------------------------------------------------------------
// A unit is two row tiles (256 rows) of one sequence, unit = b * pairs_per_seq + pair; its
// work is key blocks 0 .. nblk(b) - 1, taken in order. With C clusters:
//  * when every sequence has the same block count, the first (units / C) * C units go out
//    whole, round robin (cluster c takes units c, c + C, ...): the clusters running at the
//    same time then walk the same few sequences' keys in step and share them in L2;
//  * the remaining units (all of them when lengths differ) form the tail, cut into C
//    contiguous ranges of equal COST, units in order: when lengths differ a unit costs its
//    key blocks plus kItemCost blocks for the item boundary (the epilogue, the next Q load
//    and the pipeline refill between two items take about as long as that many blocks).
//    In "virtual blocks" unit u spans kov boundary blocks followed by its key blocks, the
//    tail spans Wv of them, and cluster c takes the key blocks whose virtual positions fall
//    in [Wv c / C, Wv (c + 1) / C). Equal block counts alone left clusters that met many
//    short units (ragged prefixes) with several more boundaries than others.
// Everything is derived from prefix_len on the device, the same way in every CTA. A tail
// unit cut by a range boundary is processed in pieces: each piece writes its normalised
// partial state (o, lse) into slot 2c (the first item of the cluster's tail range) or
// 2c + 1 (its last item), and a merge pass combines them.
__device__ __forceinline__ int seq_blocks(const TcParams &p, int b) {
    return (p.prefix_len[b] + p.T + kKeys - 1) / kKeys;
}

// Key blocks of sequence b, from a shared-memory table of the first kSeqTable sequences
// when the batch fits in it (the schedule reads them many times), else from prefix_len.
struct SeqBlocks {
    const TcParams &p;
    const int *tab;
    __device__ __forceinline__ int operator()(int b) const { return tab ? tab[b] : seq_blocks(p, b); }
};


// Boundary blocks charged per unit when lengths differ: an item boundary takes about as
// long as kItemCost key blocks. With equal lengths every unit costs the same and the
// plain block split is already balanced, so no boundary blocks are charged.
constexpr int kItemCost = 6;

// Where virtual position s of the tail falls: unit u, that unit's first key block in the
// tail's key-block numbering (start), its block count, and pos = the first key block at
// or after s (start when s lies in the unit's boundary part). s = Wv gives u = units and
// pos = the tail's key-block count.
__device__ __forceinline__ void locate_vblock(const TcParams &p, const SeqBlocks &nbs, int u_first, int kov,
                                              int64_t s, int &u, int64_t &start, int &nblk, int64_t &pos) {
    int64_t acc_v = 0, acc_r = 0;
    for (int b = u_first / p.pairs_per_seq, k0 = u_first % p.pairs_per_seq; b < p.B; ++b, k0 = 0) {
        const int nb = nbs(b);
        const int64_t vs = kov + nb;                          // virtual size of one unit
        const int64_t k = p.pairs_per_seq - k0;               // tail units of this sequence
        if (s < acc_v + k * vs) {
            const int64_t kk = (s - acc_v) / vs;
            u = b * p.pairs_per_seq + k0 + (int)kk;
            start = acc_r + kk * nb;
            nblk = nb;
            const int64_t into = s - acc_v - kk * vs - kov;         // key blocks of the unit before s
            pos = start + (into > 0 ? into : 0);
            return;
        }
        acc_v += k * vs;
        acc_r += k * nb;
    }
    u = p.B * p.pairs_per_seq;
    start = acc_r;
    nblk = 0;
    pos = acc_r;
}


// The schedule of all C clusters, computed by one whole warp (every lane gets R and kov):
//  * R rounds of whole units: in round k cluster c takes unit kC + c. With equal lengths
//    R = units / C. Otherwise rounds are added while every cluster's cost stays below its
//    fair share (the total cost / C, less one block), so the clusters running at the same
//    time work on consecutive units -- the same one or two sequences -- and share their
//    keys in L2.
//  * the tail, units RC .. : its virtual blocks are cut at B[0] = 0 <= B[1] <= .. <= B[C]
//    (written to shared memory), cluster c taking [B[c], B[c+1]): B[c] = (c S) / C - L[c]
//    with S the total cost and L[c] the whole-unit cost of clusters 0 .. c-1, so each
//    cluster's tail fills the rest of its fair share. With equal lengths this is the
//    plain cut (Wt c) / C of the tail.
__device__ __forceinline__ int cluster_schedule(const TcParams &p, const SeqBlocks &nbs, int C, int lane,
                                                int64_t *B, int &kov) {
    const int U = p.B * p.pairs_per_seq;
    const int nb0 = nbs(0);
    bool same = true;
    for (int b = lane; b < p.B; b += 32) same = same && nbs(b) == nb0;
    const bool uniform = __all_sync(0xffffffffu, same);
    kov = uniform ? 0 : kItemCost;
    const int c0 = lane, c1 = lane + 32;                      // this lane's clusters (C <= 48)
    int64_t S = 0;                                            // total cost of all units
    for (int b = lane; b < p.B; b += 32) S += (int64_t)p.pairs_per_seq * (kov + nbs(b));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) S += __shfl_xor_sync(0xffffffffu, S, off);
    int64_t l0 = 0, l1 = 0;                                   // whole-unit cost of clusters c0, c1
    int R;
    if (uniform) {
        R = U / C;
        l0 = c0 < C ? (int64_t)R * nb0 : 0;
        l1 = c1 < C ? (int64_t)R * nb0 : 0;
    } else {
        const int64_t fair = S / C;
        R = 0;
        for (int k = 0; k < U / C; ++k) {
            const int64_t n0 = c0 < C ? l0 + kov + nbs((k * C + c0) / p.pairs_per_seq) : 0;
            const int64_t n1 = c1 < C ? l1 + kov + nbs((k * C + c1) / p.pairs_per_seq) : 0;
            int64_t mx = n0 > n1 ? n0 : n1;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const int64_t o = __shfl_xor_sync(0xffffffffu, mx, off);
                mx = o > mx ? o : mx;
            }
            if (mx > fair - 1) break;
            l0 = n0;
            l1 = n1;
            R = k + 1;
        }
    }
    // L[c] = sum of the whole-unit costs of clusters before c (exclusive scan over 2 x 32)
    int64_t x0 = l0, x1 = l1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int64_t y0 = __shfl_up_sync(0xffffffffu, x0, off), y1 = __shfl_up_sync(0xffffffffu, x1, off);
        if (lane >= off) {
            x0 += y0;
            x1 += y1;
        }
    }
    const int64_t total0 = __shfl_sync(0xffffffffu, x0, 31);
    const int64_t L0 = x0 - l0, L1 = total0 + x1 - l1;
    if (c0 < C) B[c0] = S * c0 / C - L0;
    if (c1 < C) B[c1] = S * c1 / C - L1;
    const int64_t all = total0 + __shfl_sync(0xffffffffu, x1, 31);
    if (lane == 0) B[C] = S - all;
    return R;
}

struct Item {
    int b, rt0;            // sequence; first of the unit's two row tiles
    int P, nblk, key_base; // prefix length, key blocks of the unit, first key of block 0 (<= 0)
    int kb0, nb;           // blocks [kb0, kb0 + nb) of the unit
    bool whole;            // the unit's whole key range: write the final rows
    int slot;              // partial-state slot otherwise
};

struct WorkIter {
    int wu, wleft;         // next whole unit (stride C) and whole units left
    int u, kb, left, taken;   // tail range: unit, block, blocks left, tail items taken
};

__device__ __forceinline__ void fill_item(const TcParams &p, int u, Item &it) {
    const int b = u / p.pairs_per_seq;
    it.b = b;
    it.rt0 = 2 * (u % p.pairs_per_seq);
    it.P = p.prefix_len[b];
    const int kv_len = it.P + p.T;
    it.nblk = (kv_len + kKeys - 1) / kKeys;
    it.key_base = kv_len - it.nblk * kKeys;
}

__device__ __forceinline__ bool next_item(const TcParams &p, WorkIter &w, int c, int C, Item &it) {
    if (w.wleft > 0) {
        fill_item(p, w.wu, it);
        it.kb0 = 0;
        it.nb = it.nblk;
        it.whole = true;
        it.slot = 0;
        w.wu += C;
        --w.wleft;
        return true;
    }
    if (w.left <= 0) return false;
    fill_item(p, w.u, it);
    it.kb0 = w.kb;
    it.nb = min(it.nblk - w.kb, w.left);
    it.whole = it.kb0 == 0 && it.nb == it.nblk;
    it.slot = 2 * c + (w.taken == 0 ? 0 : 1);
    w.left -= it.nb;
    ++w.taken;
    if (w.kb + it.nb == it.nblk) {
        ++w.u;
        w.kb = 0;
    } else {
        w.kb += it.nb;
    }
    return true;
}

__device__ __forceinline__ bool aborted(const Barriers &bar) {
    return *reinterpret_cast<const volatile int *>(&bar.abort_flag) != 0;
}

// Wait until every tcgen05 operation this (MMA-issuing) thread issued has completed;
// the completion also arrives on the drain barrier of the other CTAs in `mask`.
__device__ __forceinline__ void drain_mmas(Barriers &bar, uint16_t mask) {
    mma_commit_pair(&bar.drain, mask);
    mbar_wait(&bar.drain, 0, bar.wait_ns);
}

__device__ __forceinline__ void set_abort(Barriers &bar, int32_t *err, int code) {
    bar.abort_flag = 1;
    if (err) atomicCAS(err, 0, code);
}

// Waits come in two scopes. Hand-offs that publish no memory of their own (TMA and MMA
// completions, "done reading" signals) wait with the default CTA-scope acquire, which
// is much cheaper on the MMA threads' critical path; hand-offs that publish a remote
// store (flags, commands, statistics) wait with cluster-scope acquire.
__device__ __forceinline__ bool wait_or_abort(Barriers &bar, uint64_t *b, uint32_t parity, int32_t *err, int code) {
    if (*reinterpret_cast<volatile int *>(&bar.abort_flag)) return false;
    if (mbar_wait(b, parity, bar.wait_ns)) return true;
    set_abort(bar, err, code);
    return false;
}

__device__ __forceinline__ bool wait_cluster_or_abort(Barriers &bar, uint64_t *b, uint32_t parity, int32_t *err,
                                                      int code) {
    if (*reinterpret_cast<volatile int *>(&bar.abort_flag)) return false;
    if (mbar_wait_cluster(b, parity, bar.wait_ns)) return true;
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

// Position in a ring of `kSlots` buffers: slot, its phase parity, uses so far.
struct RingPos {
    int slot = 0;
    uint32_t phase = 0;
    int n = 0;
};

template <int kSlots>
__device__ __forceinline__ void ring_advance(RingPos &r) {
    ++r.n;
    if (++r.slot == kSlots) {
        r.slot = 0;
        r.phase ^= 1;
    }
}

// Wait until the releases of the last (up to kSlots) uses of a ring have arrived: the
// copies into those slots have landed and been read, and no arrival is still in flight.
template <int kSlots>
__device__ __forceinline__ void ring_drain(uint64_t *empty, const RingPos &r, uint64_t limit_ns) {
    const int outstanding = r.n < kSlots ? r.n : kSlots;
    int s = r.slot;
    uint32_t ph = r.phase;
    for (int k = 0; k < outstanding; ++k) {
        if (--s < 0) {
            s = kSlots - 1;
            ph ^= 1;
        }
        mbar_wait(&empty[s], ph, limit_ns);
    }
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

// Visibility of keys [key0, key0 + 64) for one query row as a 64-bit mask (bit c: key
// key0 + c): keys before 0 are padding (hidden), prefix keys [0, P) are visible, and tree
// key P + t is visible when bit t of the row's packed ancestor bits is set. The tree part
// of a window spans at most three 32-bit words.
__device__ __forceinline__ uint64_t vis_mask64(const uint32_t *visrow, int W, int key0, int P) {
    uint64_t m = 0;
    const int p_lo = max(key0, 0) - key0, p_hi = min(key0 + 64, P) - key0;   // prefix keys, as c
    if (p_hi > p_lo) {
        const uint64_t below_hi = p_hi >= 64 ? ~0ull : ((1ull << p_hi) - 1);
        m |= below_hi & ~((1ull << p_lo) - 1);
    }
    const int c_lo = max(key0, P) - key0;                                      // first tree key, as c
    if (c_lo < 64) {
        const int ta = key0 + c_lo - P;                                        // its tree index (>= 0)
        const int wi = ta >> 5, sh = ta & 31;
        const uint64_t w0 = wi < W ? __ldg(visrow + wi) : 0u;
        const uint64_t w1 = wi + 1 < W ? __ldg(visrow + wi + 1) : 0u;
        const uint64_t w2 = wi + 2 < W ? __ldg(visrow + wi + 2) : 0u;
        const uint64_t bits = ((w0 | (w1 << 32)) >> sh) | (sh ? (w2 << (64 - sh)) : 0ull);   // tree bits ta..ta+63
        m |= bits << c_lo;
    }
    return m;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Largest scaled score of a row's 64 raw scores (scale > 0: scale * max; else scale * min).
__device__ __forceinline__ float scaled_max64(const float (&x)[64], float scale) {
    float r;
    if (scale >= 0.f) {
        r = fmax3(x[0], x[1], x[2]);
#pragma unroll
        for (int c = 3; c < 63; c += 2) r = fmax3(r, x[c], x[c + 1]);
        r = fmaxf(r, x[63]);
    } else {
        r = fmin3(x[0], x[1], x[2]);
#pragma unroll
        for (int c = 3; c < 63; c += 2) r = fmin3(r, x[c], x[c + 1]);
        r = fminf(r, x[63]);
    }
    return r * scale;
}

// p = 2^(scale * x - m) for 64 keys of one row, packed to bf16 into a 128-byte
// swizzled row of a P tile; returns the fp32 sum of the p. kScaled: x already holds
// scale * score (hidden keys -inf) and m may be -inf (all hidden so far: p = 0).
template <bool kScaled>
__device__ __forceinline__ float stage_p_row(const float (&x)[64], float scale, float m, unsigned char *dst_row,
                                             int row) {
    float lsum = 0.f;
    const bool live = !kScaled || m > -INFINITY;
    const float nm = -m;
#pragma unroll
    for (int u = 0; u < 8; ++u) {                          // 8 chunks of 8 keys
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float e0, e1;
            if (kScaled) {
                e0 = live ? fast_exp2(x[u * 8 + 2 * q] + nm) : 0.f;
                e1 = live ? fast_exp2(x[u * 8 + 2 * q + 1] + nm) : 0.f;
            } else {
                e0 = fast_exp2(fmaf(x[u * 8 + 2 * q], scale, nm));
                e1 = fast_exp2(fmaf(x[u * 8 + 2 * q + 1], scale, nm));
            }
            lsum += e0 + e1;
            w[q] = pack_bf16x2(e0, e1);
        }
        *reinterpret_cast<uint4 *>(dst_row + ((u ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    return lsum;
}

// TMEM-address helpers: lane field in bits [31:16].
__device__ __forceinline__ uint32_t tmem_lane_addr(uint32_t base, int warp, uint32_t col) {
    return base + ((uint32_t)(32 * (warp & 3)) << 16) + col;
}

__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(kThreads, 1)
    verify_tc_kernel(const __grid_constant__ CUtensorMap map_ks, const __grid_constant__ CUtensorMap map_vs,
                     const __grid_constant__ CUtensorMap map_kpe, const __grid_constant__ CUtensorMap map_qpe,
                     const TcParams p) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ Barriers bar;
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~static_cast<uintptr_t>(1023));
    const uint32_t rank = cluster_ctarank();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- roles ------------------------------------------------------------------------
    const bool s_role = rank < 2;                  // ranks 0, 1: S pair; 2, 3: O pair
    const int kpair = (int)(rank & 1);            // row tile of the unit = position in the pair
    const bool leader = kpair == 0;               // issues the pair's MMAs
    const uint32_t lead_rank = rank & ~1u;
    const uint32_t o_rank = 2u + (uint32_t)kpair;  // the O-CTA an S-CTA feeds
    constexpr uint16_t kMaskS = 0x3, kMaskO = 0xC, kMaskAll = 0xF;

    // Before the set-up: warm L2 with this CTA's rows of Q for unit c, the cluster's first
    // item whenever a round of whole units goes out first (every unit costs the same, or
    // the first round fits the fair share); otherwise the request is merely unused. The
    // first Q load then reads L2 instead of DRAM.
    if (s_role && warp == 4 && lane == 0) {
        const int c = (int)(blockIdx.x >> 2), C = (int)(gridDim.x >> 2);
        if (p.B * p.pairs_per_seq >= C) {
            const int b = c / p.pairs_per_seq;
            const int r0 = (2 * (c % p.pairs_per_seq) + kpair) * kRows;
            if (r0 < p.rows_seq) {
                const int nrows = min(kRows, p.rows_seq - r0);
                const unsigned char *qsrc =
                    reinterpret_cast<const unsigned char *>(p.q_nope + ((int64_t)b * p.rows_seq + r0) * p.q_stride);
                const uint32_t bytes = (uint32_t)((nrows - 1) * p.q_stride + kDc) * 2;
                for (uint32_t o = 0; o < bytes; o += kQPrefetchChunk)
                    prefetch_l2_bulk(qsrc + o, min(kQPrefetchChunk, bytes - o));
            }
        }
    }

    // ---- set-up: this cluster's work, barriers, TMEM ---------------------------------
    if (warp == 0) {
        const int c = (int)(blockIdx.x >> 2), C = (int)(gridDim.x >> 2);
        // the sequences' block counts, read from prefix_len once (all lanes at a time)
        const bool tab = p.B <= kSeqTable;
        if (tab)
            for (int b = lane; b < p.B; b += 32) bar.nb_tab[b] = seq_blocks(p, b);
        __syncwarp();
        const SeqBlocks nbs{p, tab ? bar.nb_tab : nullptr};
        int kov;
        const int R = cluster_schedule(p, nbs, C, lane, bar.sched_B, kov);
        __syncwarp();
        if (blockIdx.x == 0 && p.sched) {       // the cut points, for the merge pass
            for (int k = lane; k <= C; k += 32) p.sched[2 + k] = bar.sched_B[k];
            if (lane == 0) {
                p.sched[0] = R;
                p.sched[1] = kov;
            }
        }
        if (lane == 0) {
            const int u_first = R * C;
            int u0, nblk0, u1, nblk1;
            int64_t start0, pos0, start1, pos1;
            locate_vblock(p, nbs, u_first, kov, bar.sched_B[c], u0, start0, nblk0, pos0);
            locate_vblock(p, nbs, u_first, kov, bar.sched_B[c + 1], u1, start1, nblk1, pos1);
            int whole_blocks = 0;
            for (int k = 0; k < R; ++k) whole_blocks += nbs((k * C + c) / p.pairs_per_seq);
            bar.work_wleft = R;
            bar.work_u0 = u0;
            bar.work_kb0 = (int)(pos0 - start0);
            bar.work_left = (int)(pos1 - pos0);
            bar.work_count = whole_blocks + bar.work_left;
        }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kNK; ++i) { mbar_init(&bar.kfull[i], 1); mbar_init(&bar.kempty[i], 1); }
        for (int i = 0; i < kNR; ++i) { mbar_init(&bar.rfull[i], 1); mbar_init(&bar.rempty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&bar.sfull[i], 1); mbar_init(&bar.sempty[i], 16); }
        mbar_init(&bar.qpe_full, 1);
        mbar_init(&bar.qpe_empty, 1);
        mbar_init(&bar.q_ready, 16);
        for (int i = 0; i < kNP; ++i) {
            mbar_init(&bar.pempty[i], 1);
            mbar_init(&bar.pfull[i], 1);
            mbar_init(&bar.pready[i], 2);
            bar.need[0][i] = bar.need[1][i] = 0;
        }
        for (int i = 0; i < kNS; ++i) {
            mbar_init(&bar.sfree[i], 1);
            mbar_init(&bar.staged[i][0], 4);
            mbar_init(&bar.staged[i][1], 4);
        }
        for (int i = 0; i < kNV; ++i) { mbar_init(&bar.vfull[i], 1); mbar_init(&bar.vempty[i], 1); }
        mbar_init(&bar.go, 1);
        mbar_init(&bar.rescaled, 2);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar.stats_full[i], 4 * 32);
            mbar_init(&bar.stats_empty[i], kEpiWarps);
        }
        mbar_init(&bar.o_done, 1);
        mbar_init(&bar.o_free, 2 * kEpiWarps);
        bar.kseen[0] = bar.kseen[1] = -1;
        mbar_init(&bar.sync_bar, 1);
        // one drain commit per MMA issuer that runs: two in the S leader (one for a single
        // block), one in the O leader
        mbar_init(&bar.drain, (s_role && bar.work_count > 1) ? 2 : 1);
        bar.cmd = 0;
        bar.abort_flag = 0;
        bar.wait_ns = p.wait_ns;
        fence_mbar_init();
    }
    if (warp == 0) {           // collective over the pair: both CTAs get the same columns
        tmem_alloc_pair(&bar.tmem_base, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();            // every barrier of the cluster initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem = bar.tmem_base;

    // Every role walks the same sequence of items of this cluster's work range; per-block
    // state (ring slots, buffers, parities) follows the cluster-wide block counter g.
    const int cl = blockIdx.x >> 2, ncl = gridDim.x >> 2;
    const WorkIter w0 = {cl, bar.work_wleft, bar.work_u0, bar.work_kb0, bar.work_left, 0};
    const int G = bar.work_count;                  // key blocks of this cluster

    if (s_role) {
        // =============================== S-CTA ===============================
        unsigned char *qpe_tile = smem + kOffQpe;
        unsigned char *kring = smem + kOffKRing;
        unsigned char *rring = smem + kOffRRing;
        const uint32_t tmem_q = tmem;                 // Q_nope: columns [0, 256)
        const uint32_t tmem_s0 = tmem + 256;          // score buffers at 256 and 384
        if (warp == 0) {
            // ------- Q_pe per item; the leader arms the key rings ---------------------------
            // The key chunks are loaded by the O-CTAs (their copy engines carry less than
            // this one, which sends P); the leader only arms the pair's barriers: a slot's
            // next use is armed once the pair's MMAs have released it.
            if (elect_one() && G > 0) {
                RingPos kr, rr;
                bool going = true;
                WorkIter w = w0;
                Item it;
                int ii = 0;
                while (going && !aborted(bar) && next_item(p, w, cl, ncl, it)) {
                    // this CTA's Q_pe tile is free once the previous item's rope MMAs read it
                    if (ii > 0 && !(going = wait_or_abort(bar, &bar.qpe_empty, (uint32_t)(ii - 1) & 1, p.err, -24)))
                        break;
                    if (leader) mbar_arrive_expect_tx(&bar.qpe_full, 2 * kQpeBytes);
                    tma_load_2d_pair(qpe_tile, &map_qpe, map_to_rank(&bar.qpe_full, lead_rank), 0,
                                     (int)((int64_t)it.b * p.rows_seq + (it.rt0 + kpair) * kRows));
                    KDT_TC_TRACE(kEvQpeIssued, ii);
                    ++ii;
                    // a few blocks before the item ends, warm L2 with the next item's rows of Q
                    // (the pair's 256 rows are contiguous): its load then sits between two
                    // items on the tensor pipes' critical path
                    const int j_pf = it.nb > kQPrefetchBlocks ? it.nb - kQPrefetchBlocks : 0;
                    for (int j = 0; leader && j < it.nb && going; ++j) {
                        if (j == j_pf) {
                            WorkIter wn = w;
                            Item nx;
                            if (next_item(p, wn, cl, ncl, nx)) {
                                const int r0 = nx.rt0 * kRows;
                                const int nrows = min(2 * kRows, p.rows_seq - r0);
                                const unsigned char *qsrc = reinterpret_cast<const unsigned char *>(
                                    p.q_nope + ((int64_t)nx.b * p.rows_seq + r0) * p.q_stride);
                                const uint32_t bytes = (uint32_t)((nrows - 1) * p.q_stride + kDc) * 2;
                                for (uint32_t o = 0; o < bytes; o += kQPrefetchChunk)
                                    prefetch_l2_bulk(qsrc + o, min(kQPrefetchChunk, bytes - o));
                                for (int k = 0; k < 2 && r0 + k * kRows < p.rows_seq; ++k)
                                    tma_prefetch_2d(&map_qpe, 0, (int)((int64_t)nx.b * p.rows_seq + r0 + k * kRows));
                            }
                        }
                        for (int c = 0; c < kKChunks && going; ++c) {
                            if (kr.n >= kNK &&
                                !(going = wait_or_abort(bar, &bar.kempty[kr.slot], kr.phase ^ 1, p.err, -2)))
                                break;
                            if (kr.n >= kNK) KDT_TC_TRACE(kEvKEmpty, kr.n - kNK);
                            mbar_arrive_expect_tx(&bar.kfull[kr.slot], 2 * kKSlotBytes);
                            ring_advance<kNK>(kr);
                        }
                        if (!going) break;
                        if (rr.n >= kNR &&
                            !(going = wait_or_abort(bar, &bar.rempty[rr.slot], rr.phase ^ 1, p.err, -2)))
                            break;
                        mbar_arrive_expect_tx(&bar.rfull[rr.slot], 2 * kKSub);
                        ring_advance<kNR>(rr);
                    }
                }
                // drain (both S-CTAs): the MMA commits for the last uses of every slot mean
                // the copies into this CTA have landed and been read
                if (!leader) {
                    kr = RingPos{};
                    rr = RingPos{};
                    for (int u = 0; u < kKChunks * G; ++u) ring_advance<kNK>(kr);
                    for (int u = 0; u < G; ++u) ring_advance<kNR>(rr);
                }
                ring_drain<kNK>(bar.kempty, kr, bar.wait_ns);
                ring_drain<kNR>(bar.rempty, rr, bar.wait_ns);
                if (ii > 0) mbar_wait(&bar.qpe_empty, (uint32_t)(ii - 1) & 1, bar.wait_ns);
            }
        } else if (warp == 1 || warp == 2) {
            // ---------------- MMA issuers (leader): S = Q K^T for 256 rows -----------------
            // Two issuing threads, warp 1 for even blocks and warp 2 for odd ones: the tensor
            // queue is shallow, so while one thread waits on a barrier or commits, the other's
            // MMAs keep the pipe busy. Latent ring slots serve both threads in turn, so before
            // waiting on a slot's use u a thread makes sure the other thread has already seen
            // use u - kNK land (a parity wait can only tell adjacent phases apart). Rope slots
            // and score buffers follow block parity.
            const int par = warp - 1;
            if (leader && elect_one() && G > par) {
                const uint32_t idesc = idesc_bf16_f32(2 * kRows, kKeys, 0, 0);
                volatile int *seen_mine = &bar.kseen[par];
                volatile int *seen_other = &bar.kseen[par ^ 1];
                bool ok = true;
                WorkIter w = w0;
                Item it;
                int ii = 0, g = 0;
                while (ok && next_item(p, w, cl, ncl, it)) {
                    // this item's rows of Q are in tensor memory and its Q_pe tile landed
                    ok = wait_or_abort(bar, &bar.q_ready, (uint32_t)ii & 1, p.err, -3) &&
                         wait_or_abort(bar, &bar.qpe_full, (uint32_t)ii & 1, p.err, -3);
                    tc_fence_after();
                    for (int j = 0; j < it.nb && ok; ++j, ++g) {
                        if ((g & 1) != par) continue;
                        const int buf = g & 1;
                        if (g >= 2 && !(ok = wait_or_abort(bar, &bar.sempty[buf], (uint32_t)((g >> 1) - 1) & 1, p.err, -4)))
                            break;
                        tc_fence_after();
                        KDT_TC_TRACE(kEvSMmaStart, g);
                        const uint32_t d = tmem_s0 + buf * kKeys;
                        for (int c = 0; c < kKChunks; ++c) {
                            const int u = kKChunks * g + c;         // latent chunk use
                            const int slot = u % kNK;
                            // the slot's previous use belongs to the other thread when its block
                            // has the other parity: wait until that thread has seen it land
                            const int prev = u - kNK;
                            if (prev >= 0 && (((prev / kKChunks) & 1) != par)) {
                                const uint64_t t0 = global_ns();
                                while (*seen_other < prev) {
                                    if (aborted(bar) || global_ns() - t0 > bar.wait_ns) {
                                        set_abort(bar, p.err, -25);
                                        ok = false;
                                        break;
                                    }
                                }
                                if (!ok) break;
                            }
                            if (!(ok = wait_or_abort(bar, &bar.kfull[slot], (uint32_t)(u / kNK) & 1, p.err, -5))) break;
                            *seen_mine = u;
                            tc_fence_after();
                            KDT_TC_TRACE(kEvKFull, u);
                            // descriptors as a base plus compile-time offsets: the issue loop is a
                            // few adds per MMA, so one thread keeps up with the tensor pipe
                            const uint64_t bdesc0 = sdesc_sw128(smem_u32(kring + slot * kKSlotBytes), 16, 1024);
                            const uint32_t acol = tmem_q + 32 * kKSubPerChunk * c;
                            const uint32_t acc0 = c > 0 ? 1u : 0u;
#pragma unroll
                            for (int t = 0; t < kKSubPerChunk; ++t)   // sub-tile t: dims 64 (kKSubPerChunk c + t) .. +64
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    mma_ts_pair(d, acol + 32 * t + 8 * kk, bdesc0 + (uint64_t)((t * kKSub + kk * 32) >> 4),
                                                idesc, (t > 0 || kk > 0) ? 1u : acc0);
                            KDT_TC_TRACE(kEvKIssued, u);
                            mma_commit_pair(&bar.kempty[slot], kMaskAll);   // slot free: S-CTAs and their loaders
                        }
                        if (!ok) break;
                        const int rslot = g % kNR;
                        if (!(ok = wait_or_abort(bar, &bar.rfull[rslot], (uint32_t)(g / kNR) & 1, p.err, -5))) break;
                        tc_fence_after();
                        KDT_TC_TRACE(kEvRFull, g);
                        const uint64_t qdesc0 = sdesc_sw128(smem_u32(qpe_tile), 16, 1024);
                        const uint64_t rdesc0 = sdesc_sw128(smem_u32(rring + rslot * kKSub), 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)             // rope dims
                            mma_ss_pair(d, qdesc0 + (uint64_t)(kk * 2), rdesc0 + (uint64_t)(kk * 2), idesc, 1u);
                        mma_commit_pair(&bar.rempty[rslot], kMaskAll);
                        mma_commit_pair(&bar.sfull[buf], kMaskS);
                        // the item's last block: both CTAs' Q_pe tiles may be refilled once it ran
                        if (j == it.nb - 1) mma_commit_pair(&bar.qpe_empty, kMaskS);
                        KDT_TC_TRACE(kEvSMmaIssued, g);
                    }
                    ++ii;
                }
                drain_mmas(bar, 0x1);
            }
        } else if (warp == 3) {
            // ---------------- P copier: each half of P to the O-CTA once staged ---------------
            if (elect_one()) {
                for (int g = 0; g < G; ++g) {
                    const int ss = g % kNS, ps = g % kNP;
                    const uint32_t par = (uint32_t)(g / kNS) & 1;
                    bool ok = true;
                    for (int h = 0; h < 2 && ok; ++h) {
                        if (!(ok = wait_or_abort(bar, &bar.staged[ss][h], par, p.err, -22))) break;
                        const uint32_t off = (uint32_t)h * (kPBytes / 2);
                        bulk_copy_to_peer(smem_u32(smem + kOffP + ps * kPSlotBytes + off),
                                          smem + kOffPStage + ss * kPSlotBytes + off,
                                          h == 0 ? kPBytes / 2 : kPBytes / 2 + kRows * 4, &bar.pfull[ps], o_rank);
                        if (h == 0) KDT_TC_TRACE(kEvSoftmaxSent, g);
                    }
                    if (!ok) break;
                }
            }
        } else if (warp >= 4) {
            // ---------------- per item: Q_nope -> TMEM, softmax, statistics -----------------
            // Eight warps: warp w serves the 32 rows of TMEM lane quadrant (w % 4); warps 4-7
            // take keys 0..63 of each block, warps 8-11 keys 64..127.
            const int half = (warp - 4) >> 2;
            const int row = 32 * (warp & 3) + lane;
            float *rowmax_s = reinterpret_cast<float *>(smem + kOffRowMax);
            float *lsum_s = reinterpret_cast<float *>(smem + kOffLSum);
            bool ok = true;
            bool fail = false;
            bool vis_ready = false;                    // the visibility bits are known to be written
            // Q_nope of an item's rows into tensor memory, 16 loads in flight per thread
            auto load_q = [&](const Item &q, bool withhold) {
                const int Rq = (q.rt0 + kpair) * kRows + row;
                const bool valid = Rq < p.rows_seq;
                const uint4 *src =
                    reinterpret_cast<const uint4 *>(p.q_nope + ((int64_t)q.b * p.rows_seq + Rq) * p.q_stride) + 32 * half;
#pragma unroll
                for (int r2 = 0; r2 < 2; ++r2) {
                    uint4 v[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) v[k] = valid ? __ldg(src + 16 * r2 + k) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t wq[32];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            wq[4 * k] = v[8 * h + k].x;
                            wq[4 * k + 1] = v[8 * h + k].y;
                            wq[4 * k + 2] = v[8 * h + k].z;
                            wq[4 * k + 3] = v[8 * h + k].w;
                        }
                        tmem_st32(tmem_lane_addr(tmem_q, warp, (4 * half + 2 * r2 + h) * 32), wq);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && !withhold) mbar_arrive_remote_cta(&bar.q_ready, lead_rank);
            };
            WorkIter w = w0;
            Item it;
            int ii = 0, g = 0;
            bool have = next_item(p, w, cl, ncl, it);
            if (have) {
                load_q(it, p.fault == 1);                  // the test hook leaves Q-ready one arrival short
                if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvQReady, 0);
            }
            while (!fail && have) {
                const int R = (it.rt0 + kpair) * kRows + row;
                const int qi = min(R, p.rows_seq - 1) / p.H;
                const uint32_t *visrow = p.vis + ((int64_t)it.b * p.T + qi) * p.W;
                float m_run = -INFINITY;                           // log2 units, same in both halves
                float l_run = 0.f;                                 // this half's share of the row sum
                for (int j = 0; j < it.nb; ++j, ++g) {
                    // No warp leaves this loop on its own: every iteration meets the other seven
                    // at the named barrier, which ORs their failures.
                    const int buf = g & 1;
                    const int ss = g % kNS;                        // staging slot here
                    const int ps = g % kNP;                        // P slot in the O-CTA
                    ok = ok && warp_wait(bar, &bar.sfull[buf], (uint32_t)(g >> 1) & 1, p.err, -6);
                    float x[64];
                    float mx = -INFINITY;
                    bool masked = false;                            // block half holds hidden keys
                    if (ok) {
                        tc_fence_after();
                        if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvSoftmaxIn, g);
                        uint32_t r0v[32], r1v[32];
                        const uint32_t sbase = tmem_s0 + buf * kKeys + 64 * half;
                        tmem_ld32(tmem_lane_addr(sbase, warp, 0), r0v);
                        tmem_ld32(tmem_lane_addr(sbase, warp, 32), r1v);
                        tmem_wait_ld();
                        if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvSoftmaxLd, g);
#pragma unroll
                        for (int q = 0; q < 32; ++q) {             // raw scores
                            x[q] = __uint_as_float(r0v[q]);
                            x[32 + q] = __uint_as_float(r1v[q]);
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_remote_cta(&bar.sempty[buf], lead_rank);   // buffer may be overwritten
                        if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvSoftmaxLoaded, g);
                        const int key0 = it.key_base + (it.kb0 + j) * kKeys + 64 * half;
                        masked = key0 < 0 || key0 + 64 > it.P;     // leading pad or tree keys
                        if (masked) {   // scale now, hidden keys -inf (also right for scale 0)
                            // the bits may come from the visibility kernel launched just before
                            // this one: wait for it before the first window with tree keys
                            if (!vis_ready && key0 + 64 > it.P) {
                                griddep_wait();
                                vis_ready = true;
                            }
                            const uint64_t vm = vis_mask64(visrow, p.W, key0, it.P);
#pragma unroll
                            for (int c = 0; c < 64; ++c) x[c] = ((vm >> c) & 1ull) ? x[c] * p.scale_log2 : -INFINITY;
#pragma unroll
                            for (int c = 0; c < 64; ++c) mx = fmaxf(mx, x[c]);
                        } else {        // all visible: raw scores kept, the scale goes into the exponent
                            mx = scaled_max64(x, p.scale_log2);
                        }
                        rowmax_s[(buf * 2 + half) * kRows + row] = mx;
                    }
                    if (barrier_or<2, 256>(!ok)) {
                        fail = true;
                        break;
                    }
                    if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvSoftmaxMax, g);
                    mx = fmaxf(mx, rowmax_s[(buf * 2 + (half ^ 1)) * kRows + row]);
                    float alpha = 1.f;
                    if (mx > m_run + kRescaleThreshold || (m_run == -INFINITY && mx > -INFINITY)) {
                        alpha = (m_run == -INFINITY) ? 1.f : fast_exp2(m_run - mx);
                        m_run = mx;
                        l_run *= alpha;
                    }
                    // the O-CTA's P slot is free once P.V of block g - kNP has run; this CTA's
                    // staging slot once the copy of block g - kNS has landed
                    ok = (g < kNP || warp_wait(bar, &bar.pempty[ps], (uint32_t)((g / kNP) - 1) & 1, p.err, -7)) &&
                         (g < kNS || warp_wait(bar, &bar.sfree[ss], (uint32_t)((g / kNS) - 1) & 1, p.err, -19));
                    if (ok) {
                        if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvSoftmaxSlot, g);
                        unsigned char *slot_base = smem + kOffPStage + ss * kPSlotBytes;
                        unsigned char *stage_row = slot_base + half * (kPBytes / 2) + row * 128;
                        // an all-visible half has finite scores, so m_run is finite here
                        l_run += masked ? stage_p_row<true>(x, p.scale_log2, m_run, stage_row, row)
                                        : stage_p_row<false>(x, p.scale_log2, m_run, stage_row, row);
                        // the rescale factors follow the second half of P, which carries them
                        if (half == 1) reinterpret_cast<float *>(slot_base + kPBytes)[row] = alpha;
                        fence_proxy_async_smem();                  // staging visible to the copy engine
                        __syncwarp();
                        // hand the rows to the copy thread without waiting for the other warps
                        if (lane == 0) mbar_arrive(&bar.staged[ss][half]);
                        if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvSoftmaxStaged, g);
                    }
                }
                if (fail) break;
                // this item's statistics for the O-CTA epilogue: (m, l), l over both halves
                if (half == 1) lsum_s[row] = l_run;
                if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvItemEnd0, ii);
                if (warp == 8 && lane == 0) KDT_TC_TRACE(kEvItemEnd1, ii);
                fail = barrier_or<2, 256>(!ok);
                if (fail) break;
                if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvItemBar, ii);
                const int sb = ii & 1;                            // statistics buffer of this item
                if (half == 0) {
                    // the O-CTA has read this buffer's previous contents (item ii - 2)
                    ok = ii < 2 || warp_wait(bar, &bar.stats_empty[sb], (uint32_t)((ii >> 1) - 1) & 1, p.err, -26);
                    if (ok) {
                        const uint32_t dst = map_to_rank(smem + kOffStats + (sb * kRows + row) * 8, o_rank);
                        st_cluster_f32(dst, m_run);
                        st_cluster_f32(dst + 4, l_run + lsum_s[row]);
                        // every lane releases its own two stores: no fence on this path
                        mbar_arrive_remote(&bar.stats_full[sb], o_rank);
                    }
                    if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvStatsSent, ii);
                }
                ++ii;
                // the next item's Q_nope: tensor memory is free, every MMA of this item ran
                // before its last scores could be read
                have = next_item(p, w, cl, ncl, it);
                if (have && ok) {
                    load_q(it, false);
                    if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvQReady, ii);
                }
                // lsum_s is rewritten at the end of the next item only after this barrier
                fail = barrier_or<2, 256>(!ok);
            }
            // The O pair's MMA commits (pempty), the O-CTA's watcher (sfree) and its epilogue
            // (stats_empty) arrive here; the arrivals still due are consumed before this CTA
            // may leave, so none can land in the shared memory of a CTA that later runs here.
            if (!fail && ok && warp == 4) {
                for (int ps = 0; ps < kNP && ps < G; ++ps) {
                    const int g_last = ps + ((G - 1 - ps) / kNP) * kNP;
                    ok = warp_wait(bar, &bar.pempty[ps], (uint32_t)(g_last / kNP) & 1, p.err, -18) && ok;
                }
                for (int ss = 0; ss < kNS && ss < G; ++ss) {
                    const int g_last = ss + ((G - 1 - ss) / kNS) * kNS;
                    ok = warp_wait(bar, &bar.sfree[ss], (uint32_t)(g_last / kNS) & 1, p.err, -20) && ok;
                }
                for (int sb = 0; sb < 2 && sb < ii; ++sb) {
                    const int i_last = sb + ((ii - 1 - sb) / 2) * 2;
                    ok = warp_wait(bar, &bar.stats_empty[sb], (uint32_t)(i_last >> 1) & 1, p.err, -27) && ok;
                }
            }
        }
    } else {
        // =============================== O-CTA ===============================
        unsigned char *pbase = smem + kOffP;
        unsigned char *vbase = smem + kOffV;
        const float2 *stats_s = reinterpret_cast<const float2 *>(smem + kOffStats);
        if (warp == 0) {
            // ------- TMA producer: this CTA's 128 of each 256 latent columns of V -------
            if (elect_one() && G > 0) {
                tma_prefetch_desc(&map_vs);
                RingPos vr;
                bool going = true;
                WorkIter w = w0;
                Item it;
                while (going && !aborted(bar) && next_item(p, w, cl, ncl, it)) {
                    for (int j = 0; j < it.nb && going; ++j) {
                        const int key0 = it.key_base + (it.kb0 + j) * kKeys;
                        for (int h = 0; h < kVChunks; ++h) {
                            if (vr.n >= kNV &&
                                !(going = wait_or_abort(bar, &bar.vempty[vr.slot], vr.phase ^ 1, p.err, -8)))
                                break;
                            if (leader) mbar_arrive_expect_tx(&bar.vfull[vr.slot], 2 * kVSlotBytes);
                            // chunk h of the pair spans 2 kVSubPerChunk sub-tiles of latent dims, the
                            // first kVSubPerChunk from O-CTA 0, the rest from O-CTA 1: one request
                            tma_load_4d_pair(vbase + vr.slot * kVSlotBytes, &map_vs, map_to_rank(&bar.vfull[vr.slot], lead_rank),
                                             0, key0, (2 * h + kpair) * kVSubPerChunk, it.b);
                            KDT_TC_TRACE(kEvVIssue, vr.n);
                            ring_advance<kNV>(vr);
                        }
                    }
                }
                ring_drain<kNV>(bar.vempty, vr, bar.wait_ns);
            }
        } else if (warp == 1) {
            // ---------------- MMA issuer (leader): O += P V for 256 rows --------------------
            if (leader && elect_one() && G > 0) {
                const uint32_t idesc = idesc_bf16_f32(2 * kRows, 128 * kVSubPerChunk, 0, 1);
                RingPos vr;
                uint32_t rs_phase = 0, sync_phase = 0;
                bool ok = true;
                WorkIter w = w0;
                Item it;
                int ii = 0, g = 0;
                while (ok && next_item(p, w, cl, ncl, it)) {
                    // the previous item's epilogue has read O out of tensor memory
                    if (ii > 0 && !(ok = wait_cluster_or_abort(bar, &bar.o_free, (uint32_t)(ii - 1) & 1, p.err, -28)))
                        break;
                    KDT_TC_TRACE(kEvOFree, ii);
                    for (int j = 0; j < it.nb && ok; ++j, ++g) {
                        const int ps = g % kNP;
                        if (!(ok = wait_cluster_or_abort(bar, &bar.pready[ps], (uint32_t)(g / kNP) & 1, p.err, -9))) break;
                        KDT_TC_TRACE(kEvOMmaStart, g);
                        const uint32_t n0 = *reinterpret_cast<volatile uint32_t *>(&bar.need[0][ps]);
                        const uint32_t n1 = *reinterpret_cast<volatile uint32_t *>(&bar.need[1][ps]);
                        if (n0 | n1) {
                            // let every P.V issued so far finish, then hand O to the CTAs whose
                            // rows need the rescale (the others count as done at once)
                            mma_commit_pair(&bar.sync_bar, 0x4);
                            if (!(ok = wait_or_abort(bar, &bar.sync_bar, sync_phase, p.err, -15))) break;
                            sync_phase ^= 1;
                            tc_fence_before();
                            for (uint32_t k = 0; k < 2; ++k) {
                                if (k == 0 ? n0 : n1) {
                                    st_cluster_u32(map_to_rank(&bar.cmd, 2 + k), (uint32_t)ps);
                                    mbar_arrive_remote(&bar.go, 2 + k);      // release: command first
                                } else {
                                    mbar_arrive(&bar.rescaled);
                                }
                            }
                            if (!(ok = wait_cluster_or_abort(bar, &bar.rescaled, rs_phase, p.err, -16))) break;
                            rs_phase ^= 1;
                        }
                        tc_fence_after();
                        const uint64_t adesc0 = sdesc_sw128(smem_u32(pbase + ps * kPSlotBytes), 16, 1024);
                        const uint32_t acc0 = j > 0 ? 1u : 0u;
                        for (int h = 0; h < kVChunks; ++h) {
                            if (!(ok = wait_or_abort(bar, &bar.vfull[vr.slot], vr.phase, p.err, -10))) break;
                            tc_fence_after();
                            KDT_TC_TRACE(kEvVFull, vr.n);
                            const uint64_t bdesc0 = sdesc_sw128(smem_u32(vbase + vr.slot * kVSlotBytes), kVSub, 1024);
                            const uint32_t dcol = tmem + 128 * kVSubPerChunk * h;
#pragma unroll
                            for (int kk = 0; kk < kKeys / 16; ++kk)   // the item's first block starts O afresh
                                mma_ss_pair(dcol, adesc0 + (uint64_t)(((kk >> 2) * (kPBytes / 2) + (kk & 3) * 32) >> 4),
                                            bdesc0 + (uint64_t)((kk * 2048) >> 4), idesc, kk > 0 ? 1u : acc0);
                            mma_commit_pair(&bar.vempty[vr.slot], kMaskO);   // slot free in both O-CTAs
                            ring_advance<kNV>(vr);
                        }
                        if (!ok) break;
                        KDT_TC_TRACE(kEvOMmaIssued, g);
                        // P slot ps of both O-CTAs is free again: tell both S-CTAs
                        mma_commit_pair(&bar.pempty[ps], kMaskS);
                    }
                    if (!ok) break;
                    // the item's P.V is complete once this arrives; the epilogues then read O
                    mma_commit_pair(&bar.o_done, kMaskO);
                    for (uint32_t k = 0; k < 2; ++k) {   // end the correction loop of this item
                        st_cluster_u32(map_to_rank(&bar.cmd, 2 + k), kCmdDone);
                        mbar_arrive_remote(&bar.go, 2 + k);
                    }
                    ++ii;
                }
                if (!ok) {   // release the correction warps of an item left unfinished
                    for (uint32_t k = 0; k < 2; ++k) {
                        st_cluster_u32(map_to_rank(&bar.cmd, 2 + k), kCmdDone);
                        mbar_arrive_remote(&bar.go, 2 + k);
                    }
                }
                drain_mmas(bar, kMaskO);
            }
        } else if (warp == 3) {
            // ------- key loader: S-CTA k's half of each key block, into its shared memory -------
            // Multicast to that one CTA with pair semantics: the bytes complete on the S
            // leader's barrier, which counts both S-CTAs' halves.
            if (elect_one() && G > 0) {
                tma_prefetch_desc(&map_ks);
                tma_prefetch_desc(&map_kpe);
                const uint16_t dst_mask = (uint16_t)(1u << kpair);
                unsigned char *kring = smem + kOffKRing;     // same offsets as in the S-CTA
                unsigned char *rring = smem + kOffRRing;
                RingPos kr, rr;
                bool going = true;
                // L2 prefetch cursor, kKvPrefetchBlocks blocks ahead of the loads: the clusters
                // on one sequence ask for each block at about the same time, so without it every
                // one of them waits for the same DRAM fetch
                WorkIter wp = w0;
                Item ip;
                int jp = 0;
                bool pf = next_item(p, wp, cl, ncl, ip);
                auto prefetch_block = [&]() {
                    if (!pf) return;
                    const int pk0 = ip.key_base + (ip.kb0 + jp) * kKeys + kpair * kHalfKeys;
                    for (int c = 0; c < kKChunks; ++c) tma_prefetch_4d(&map_ks, 0, pk0, kKSubPerChunk * c, ip.b);
                    tma_prefetch_3d(&map_kpe, 0, pk0, ip.b);
                    if (++jp == ip.nb) {
                        jp = 0;
                        pf = next_item(p, wp, cl, ncl, ip);
                    }
                };
                for (int k = 0; k < kKvPrefetchBlocks; ++k) prefetch_block();
                WorkIter w = w0;
                Item it;
                while (going && !aborted(bar) && next_item(p, w, cl, ncl, it)) {
                    for (int j = 0; j < it.nb && going; ++j) {
                        prefetch_block();
                        const int key0 = it.key_base + (it.kb0 + j) * kKeys + kpair * kHalfKeys;   // S-CTA k's 64 keys
                        for (int c = 0; c < kKChunks && going; ++c) {   // latent sub-tiles [kKSubPerChunk c, +kKSubPerChunk)
                            if (kr.n >= kNK &&
                                !(going = wait_or_abort(bar, &bar.kempty[kr.slot], kr.phase ^ 1, p.err, -21)))
                                break;
                            tma_load_4d_pair_mc(kring + kr.slot * kKSlotBytes, &map_ks,
                                                map_to_rank(&bar.kfull[kr.slot], 0), 0, key0, kKSubPerChunk * c, it.b, dst_mask);
                            KDT_TC_TRACE(kEvKIssue, kr.n);
                            ring_advance<kNK>(kr);
                        }
                        if (!going) break;
                        if (rr.n >= kNR &&
                            !(going = wait_or_abort(bar, &bar.rempty[rr.slot], rr.phase ^ 1, p.err, -21)))
                            break;
                        tma_load_3d_pair_mc(rring + rr.slot * kKSub, &map_kpe, map_to_rank(&bar.rfull[rr.slot], 0), 0,
                                            key0, it.b, dst_mask);
                        ring_advance<kNR>(rr);
                    }
                }
                // every copy this CTA issued has landed and been read before it may exit
                ring_drain<kNK>(bar.kempty, kr, bar.wait_ns);
                ring_drain<kNR>(bar.rempty, rr, bar.wait_ns);
            }
        } else if (warp == 2) {
            // ---------------- P watcher: P of each block landed, and does O need a rescale? --
            for (int g = 0; g < G; ++g) {
                const int ps = g % kNP;
                if (lane == 0) mbar_arrive_expect_tx(&bar.pfull[ps], kPTx);   // P + alpha of block g
                if (!warp_wait(bar, &bar.pfull[ps], (uint32_t)(g / kNP) & 1, p.err, -11)) break;
                if (lane == 0) KDT_TC_TRACE(kEvCorrIn, g);
                // factors other than 1 only occur once a row has a running maximum, i.e. not in
                // the first block of an item, whose P.V starts O afresh
                const float4 a4 = reinterpret_cast<const float4 *>(pbase + ps * kPSlotBytes + kPBytes)[lane];
                const bool need = __any_sync(0xffffffffu, a4.x != 1.f || a4.y != 1.f || a4.z != 1.f || a4.w != 1.f);
                if (lane == 0) {
                    mbar_arrive_remote_cta(&bar.sfree[g % kNS], (uint32_t)kpair);   // its staging slot is reusable
                    st_cluster_u32(map_to_rank(&bar.need[kpair][ps], lead_rank), need ? 1u : 0u);
                    mbar_arrive_remote(&bar.pready[ps], lead_rank);                 // release: flag first
                }
                __syncwarp();
            }
        } else if (warp >= 4 && warp < 4 + kEpiWarps) {
            // ---------------- correction (rare rescale) and epilogue, per item ----------------
            // Warp w serves the 32 rows of TMEM lane quadrant (w % 4) and the columns
            // [col0, col0 + kEpiGroupCols); named barrier 1 counts these warps. They sleep on
            // `go` until the MMA thread hands O over for a rescale or ends the item.
            const int row = 32 * (warp & 3) + lane;
            const int col0 = ((warp - 4) >> 2) * kEpiGroupCols;
            bool ok = true;
            uint32_t e = 0;                                     // `go` events so far
            WorkIter w = w0;
            Item it;
            int ii = 0;
            while (ok && next_item(p, w, cl, ncl, it)) {
                for (;; ++e) {
                    ok = warp_wait_cluster(bar, &bar.go, e & 1, p.err, -12);
                    if (barrier_or<1, 32 * kEpiWarps>(!ok)) {
                        ok = false;
                        break;
                    }
                    const uint32_t cmd = *reinterpret_cast<volatile uint32_t *>(&bar.cmd);
                    if (cmd == kCmdDone) {
                        ++e;
                        break;
                    }
                    // every P.V before the block in P slot `cmd` has completed: rescale this
                    // CTA's rows of O by that block's factors (rows that need none multiply by 1)
                    const float a = reinterpret_cast<const float *>(pbase + (cmd % kNP) * kPSlotBytes + kPBytes)[row];
                    tc_fence_after();
                    for (int c = 0; c < kEpiGroupCols / 32; ++c) {
                        uint32_t r[32];
                        const uint32_t addr = tmem_lane_addr(tmem, warp, col0 + c * 32);
                        tmem_ld32(addr, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 32; ++q) r[q] = __float_as_uint(__uint_as_float(r[q]) * a);
                        tmem_st32(addr, r);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    barrier_or<1, 32 * kEpiWarps>(false);  // every warp's stores done
                    if (threadIdx.x == 128) mbar_arrive_remote(&bar.rescaled, lead_rank);
                }
                if (!ok) break;
                // epilogue of the item: o = O / l, lse = ln2 (m + log2 l); whole units write the
                // final rows, pieces their partial state
                const int sb = ii & 1;
                ok = warp_wait(bar, &bar.o_done, (uint32_t)ii & 1, p.err, -13) &&
                     warp_wait_cluster(bar, &bar.stats_full[sb], (uint32_t)(ii >> 1) & 1, p.err, -14);
                if (barrier_or<1, 32 * kEpiWarps>(!ok)) {
                    ok = false;
                    break;
                }
                if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvEpiIn, ii);
                tc_fence_after();
                const int R = (it.rt0 + kpair) * kRows + row;
                const int64_t grow = (int64_t)it.b * p.rows_seq + R;
                float *orow, *lrow;
                if (it.whole) {
                    orow = p.out + grow * kDc;
                    lrow = p.lse ? p.lse + grow : nullptr;
                } else {
                    const int64_t k = (int64_t)it.slot * (2 * kRows) + kpair * kRows + row;
                    orow = p.part_o + k * kDc;
                    lrow = p.part_lse + k;
                }
                const float2 st = stats_s[sb * kRows + row];
                const float inv = st.y > 0.f ? 1.f / st.y : 0.f;
                // Each thread holds one row; the rows go out through a per-warp transpose in
                // shared memory so that every store instruction writes whole 32-byte sectors
                // (eight rows x 64 bytes). 16-byte slot q of staged row r sits at
                // q ^ ((r >> 1) & 3), which keeps both the row-wise writes and the
                // sector-wise reads at the minimum number of shared-memory wavefronts.
                static_assert(kEpiCols == 16, "the transpose below stages 16 columns");
                float *stg = reinterpret_cast<float *>(smem + kOffEpi) + (warp - 4) * 32 * kEpiCols;
                const int rsub = lane >> 2, qsub = lane & 3;      // read side: row 8i + rsub, slot qsub
                float *orow0 = orow - (int64_t)lane * kDc + col0; // row 0 of this warp's 32, its first column
                const int rows_ok = p.rows_seq - (R - lane);      // rows of the 32 that exist
                for (int c = 0; c < kEpiGroupCols / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tmem_lane_addr(tmem, warp, col0 + c * 32), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<float4 *>(stg + lane * kEpiCols + ((q ^ ((lane >> 1) & 3)) << 2)) =
                                make_float4(__uint_as_float(r[16 * hh + 4 * q]) * inv, __uint_as_float(r[16 * hh + 4 * q + 1]) * inv,
                                            __uint_as_float(r[16 * hh + 4 * q + 2]) * inv,
                                            __uint_as_float(r[16 * hh + 4 * q + 3]) * inv);
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int rr = 8 * i + rsub;
                            const float4 v =
                                *reinterpret_cast<const float4 *>(stg + rr * kEpiCols + ((qsub ^ ((rr >> 1) & 3)) << 2));
                            if (rr < rows_ok)
                                *reinterpret_cast<float4 *>(orow0 + (int64_t)rr * kDc + c * 32 + hh * 16 + 4 * qsub) = v;
                        }
                        __syncwarp();
                    }
                }
                if (col0 == 0 && R < p.rows_seq && lrow) *lrow = st.y > 0.f ? 0.6931471805599453f * (st.x + log2f(st.y)) : -INFINITY;
                // O may be overwritten and the statistics buffer refilled
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_remote(&bar.o_free, lead_rank);
                    mbar_arrive_remote_cta(&bar.stats_empty[sb], (uint32_t)kpair);
                }
                if (warp == 4 && lane == 0) KDT_TC_TRACE(kEvEpiOut, ii);
                ++ii;
            }
        }
    }

    // ---- teardown ------------------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (aborted(bar)) {
        // Error path only: copies another CTA issued before it noticed may still be in
        // flight; give them time to land (they take microseconds) before any CTA of the
        // cluster can leave.
        const uint64_t t0 = global_ns();
        do {
            __nanosleep(1000);
        } while (global_ns() - t0 < 200000ull);
    }
    griddep_launch_dependents();   // the merge pass may launch once every CTA got here
    cluster_sync();            // no CTA leaves while another may still touch its shared memory
    tc_fence_after();
    if (warp == 0) tmem_dealloc_pair(tmem, 512);
}

// Combines the pieces of each unit cut by a boundary of the work split. Block (c - 1, y)
// serves boundary c when c is the first boundary inside its unit, rows 8y .. 8y + 7 of
// the unit's 256 (one warp per row, 16 columns per lane): the normalised partial states
// (o_k, lse_k) of the pieces combine exactly as the log-sum-exp merge of disjoint key
// sets, o = sum_k e^(lse_k - M) o_k / sum_k e^(lse_k - M) with M the largest lse_k.
__global__ void __launch_bounds__(256) merge_pieces_kernel(const TcParams p, int C) {
    __shared__ int s_valid, s_n, s_b, s_rt0;
    __shared__ int s_slot[kMaxClusters + 1];
    __shared__ int s_nb[kSeqTable];
    const int c = blockIdx.x + 1;
    const bool tab = p.B <= kSeqTable;
    if (tab)
        for (int b = threadIdx.x; b < p.B; b += blockDim.x) s_nb[b] = seq_blocks(p, b);
    // launched to overlap the attention kernel's end: its pieces and cut points are read
    // only after it completed
    griddep_wait();
    __syncthreads();
    if (threadIdx.x == 0) {
        s_valid = 0;
        // the cut points the kernel computed and wrote
        const int R = (int)p.sched[0], kov = (int)p.sched[1];
        const int64_t *B = p.sched + 2;
        const int u_first = R * C;
        const SeqBlocks nbs{p, tab ? s_nb : nullptr};
        // key-block position of range boundary k, as the kernel computes it
        auto boundary = [&](int k, int &uu, int64_t &st, int &nb) {
            int64_t pos;
            locate_vblock(p, nbs, u_first, kov, B[k], uu, st, nb, pos);
            return pos;
        };
        int u, nblk, ud, nd;
        int64_t start, sd;
        const int64_t sc = boundary(c, u, start, nblk);
        const int64_t sprev = boundary(c - 1, ud, sd, nd);
        if (nblk > 0 && sc > start && sprev <= start) {
            int n = 0;
            s_slot[n++] = 2 * (c - 1) + (sprev == start ? 0 : 1);   // the piece that starts the unit
            for (int cc = c; cc < C && n <= kMaxClusters; ++cc) {
                const int64_t lo = boundary(cc, ud, sd, nd), hi = boundary(cc + 1, ud, sd, nd);
                if (lo >= start + nblk) break;
                if (hi > lo) s_slot[n++] = 2 * cc;                 // pieces that start a cluster's tail range
            }
            s_n = n;
            s_b = u / p.pairs_per_seq;
            s_rt0 = 2 * (u % p.pairs_per_seq);
            s_valid = 1;
        }
    }
    __syncthreads();
    if (!s_valid) return;
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.y * 8 + (threadIdx.x >> 5);        // row of the unit, 0..255
    const int R = s_rt0 * kRows + r;
    if (R >= p.rows_seq) return;
    // the pieces' lse, 32 at a time across the lanes (one round trip for the weights), then
    // their rows of o weighted and summed (independent loads)
    const int n = s_n;
    float M = -INFINITY;
    for (int base = 0; base < n; base += 32) {
        const float l = base + lane < n ? p.part_lse[(int64_t)s_slot[base + lane] * (2 * kRows) + r] : -INFINITY;
        float m = l;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        M = fmaxf(M, m);
    }
    float sum = 0.f;
    float4 acc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = 0; base < n && M > -INFINITY; base += 32) {
        const float l = base + lane < n ? p.part_lse[(int64_t)s_slot[base + lane] * (2 * kRows) + r] : -INFINITY;
        const float w = l == -INFINITY ? 0.f : expf(l - M);   // a piece with no visible key weighs 0
        float ws = w;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, off);
        sum += ws;
        const int cnt = n - base < 32 ? n - base : 32;
#pragma unroll 4
        for (int k = 0; k < cnt; ++k) {
            const float wk = __shfl_sync(0xffffffffu, w, k);
            if (wk == 0.f) continue;
            const float4 *src =
                reinterpret_cast<const float4 *>(p.part_o + ((int64_t)s_slot[base + k] * (2 * kRows) + r) * kDc);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 v = __ldg(src + lane + 32 * q);
                acc[q] = make_float4(fmaf(wk, v.x, acc[q].x), fmaf(wk, v.y, acc[q].y), fmaf(wk, v.z, acc[q].z),
                                     fmaf(wk, v.w, acc[q].w));
            }
        }
    }
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    const int64_t grow = (int64_t)s_b * p.rows_seq + R;
    float4 *dst = reinterpret_cast<float4 *>(p.out + grow * kDc);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        dst[lane + 32 * q] = make_float4(acc[q].x * inv, acc[q].y * inv, acc[q].z * inv, acc[q].w * inv);
    if (lane == 0 && p.lse) p.lse[grow] = sum > 0.f ? M + logf(sum) : -INFINITY;
}

}  // namespace

int tc_rows_per_unit() { return 2 * kRows; }
int tc_keys_per_block() { return kKeys; }

int tc_max_clusters() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return sm_count() / 4 > 0 ? sm_count() / 4 : 1;
    const int slot = dev & 63;
    int n = cached[slot].load(std::memory_order_relaxed);
    if (n > 0) return n;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 4;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaFuncSetAttribute(verify_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, verify_tc_kernel, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();    // clear the query's error; plan with the SM count instead
        const int f = sm_count() / 4;
        return f < 1 ? 1 : (f > kMaxClusters ? kMaxClusters : f);
    }
    if (n > kMaxClusters) n = kMaxClusters;
    cached[slot].store(n, std::memory_order_relaxed);
    return n;
}

namespace {

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


cudaError_t launch_verify_tc(const VerifyParams &vp, cudaStream_t s) {
    CUtensorMap map_ks, map_vs, map_kpe, map_qpe;
    const cuuint64_t L = (cuuint64_t)vp.L;
    {
        // c_kv viewed as [B][8 dim-blocks][L keys][64]: a box of (64, n keys, m blocks)
        // lands as m consecutive [n x 64] 128B-swizzled sub-tiles.
        cuuint64_t dims[4] = {64, L, (cuuint64_t)(kDc / 64), (cuuint64_t)vp.B};
        cuuint64_t strides[3] = {(cuuint64_t)kDc * 2, 128, L * kDc * 2};
        cuuint32_t box_k[4] = {64, kHalfKeys, kKSubPerChunk, 1};   // S-CTA: its 64 keys x one chunk of dims
        cuuint32_t box_v[4] = {64, kKeys, kVSubPerChunk, 1};       // O-CTA: 128 keys x its dims of one chunk
        if (!make_map(&map_ks, vp.c_kv, 4, dims, strides, box_k)) return cudaErrorInvalidValue;
        if (!make_map(&map_vs, vp.c_kv, 4, dims, strides, box_v)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[3] = {(cuuint64_t)kDr, L, (cuuint64_t)vp.B};
        cuuint64_t strides[2] = {(cuuint64_t)kDr * 2, L * kDr * 2};
        cuuint32_t box[3] = {64, kHalfKeys, 1};
        if (!make_map(&map_kpe, vp.k_pe, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)kDr, (cuuint64_t)vp.rows_total};
        cuuint64_t strides[1] = {(cuuint64_t)vp.q_pe_stride * 2};   // rows may sit inside a combined buffer
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
    p.rows_total = vp.rows_total;
    p.q_nope = static_cast<const __nv_bfloat16 *>(vp.q_nope);
    p.q_stride = vp.q_nope_stride;
    p.prefix_len = vp.prefix_len;
    p.vis = vp.vis;
    p.scale_log2 = vp.scale_log2;
    p.out = vp.out;
    p.lse = vp.lse;
    p.part_o = vp.part_o;
    p.part_lse = vp.part_lse;
    p.err = vp.err;
    p.pairs_per_seq = (p.row_tiles + 1) / 2;
    p.wait_ns = vp.wait_ns ? vp.wait_ns : kWaitLimit;
    p.fault = vp.fault;
    p.sched = vp.tc_sched;
    const int C = vp.tc_clusters;
    if (C < 1 || C > kMaxClusters || (C > 1 && (!p.part_o || !p.part_lse || !p.sched))) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(verify_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    // Programmatic dependent launch: this kernel overlaps the visibility kernel launched
    // just before it in the same call (it waits for it before reading the bits), and the
    // merge pass overlaps this kernel's end (it waits before reading the pieces).
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(4 * C));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = vp.overlap_vis ? 1 : 0;
    if ((e = cudaLaunchKernelEx(&cfg, verify_tc_kernel, map_ks, map_vs, map_kpe, map_qpe, p)) != cudaSuccess) return e;
    if (C > 1) {
        cudaLaunchConfig_t mc = {};
        mc.gridDim = dim3((unsigned)(C - 1), 2 * kRows / 8);
        mc.blockDim = dim3(256);
        mc.stream = s;
        mc.attrs = pdl;
        mc.numAttrs = 1;
        e = cudaLaunchKernelEx(&mc, merge_pieces_kernel, p, C);
    }
    return e;
}

}  // namespace kdt
