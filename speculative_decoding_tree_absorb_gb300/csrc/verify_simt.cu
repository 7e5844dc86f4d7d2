// K3: SIMT tree-verify MLA-absorb attention (fp32 arithmetic; fp32 or bf16 inputs).
//
// Computes, for every row r = (i, h) of sequence b (rows of one sequence are the
// contiguous [T*H] block of q), the score of each visible key
//   s_j = scale * (q_nope[r] . c_kv[j] + q_pe[r] . k_pe[j])
// (page "The Verify-Attn Kernel: A Single File Write ...", section "The Design
// Journey: From Concept to CUDA"), masks keys outside prefix + ancestors + self,
// and accumulates softmax(s) . c_kv with an online (running-max) softmax over key
// blocks -- the tiling that page's "Design Decisions and Trade-Offs" section
// names for contexts beyond the single shared-memory score array.
//
// Design (differs from the pages' one-block-per-(b,h,i) kernel): a CTA owns consecutive
// rows of one sequence -- all heads of a few tree queries -- so each cache row it stages
// in shared memory serves all of them instead of one row. Two tiles:
//  * the small-shape tile, 16 rows (128 threads, 2 rows a thread, 64-key blocks): scores
//    as a 2 x 4 register tile (keys tx, tx + 16, tx + 32, tx + 48 of the 16 key lanes, so
//    that a warp's key reads are consecutive rows), the output as 2 rows x 32 columns;
//  * the 64-row tile (512 threads, 128-key blocks), the fp32 path: 8 x 8 register tiles
//    in both contractions, the output tile parked in tensor memory while the scores of
//    the next block use the registers (see verify_simt_tm_kernel below).
//  * Every operand reaches shared memory by cp.async (16-byte copies, rows past the
//    sequence zero-filled, never read), in one ring filled in the order the block
//    consumes it: per key block, 9 chunks of 64 dims of Q and K for the scores, then
//    slices of 16 value rows (the latent rows again) for P.V. So the next block's first
//    chunks load while this block's P.V runs, and the loads ahead of the one in use hide
//    the L2/DRAM latency; operands stay in their row-major global layout.
//  * No atomics: every output element has one owner.
// Split-KV: blockIdx.y takes a contiguous range of key blocks; with more than one split
// the CTA writes a normalised partial (o_s, lse_s) that K2 merges.
#include "kdt_internal.cuh"
#include "tc_ptx.cuh"

#include <math.h>

namespace kdt {
namespace {
// (o0, o1) += p * (v0, v1) as one packed fp32x2 FMA (each lane an IEEE fma, as fmaf).
__device__ __forceinline__ void fma2_bcast(float &o0, float &o1, float p, float v0, float v1) {
    asm("{\n\t.reg .b64 acc, pp, vv;\n\t"
        "mov.b64 acc, {%0, %1};\n\t"
        "mov.b64 pp, {%2, %2};\n\t"
        "mov.b64 vv, {%3, %4};\n\t"
        "fma.rn.f32x2 acc, pp, vv, acc;\n\t"
        "mov.b64 {%0, %1}, acc;\n\t}"
        : "+f"(o0), "+f"(o1)
        : "f"(p), "f"(v0), "f"(v1));
}

constexpr int kKeys = kSimtKeys;       // 64 keys per block
constexpr int kDChunk = 64;            // dims per score chunk (fewer, larger steps: each step ends at a barrier)
constexpr int kQKChunks = kDqk / kDChunk;      // 9; a chunk lies wholly in the latent or the rope dims

// Element-type traits: shared-memory row pads (keep 16-byte alignment and spread the
// rows over the banks) and 4-wide loads widened to fp32.
template <typename T> struct Elt;
template <> struct Elt<float> {
    static constexpr int kPadQK = 4, kPadV = 4;
    __device__ static float4 get4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
};
template <> struct Elt<__nv_bfloat16> {
    static constexpr int kPadQK = 8, kPadV = 8;
    __device__ static float4 get4(const __nv_bfloat16 *p) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
    }
};

// kRows query rows a CTA: 64 (512 threads) or the small-shape tile of 16 (128 threads).
// Two rows a thread in both: one row a thread (twice the threads, 8-row value slices, a
// 6-slot ring) measured slower on small shapes (the score loop then issues 5 shared-memory
// loads per 16 FMAs and waits on shared memory).
template <typename T, int kRows> struct Layout {
    static constexpr int kRPT = 2;                                     // query rows a thread
    static constexpr int kThreads = 16 * kRows / kRPT;
    static constexpr int kVKeys = 16;                                  // value rows per P.V slice
    static constexpr int kSteps = kQKChunks + kKeys / kVKeys;          // loads per key block
    static constexpr int kNS = 4;                                      // ring slots
    static constexpr int kQKRow = kDChunk + Elt<T>::kPadQK;            // elements per staged Q/K row
    static constexpr int kVRow = kDc + Elt<T>::kPadV;                  // elements per staged value row
    static constexpr int kQKBytes = (kRows + kKeys) * kQKRow * (int)sizeof(T);
    static constexpr int kVBytes = kVKeys * kVRow * (int)sizeof(T);
    static constexpr int kSlot = ((kQKBytes > kVBytes ? kQKBytes : kVBytes) + 127) / 128 * 128;
    static constexpr int kPRow = kKeys + 4;                            // floats per P row
    static constexpr int kSmem = kNS * kSlot + kRows * kPRow * 4;
};

// 16-byte asynchronous copy global -> shared; src_bytes 0 fills the 16 bytes with zeros
// (the source address is then not read).
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <typename Tin, int kRows>
__global__ void __launch_bounds__(Layout<Tin, kRows>::kThreads, kRows == 16 ? 2 : 1)
    verify_simt_kernel(const VerifyParams p) {
    using L = Layout<Tin, kRows>;
    constexpr int kThreads = L::kThreads, kRPT = L::kRPT, kVKeys = L::kVKeys, kSteps = L::kSteps, kNS = L::kNS;
    constexpr int kEl16 = 16 / (int)sizeof(Tin);       // elements per 16-byte copy
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *ps = reinterpret_cast<float *>(smem_raw + kNS * L::kSlot);     // P [kRows][68]

    const int tid = threadIdx.x;
    const int tx = tid & 15;          // key lane (S) / column group (O)
    const int ty = tid >> 4;          // rows kRPT ty .. kRPT ty + kRPT - 1
    const int b = blockIdx.z;
    const int split = blockIdx.y;
    const int rows_seq = p.T * p.H;
    const int r0 = blockIdx.x * kRows;

    const Tin *q_nope = static_cast<const Tin *>(p.q_nope);
    const Tin *q_pe = static_cast<const Tin *>(p.q_pe);
    const Tin *c_kv = static_cast<const Tin *>(p.c_kv);
    const Tin *k_pe = static_cast<const Tin *>(p.k_pe);

    const int P = p.prefix_len[b];
    const int kv_len = P + p.T;
    const int nblk = (kv_len + kKeys - 1) / kKeys;
    const int kb0 = split * p.blocks_per_split;
    const int kb1 = min(nblk, kb0 + p.blocks_per_split);
    const int key_end = min(kv_len, kb1 * kKeys);
    const int64_t q_row0 = (int64_t)b * rows_seq + r0;
    const int64_t kv_row0 = (int64_t)b * p.L;
    const int total = kb1 > kb0 ? (kb1 - kb0) * kSteps : 0;

    // Copies of one load, spread over the threads: 16-byte pieces of the Q rows, then of the
    // key rows (a Q/K chunk), or of the value rows (a value slice).
    constexpr int kQKPieces = kDChunk / kEl16;                 // 16-byte pieces per chunk row
    constexpr int kQPieces = kRows * kQKPieces;
    constexpr int kVPieces = kDc / kEl16;                      // 16-byte pieces per value row

    // Queue load g of the sequence (block kb0 + g / kSteps, step g % kSteps) into its slot;
    // one commit group per load, empty past the end, so that the wait counts stay uniform.
    auto issue = [&](int g) {
        if (g < total) {
            const int kb = kb0 + g / kSteps, step = g % kSteps;
            Tin *slot = reinterpret_cast<Tin *>(smem_raw + (g % kNS) * L::kSlot);
            if (step < kQKChunks) {
                // Q rows r0.. and K rows kb*64.. of dims [32 step, 32 step + 32)
                const int d0 = step * kDChunk;
                const bool nope = d0 < kDc;
                const Tin *qbase = nope ? q_nope + d0 : q_pe + (d0 - kDc);
                const int64_t qstride = nope ? p.q_nope_stride : p.q_pe_stride;
#pragma unroll
                for (int i = tid; i < kQPieces; i += kThreads) {
                    const int rr = i / kQKPieces, pc = i % kQKPieces;
                    const bool ok = r0 + rr < rows_seq;
                    cp_async16(slot + rr * L::kQKRow + pc * kEl16, qbase + (q_row0 + (ok ? rr : 0)) * qstride + pc * kEl16,
                               ok ? 16u : 0u);
                }
                const Tin *kbase = nope ? c_kv + d0 : k_pe + (d0 - kDc);
                const int kstride = nope ? kDc : kDr;
#pragma unroll
                for (int i = tid; i < kKeys * kQKPieces; i += kThreads) {
                    const int rr = i / kQKPieces, pc = i % kQKPieces;
                    const int key = kb * kKeys + rr;
                    const bool ok = key < key_end;
                    cp_async16(slot + (kRows + rr) * L::kQKRow + pc * kEl16,
                               kbase + (kv_row0 + (ok ? key : 0)) * kstride + pc * kEl16, ok ? 16u : 0u);
                }
            } else {
                // value rows kb*64 + 16 (step - kQKChunks) .. + 16, all 512 latent dims
                const int k0 = kb * kKeys + (step - kQKChunks) * kVKeys;
#pragma unroll
                for (int i = tid; i < kVKeys * kVPieces; i += kThreads) {
                    const int kk = i / kVPieces, pc = i % kVPieces;
                    const int key = k0 + kk;
                    const bool ok = key < key_end;
                    cp_async16(slot + kk * L::kVRow + pc * kEl16, c_kv + (kv_row0 + (ok ? key : 0)) * kDc + pc * kEl16,
                               ok ? 16u : 0u);
                }
            }
        }
        cp_async_commit();
    };

    // query index of each of this thread's 2 rows (for the tree mask)
    int qidx[kRPT];
#pragma unroll
    for (int i = 0; i < kRPT; ++i) qidx[i] = min(r0 + kRPT * ty + i, rows_seq - 1) / p.H;

    float o[kRPT][32];
    float m2[kRPT], lpart[kRPT];
#pragma unroll
    for (int i = 0; i < kRPT; ++i) {
#pragma unroll
        for (int c = 0; c < 32; ++c) o[i][c] = 0.f;
        m2[i] = -INFINITY;
        lpart[i] = 0.f;
    }
    float acc[kRPT][4];
    bool vis_ready = false;            // the visibility bits are known to be written

#pragma unroll
    for (int g = 0; g < kNS - 1; ++g) issue(g);
    for (int g = 0; g < total; ++g) {
        cp_async_wait<kNS - 2>();      // this thread's copies of load g have landed
        __syncthreads();               // everyone's have; everyone is done with load g - 1's slot
        issue(g + kNS - 1);            // into the slot load g - 1 used
        const int step = g % kSteps;
        const int k0 = (kb0 + g / kSteps) * kKeys;
        const Tin *slot = reinterpret_cast<const Tin *>(smem_raw + (g % kNS) * L::kSlot);
        if (step < kQKChunks) {
            // ---------------- S += Q K^T over 64 dims: rows 2ty+i, keys tx + 16 j -------------
            if (step == 0) {
#pragma unroll
                for (int i = 0; i < kRPT; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
            }
            const Tin *qs = slot + (kRPT * ty) * L::kQKRow;
            const Tin *ks = slot + (kRows + tx) * L::kQKRow;
#pragma unroll
            for (int d = 0; d < kDChunk; d += 4) {
                float4 a[kRPT];
#pragma unroll
                for (int i = 0; i < kRPT; ++i) a[i] = Elt<Tin>::get4(qs + i * L::kQKRow + d);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 k = Elt<Tin>::get4(ks + 16 * j * L::kQKRow + d);
#pragma unroll
                    for (int i = 0; i < kRPT; ++i)
                        acc[i][j] = fmaf(a[i].x, k.x, fmaf(a[i].y, k.y, fmaf(a[i].z, k.z, fmaf(a[i].w, k.w, acc[i][j]))));
                }
            }
            if (step == kQKChunks - 1) {
                // ---------------- mask, online softmax, P to shared memory -------------------
                // the bits may come from the visibility kernel launched just before this one:
                // wait for it before the first block with tree keys
                if (!vis_ready && k0 + kKeys > P) {
                    tc::griddep_wait();
                    vis_ready = true;
                }
#pragma unroll
                for (int i = 0; i < kRPT; ++i) {
                    float s[4];
                    float mx = -INFINITY;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int key = k0 + tx + 16 * j;
                        bool visible = key < key_end;
                        if (visible && key >= P) {
                            const int t = key - P;
                            const uint32_t w = p.vis[((int64_t)b * p.T + qidx[i]) * p.W + (t >> 5)];
                            visible = (w >> (t & 31)) & 1u;
                        }
                        s[j] = visible ? acc[i][j] * p.scale_log2 : -INFINITY;
                        mx = fmaxf(mx, s[j]);
                    }
#pragma unroll
                    for (int off = 8; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    const float mnew = fmaxf(m2[i], mx);
                    // a row with nothing visible so far keeps m = -inf: weights 0, no rescale
                    const float alpha = (mnew == -INFINITY) ? 1.f : exp2f(m2[i] - mnew);
                    float rs = 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float pj = (mnew == -INFINITY) ? 0.f : exp2f(s[j] - mnew);
                        ps[(kRPT * ty + i) * L::kPRow + tx + 16 * j] = pj;
                        rs += pj;
                    }
                    lpart[i] = lpart[i] * alpha + rs;
                    m2[i] = mnew;
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[i][c] *= alpha;
                }
                // P is read after the next load's barrier
            }
        } else {
            // ---------------- O += P V for 16 keys: rows 2ty+i, columns 64 c + 4 tx ------------
            const int kk0 = (step - kQKChunks) * kVKeys;
#pragma unroll 2
            for (int kk = 0; kk < kVKeys; ++kk) {
                float pr[kRPT];
#pragma unroll
                for (int i = 0; i < kRPT; ++i) pr[i] = ps[(kRPT * ty + i) * L::kPRow + kk0 + kk];
                const Tin *vrow = slot + kk * L::kVRow + 4 * tx;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 v = Elt<Tin>::get4(vrow + 64 * c);
#pragma unroll
                    for (int i = 0; i < kRPT; ++i) {
                        o[i][4 * c + 0] = fmaf(pr[i], v.x, o[i][4 * c + 0]);
                        o[i][4 * c + 1] = fmaf(pr[i], v.y, o[i][4 * c + 1]);
                        o[i][4 * c + 2] = fmaf(pr[i], v.z, o[i][4 * c + 2]);
                        o[i][4 * c + 3] = fmaf(pr[i], v.w, o[i][4 * c + 3]);
                    }
                }
            }
        }
    }
    cp_async_wait<0>();
    tc::griddep_launch_dependents();   // the split merge may launch; it waits for this kernel's end

    // ---------------- epilogue: o = O / l, lse = ln2 * (m2 + log2 l) -------------------------
    const bool partial = p.num_splits > 1;
    float *obase = partial ? p.part_o + (int64_t)split * p.rows_total * kDc : p.out;
    float *lbase = partial ? p.part_lse + (int64_t)split * p.rows_total : p.lse;
#pragma unroll
    for (int i = 0; i < kRPT; ++i) {
        float l = lpart[i];
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        const int r = r0 + kRPT * ty + i;
        if (r >= rows_seq) continue;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int64_t grow = (int64_t)b * rows_seq + r;
        float *orow = obase + grow * kDc;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4 *>(orow + c * 64 + tx * 4) =
                make_float4(o[i][c * 4] * inv, o[i][c * 4 + 1] * inv, o[i][c * 4 + 2] * inv, o[i][c * 4 + 3] * inv);
        if (tx == 0 && lbase) lbase[grow] = (l > 0.f) ? 0.6931471805599453f * (m2[i] + log2f(l)) : -INFINITY;
    }
}

// The 64-row tile with 128-key blocks and 8 x 8 register tiles in both contractions. A
// warp-wide 16- or 8-byte shared load costs one 128-byte wavefront per 8 or 16 lanes
// however many lanes share an address, so a lane receives at most 4 bytes a wavefront
// while the SM issues four FMA instructions a cycle: only a tile whose every loaded
// operand feeds 8 FMAs (8 x 8) keeps the FMA pipes busy. The 64 output accumulators and
// the 64 score accumulators do not both fit in 128 registers, so the output tile waits in
// tensor memory (256 columns, each thread its own lane and 64 columns) while the scores
// of the next block are computed:
//  * scores: warp w takes rows 8 (w / 2) .. + 8 and keys 64 (w % 2) .. + 64 of the block;
//    lane = 8 dg + kt computes those 8 rows x keys kt + 8 j (j < 8) over the dim pairs
//    2 dg + 8 u of every 64-dim chunk; the four dim groups' partial sums meet by two shuffle rounds,
//    after which a lane holds rows 2 dg, 2 dg + 1 of its warp's 8 (8 keys each).
//  * output: warp w takes rows 32 (w / 8) .. + 32 and columns 64 (w % 8) .. + 64; lane =
//    8 rt + ct holds rows 8 rt .. + 8 of those and columns 4 ct + 32 q (q < 2, 4 each),
//    reading P transposed ([key][row]) and 16-key value slices.
template <typename T> struct LayoutTm {
    static constexpr int kRows = 64, kKB = kSimtKeysTm, kThreads = 512, kVKeys = 16, kNS = 3;
    static constexpr int kQK = kQKChunks, kSteps = kQKChunks + kKB / kVKeys;   // 9 + 8 loads a block
    static constexpr int kQKRow = kDChunk + Elt<T>::kPadQK;
    static constexpr int kVRow = kDc + Elt<T>::kPadV;
    static constexpr int kQKBytes = (kRows + kKB) * kQKRow * (int)sizeof(T);
    static constexpr int kVBytes = kVKeys * kVRow * (int)sizeof(T);
    static constexpr int kSlot = ((kQKBytes > kVBytes ? kQKBytes : kVBytes) + 127) / 128 * 128;
    static constexpr int kPtRow = kRows + 4;
    static constexpr int kOffPt = kNS * kSlot;
    static constexpr int kOffRed = kOffPt + kKB * kPtRow * 4;     // [2 key halves][64 rows]
    static constexpr int kOffAlpha = kOffRed + 2 * kRows * 4;     // [64]
    static constexpr int kOffTmem = kOffAlpha + kRows * 4;        // tensor-memory base address
    static constexpr int kOffWork = kOffTmem + 16;                // this CTA's work range (5 x int64)
    static constexpr int kSmem = kOffWork + 5 * 8;
    static constexpr uint32_t kTmemCols = 256;
};

// Two consecutive elements widened to fp32.
template <typename T> __device__ __forceinline__ float2 get2(const T *p);
template <> __device__ __forceinline__ float2 get2<float>(const float *p) { return *reinterpret_cast<const float2 *>(p); }
template <> __device__ __forceinline__ float2 get2<__nv_bfloat16>(const __nv_bfloat16 *p) {
    const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

// Key blocks of sequence b for blocks of kb keys.
__device__ __forceinline__ int seq_blocks_of(const VerifyParams &p, int b, int kb) {
    return (p.prefix_len[b] + p.T + kb - 1) / kb;
}

// The work of the 64-row tile is the list of (row tile, key block) pairs, sequence-major,
// then tile-major, then in key order: W = tiles_seq * sum_b blocks(b) of them. CTA c of C
// takes positions [W c / C, W (c + 1) / C). One warp computes W, the range and the
// (sequence, tile, block) of its first position; lane 0 writes {s0, s1, b, tile, block}.
__device__ __forceinline__ void locate_work(const VerifyParams &p, int tiles_seq, int kb, int64_t C, int64_t c,
                                            int lane, int64_t *out) {
    int64_t W = 0;
    for (int b = lane; b < p.B; b += 32) W += (int64_t)tiles_seq * seq_blocks_of(p, b, kb);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
    const int64_t s0 = W * c / C, s1 = W * (c + 1) / C;
    int fb = -1, fnb = 1;
    int64_t fbefore = 0, acc = 0;
    for (int base = 0; base < p.B && fb < 0; base += 32) {
        const int b = base + lane;
        const int nbk = b < p.B ? seq_blocks_of(p, b, kb) : 1;
        const int64_t w = b < p.B ? (int64_t)tiles_seq * nbk : 0;
        int64_t incl = w;                            // inclusive scan over the lanes
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        const int64_t before = acc + incl - w;
        const unsigned hit = __ballot_sync(0xffffffffu, b < p.B && s0 >= before && s0 < before + w);
        if (hit) {
            const int src = __ffs(hit) - 1;
            fb = base + src;
            fbefore = __shfl_sync(0xffffffffu, before, src);
            fnb = __shfl_sync(0xffffffffu, nbk, src);
        }
        acc += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
        const int64_t off = fb >= 0 ? s0 - fbefore : 0;
        out[0] = s0;
        out[1] = s1;
        out[2] = fb >= 0 ? fb : 0;
        out[3] = off / fnb;
        out[4] = off % fnb;
    }
}

template <typename Tin>
__global__ void __launch_bounds__(512, 1) verify_simt_tm_kernel(const VerifyParams p) {
    using L = LayoutTm<Tin>;
    constexpr int kThreads = L::kThreads, kVKeys = L::kVKeys, kSteps = L::kSteps, kNS = L::kNS, kR = L::kRows,
                  kKB = L::kKB;
    constexpr int kEl16 = 16 / (int)sizeof(Tin);
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *pt = reinterpret_cast<float *>(smem_raw + L::kOffPt);       // P^T [128 keys][68]
    float *red = reinterpret_cast<float *>(smem_raw + L::kOffRed);     // [2][64]
    float *alpha_s = reinterpret_cast<float *>(smem_raw + L::kOffAlpha);
    uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(smem_raw + L::kOffTmem);
    int64_t *work_s = reinterpret_cast<int64_t *>(smem_raw + L::kOffWork);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // score tile
    const int kh = warp & 1, dg = lane >> 3, kt = lane & 7;
    const int srow = 8 * (warp >> 1);                 // first of the warp's 8 rows
    const int skey = 64 * kh + kt;                    // keys skey + 8 j of the block
    const int mrow = srow + 2 * dg;                   // rows mrow, mrow + 1 after the reduction
    // output tile
    const int orow = 32 * (warp >> 3) + 8 * (lane >> 3);
    const int ocol = 64 * (warp & 7) + 4 * (lane & 7);

    const int rows_seq = p.T * p.H;
    const int tiles_seq = (rows_seq + kR - 1) / kR;      // row tiles of a sequence
    const Tin *q_nope = static_cast<const Tin *>(p.q_nope);
    const Tin *q_pe = static_cast<const Tin *>(p.q_pe);
    const Tin *c_kv = static_cast<const Tin *>(p.c_kv);
    const Tin *k_pe = static_cast<const Tin *>(p.k_pe);

    // tensor memory for the output tile between blocks: warp w uses lanes 32 (w % 4) ..
    // and columns 64 (w / 4) .. + 64
    if (warp == 0) {
        tc::tmem_alloc(tmem_base_s, L::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_o = *tmem_base_s + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(64 * (warp >> 2));

    // ---- this CTA's share of the work: (row tile, key block) pairs in sequence-major,
    // tile-major, key-block order, W of them, cut into gridDim.x equal contiguous ranges;
    // a range is processed as segments of one tile each
    const int C = gridDim.x, c = blockIdx.x;
    if (warp == 0) locate_work(p, tiles_seq, kKB, (int64_t)C, (int64_t)c, lane, work_s);
    __syncthreads();
    const int64_t s_begin = work_s[0], s_end = work_s[1];
    int b = (int)work_s[2], rt = (int)work_s[3], kb_at = (int)work_s[4];
    bool vis_ready = false;
    bool first_seg = true;
    for (int64_t pos = s_begin; pos < s_end;) {
    const int r0 = rt * kR;
    const int P = p.prefix_len[b];
    const int kv_len = P + p.T;
    const int nblk = (kv_len + kKB - 1) / kKB;
    const int kb0 = kb_at;
    const int kb1 = (int)min((int64_t)nblk, (int64_t)kb0 + (s_end - pos));
    const int key_end = min(kv_len, kb1 * kKB);
    const int64_t q_row0 = (int64_t)b * rows_seq + r0;
    const int64_t kv_row0 = (int64_t)b * p.L;
    const int nb = kb1 - kb0;
    const int total = nb * kSteps;
    const bool whole = kb0 == 0 && kb1 == nblk;

    // Queue load g (block kb0 + g / kSteps, step g % kSteps) into its ring slot: Q rows and
    // the block's 128 key rows of one 64-dim chunk, or 16 value rows; one commit group a
    // load, empty past the end, so that the wait counts stay uniform.
    constexpr int kQKPieces = kDChunk / kEl16;
    constexpr int kVPieces = kDc / kEl16;
    auto issue = [&](int g) {
        if (g < total) {
            const int kb = kb0 + g / kSteps, step = g % kSteps;
            Tin *slot = reinterpret_cast<Tin *>(smem_raw + (g % kNS) * L::kSlot);
            if (step < L::kQK) {
                const int d0 = step * kDChunk;
                const bool nope = d0 < kDc;
                const Tin *qbase = nope ? q_nope + d0 : q_pe + (d0 - kDc);
                const int64_t qstride = nope ? p.q_nope_stride : p.q_pe_stride;
#pragma unroll
                for (int i = tid; i < kR * kQKPieces; i += kThreads) {
                    const int rr = i / kQKPieces, pc = i % kQKPieces;
                    const bool ok = r0 + rr < rows_seq;
                    cp_async16(slot + rr * L::kQKRow + pc * kEl16, qbase + (q_row0 + (ok ? rr : 0)) * qstride + pc * kEl16,
                               ok ? 16u : 0u);
                }
                const Tin *kbase = nope ? c_kv + d0 : k_pe + (d0 - kDc);
                const int kstride = nope ? kDc : kDr;
#pragma unroll
                for (int i = tid; i < kKB * kQKPieces; i += kThreads) {
                    const int rr = i / kQKPieces, pc = i % kQKPieces;
                    const int key = kb * kKB + rr;
                    const bool ok = key < key_end;
                    cp_async16(slot + (kR + rr) * L::kQKRow + pc * kEl16,
                               kbase + (kv_row0 + (ok ? key : 0)) * kstride + pc * kEl16, ok ? 16u : 0u);
                }
            } else {
                const int k0 = kb * kKB + (step - L::kQK) * kVKeys;
#pragma unroll
                for (int i = tid; i < kVKeys * kVPieces; i += kThreads) {
                    const int kk = i / kVPieces, pc = i % kVPieces;
                    const int key = k0 + kk;
                    const bool ok = key < key_end;
                    cp_async16(slot + kk * L::kVRow + pc * kEl16, c_kv + (kv_row0 + (ok ? key : 0)) * kDc + pc * kEl16,
                               ok ? 16u : 0u);
                }
            }
        }
        cp_async_commit();
    };

    int qidx[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) qidx[i] = min(r0 + mrow + i, rows_seq - 1) / p.H;
    float m2[2] = {-INFINITY, -INFINITY}, lpart[2] = {0.f, 0.f};
    float o[8][8];
    int g = 0;                                        // loads consumed so far

#pragma unroll
    for (int k = 0; k < kNS - 1; ++k) issue(k);
    // wait for load g, then refill the slot load g - 1 used
    auto next_load = [&]() -> const Tin * {
        cp_async_wait<kNS - 2>();
        __syncthreads();
        issue(g + kNS - 1);
        return reinterpret_cast<const Tin *>(smem_raw + (g % kNS) * L::kSlot);
    };

    for (int blk = 0; blk < nb; ++blk) {
        const int k0 = (kb0 + blk) * kKB;
        // ---------------- S partial = Q K^T over this lane's 16 dims of each chunk -------------
        float acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
        for (int c = 0; c < L::kQK; ++c, ++g) {
            const Tin *slot = next_load();
            // lane group dg takes the dim pairs 2 dg + 8 u: the two groups of a half-warp
            // then read disjoint banks of the 8 consecutive key rows
            const Tin *qs = slot + srow * L::kQKRow + 2 * dg;
            const Tin *ks = slot + (kR + skey) * L::kQKRow + 2 * dg;
#pragma unroll 1
            for (int d = 0; d < kDChunk; d += 8) {
                float2 a[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) a[i] = get2(qs + i * L::kQKRow + d);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float2 k = get2(ks + 8 * j * L::kQKRow + d);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i][j] = fmaf(a[i].x, k.x, fmaf(a[i].y, k.y, acc[i][j]));
                }
            }
        }
        // ---------------- the four dim groups' sums: two transposing shuffle rounds ----------
        // round 1 (partner dg ^ 2): keep rows 4 (dg >> 1) .. + 4; round 2 (dg ^ 1): keep 2.
        float s4[4][8];
        const bool up2 = (dg & 2) != 0, up1 = (dg & 1) != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float send = up2 ? acc[i][j] : acc[4 + i][j];
                const float keep = up2 ? acc[4 + i][j] : acc[i][j];
                s4[i][j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
            }
        float s[2][8];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float send = up1 ? s4[i][j] : s4[2 + i][j];
                const float keep = up1 ? s4[2 + i][j] : s4[i][j];
                s[i][j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
            }
        // ---------------- mask, scale, row maxima of this warp's 64 keys ------------------------
        if (!vis_ready && k0 + kKB > P) {            // the bits may come from the kernel just before
            tc::griddep_wait();
            vis_ready = true;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int key = k0 + skey + 8 * j;
                bool visible = key < key_end;
                if (visible && key >= P) {
                    const int t = key - P;
                    const uint32_t w = p.vis[((int64_t)b * p.T + qidx[i]) * p.W + (t >> 5)];
                    visible = (w >> (t & 31)) & 1u;
                }
                s[i][j] = visible ? s[i][j] * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, s[i][j]);
            }
#pragma unroll
            for (int off = 4; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            if (kt == 0) red[kh * kR + mrow + i] = mx;
        }
        // ---------------- first value slice: online softmax, P^T, rescale factors --------------
        const Tin *vslot = next_load();              // its barrier also publishes the maxima
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float mx = fmaxf(red[mrow + i], red[kR + mrow + i]);
            const float mnew = fmaxf(m2[i], mx);
            const float al = (mnew == -INFINITY) ? 1.f : exp2f(m2[i] - mnew);
            float rs = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float pj = (mnew == -INFINITY) ? 0.f : exp2f(s[i][j] - mnew);
                pt[(skey + 8 * j) * L::kPtRow + mrow + i] = pj;
                rs += pj;
            }
            lpart[i] = lpart[i] * al + rs;
            m2[i] = mnew;
            if (kh == 0 && kt == 0) alpha_s[mrow + i] = al;
        }
        __syncthreads();                             // P^T and every row's factor are written
        // the output tile back from tensor memory (zero before the first block), rescaled
        if (blk == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int c = 0; c < 8; ++c) o[i][c] = 0.f;
        } else {
            uint32_t t0[32], t1[32];
            tc::tmem_ld32(tmem_o, t0);
            tc::tmem_ld32(tmem_o + 32, t1);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    o[i][c] = __uint_as_float(t0[8 * i + c]);
                    o[4 + i][c] = __uint_as_float(t1[8 * i + c]);
                }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float al = alpha_s[orow + i];
#pragma unroll
            for (int c = 0; c < 8; ++c) o[i][c] *= al;
        }
        // ---------------- O += P V, 16 keys a slice ---------------------------------------------
        for (int v = 0; v < kKB / kVKeys; ++v) {
            if (v > 0) vslot = next_load();
            const int kk0 = v * kVKeys;
#pragma unroll 4
            for (int kk = 0; kk < kVKeys; ++kk) {
                const float4 pa = *reinterpret_cast<const float4 *>(pt + (kk0 + kk) * L::kPtRow + orow);
                const float4 pb = *reinterpret_cast<const float4 *>(pt + (kk0 + kk) * L::kPtRow + orow + 4);
                const float pr[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
                const Tin *vrow = vslot + kk * L::kVRow + ocol;
                const float4 va = Elt<Tin>::get4(vrow), vb = Elt<Tin>::get4(vrow + 32);
                const float vv[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int c = 0; c < 8; c += 2) fma2_bcast(o[i][c], o[i][c + 1], pr[i], vv[c], vv[c + 1]);
            }
            ++g;
        }
        // the tile waits in tensor memory while the next block's scores use the registers
        if (blk + 1 < nb) {
            uint32_t t0[32], t1[32];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    t0[8 * i + c] = __float_as_uint(o[i][c]);
                    t1[8 * i + c] = __float_as_uint(o[4 + i][c]);
                }
            tc::tmem_st32(tmem_o, t0);
            tc::tmem_st32(tmem_o + 32, t1);
            tc::tmem_wait_st();
        }
    }
    cp_async_wait<0>();

    // ---------------- segment epilogue: o = O / l, lse = ln2 * (m2 + log2 l) ---------------
    __syncthreads();           // every read of the maxima buffer and of the ring is done
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float l = lpart[i];
#pragma unroll
        for (int off = 4; off >= 1; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (kt == 0) red[kh * kR + mrow + i] = l;
    }
    __syncthreads();
    // a whole tile writes its final rows; a piece of one its normalised state, in slot 2c
    // when it is the first segment of this CTA's range, else (its last) in slot 2c + 1
    float *obase = p.out, *lbase = p.lse;
    int64_t rowbase = (int64_t)b * rows_seq + r0;
    if (!whole) {
        obase = p.part_o;
        lbase = p.part_lse;
        rowbase = (int64_t)(first_seg ? 2 * c : 2 * c + 1) * kR;
    }
    if (kh == 0 && kt == 0 && lbase) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float l = red[mrow + i] + red[kR + mrow + i];
            if (r0 + mrow + i < rows_seq)
                lbase[rowbase + mrow + i] = (l > 0.f) ? 0.6931471805599453f * (m2[i] + log2f(l)) : -INFINITY;
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (r0 + orow + i >= rows_seq) continue;
        const float l = red[orow + i] + red[kR + orow + i];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float *orow_p = obase + (rowbase + orow + i) * kDc + ocol;
        *reinterpret_cast<float4 *>(orow_p) = make_float4(o[i][0] * inv, o[i][1] * inv, o[i][2] * inv, o[i][3] * inv);
        *reinterpret_cast<float4 *>(orow_p + 32) = make_float4(o[i][4] * inv, o[i][5] * inv, o[i][6] * inv, o[i][7] * inv);
    }
    // the next segment: the rest of this tile cannot follow (a segment ends at the tile's
    // last block or at the end of the range), so the next tile
    pos += nb;
    first_seg = false;
    kb_at = kb1;
    if (kb_at == nblk) {
        kb_at = 0;
        if (++rt == tiles_seq) {
            rt = 0;
            ++b;
        }
    }
    }   // segments
    tc::griddep_launch_dependents();   // the piece merge may launch; it waits for this kernel's end
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(*tmem_base_s, L::kTmemCols);
}

template <typename Tin>
cudaError_t launch_typed_tm(const VerifyParams &p, cudaStream_t s) {
    using L = LayoutTm<Tin>;
    cudaError_t e = cudaFuncSetAttribute(verify_simt_tm_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
    if (e != cudaSuccess) return e;
    // programmatic dependent launch after the visibility kernel of the same call
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.simt_ctas > 0 ? p.simt_ctas : 1);
    cfg.blockDim = dim3(L::kThreads);
    cfg.dynamicSmemBytes = L::kSmem;
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = p.overlap_vis ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, verify_simt_tm_kernel<Tin>, p);
}

// Shapes whose every sequence fits one block of at most 64 keys (prefix + tree): one pass,
// no key loop. A CTA takes R = 1, 2 or 4 rows of one sequence; it loads their queries and
// ALL the sequence's cache rows as a few bulk copies on one mbarrier, builds the rows'
// visibility from the parent array itself while they land (no separate visibility
// launch), and computes the scores, the softmax and P.V from shared memory, the value rows
// being the staged latent rows. A shape this small is bound by latency, not by any pipe:
// the launch takes the fewest rows a CTA whose grid the device holds at once, so each CTA
// is as short as the one-wave budget allows (on Tiny 2 rows a CTA instead of 4 cut the CTA
// from 5.4 to 4.5 us; fewer rows only pay within one wave, as every CTA loads the whole
// key block).
//  * scores: lane (key lane kg, dim slot 4 w + sl) computes all R rows x 8 keys (kg + 8 j)
//    over the dim pairs pr + 32 s, pr = (4 w + sl + 2 kg) mod 32: the 16 lanes of a
//    half-warp then read 16 different pair columns, so every 8-byte key or query read is
//    one conflict-free shared-memory wavefront of distinct bytes. The number of 8-key
//    groups (2, 4, 6 or 8, covering the block's keys) is a compile-time count picked once:
//    a runtime bound around each group kept its loads and FMAs from overlapping and cost
//    a third of the phase. The 32 slots' partials meet through two shuffle steps and
//    shared memory.
//  * softmax: warp r < R sums row r's partials and takes its softmax (keys lane, lane + 32).
//  * output: thread t the columns 2 t, 2 t + 1 of the R rows.
__device__ __forceinline__ float fast_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fast_lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr int kOneKeys = 64;
constexpr int kOneThreads = 256;

// Operands land unpadded, as the few large bulk copies of whole row ranges (a copy's cost
// is per request); lane (group, key lane) walks the dim pairs in an order rotated by its
// key lane, so the 8 key rows a half-warp reads sit in different banks all the same.
template <typename T, int R> struct LayoutOne {
    static constexpr int kOffQn = 0;                                                 // [R][512]
    static constexpr int kOffQp = kOffQn + R * kDc * (int)sizeof(T);                 // [R][64]
    static constexpr int kOffKn = kOffQp + R * kDr * (int)sizeof(T);                 // [64][512]
    static constexpr int kOffKp = kOffKn + kOneKeys * kDc * (int)sizeof(T);          // [64][64]
    static constexpr int kOffRed = kOffKp + kOneKeys * kDr * (int)sizeof(T);         // [8][R][64] partials
    static constexpr int kOffPt = kOffRed + 8 * R * kOneKeys * 4;                    // [64][R] P^T
    static constexpr int kOffRow = kOffPt + kOneKeys * R * 4;                        // [R] masks, [R] l
    static constexpr int kOffBar = (kOffRow + R * 12 + 7) & ~7;                      // copy barrier
    static constexpr int kSmem = kOffBar + 8;
};

// Partial scores of one lane: rows 0..R-1 x keys kg + 8 j (j < KJ) over the latent pairs
// pr + 32 s (s < 8) and the rope pair pr, accumulated into acc.
template <int KJ, int R, typename Tin>
__device__ __forceinline__ void one_scores(float (&acc)[R][8], const Tin *qn, const Tin *qp, const Tin *kn,
                                           const Tin *kp, int pr, int kg) {
    auto part = [&](const Tin *q, const Tin *k, int width, int nsteps) {
        const Tin *qa = q + 2 * pr;
        const Tin *kb = k + kg * width + 2 * pr;
#pragma unroll 2
        for (int u = 0; u < nsteps; ++u) {
            float2 a[R];
#pragma unroll
            for (int i = 0; i < R; ++i) a[i] = get2(qa + i * width + 64 * u);
#pragma unroll
            for (int j = 0; j < KJ; ++j) {
                const float2 kk = get2(kb + 8 * j * width + 64 * u);
#pragma unroll
                for (int i = 0; i < R; ++i) acc[i][j] = fmaf(a[i].x, kk.x, fmaf(a[i].y, kk.y, acc[i][j]));
            }
        }
    };
    part(qn, kn, kDc, kDc / 64);
    part(qp, kp, kDr, kDr / 64);
}

// check_all: this grid is small enough that CTA (0, 0) checks every parent entry of the
// batch and writes the error word (0 if none; no clearing before the launch); otherwise
// the word was cleared and each sequence's first CTA records its malformed entries.
template <typename Tin, int R>
__global__ void __launch_bounds__(kOneThreads, 1) verify_simt_one_kernel(const VerifyParams p,
                                                                         const int32_t *parent, bool check_all) {
    constexpr int kOneRows = R;
    using L = LayoutOne<Tin, R>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Tin *qn_s = reinterpret_cast<Tin *>(smem_raw + L::kOffQn);
    Tin *qp_s = reinterpret_cast<Tin *>(smem_raw + L::kOffQp);
    Tin *kn_s = reinterpret_cast<Tin *>(smem_raw + L::kOffKn);
    Tin *kp_s = reinterpret_cast<Tin *>(smem_raw + L::kOffKp);
    float *red = reinterpret_cast<float *>(smem_raw + L::kOffRed);
    float *pt = reinterpret_cast<float *>(smem_raw + L::kOffPt);
    uint64_t *mask_s = reinterpret_cast<uint64_t *>(smem_raw + L::kOffRow);
    float *l_s = reinterpret_cast<float *>(smem_raw + L::kOffRow + kOneRows * 8);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem_raw + L::kOffBar);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.y;
    const int rows_seq = p.T * p.H;
    const int r0 = blockIdx.x * kOneRows;
    const int nq = min(kOneRows, rows_seq - r0);
    constexpr uint32_t kNopeBytes = kDc * sizeof(Tin), kPeBytes = kDr * sizeof(Tin);
    if (tid == 0) {
        tc::mbar_init(bar, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    // ---- every operand by bulk copies on one barrier: the rows of the 4 queries that exist
    // (one copy per part when the rows are contiguous) and the sequence's first max_kv
    // (<= 64) cache rows, whatever its own length (one copy per part). Rows past them are
    // never read as operands (their scores are masked, their outputs unused).
    const Tin *q_nope = static_cast<const Tin *>(p.q_nope);
    const Tin *q_pe = static_cast<const Tin *>(p.q_pe);
    const Tin *c_kv = static_cast<const Tin *>(p.c_kv);
    const Tin *k_pe = static_cast<const Tin *>(p.k_pe);
    const int nkv = p.max_kv;
    if (tid == 0) {
        tc::mbar_arrive_expect_tx(bar, (uint32_t)(nq + nkv) * (kNopeBytes + kPeBytes));
        const int64_t g0 = (int64_t)b * rows_seq + r0;
        if (p.q_nope_stride == kDc) {
            tc::bulk_load_1d(qn_s, q_nope + g0 * kDc, (uint32_t)nq * kNopeBytes, bar);
        } else {
            for (int rr = 0; rr < nq; ++rr) tc::bulk_load_1d(qn_s + rr * kDc, q_nope + (g0 + rr) * p.q_nope_stride, kNopeBytes, bar);
        }
        if (p.q_pe_stride == kDr) {
            tc::bulk_load_1d(qp_s, q_pe + g0 * kDr, (uint32_t)nq * kPeBytes, bar);
        } else {
            for (int rr = 0; rr < nq; ++rr) tc::bulk_load_1d(qp_s + rr * kDr, q_pe + (g0 + rr) * p.q_pe_stride, kPeBytes, bar);
        }
        tc::bulk_load_1d(kn_s, c_kv + (int64_t)b * p.L * kDc, (uint32_t)nkv * kNopeBytes, bar);
        tc::bulk_load_1d(kp_s, k_pe + (int64_t)b * p.L * kDr, (uint32_t)nkv * kPeBytes, bar);
    }
    const int P = p.prefix_len[b];
    const int kv = min(P + p.T, nkv);                // <= max_kv <= 64 (the caller's bound; clamped for safety)
    const int nk = (kv + 7) & ~7;                    // keys computed: kv rounded up to 8
    // ---- meanwhile: the rows' visible keys (prefix, ancestors, self) as 64-bit masks
    if (warp == 0) {
        if (lane < kOneRows) {
            const int r = min(r0 + lane, rows_seq - 1);
            const int qi = r / p.H;
            uint64_t m = P > 0 ? (~0ull >> (64 - P)) : 0ull;          // P <= 63 here (kv <= 64, T >= 1)
            if (parent) {
                const int32_t *par = parent + (int64_t)b * p.T;
                int j = qi;
                while (true) {                        // parents strictly decrease: <= T steps
                    m |= 1ull << (P + j);
                    const int pj = par[j];
                    if (pj < -1 || pj >= j || pj < 0) break;   // malformed entries are recorded below
                    j = pj;
                }
            } else {
                const uint32_t *vrow = p.vis + ((int64_t)b * p.T + qi) * p.W;
                const uint64_t bits = (uint64_t)vrow[0] | (p.W > 1 ? (uint64_t)vrow[1] << 32 : 0ull);
                m |= (p.T >= 64 ? bits : (bits & ((1ull << p.T) - 1))) << P;
            }
            mask_s[lane] = m;
        }
        // the error word gets the first malformed parent entry over all sequences, as the
        // visibility kernel reports it
        if (check_all) {
            if (blockIdx.x == 0 && blockIdx.y == 0 && p.err) {
                int first = 0x7fffffff;
                if (parent)
#pragma unroll 8
                    for (int j = lane; j < p.B * p.T; j += 32) {
                        const int pj = parent[j], jj = j % p.T;
                        if ((pj < -1 || pj >= jj) && j + 1 < first) first = j + 1;
                    }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) first = min(first, __shfl_xor_sync(0xffffffffu, first, off));
                if (lane == 0) *p.err = first == 0x7fffffff ? 0 : first;
            }
        } else if (parent && blockIdx.x == 0) {
            const int32_t *par = parent + (int64_t)b * p.T;
            for (int j = lane; j < p.T; j += 32) {
                const int pj = par[j];
                if (pj < -1 || pj >= j) record_error(p.err, (int32_t)((int64_t)b * p.T + j + 1));
            }
        }
    }
    // every thread sees the copies land (bounded: a lost completion ends the call with an
    // error, after a second wait for copies still in flight)
    const bool landed = tc::mbar_wait(bar, 0, 200000000ull);
    if (__syncthreads_or(!landed)) {
        if (tid == 0 && p.err) atomicCAS(p.err, 0, -40);
        tc::mbar_wait(bar, 0, 200000000ull);
        return;
    }

    // ---- partial scores of this lane's dim slot: all R rows x 8 keys
    const int kg = lane & 7, sl = lane >> 3;         // key lane (keys kg + 8 j), slot in the warp
    const int pr = (4 * warp + sl + 2 * kg) & 31;    // dim pairs pr + 32 s of the latent, pr of the rope
    float acc[kOneRows][8];
#pragma unroll
    for (int i = 0; i < kOneRows; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    // the key groups computed (a multiple of 2 covering nk) are fixed at compile time:
    // a runtime bound around each group's loads and FMAs serialises them
    switch ((nk + 15) >> 4) {
        case 1:
            one_scores<2, R>(acc, qn_s, qp_s, kn_s, kp_s, pr, kg);
            break;
        case 2:
            one_scores<4, R>(acc, qn_s, qp_s, kn_s, kp_s, pr, kg);
            break;
        case 3:
            one_scores<6, R>(acc, qn_s, qp_s, kn_s, kp_s, pr, kg);
            break;
        default:
            one_scores<8, R>(acc, qn_s, qp_s, kn_s, kp_s, pr, kg);
            break;
    }
    // the warp's 4 slots in two transposing shuffle steps (partner lane ^ 16, then lane ^ 8),
    // each trading half of what a lane holds, then the 8 warps through shared memory:
    //  R = 4: rows 0-1 against 2-3, then row 2 a against 2 a + 1: lane (kg, sl) keeps row sl;
    //  R = 2: row 0 against row 1, then keys j < 4 against j >= 4;
    //  R = 1: keys j < 4 against j >= 4, then j < 2 against j >= 2 of those.
    const bool up2 = (sl & 2) != 0, up1 = (sl & 1) != 0;
    if constexpr (R == 4) {
        float s2[2][8];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float give = up2 ? acc[i][j] : acc[2 + i][j];
                const float keep = up2 ? acc[2 + i][j] : acc[i][j];
                s2[i][j] = keep + __shfl_xor_sync(0xffffffffu, give, 16);
            }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float give = up1 ? s2[0][j] : s2[1][j];
            const float keep = up1 ? s2[1][j] : s2[0][j];
            red[(warp * R + sl) * kOneKeys + kg + 8 * j] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
        }
    } else if constexpr (R == 2) {
        float s1[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float give = up2 ? acc[0][j] : acc[1][j];
            const float keep = up2 ? acc[1][j] : acc[0][j];
            s1[j] = keep + __shfl_xor_sync(0xffffffffu, give, 16);
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float give = up1 ? s1[t] : s1[4 + t];
            const float keep = up1 ? s1[4 + t] : s1[t];
            red[(warp * R + (up2 ? 1 : 0)) * kOneKeys + kg + 8 * (4 * (up1 ? 1 : 0) + t)] =
                keep + __shfl_xor_sync(0xffffffffu, give, 8);
        }
    } else {
        static_assert(R == 1, "rows a CTA: 1, 2 or 4");
        float s1[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float give = up2 ? acc[0][t] : acc[0][4 + t];
            const float keep = up2 ? acc[0][4 + t] : acc[0][t];
            s1[t] = keep + __shfl_xor_sync(0xffffffffu, give, 16);
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const float give = up1 ? s1[t] : s1[2 + t];
            const float keep = up1 ? s1[2 + t] : s1[t];
            red[warp * kOneKeys + kg + 8 * (4 * (up2 ? 1 : 0) + 2 * (up1 ? 1 : 0) + t)] =
                keep + __shfl_xor_sync(0xffffffffu, give, 8);
        }
    }
    __syncthreads();
    // ---- scores summed over the 8 warps, masked, and the softmax: one warp a row
    if (warp < kOneRows) {
        const int r = warp;
        float x[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int key = lane + 32 * h;
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) sum += red[(w * kOneRows + r) * kOneKeys + key];
            const bool visible = key < kv && ((mask_s[r] >> key) & 1ull);
            x[h] = visible ? sum * p.scale_log2 : -INFINITY;
        }
        float m = fmaxf(x[0], x[1]);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        // the hardware base-2 exponential and logarithm (relative error about 2^-22)
        const float p0 = m == -INFINITY ? 0.f : fast_ex2(x[0] - m), p1 = m == -INFINITY ? 0.f : fast_ex2(x[1] - m);
        pt[lane * kOneRows + r] = p0;
        pt[(lane + 32) * kOneRows + r] = p1;
        float l = p0 + p1;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (lane == 0) {
            l_s[r] = l;
            const int gr = r0 + r;
            if (gr < rows_seq && p.lse)
                p.lse[(int64_t)b * rows_seq + gr] = l > 0.f ? 0.6931471805599453f * (m + fast_lg2(l)) : -INFINITY;
        }
    }
    __syncthreads();
    // ---- O = P V over the visible block, columns 2 tid, 2 tid + 1 of the R rows
    float o[kOneRows][2];
#pragma unroll
    for (int i = 0; i < kOneRows; ++i) o[i][0] = o[i][1] = 0.f;
#pragma unroll 4
    for (int key = 0; key < kv; ++key) {
        float pr[R];
        if constexpr (R == 4) {
            const float4 q4 = *reinterpret_cast<const float4 *>(pt + key * R);
            pr[0] = q4.x;
            pr[1] = q4.y;
            pr[2] = q4.z;
            pr[3] = q4.w;
        } else if constexpr (R == 2) {
            const float2 q2 = *reinterpret_cast<const float2 *>(pt + key * R);
            pr[0] = q2.x;
            pr[1] = q2.y;
        } else {
            pr[0] = pt[key];
        }
        const float2 v = get2(kn_s + key * kDc + 2 * tid);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            o[i][0] = fmaf(pr[i], v.x, o[i][0]);
            o[i][1] = fmaf(pr[i], v.y, o[i][1]);
        }
    }
#pragma unroll
    for (int i = 0; i < kOneRows; ++i) {
        const int gr = r0 + i;
        if (gr >= rows_seq) continue;
        const float inv = l_s[i] > 0.f ? 1.f / l_s[i] : 0.f;
        *reinterpret_cast<float2 *>(p.out + ((int64_t)b * rows_seq + gr) * kDc + 2 * tid) =
            make_float2(o[i][0] * inv, o[i][1] * inv);
    }
}

template <typename Tin, int R>
cudaError_t launch_one_rows(const VerifyParams &p, const int32_t *parent, bool check_all, cudaStream_t s) {
    using L = LayoutOne<Tin, R>;
    cudaError_t e =
        cudaFuncSetAttribute(verify_simt_one_kernel<Tin, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
    if (e != cudaSuccess) return e;
    const int rows_seq = p.T * p.H;
    dim3 grid((rows_seq + R - 1) / R, p.B);
    verify_simt_one_kernel<Tin, R><<<grid, kOneThreads, L::kSmem, s>>>(p, parent, check_all);
    return cudaGetLastError();
}

// CTAs of R rows the device holds at once: by shared memory (the key block dominates),
// at most 3 an SM (the register file, 256 threads of at most 80 registers).
template <typename Tin, int R> int64_t one_wave_ctas() {
    int dev = 0, smem_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        smem_sm <= 0)
        smem_sm = 228 * 1024;
    int per_sm = smem_sm / (LayoutOne<Tin, R>::kSmem + 1024);   // 1 KB reserved a CTA
    per_sm = per_sm < 1 ? 1 : (per_sm > 3 ? 3 : per_sm);
    return (int64_t)sm_count() * per_sm;
}

template <typename Tin> int one_rows_typed(int64_t B, int64_t rows_seq) {
    if (B * rows_seq <= one_wave_ctas<Tin, 1>()) return 1;
    if (B * ((rows_seq + 1) / 2) <= one_wave_ctas<Tin, 2>()) return 2;
    return 4;
}

template <typename Tin, int kRows>
cudaError_t launch_typed(const VerifyParams &p, cudaStream_t s) {
    using L = Layout<Tin, kRows>;
    const int rows_seq = p.T * p.H;
    cudaError_t e = cudaFuncSetAttribute(verify_simt_kernel<Tin, kRows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kSmem);
    if (e != cudaSuccess) return e;
    // programmatic dependent launch after the visibility kernel of the same call: the kernel
    // waits for it before its first block with tree keys
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((rows_seq + kRows - 1) / kRows, p.num_splits, p.B);
    cfg.blockDim = dim3(L::kThreads);
    cfg.dynamicSmemBytes = L::kSmem;
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = p.overlap_vis ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, verify_simt_kernel<Tin, kRows>, p);
}

// Combines the pieces of every row tile that the work split of the 64-row tile cut: CTA
// (tile, y) merges rows 8 y .. 8 y + 7 of the tile, one warp a row. The tile spans work
// positions [T0, T1); the CTAs whose ranges meet it are c_a = cta_of(T0) .. c_b =
// cta_of(T1 - 1) (one CTA: the tile was written whole), each with a normalised state
// (o, lse) in slot 2c (its range starts inside the tile) or 2c + 1 (its range starts
// before). Merge by log-sum-exp: lse = log sum_k e^lse_k, o = sum_k e^(lse_k - lse) o_k.
__global__ void __launch_bounds__(256) merge_simt_pieces_kernel(const VerifyParams p) {
    tc::griddep_wait();                       // the pieces are written by the kernel before
    constexpr int kR = kSimtRows, kKB = kSimtKeysTm;
    const int rows_seq = p.T * p.H;
    const int tiles_seq = (rows_seq + kR - 1) / kR;
    const int tile = blockIdx.x, b = tile / tiles_seq, rt = tile % tiles_seq;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t C = p.simt_ctas;
    // W and the positions before sequence b, over all threads
    int64_t tot = 0, bef = 0;
    for (int bb = threadIdx.x; bb < p.B; bb += blockDim.x) {
        const int64_t w = (int64_t)tiles_seq * seq_blocks_of(p, bb, kKB);
        tot += w;
        if (bb < b) bef += w;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, off);
        bef += __shfl_xor_sync(0xffffffffu, bef, off);
    }
    __shared__ int64_t part[2][8];
    if (lane == 0) {
        part[0][warp] = tot;
        part[1][warp] = bef;
    }
    __syncthreads();
    int64_t W = 0, before = 0;
    for (int k = 0; k < (int)(blockDim.x >> 5); ++k) {
        W += part[0][k];
        before += part[1][k];
    }
    const int nblk = seq_blocks_of(p, b, kKB);
    const int64_t T0 = before + (int64_t)rt * nblk, T1 = T0 + nblk;
    auto cta_of = [&](int64_t x) { return ((x + 1) * C - 1) / W; };   // largest c with W c / C <= x
    auto start_of = [&](int64_t cc) { return W * cc / C; };
    const int64_t ca = cta_of(T0), cb = cta_of(T1 - 1);
    if (ca == cb) return;
    const int row = blockIdx.y * 8 + warp;
    const int r = rt * kR + row;
    if (row >= kR || r >= rows_seq) return;
    // the pieces' lse, 32 at a time (lane k: CTA base + k), in one round trip each
    auto slot_of = [&](int64_t cc) -> int64_t {                      // -1: an empty range
        if (cc > cb || start_of(cc) == start_of(cc + 1)) return -1;
        return start_of(cc) >= T0 ? 2 * cc : 2 * cc + 1;
    };
    float M = -INFINITY;
    for (int64_t base = ca; base <= cb; base += 32) {
        const int64_t sl = slot_of(base + lane);
        if (sl >= 0) M = fmaxf(M, p.part_lse[sl * kR + row]);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float4 acc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    float S = 0.f;
    if (M > -INFINITY) {
        for (int64_t base = ca; base <= cb; base += 32) {
            const int64_t sl = slot_of(base + lane);
            const float w = sl >= 0 ? __expf(p.part_lse[sl * kR + row] - M) : 0.f;
            S += w;
            const int cnt = (int)(cb - base + 1 < 32 ? cb - base + 1 : 32);
            // the pieces' rows as independent loads, the weights broadcast from their lanes
#pragma unroll 4
            for (int k = 0; k < cnt; ++k) {
                const float wk = __shfl_sync(0xffffffffu, w, k);
                const int64_t slk = __shfl_sync(0xffffffffu, sl, k);
                if (slk < 0) continue;                                // the same for the whole warp
                const float4 *src = reinterpret_cast<const float4 *>(p.part_o + (slk * kR + row) * kDc) + lane;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 v = src[32 * q];
                    acc[q].x = fmaf(wk, v.x, acc[q].x);
                    acc[q].y = fmaf(wk, v.y, acc[q].y);
                    acc[q].z = fmaf(wk, v.z, acc[q].z);
                    acc[q].w = fmaf(wk, v.w, acc[q].w);
                }
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) S += __shfl_xor_sync(0xffffffffu, S, off);
    }
    const float inv = S > 0.f ? 1.f / S : 0.f;
    float4 *dst = reinterpret_cast<float4 *>(p.out + ((int64_t)b * rows_seq + r) * kDc) + lane;
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[32 * q] = make_float4(acc[q].x * inv, acc[q].y * inv, acc[q].z * inv, acc[q].w * inv);
    if (lane == 0 && p.lse) p.lse[(int64_t)b * rows_seq + r] = S > 0.f ? M + __logf(S) : -INFINITY;
}

}  // namespace

cudaError_t launch_verify_simt(const VerifyParams &p, kdt_dtype dt, int rows_per_cta, cudaStream_t s) {
    if (rows_per_cta == kSimtSmallRows)
        return dt == KDT_F32 ? launch_typed<float, kSimtSmallRows>(p, s) : launch_typed<__nv_bfloat16, kSimtSmallRows>(p, s);
    return dt == KDT_F32 ? launch_typed_tm<float>(p, s) : launch_typed_tm<__nv_bfloat16>(p, s);
}

int simt_one_rows(kdt_dtype dt, int64_t B, int64_t rows_seq) {
    return dt == KDT_F32 ? one_rows_typed<float>(B, rows_seq) : one_rows_typed<__nv_bfloat16>(B, rows_seq);
}

cudaError_t launch_verify_simt_one(const VerifyParams &p, kdt_dtype dt, const int32_t *parent, bool check_all,
                                   int rows_per_cta, cudaStream_t s) {
    if (dt == KDT_F32) {
        return rows_per_cta == 1   ? launch_one_rows<float, 1>(p, parent, check_all, s)
               : rows_per_cta == 2 ? launch_one_rows<float, 2>(p, parent, check_all, s)
                                   : launch_one_rows<float, 4>(p, parent, check_all, s);
    }
    return rows_per_cta == 1   ? launch_one_rows<__nv_bfloat16, 1>(p, parent, check_all, s)
           : rows_per_cta == 2 ? launch_one_rows<__nv_bfloat16, 2>(p, parent, check_all, s)
                               : launch_one_rows<__nv_bfloat16, 4>(p, parent, check_all, s);
}

cudaError_t launch_merge_simt_pieces(const VerifyParams &p, cudaStream_t s) {
    const int rows_seq = p.T * p.H;
    const int tiles_seq = (rows_seq + kSimtRows - 1) / kSimtRows;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)p.B * tiles_seq), kSimtRows / 8);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_simt_pieces_kernel, p);
}

}  // namespace kdt
