// K4: per-head value up-projection of the latent attention output (tcgen05).
//
// The verify kernel returns the latent o[r, h, :512] (r = b*T + i); the head's value
// is v[r, h, :] = o[r, h, :] . w_vc[h] with w_vc[h] of shape [512, D_v], a GEMM kept
// apart from the attention kernel (page "The Verify-Attn Kernel: A Single File Write
// ...", section "Design Decisions and Trade-Offs").
//
// GB300 design:
//  * Per head this is a dense contraction M = rows x N = D_v x K = 512. Its arithmetic
//    intensity is low (about 47 FLOP/B at D_v = 128, fp32 o read once): the kernel is
//    HBM-bound, and the tensor cores are what keeps the contraction below the memory
//    time (fp32 FMA alone would take four times longer than the bytes).
//  * Precision: o is fp32 and w_vc bf16. Each o element is split into two bf16 parts,
//    hi = bf16(o) and lo = bf16(o - hi), so o = hi + lo to within 2^-16 |o| (bf16's unit
//    roundoff 2^-8, squared: |o - hi| <= 2^-8 |o| and lo rounds that again); both parts
//    are multiplied by the (exact) bf16 weights on the tensor cores, accumulating in
//    fp32 in tensor memory. The result meets the fp32 path's bound at twice the MMA
//    work, which still hides under the memory time.
//  * Work: tiles of 128 rows of one head (M = 128, cta_group::1), persistent CTAs (one
//    per SM) taking tiles in head-major order, so the CTAs running at once share a few
//    heads' weights in L2. Per 64-wide latent chunk the fp32 rows arrive by TMA (two
//    128B-swizzled [128 x 32] boxes) into a 4-slot staging ring and the weights into a
//    4-slot ring, so 128 KB of rows and 64 KB of weights per SM are in flight; eight
//    converter warps (one row per thread, half a chunk per warp) write hi and lo into
//    tensor memory with tcgen05.st, where the MMA reads its A operand, so shared memory
//    holds only the staging, the weights and the epilogue transpose. The weights arrive by TMA as MN-major tiles; one thread issues the MMAs.
//    The accumulator is double-buffered in tensor memory (2 x 128 columns, next to two
//    64-column A slots) so one tile's epilogue (four warps, rows transposed through
//    shared memory into whole 128-byte line stores) overlaps the next tile's loads.
//  * Measured and not kept: equal shares of 8-row groups per CTA instead of whole tiles
//    (a share then spans up to three partial tiles, each streaming the head's full
//    weights: slower on both shapes timed although it evens out the last wave), and an
//    L2 bulk prefetch of a tile's whole 2 KB rows ahead of its chunk loads (slower).
#include "kdt_internal.cuh"
#include "tc_ptx.cuh"

#include <string.h>

namespace kdt {
namespace {

using namespace tc;

constexpr int kVRows = 128;                  // rows of a tile (MMA M)
constexpr int kVChunk = 64;                  // latent dims per chunk (one 128-byte bf16 row)
constexpr int kVChunks = kDc / kVChunk;      // 8
constexpr int kVThreads = 512;               // 16 warps
constexpr int kNF = 4;                       // fp32 staging slots
constexpr int kNA = 2;                       // tensor-memory A slots (hi + lo of one chunk)
constexpr int kNW = 4;                       // weight slots
constexpr int kConvWarps = 8;                // converter warps 4..11
constexpr int kF32Box = kVRows * 32 * 4;            // [128 rows x 32 fp32], 128B-swizzled: 16 KB
constexpr int kF32Bytes = 2 * kF32Box;              // one chunk: 32 KB
constexpr int kWSub = kVChunk * 128;                // [64 latent rows x 64 value cols] bf16: 8 KB
constexpr int kMaxDv = 128;
constexpr int kWSlot = (kMaxDv / 64) * kWSub;       // 16 KB
constexpr int kOffF = 0;
constexpr int kOffW = kOffF + kNF * kF32Bytes;
constexpr int kOffEpi = kOffW + kNW * kWSlot;
constexpr int kVTile = kOffEpi + 4 * 32 * 32 * 4;
constexpr int kVSmem = kVTile + 1024;
static_assert(kVSmem <= 227 * 1024, "shared memory budget");
// Tensor memory: accumulators at columns [0, 256), A slot s at 256 + 64 s (hi: 32 columns
// of packed bf16 pairs, then lo).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = kMaxDv;
constexpr uint32_t kACol0 = 2 * kAccCols;
constexpr uint64_t kVWaitLimit = 200000000ull;      // ns a wait may poll before giving up

struct VBars {
    uint64_t f_full[kNF], f_empty[kNF];
    uint64_t a_full[kNA], a_empty[kNA];
    uint64_t w_full[kNW], w_empty[kNW];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

struct VParams {
    int R, H, Dv;
    int row_tiles, tiles;
    float *v;
    int32_t *err;
};

__device__ __forceinline__ bool v_aborted(const VBars &b) {
    return *reinterpret_cast<const volatile int *>(&b.abort_flag) != 0;
}

__device__ __forceinline__ bool v_wait(VBars &b, uint64_t *bar, uint32_t parity, int32_t *err, int code) {
    if (v_aborted(b)) return false;
    if (mbar_wait(bar, parity, kVWaitLimit)) return true;
    b.abort_flag = 1;
    if (err) atomicCAS(err, 0, code);
    return false;
}

// bf16 round-to-nearest-even of two floats packed (lo element in the low half).
__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

__device__ __forceinline__ float bf16_lo_as_f32(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf16_hi_as_f32(uint32_t p) { return __uint_as_float(p & 0xFFFF0000u); }

// 32 lanes x 16 consecutive 32-bit columns: thread t of the warp writes lane (base + t).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__global__ void __launch_bounds__(kVThreads, 1)
    vc_proj_kernel(const __grid_constant__ CUtensorMap map_o, const __grid_constant__ CUtensorMap map_w,
                   const VParams p) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ VBars bar;
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_sub = p.Dv / 64;                       // 64-column weight sub-tiles per chunk
    const uint32_t w_bytes = (uint32_t)n_sub * kWSub;
    // tiles of this CTA: blockIdx.x, blockIdx.x + gridDim.x, ...
    const int my_tiles = p.tiles > (int)blockIdx.x ? (p.tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNF; ++i) { mbar_init(&bar.f_full[i], 1); mbar_init(&bar.f_empty[i], kConvWarps); }
        for (int i = 0; i < kNA; ++i) { mbar_init(&bar.a_full[i], kConvWarps); mbar_init(&bar.a_empty[i], 1); }
        for (int i = 0; i < kNW; ++i) { mbar_init(&bar.w_full[i], 1); mbar_init(&bar.w_empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&bar.acc_full[i], 1); mbar_init(&bar.acc_empty[i], 4); }
        mbar_init(&bar.drain, 1);
        bar.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&bar.tmem_base, kTmemCols);         // two accumulators, two A slots
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem_base;

    if (warp == 0 || warp == 2) {
        // ---------------- TMA producers: warp 0 the fp32 rows of o, warp 2 the weights -------
        // (separate threads, so the shallower weight ring never holds up the row loads)
        if (elect_one() && my_tiles > 0) {
            const bool rows = warp == 0;
            tma_prefetch_desc(rows ? &map_o : &map_w);
            const int depth = rows ? kNF : kNW;
            uint64_t *full = rows ? bar.f_full : bar.w_full;
            uint64_t *empty = rows ? bar.f_empty : bar.w_empty;
            bool ok = true;
            int n = 0;                                   // loads issued
            for (int k = 0; k < my_tiles && ok; ++k) {
                const int t = (int)blockIdx.x + k * (int)gridDim.x;
                const int h = t / p.row_tiles, r0 = (t % p.row_tiles) * kVRows;
                for (int c = 0; c < kVChunks; ++c) {
                    const int g = k * kVChunks + c;
                    const int sl = g % depth;
                    if (g >= depth &&
                        !(ok = v_wait(bar, &empty[sl], (uint32_t)((g / depth) - 1) & 1, p.err, rows ? -31 : -32)))
                        break;
                    if (rows) {
                        mbar_arrive_expect_tx(&full[sl], kF32Bytes);
                        for (int hh = 0; hh < 2; ++hh)
                            tma_load_3d(smem + kOffF + sl * kF32Bytes + hh * kF32Box, &map_o, &full[sl],
                                        c * kVChunk + 32 * hh, h, r0);
                    } else {
                        mbar_arrive_expect_tx(&full[sl], w_bytes);
                        for (int nn = 0; nn < n_sub; ++nn)
                            tma_load_3d(smem + kOffW + sl * kWSlot + nn * kWSub, &map_w, &full[sl], 64 * nn,
                                        c * kVChunk, h);
                    }
                    ++n;
                }
            }
            // every copy issued has landed and been consumed before the CTA may leave
            // (bounded: on the error path a use nobody consumes times out)
            for (int g = n - depth > 0 ? n - depth : 0; g < n; ++g)
                mbar_wait(&empty[g % depth], (uint32_t)(g / depth) & 1, kVWaitLimit);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: acc (+)= hi . W + lo . W over the 8 chunks --------------
        if (elect_one() && my_tiles > 0) {
            const uint32_t idesc = idesc_bf16_f32(kVRows, (uint32_t)p.Dv, 0, 1);
            bool ok = true;
            for (int k = 0; k < my_tiles && ok; ++k) {
                const int buf = k & 1;
                if (k >= 2 && !(ok = v_wait(bar, &bar.acc_empty[buf], (uint32_t)((k >> 1) - 1) & 1, p.err, -33)))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)buf * kAccCols;
                for (int c = 0; c < kVChunks && ok; ++c) {
                    const int g = k * kVChunks + c;
                    const int as = g % kNA, ws = g % kNW;
                    if (!(ok = v_wait(bar, &bar.a_full[as], (uint32_t)(g / kNA) & 1, p.err, -34))) break;
                    if (!(ok = v_wait(bar, &bar.w_full[ws], (uint32_t)(g / kNW) & 1, p.err, -35))) break;
                    tc_fence_after();
                    const uint32_t a0 = tmem + kACol0 + (uint32_t)(as * 64);
                    const uint32_t w0 = smem_u32(smem + kOffW + ws * kWSlot);
                    for (int part = 0; part < 2; ++part)
                        for (int kk = 0; kk < kVChunk / 16; ++kk) {
                            const uint64_t bdesc = sdesc_sw128(w0 + kk * 2048, kWSub, 1024);
                            mma_ts(d, a0 + 32 * part + 8 * kk, bdesc, idesc, (c > 0 || part > 0 || kk > 0) ? 1u : 0u);
                        }
                    mma_commit(&bar.a_empty[as]);
                    mma_commit(&bar.w_empty[ws]);
                }
                if (ok) mma_commit(&bar.acc_full[buf]);
            }
            mma_commit(&bar.drain);                   // every MMA of this CTA has completed
            mbar_wait(&bar.drain, 0, kVWaitLimit);
        }
    } else if (warp >= 4 && warp < 4 + kConvWarps) {
        // ---------------- converters: fp32 -> bf16 hi and lo into tensor memory ---------------
        // Warp w serves TMEM lane quadrant w % 4 (rows 32 (w % 4) + lane, one per thread) and
        // latent dims [32 hh, 32 hh + 32) of each chunk, hh = (w - 4) / 4: its rows of the
        // staged box hh, 128B-swizzled (16-byte unit u of row r at u ^ (r % 8)).
        const int q = warp & 3, hh = (warp - 4) >> 2;
        const int row = 32 * q + lane;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        bool ok = true;
        for (int k = 0; k < my_tiles && ok; ++k) {
            for (int c = 0; c < kVChunks && ok; ++c) {
                const int g = k * kVChunks + c;
                const int fs = g % kNF, as = g % kNA;
                ok = __all_sync(0xffffffffu, v_wait(bar, &bar.f_full[fs], (uint32_t)(g / kNF) & 1, p.err, -36));
                if (ok && g >= kNA)
                    ok = __all_sync(0xffffffffu,
                                    v_wait(bar, &bar.a_empty[as], (uint32_t)((g / kNA) - 1) & 1, p.err, -37));
                if (!ok) break;
                tc_fence_after();
                const unsigned char *src = smem + kOffF + fs * kF32Bytes + hh * kF32Box + row * 128;
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float4 x = *reinterpret_cast<const float4 *>(src + ((u ^ (row & 7)) << 4));
                    const uint32_t h01 = pack2_bf16(x.x, x.y), h23 = pack2_bf16(x.z, x.w);
                    hi[2 * u] = h01;
                    hi[2 * u + 1] = h23;
                    lo[2 * u] = pack2_bf16(x.x - bf16_lo_as_f32(h01), x.y - bf16_hi_as_f32(h01));
                    lo[2 * u + 1] = pack2_bf16(x.z - bf16_lo_as_f32(h23), x.w - bf16_hi_as_f32(h23));
                }
                const uint32_t a0 = tmem + lane_base + kACol0 + (uint32_t)(as * 64 + 16 * hh);
                tmem_st16(a0, hi);
                tmem_st16(a0 + 32, lo);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bar.a_full[as]);
                    mbar_arrive(&bar.f_empty[fs]);
                }
            }
        }
    } else if (warp >= 4 + kConvWarps) {
        // ---------------- epilogue: accumulator rows -> v[r, h, :] ----------------------------
        const int q = warp & 3;                              // TMEM lane quadrant of this warp
        float *stg = reinterpret_cast<float *>(smem + kOffEpi) + q * 32 * 32;
        const int rsub = lane >> 3, qsub = lane & 7;
        bool ok = true;
        for (int k = 0; k < my_tiles && ok; ++k) {
            const int buf = k & 1;
            const int t = (int)blockIdx.x + k * (int)gridDim.x;
            const int h = t / p.row_tiles, r0 = (t % p.row_tiles) * kVRows + 32 * q;
            ok = __all_sync(0xffffffffu, v_wait(bar, &bar.acc_full[buf], (uint32_t)(k >> 1) & 1, p.err, -38));
            if (!ok) break;
            tc_fence_after();
            const int rows_ok = p.R - r0;                    // rows of this warp's 32 that exist
            const int64_t rstride = (int64_t)p.H * p.Dv;
            float *vrow0 = p.v + ((int64_t)r0 * p.H + h) * p.Dv;
            for (int cc = 0; cc < p.Dv / 32; ++cc) {
                uint32_t rv[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)buf * kAccCols + (uint32_t)(32 * cc), rv);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    *reinterpret_cast<float4 *>(stg + lane * 32 + ((u ^ (lane & 7)) << 2)) =
                        make_float4(__uint_as_float(rv[4 * u]), __uint_as_float(rv[4 * u + 1]),
                                    __uint_as_float(rv[4 * u + 2]), __uint_as_float(rv[4 * u + 3]));
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int rr = 4 * i + rsub;
                    const float4 val = *reinterpret_cast<const float4 *>(stg + rr * 32 + ((qsub ^ (rr & 7)) << 2));
                    if (rr < rows_ok)
                        *reinterpret_cast<float4 *>(vrow0 + (int64_t)rr * rstride + cc * 32 + 4 * qsub) = val;
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.acc_empty[buf]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn v_encode_fn() {
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

}  // namespace

cudaError_t launch_vc_proj(const float *o, const void *w_vc, int R, int H, int Dv, float *v, int32_t *err,
                           cudaStream_t s) {
    EncodeTiledFn fn = v_encode_fn();
    if (!fn) return cudaErrorInvalidValue;
    CUtensorMap map_o, map_w;
    memset(&map_o, 0, sizeof(map_o));
    memset(&map_w, 0, sizeof(map_w));
    {
        // o as [R rows][H heads][512] fp32; a box is 32 dims (128 bytes) of one head's 128 rows
        const cuuint64_t dims[3] = {(cuuint64_t)kDc, (cuuint64_t)H, (cuuint64_t)R};
        const cuuint64_t strides[2] = {(cuuint64_t)kDc * 4, (cuuint64_t)H * kDc * 4};
        const cuuint32_t box[3] = {32, 1, kVRows};
        const cuuint32_t es[3] = {1, 1, 1};
        if (fn(&map_o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(o), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // w_vc as [H][512 latent rows][Dv] bf16; a box is [64 latent rows x 64 value cols]
        const cuuint64_t dims[3] = {(cuuint64_t)Dv, (cuuint64_t)kDc, (cuuint64_t)H};
        const cuuint64_t strides[2] = {(cuuint64_t)Dv * 2, (cuuint64_t)kDc * Dv * 2};
        const cuuint32_t box[3] = {64, kVChunk, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        if (fn(&map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(w_vc), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    VParams p;
    p.R = R;
    p.H = H;
    p.Dv = Dv;
    p.row_tiles = (R + kVRows - 1) / kVRows;
    p.tiles = p.row_tiles * H;
    p.v = v;
    p.err = err;
    const int grid = p.tiles < sm_count() ? p.tiles : sm_count();
    cudaError_t e = cudaFuncSetAttribute(vc_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kVSmem);
    if (e != cudaSuccess) return e;
    vc_proj_kernel<<<grid, kVThreads, kVSmem, s>>>(map_o, map_w, p);
    return cudaGetLastError();
}

}  // namespace kdt
