// K4: per-head value up-projection of the latent attention output (tcgen05).
//
// The verify kernel returns the latent o[r, h, :512] (r = b*T + i); the head's value
// is v[r, h, :] = o[r, h, :] . w_vc[h] with w_vc[h] of shape [512, D_v]: "a follow-up
// matrix multiply applies the per-head value weights" (page "The Verify-Attn Kernel:
// A Single File Write ...", section "Design Decisions and Trade-Offs").
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
//    heads' weights in L2. Per 64-wide latent chunk: the fp32 rows arrive by TMA into a
//    2-slot staging ring, four converter warps write hi and lo as 128B-swizzled K-major
//    bf16 tiles, the weights arrive by TMA as MN-major tiles, and one thread issues the
//    MMAs. The accumulator is double-buffered in tensor memory (2 x D_v columns) so one
//    tile's epilogue (four warps, rows transposed through shared memory into whole
//    128-byte line stores) overlaps the next tile's loads and MMAs.
//  * Every wait is bounded; on expiry the kernel records a negative code in the error
//    word, lets the other roles leave, drains its MMAs, frees tensor memory and returns.
#include "kdt_internal.cuh"
#include "tc_ptx.cuh"

#include <string.h>

namespace kdt {
namespace {

using namespace tc;

constexpr int kVRows = 128;                  // rows of a tile (MMA M)
constexpr int kVChunk = 64;                  // latent dims per chunk (one 128-byte bf16 row)
constexpr int kVChunks = kDc / kVChunk;      // 8
constexpr int kVThreads = 384;               // 12 warps
constexpr int kNF = 2;                       // fp32 staging slots
constexpr int kNA = 2;                       // bf16 operand slots (hi + lo)
constexpr int kNW = 3;                       // weight slots
constexpr int kF32Bytes = kVRows * kVChunk * 4;     // 32 KB
constexpr int kAHalf = kVRows * kVChunk * 2;        // 16 KB: one bf16 part
constexpr int kASlot = 2 * kAHalf;                  // hi then lo
constexpr int kWSub = kVChunk * 128;                // [64 latent rows x 64 value cols] bf16: 8 KB
constexpr int kMaxDv = 128;
constexpr int kWSlot = (kMaxDv / 64) * kWSub;       // 16 KB
constexpr int kOffF = 0;
constexpr int kOffA = kOffF + kNF * kF32Bytes;
constexpr int kOffW = kOffA + kNA * kASlot;
constexpr int kOffEpi = kOffW + kNW * kWSlot;
constexpr int kVTile = kOffEpi + 4 * 32 * 32 * 4;
constexpr int kVSmem = kVTile + 1024;
static_assert(kVSmem <= 227 * 1024, "shared memory budget");
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
        for (int i = 0; i < kNF; ++i) { mbar_init(&bar.f_full[i], 1); mbar_init(&bar.f_empty[i], 4); }
        for (int i = 0; i < kNA; ++i) { mbar_init(&bar.a_full[i], 4); mbar_init(&bar.a_empty[i], 1); }
        for (int i = 0; i < kNW; ++i) { mbar_init(&bar.w_full[i], 1); mbar_init(&bar.w_empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&bar.acc_full[i], 1); mbar_init(&bar.acc_empty[i], 4); }
        mbar_init(&bar.drain, 1);
        bar.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&bar.tmem_base, 256);               // two accumulators of up to 128 columns
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar.tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer: fp32 rows of o and the head's weights ----------------
        if (elect_one() && my_tiles > 0) {
            tma_prefetch_desc(&map_o);
            tma_prefetch_desc(&map_w);
            bool ok = true;
            int nf = 0, nw = 0;                          // staging and weight loads issued
            for (int k = 0; k < my_tiles && ok; ++k) {
                const int t = (int)blockIdx.x + k * (int)gridDim.x;
                const int h = t / p.row_tiles, r0 = (t % p.row_tiles) * kVRows;
                for (int c = 0; c < kVChunks && ok; ++c) {
                    const int g = k * kVChunks + c;
                    const int fs = g % kNF, ws = g % kNW;
                    if (g >= kNF && !(ok = v_wait(bar, &bar.f_empty[fs], (uint32_t)((g / kNF) - 1) & 1, p.err, -31)))
                        break;
                    mbar_arrive_expect_tx(&bar.f_full[fs], kF32Bytes);
                    tma_load_3d(smem + kOffF + fs * kF32Bytes, &map_o, &bar.f_full[fs], c * kVChunk, h, r0);
                    ++nf;
                    if (g >= kNW && !(ok = v_wait(bar, &bar.w_empty[ws], (uint32_t)((g / kNW) - 1) & 1, p.err, -32)))
                        break;
                    mbar_arrive_expect_tx(&bar.w_full[ws], w_bytes);
                    for (int n = 0; n < n_sub; ++n)
                        tma_load_3d(smem + kOffW + ws * kWSlot + n * kWSub, &map_w, &bar.w_full[ws], 64 * n,
                                    c * kVChunk, h);
                    ++nw;
                }
            }
            // every copy issued has landed and been consumed before the CTA may leave
            // (bounded: on the error path a use nobody consumes times out)
            for (int g = nf - kNF > 0 ? nf - kNF : 0; g < nf; ++g)
                mbar_wait(&bar.f_empty[g % kNF], (uint32_t)(g / kNF) & 1, kVWaitLimit);
            for (int g = nw - kNW > 0 ? nw - kNW : 0; g < nw; ++g)
                mbar_wait(&bar.w_empty[g % kNW], (uint32_t)(g / kNW) & 1, kVWaitLimit);
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
                const uint32_t d = tmem + (uint32_t)(buf * kMaxDv);
                for (int c = 0; c < kVChunks && ok; ++c) {
                    const int g = k * kVChunks + c;
                    const int as = g % kNA, ws = g % kNW;
                    if (!(ok = v_wait(bar, &bar.a_full[as], (uint32_t)(g / kNA) & 1, p.err, -34))) break;
                    if (!(ok = v_wait(bar, &bar.w_full[ws], (uint32_t)(g / kNW) & 1, p.err, -35))) break;
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(smem + kOffA + as * kASlot);
                    const uint32_t w0 = smem_u32(smem + kOffW + ws * kWSlot);
                    for (int part = 0; part < 2; ++part)
                        for (int kk = 0; kk < kVChunk / 16; ++kk) {
                            const uint64_t adesc = sdesc_sw128(a0 + part * kAHalf + kk * 32, 16, 1024);
                            const uint64_t bdesc = sdesc_sw128(w0 + kk * 2048, kWSub, 1024);
                            mma_ss(d, adesc, bdesc, idesc, (c > 0 || part > 0 || kk > 0) ? 1u : 0u);
                        }
                    mma_commit(&bar.a_empty[as]);
                    mma_commit(&bar.w_empty[ws]);
                }
                if (ok) mma_commit(&bar.acc_full[buf]);
            }
            mma_commit(&bar.drain);                   // every MMA of this CTA has completed
            mbar_wait(&bar.drain, 0, kVWaitLimit);
        }
    } else if (warp >= 4 && warp < 8) {
        // ---------------- converters: fp32 -> bf16 hi and lo, 128B-swizzled K-major -----------
        const int tid = threadIdx.x - 128;
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
                const float4 *src = reinterpret_cast<const float4 *>(smem + kOffF + fs * kF32Bytes);
                unsigned char *hi = smem + kOffA + as * kASlot;
                unsigned char *lo = hi + kAHalf;
#pragma unroll 4
                for (int j = 0; j < 16; ++j) {
                    const int f = tid + 128 * j;            // float4 f of the [128 x 64] chunk
                    const int r = f >> 4, c4 = f & 15;
                    const float4 x = src[f];
                    const uint32_t h01 = pack2_bf16(x.x, x.y), h23 = pack2_bf16(x.z, x.w);
                    const uint32_t l01 = pack2_bf16(x.x - bf16_lo_as_f32(h01), x.y - bf16_hi_as_f32(h01));
                    const uint32_t l23 = pack2_bf16(x.z - bf16_lo_as_f32(h23), x.w - bf16_hi_as_f32(h23));
                    // element 4 c4 of row r: 16-byte unit c4 / 2 of the row, swizzled by row % 8
                    const uint32_t off = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((c4 >> 1) ^ (r & 7))) << 4) +
                                                    (c4 & 1) * 8);
                    *reinterpret_cast<uint2 *>(hi + off) = make_uint2(h01, h23);
                    *reinterpret_cast<uint2 *>(lo + off) = make_uint2(l01, l23);
                }
                fence_proxy_async_smem();                    // the MMA reads through the async proxy
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bar.a_full[as]);
                    mbar_arrive(&bar.f_empty[fs]);
                }
            }
        }
    } else if (warp >= 8) {
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
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * kMaxDv + 32 * cc), rv);
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
    if (warp == 0) tmem_dealloc(tmem, 256);
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
        // o as [R rows][H heads][512] fp32; a box is one head's 64-dim chunk of 128 rows
        const cuuint64_t dims[3] = {(cuuint64_t)kDc, (cuuint64_t)H, (cuuint64_t)R};
        const cuuint64_t strides[2] = {(cuuint64_t)kDc * 4, (cuuint64_t)H * kDc * 4};
        const cuuint32_t box[3] = {kVChunk, 1, kVRows};
        const cuuint32_t es[3] = {1, 1, 1};
        if (fn(&map_o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(o), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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
