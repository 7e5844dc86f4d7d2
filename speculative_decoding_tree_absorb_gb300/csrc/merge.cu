// K2: log-sum-exp merge of attention states computed over disjoint key sets.
//
// Split-KV partials are combined exactly as the pages combine a long prefix done
// by one kernel with the tree tail done by another (page "The Verify-Attn Kernel:
// A Single File Write ...", section "Design Decisions and Trade-Offs"; page "The
// Moment of Truth ...", section "The Design Journey: From Theory to Silicon"):
//   M = max_s lse_s,  w_s = exp(lse_s - M),
//   o = sum_s w_s o_s / sum_s w_s,  lse = M + ln sum_s w_s,
// where each o_s is already normalised over its own keys. A state with
// lse = -inf (no visible key) has weight 0; all -inf gives o = 0, lse = -inf.
//
// One warp per row: lane s holds split s's lse, the max and the weight sum are
// warp-shuffle reductions, and the weights are broadcast by shuffle while the
// lanes stream the 512 output columns as float4s.
#include "kdt_internal.cuh"
#include "tc_ptx.cuh"

#include <math.h>

namespace kdt {
namespace {

constexpr int kWarpsPerCta = 8;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Merge the S partial states of one row (partial s at part_o[(s*stride + k)*512],
// part_lse[s*stride + k]) into out_row / lse_out. One warp.
__device__ __forceinline__ void merge_row(const float *__restrict__ part_o, const float *__restrict__ part_lse, int S,
                                          int64_t stride, int64_t k, float *__restrict__ out_row, float *lse_out) {
    const int lane = threadIdx.x & 31;
    const float ls = lane < S ? part_lse[(int64_t)lane * stride + k] : -INFINITY;
    const float M = warp_max(ls);
    const float w = (M == -INFINITY || ls == -INFINITY) ? 0.f : expf(ls - M);
    const float wsum = warp_sum(w);
    float4 acc[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < S; ++s) {
        const float ws = __shfl_sync(0xffffffffu, w, s);
        if (ws == 0.f) continue;
        const float4 *src = reinterpret_cast<const float4 *>(part_o + ((int64_t)s * stride + k) * kDc);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float4 v = __ldg(src + lane + 32 * c);
            acc[c].x = fmaf(ws, v.x, acc[c].x);
            acc[c].y = fmaf(ws, v.y, acc[c].y);
            acc[c].z = fmaf(ws, v.z, acc[c].z);
            acc[c].w = fmaf(ws, v.w, acc[c].w);
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    float4 *dst = reinterpret_cast<float4 *>(out_row);
#pragma unroll
    for (int c = 0; c < 4; ++c)
        dst[lane + 32 * c] = make_float4(acc[c].x * inv, acc[c].y * inv, acc[c].z * inv, acc[c].w * inv);
    if (lane == 0 && lse_out) *lse_out = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

__global__ void __launch_bounds__(kWarpsPerCta * 32) merge_splits_kernel(const float *__restrict__ part_o,
                                                                         const float *__restrict__ part_lse,
                                                                         int S, int64_t rows,
                                                                         float *__restrict__ out,
                                                                         float *__restrict__ lse) {
    // launched to overlap the end of the attention kernel that wrote the partials
    tc::griddep_wait();
    const int64_t row = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    if (row >= rows) return;
    merge_row(part_o, part_lse, S, rows, row, out + row * kDc, lse ? lse + row : nullptr);
}

__global__ void __launch_bounds__(kWarpsPerCta * 32) merge_two_kernel(const float *o_a, const float *lse_a,
                                                                      const float *o_b, const float *lse_b,
                                                                      int64_t rows, int D, float *o,
                                                                      float *lse) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    if (row >= rows) return;
    const float la = lse_a[row], lb = lse_b[row];
    const float M = fmaxf(la, lb);
    const float wa = (la == -INFINITY) ? 0.f : expf(la - M);
    const float wb = (lb == -INFINITY) ? 0.f : expf(lb - M);
    const float ws = wa + wb;
    const float inv = ws > 0.f ? 1.f / ws : 0.f;
    const float4 *pa = reinterpret_cast<const float4 *>(o_a + row * D);
    const float4 *pb = reinterpret_cast<const float4 *>(o_b + row * D);
    float4 *po = reinterpret_cast<float4 *>(o + row * D);
    for (int c = lane; c < D / 4; c += 32) {
        const float4 x = pa[c], y = pb[c];
        po[c] = make_float4((wa * x.x + wb * y.x) * inv, (wa * x.y + wb * y.y) * inv,
                            (wa * x.z + wb * y.z) * inv, (wa * x.w + wb * y.w) * inv);
    }
    // every lane has read lse_a/lse_b before lane 0 may overwrite them in place
    __syncwarp();
    if (lane == 0) lse[row] = ws > 0.f ? M + logf(ws) : -INFINITY;
}

}  // namespace

cudaError_t launch_merge_splits(const float *part_o, const float *part_lse, int num_splits, int64_t rows,
                                float *out, float *lse, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int64_t ctas = (rows + kWarpsPerCta - 1) / kWarpsPerCta;
    // programmatic dependent launch after the split attention kernel (the kernel waits for
    // it before reading the partials)
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kWarpsPerCta * 32);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, merge_splits_kernel, part_o, part_lse, num_splits, rows, out, lse);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_merge_two(const float *o_a, const float *lse_a, const float *o_b, const float *lse_b,
                             int64_t rows, int D, float *o, float *lse, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int64_t ctas = (rows + kWarpsPerCta - 1) / kWarpsPerCta;
    merge_two_kernel<<<(unsigned)ctas, kWarpsPerCta * 32, 0, s>>>(o_a, lse_a, o_b, lse_b, rows, D, o, lse);
    return cudaGetLastError();
}

}  // namespace kdt
