// K0: draft-tree parent array -> packed ancestor/self visibility bits.
//
// The verify mask comes from the draft tree (page "The Moment of Truth: Validating
// a Custom CUDA Attention Kernel for Speculative Decoding", section "Context"); a
// tree query sees itself and its ancestors (page "The Verify-Attn Kernel: A Single
// File Write ...", sections "The Design Journey: From Concept to CUDA" and
// "Assumptions and the Path Forward").
//
// One CTA per sequence; thread i owns row i of the output and walks its own
// ancestor chain, so no two threads write the same word and no atomics touch the
// bits. Parent pointers must strictly decrease (-1 <= parent[i] < i); a walk
// stops at the first entry that breaks this, which bounds every walk by T steps
// and records the entry in the error word instead of trapping.
#include "kdt_internal.cuh"
#include "tc_ptx.cuh"

namespace kdt {
namespace {

__global__ void build_visibility_kernel(const int32_t *__restrict__ parent, int T, int W,
                                        uint32_t *__restrict__ vis, int32_t *err) {
    tc::griddep_launch_dependents();               // the attention kernel may start its prefix blocks
    const int b = blockIdx.x;
    const int32_t *par = parent + (int64_t)b * T;
    for (int i = threadIdx.x; i < T; i += blockDim.x) {
        uint32_t *row = vis + ((int64_t)b * T + i) * W;
        uint32_t acc[4] = {0u, 0u, 0u, 0u};           // launched only for T <= 128 (W <= 4)
        int j = i;
        while (true) {
            acc[j >> 5] |= 1u << (j & 31);
            int pj = par[j];
            if (pj < -1 || pj >= j) {                  // malformed: stop the walk here
                record_error(err, (int32_t)((int64_t)b * T + j + 1));
                break;
            }
            if (pj < 0) break;
            j = pj;
        }
        for (int w = 0; w < W; ++w) row[w] = acc[w];
    }
}

// Wide trees (T > 128): each thread zeroes its row, then sets bits word by word.
__global__ void build_visibility_wide_kernel(const int32_t *__restrict__ parent, int T, int W,
                                             uint32_t *__restrict__ vis, int32_t *err) {
    tc::griddep_launch_dependents();
    const int b = blockIdx.x;
    const int32_t *par = parent + (int64_t)b * T;
    for (int i = threadIdx.x; i < T; i += blockDim.x) {
        uint32_t *row = vis + ((int64_t)b * T + i) * W;
        for (int w = 0; w < W; ++w) row[w] = 0u;
        int j = i;
        while (true) {
            row[j >> 5] |= 1u << (j & 31);             // only this thread writes this row
            int pj = par[j];
            if (pj < -1 || pj >= j) {
                record_error(err, (int32_t)((int64_t)b * T + j + 1));
                break;
            }
            if (pj < 0) break;
            j = pj;
        }
    }
}

}  // namespace

cudaError_t launch_build_visibility(const int32_t *parent, int B, int T, uint32_t *vis, int32_t *err,
                                    cudaStream_t s) {
    if (err) {
        cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int32_t), s);
        if (e != cudaSuccess) return e;
    }
    if (B == 0) return cudaSuccess;
    const int W = (T + 31) / 32;
    const int threads = T < 256 ? ((T + 31) / 32) * 32 : 256;
    if (W <= 4) build_visibility_kernel<<<B, threads, 0, s>>>(parent, T, W, vis, err);
    else build_visibility_wide_kernel<<<B, threads, 0, s>>>(parent, T, W, vis, err);
    return cudaGetLastError();
}

}  // namespace kdt
