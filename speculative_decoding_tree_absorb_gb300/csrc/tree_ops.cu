// The steps next to tree-verify attention in a DDTree step: the NeoX rotary embedding
// of the tree's query and key rope parts before verify, and after it the greedy accept
// walk and the compaction of the cache rows of the accepted path.
//
// RoPE: page "The Query-Split Kernel: A Pivotal Edit ...", sections "The Reasoning Chain"
// (rope applied in place on the rope portion of the combined query buffer) and "Input
// Knowledge" (NeoX variant, angles in float64). Accept and compaction: page "The Moment
// of Truth: Validating a Custom CUDA Attention Kernel ...", section "Context" (a greedy
// walk deciding which draft tokens are accepted), and page "The Architecture of an
// Inference Engine ...", sections "The Context" and "Input Knowledge Required" (the
// cache is compacted after acceptance to drop the unaccepted branches).
#include <climits>

#include "kdt_internal.cuh"

namespace kdt {
namespace {

constexpr int kMaxRopeHalf = 128;   // rope widths up to 256

__device__ __forceinline__ double widen(float v) { return (double)v; }
__device__ __forceinline__ double widen(__nv_bfloat16 v) { return (double)__bfloat162float(v); }
template <typename E> __device__ __forceinline__ E narrow(double v);
template <> __device__ __forceinline__ float narrow<float>(double v) { return __double2float_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 narrow<__nv_bfloat16>(double v) { return __double2bfloat16(v); }

// One CTA per tree node (b, i). The node's angles a_j = pos * base^(-2j/d) and their
// cosines and sines are taken once in float64; then every head's query vector and the
// node's key row (cache row prefix_len[b] + i) are rotated in place: for j < d/2,
//   (x_j, x_{j+d/2}) <- (x_j c_j - x_{j+d/2} s_j,  x_{j+d/2} c_j + x_j s_j),
// each product and sum rounded in float64, the result rounded once to the element type.
// A thread owns a whole pair, so the in-place update needs no synchronisation.
template <typename E>
__global__ void rope_neox_kernel(E *q, int64_t q_stride, int H, E *k_pe, int64_t L, const int32_t *prefix_len,
                                 const int32_t *pos, int T, int d, double base) {
    __shared__ double cs[kMaxRopeHalf], sn[kMaxRopeHalf];
    const int node = blockIdx.x;                       // b * T + i
    const int b = node / T, i = node - b * T;
    const int half = d / 2;
    const double p = (double)pos[node];
    for (int j = threadIdx.x; j < half; j += blockDim.x) {
        const double a = p * pow(base, (-2.0 * (double)j) / (double)d);
        cs[j] = cos(a);
        sn[j] = sin(a);
    }
    __syncthreads();
    auto rotate = [&](E *x, int j) {
        const double x1 = widen(x[j]), x2 = widen(x[j + half]);
        const double c = cs[j], s = sn[j];
        x[j] = narrow<E>(__dsub_rn(__dmul_rn(x1, c), __dmul_rn(x2, s)));
        x[j + half] = narrow<E>(__dadd_rn(__dmul_rn(x2, c), __dmul_rn(x1, s)));
    };
    if (q)
        for (int idx = threadIdx.x; idx < H * half; idx += blockDim.x) {
            const int h = idx / half, j = idx - h * half;
            rotate(q + ((int64_t)node * H + h) * q_stride, j);
        }
    if (k_pe) {
        const int64_t row = (int64_t)prefix_len[b] + i;
        if (row >= 0 && row < L)                       // the caller's bound; never write outside
            for (int j = threadIdx.x; j < half; j += blockDim.x) rotate(k_pe + ((int64_t)b * L + row) * d, j);
    }
}

// One CTA per sequence. Each node checks whether it drafted its parent's target token;
// the lowest such child of every node is kept (atomicMin in shared memory); one thread
// then walks from the root. Matches only point from a node to a later one, so the walk
// ends within T steps even on a malformed tree (whose bad entries are skipped and
// reported like the visibility builder does).
__global__ void tree_accept_kernel(const int32_t *__restrict__ parent, const int32_t *__restrict__ tok,
                                   const int32_t *__restrict__ target, int T, int32_t *acc_nodes, int32_t *n_acc,
                                   int32_t *bonus, int32_t *err) {
    extern __shared__ int32_t next_match[];            // [T]
    const int b = blockIdx.x;
    const int64_t base = (int64_t)b * T;
    for (int i = threadIdx.x; i < T; i += blockDim.x) {
        next_match[i] = INT_MAX;
        acc_nodes[base + i] = -1;
    }
    __syncthreads();
    for (int c = threadIdx.x; c < T; c += blockDim.x) {
        const int p = parent[base + c];
        if (p < -1 || p >= c) {
            record_error(err, (int32_t)(base + c + 1));
            continue;
        }
        if (p >= 0 && tok[base + c] == target[base + p]) atomicMin(&next_match[p], c);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int cur = 0, n = 0;
        acc_nodes[base + n++] = 0;
        while (next_match[cur] != INT_MAX) {
            cur = next_match[cur];
            acc_nodes[base + n++] = cur;
        }
        n_acc[b] = n;
        bonus[b] = target[base + cur];
    }
}

// One CTA per sequence; the k-th accepted node's rows move to cache row prefix + k, in
// path order. Path nodes increase along the path (a parent precedes its children), so the
// source of step k (row prefix + path[k] >= prefix + k) is never a row an earlier step
// wrote, and the copy is safe in place with a barrier between steps. Entries outside the
// tree or the cache are not copied.
__global__ void kv_compact_kernel(uint4 *c_kv, uint4 *k_pe, int c_vec, int r_vec, int64_t L, int32_t *prefix_len,
                                  const int32_t *acc_nodes, const int32_t *n_acc, int T, int update_prefix) {
    const int b = blockIdx.x;
    const int64_t p0 = prefix_len[b];
    const int n = min(max(n_acc[b], 0), T);
    for (int k = 1; k < n; ++k) {
        const int src = acc_nodes[(int64_t)b * T + k];
        if (src == k || src < k || src >= T || p0 + src >= L || p0 < 0) continue;   // same for every thread
        const int64_t dst_row = (int64_t)b * L + p0 + k, src_row = (int64_t)b * L + p0 + src;
        for (int v = threadIdx.x; v < c_vec; v += blockDim.x) c_kv[dst_row * c_vec + v] = c_kv[src_row * c_vec + v];
        for (int v = threadIdx.x; v < r_vec; v += blockDim.x) k_pe[dst_row * r_vec + v] = k_pe[src_row * r_vec + v];
        __syncthreads();
    }
    __syncthreads();
    if (update_prefix && threadIdx.x == 0) prefix_len[b] = (int32_t)(p0 + n);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kdt

using namespace kdt;

extern "C" {

kdt_status kdt_rope_neox(const kdt_rope_args *a, cudaStream_t stream) {
    if (!a) return KDT_ERR_NULL_ARG;
    if (a->B < 0 || a->T < 1 || a->T > kMaxT || a->H < 1 || a->H > 1024) return KDT_ERR_BAD_SHAPE;
    if (a->D_r < 2 || a->D_r % 2 || a->D_r > 2 * kMaxRopeHalf) return KDT_ERR_BAD_SHAPE;
    if (a->dtype != KDT_F32 && a->dtype != KDT_BF16) return KDT_ERR_UNSUPPORTED;
    if (!(a->base > 0.0) || a->base != a->base || a->base > 1e300) return KDT_ERR_BAD_SHAPE;
    if (a->B == 0) return KDT_OK;
    if (!a->pos || (!a->q && !a->k_pe)) return KDT_ERR_NULL_ARG;
    if (a->q && a->q_row_stride < a->D_r) return KDT_ERR_BAD_SHAPE;
    if (a->k_pe && (!a->prefix_len || a->kv_row_stride < a->T)) return a->prefix_len ? KDT_ERR_BAD_SHAPE : KDT_ERR_NULL_ARG;
    const int threads = 256;
    if (a->dtype == KDT_F32)
        rope_neox_kernel<float><<<a->B * a->T, threads, 0, stream>>>(
            static_cast<float *>(a->q), a->q_row_stride, a->H, static_cast<float *>(a->k_pe), a->kv_row_stride,
            a->prefix_len, a->pos, a->T, a->D_r, a->base);
    else
        rope_neox_kernel<__nv_bfloat16><<<a->B * a->T, threads, 0, stream>>>(
            static_cast<__nv_bfloat16 *>(a->q), a->q_row_stride, a->H, static_cast<__nv_bfloat16 *>(a->k_pe),
            a->kv_row_stride, a->prefix_len, a->pos, a->T, a->D_r, a->base);
    return cudaGetLastError() == cudaSuccess ? KDT_OK : KDT_ERR_CUDA;
}

kdt_status kdt_tree_accept(const int32_t *parent, const int32_t *tok, const int32_t *target, int B, int T,
                           int32_t *acc_nodes, int32_t *n_acc, int32_t *bonus, int32_t *err, cudaStream_t stream) {
    if (B < 0 || T < 1 || T > kMaxT) return KDT_ERR_BAD_SHAPE;
    if (B == 0) return err && cudaMemsetAsync(err, 0, sizeof(int32_t), stream) != cudaSuccess ? KDT_ERR_CUDA : KDT_OK;
    if (!parent || !tok || !target || !acc_nodes || !n_acc || !bonus) return KDT_ERR_NULL_ARG;
    if (err && cudaMemsetAsync(err, 0, sizeof(int32_t), stream) != cudaSuccess) return KDT_ERR_CUDA;
    const int threads = T < 256 ? ((T + 31) / 32) * 32 : 256;
    tree_accept_kernel<<<B, threads, (size_t)T * sizeof(int32_t), stream>>>(parent, tok, target, T, acc_nodes, n_acc,
                                                                              bonus, err);
    return cudaGetLastError() == cudaSuccess ? KDT_OK : KDT_ERR_CUDA;
}

kdt_status kdt_kv_compact(void *c_kv, void *k_pe, kdt_dtype dtype, int D_c, int D_r, int B, int T,
                          int64_t kv_row_stride, int32_t *prefix_len, const int32_t *acc_nodes, const int32_t *n_acc,
                          int update_prefix, cudaStream_t stream) {
    if (B < 0 || T < 1 || T > kMaxT || D_c < 1 || D_r < 1 || kv_row_stride < T) return KDT_ERR_BAD_SHAPE;
    if (dtype != KDT_F32 && dtype != KDT_BF16) return KDT_ERR_UNSUPPORTED;
    const int esz = dtype == KDT_F32 ? 4 : 2;
    if (((int64_t)D_c * esz) % 16 || ((int64_t)D_r * esz) % 16) return KDT_ERR_BAD_SHAPE;
    if (B == 0) return KDT_OK;
    if (!c_kv || !k_pe || !prefix_len || !acc_nodes || !n_acc) return KDT_ERR_NULL_ARG;
    if (!aligned16(c_kv) || !aligned16(k_pe)) return KDT_ERR_BAD_SHAPE;
    kv_compact_kernel<<<B, 128, 0, stream>>>(static_cast<uint4 *>(c_kv), static_cast<uint4 *>(k_pe),
                                             D_c * esz / 16, D_r * esz / 16, kv_row_stride, prefix_len, acc_nodes,
                                             n_acc, T, update_prefix ? 1 : 0);
    return cudaGetLastError() == cudaSuccess ? KDT_OK : KDT_ERR_CUDA;
}

}  // extern "C"
