// The steps next to tree-verify attention in a DDTree step: the best-first draft-tree
// builder and the NeoX rotary embedding of the tree's query and key rope parts before
// verify, and after it the greedy accept walk and the compaction of the cache rows of
// the accepted path.
//
// RoPE: page "The Query-Split Kernel: A Pivotal Edit ...", sections "The Reasoning Chain"
// (rope applied in place on the rope portion of the combined query buffer) and "Input
// Knowledge" (NeoX variant, angles in float64; the engine computes in float32). Accept and compaction: page "The Moment
// of Truth: Validating a Custom CUDA Attention Kernel ...", section "Context" (a greedy
// walk deciding which draft tokens are accepted), and page "The Architecture of an
// Inference Engine ...", sections "The Context" and "Input Knowledge Required" (the
// cache is compacted after acceptance to drop the unaccepted branches; the tree is built
// best-first on the device instead of with a per-request CPU heap).
#include <climits>
#include <cmath>

#include "kdt_internal.cuh"

namespace kdt {
namespace {

constexpr int kMaxRopeHalf = 128;   // rope widths up to 256

__device__ __forceinline__ float widen(float v) { return v; }
__device__ __forceinline__ float widen(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename E> __device__ __forceinline__ E narrow(float v);
template <> __device__ __forceinline__ float narrow<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 narrow<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Angle frequencies w_j = base^(-2j/d), float64, computed on the host.
struct RopeFreqs {
    double w[kMaxRopeHalf];
};

// V consecutive elements of type E, loaded or stored as one aligned vector.
template <typename E, int V> struct alignas(sizeof(E) * V) Vec {
    E v[V];
};

// One CTA per tree node (b, i). Its angles a_j = pos * w_j are taken in float64 and their
// cosines and sines rounded once to float32; then every head's query vector and the
// node's key row (cache row prefix_len[b] + i) are rotated in place in float32: for j < d/2,
//   (x_j, x_{j+d/2}) <- (x_j c_j - x_{j+d/2} s_j,  x_{j+d/2} c_j + x_j s_j),
// each product and sum rounded to nearest on its own (no fused multiply-add), the result
// rounded once more to the element type. A thread owns V whole pairs (j .. j+V-1, moved
// as vectors when the rows allow), so the in-place update needs no synchronisation.
template <typename E, int V>
__global__ void rope_neox_kernel(E *q, int64_t q_stride, int H, E *k_pe, int64_t L, const int32_t *prefix_len,
                                 const int32_t *pos, int T, int d, const __grid_constant__ RopeFreqs freqs) {
    __shared__ float cs[kMaxRopeHalf], sn[kMaxRopeHalf];
    const int node = blockIdx.x;                       // b * T + i
    const int b = node / T, i = node - b * T;
    const int half = d / 2, groups = half / V;
    const double p = (double)pos[node];
    for (int j = threadIdx.x; j < half; j += blockDim.x) {
        const double a = p * freqs.w[j];
        cs[j] = (float)cos(a);
        sn[j] = (float)sin(a);
    }
    __syncthreads();
    auto rotate = [&](E *x, int j0) {
        Vec<E, V> a1 = *reinterpret_cast<const Vec<E, V> *>(x + j0);
        Vec<E, V> a2 = *reinterpret_cast<const Vec<E, V> *>(x + j0 + half);
#pragma unroll
        for (int t = 0; t < V; ++t) {
            const float x1 = widen(a1.v[t]), x2 = widen(a2.v[t]);
            const float c = cs[j0 + t], s = sn[j0 + t];
            a1.v[t] = narrow<E>(__fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, s)));
            a2.v[t] = narrow<E>(__fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s)));
        }
        *reinterpret_cast<Vec<E, V> *>(x + j0) = a1;
        *reinterpret_cast<Vec<E, V> *>(x + j0 + half) = a2;
    };
    if (q)
        for (int idx = threadIdx.x; idx < H * groups; idx += blockDim.x) {
            const int h = idx / groups, j0 = (idx - h * groups) * V;
            rotate(q + ((int64_t)node * H + h) * q_stride, j0);
        }
    if (k_pe) {
        const int64_t row = (int64_t)prefix_len[b] + i;
        if (row >= 0 && row < L)                       // the caller's bound; never write outside
            for (int g = threadIdx.x; g < groups; g += blockDim.x) rotate(k_pe + ((int64_t)b * L + row) * d, g * V);
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

// One CTA per sequence; the k-th accepted node's rows move to cache row prefix + k. Path
// nodes increase along the path (a parent precedes its children), so the source of step k
// (row prefix + path[k] >= prefix + k) is never a row an earlier step wrote. The path is
// moved in chunks of rows staged through shared memory: every source row of a chunk is
// read before any of its destinations is written, and later chunks read no row an
// earlier chunk wrote. Entries outside the tree or the cache are not copied.
constexpr int kCompactSmem = 40 * 1024;

__global__ void __launch_bounds__(256) kv_compact_kernel(uint4 *c_kv, uint4 *k_pe, int c_vec, int r_vec, int64_t L,
                                                         int32_t *prefix_len, const int32_t *acc_nodes,
                                                         const int32_t *n_acc, int T, int update_prefix) {
    __shared__ uint4 stage[kCompactSmem / 16];
    __shared__ int src_row[kCompactSmem / 32];
    const int b = blockIdx.x;
    const int64_t p0 = prefix_len[b];
    const int n = min(max(n_acc[b], 0), T);
    const int row_vec = c_vec + r_vec;
    const int chunk = kCompactSmem / 16 / row_vec;      // rows staged at a time
    for (int k0 = 1; k0 < n; k0 += chunk) {
        const int kn = min(chunk, n - k0);
        for (int t = threadIdx.x; t < kn; t += blockDim.x) {
            const int k = k0 + t, src = acc_nodes[(int64_t)b * T + k];
            src_row[t] = (src == k || src < k || src >= T || p0 + src >= L || p0 < 0) ? -1 : src;
        }
        __syncthreads();
        for (int v = threadIdx.x; v < kn * row_vec; v += blockDim.x) {
            const int t = v / row_vec, e = v - t * row_vec, src = src_row[t];
            if (src < 0) continue;
            const int64_t r = (int64_t)b * L + p0 + src;
            stage[v] = e < c_vec ? c_kv[r * c_vec + e] : k_pe[r * r_vec + (e - c_vec)];
        }
        __syncthreads();
        for (int v = threadIdx.x; v < kn * row_vec; v += blockDim.x) {
            const int t = v / row_vec, e = v - t * row_vec;
            if (src_row[t] < 0) continue;
            const int64_t r = (int64_t)b * L + p0 + k0 + t;
            if (e < c_vec) c_kv[r * c_vec + e] = stage[v];
            else k_pe[r * r_vec + (e - c_vec)] = stage[v];
        }
        __syncthreads();
    }
    if (update_prefix && threadIdx.x == 0) prefix_len[b] = (int32_t)(p0 + n);
}

// ------------------------------------------------------------ best-first builder --
// A frontier entry -- the candidate of rank `rank` at depth `depth` below node `par`,
// with its path score -- packed into one 64-bit key whose unsigned order is the selection
// order: higher score (high word: the float's bits mapped to an order-preserving integer,
// complemented), then lower depth, lower parent, lower rank (low word). Entries are unique
// in (depth, par, rank), so the warp minimum is one entry whatever the reduction order.
__device__ __forceinline__ uint64_t pack_key(float score, int depth, int par, int rank) {
    uint32_t u = __float_as_uint(score == 0.f ? 0.f : score);    // one zero
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);            // ascending with the float
    return ((uint64_t)(~u) << 32) | ((uint32_t)depth << 17) | ((uint32_t)par << 5) | (uint32_t)rank;
}

__device__ __forceinline__ float key_score(uint64_t key) {
    const uint32_t u = ~(uint32_t)(key >> 32);
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

constexpr int kMaxBuildDepth = 64, kMaxBuildK = 32, kMaxBuildN = kMaxT - 1;

size_t build_smem_bytes(int D, int K, int N) {
    // n_score and the frontier also stage the unranked candidates before the joins start
    const size_t lists = (size_t)D * K * 8;
    const size_t scores = ((size_t)(N + 1 > D * K ? N + 1 : D * K) * 4 + 15) / 16 * 16;
    const size_t frontier = (size_t)(N + 2 > (D * K + 1) / 2 ? N + 2 : (D * K + 1) / 2) * sizeof(uint64_t);
    return lists + scores + frontier;
}

// The candidates of every depth, staged unranked in u_lp / u_tok, ranked into s_lp / s_tok
// (log-probability descending, ties by position; NaN counts as -inf). Every lane ranks
// whole entries against the K entries of their depth, all of them at once.
__device__ __forceinline__ void rank_candidates(const float *u_lp, const int32_t *u_tok, float *s_lp,
                                                int32_t *s_tok, int D, int K, int lane) {
    for (int i = lane; i < D * K; i += 32) {
        const int d = i / K, r = i - d * K;
        float v = u_lp[i];
        if (v != v) v = -INFINITY;
        int rank = 0;
        for (int j = 0; j < K; ++j) {
            float vj = u_lp[d * K + j];
            if (vj != vj) vj = -INFINITY;
            rank += (vj > v || (vj == v && j < r)) ? 1 : 0;
        }
        s_lp[d * K + rank] = v;
        s_tok[d * K + rank] = u_tok[i];
    }
}

// One warp per sequence. The candidates of every depth are ranked first. The frontier holds, for every node
// in the tree, only its best child not yet taken: children below a node are ranked like
// the candidates, so when a node's child of rank r joins, its sibling of rank r + 1 and
// its own first child are pushed. That yields the same joins as pushing all children.
// Each join is two warp-wide minimum reductions over the packed keys.
__global__ void __launch_bounds__(32) tree_build_kernel(const int32_t *__restrict__ cand_tok,
                                                        const float *__restrict__ cand_lp, int D, int K, int N,
                                                        const int32_t *root_tok, int32_t *parent, int32_t *tok,
                                                        int32_t *depth, float *score) {
    extern __shared__ __align__(16) unsigned char bsm[];
    float *s_lp = reinterpret_cast<float *>(bsm);                      // [D][K] ranked
    int32_t *s_tok = reinterpret_cast<int32_t *>(s_lp + D * K);        // [D][K]
    float *n_score = reinterpret_cast<float *>(s_tok + D * K);         // [N + 1]
    const int n_score_len = N + 1 > D * K ? N + 1 : D * K;
    uint64_t *fr = reinterpret_cast<uint64_t *>(bsm + (size_t)D * K * 8 + ((size_t)n_score_len * 4 + 15) / 16 * 16);
    const int b = blockIdx.x, lane = threadIdx.x;
    const int T = N + 1;
    const int64_t ob = (int64_t)b * T;
    // every candidate of the sequence in one round of loads (the ranked lists are written
    // over these staged copies only after all of them have been read into registers)
    float *u_lp = n_score;                                             // [D][K] unranked, scratch
    int32_t *u_tok = reinterpret_cast<int32_t *>(fr);                  // [D][K] unranked, scratch
    for (int i = lane; i < D * K; i += 32) {
        u_lp[i] = cand_lp[(int64_t)b * D * K + i];
        u_tok[i] = cand_tok[(int64_t)b * D * K + i];
    }
    __syncwarp();
    rank_candidates(u_lp, u_tok, s_lp, s_tok, D, K, lane);
    __syncwarp();
    if (lane == 0) {
        n_score[0] = 0.f;
        parent[ob] = -1;
        tok[ob] = root_tok ? root_tok[b] : -1;
        if (depth) depth[ob] = 0;
        if (score) score[ob] = 0.f;
        fr[0] = pack_key(__fadd_rn(0.f, s_lp[0]), 1, 0, 0);
    }
    int F = 1;                                          // frontier size, the same in every lane
    __syncwarp();
    for (int n = 1; n < T && F > 0; ++n) {
        uint64_t mine = ~0ull;
        int slot = -1;
        for (int i = lane; i < F; i += 32) {
            const uint64_t k = fr[i];
            if (k < mine) {
                mine = k;
                slot = i;
            }
        }
        const uint32_t hi = __reduce_min_sync(0xffffffffu, (uint32_t)(mine >> 32));
        const uint32_t lo = __reduce_min_sync(0xffffffffu, (uint32_t)(mine >> 32) == hi ? (uint32_t)mine : ~0u);
        const uint64_t best = ((uint64_t)hi << 32) | lo;
        const int owner = __ffs(__ballot_sync(0xffffffffu, mine == best)) - 1;
        const int best_slot = __shfl_sync(0xffffffffu, slot, owner);
        const float bscore = key_score(best);
        const int bdepth = (int)(lo >> 17), bpar = (int)((lo >> 5) & 0xfffu), brank = (int)(lo & 31u);
        const bool sib = brank + 1 < K, child = bdepth < D;
        if (lane == 0) {
            fr[best_slot] = fr[F - 1];                  // take the entry out
            n_score[n] = bscore;
            parent[ob + n] = bpar;
            tok[ob + n] = s_tok[(bdepth - 1) * K + brank];
            if (depth) depth[ob + n] = bdepth;
            if (score) score[ob + n] = bscore;
            int f = F - 1;
            if (sib)
                fr[f++] = pack_key(__fadd_rn(n_score[bpar], s_lp[(bdepth - 1) * K + brank + 1]), bdepth, bpar, brank + 1);
            if (child) fr[f++] = pack_key(__fadd_rn(bscore, s_lp[bdepth * K]), bdepth + 1, n, 0);
        }
        F = F - 1 + (sib ? 1 : 0) + (child ? 1 : 0);
        __syncwarp();
    }
}

// The same joins for trees of at most 32 * R nodes with nothing but the ranked lists in
// shared memory: frontier slot s, and node n's score and fields, live in register s / 32
// (n / 32) of lane s % 32 (n % 32). A join is the two reductions, one shuffle for the
// parent's score and two reads of the ranked lists, computed alike in every lane; the
// taken slot is refilled in place with the next sibling (or, with no sibling left, the
// first child) and the child takes a fresh slot when both are pushed. The tree is
// written out once at the end, coalesced.
template <int R>
__global__ void __launch_bounds__(32) tree_build_reg_kernel(const int32_t *__restrict__ cand_tok,
                                                            const float *__restrict__ cand_lp, int D, int K, int N,
                                                            const int32_t *root_tok, int32_t *parent, int32_t *tok,
                                                            int32_t *depth, float *score) {
    extern __shared__ __align__(16) unsigned char bsm[];
    float *s_lp = reinterpret_cast<float *>(bsm);                      // [D][K] ranked
    int32_t *s_tok = reinterpret_cast<int32_t *>(s_lp + D * K);        // [D][K] ranked
    float *u_lp = reinterpret_cast<float *>(s_tok + D * K);            // [D][K] unranked
    int32_t *u_tok = reinterpret_cast<int32_t *>(u_lp + D * K);        // [D][K] unranked
    const int b = blockIdx.x, lane = threadIdx.x;
    const int T = N + 1;
    for (int i = lane; i < D * K; i += 32) {
        u_lp[i] = cand_lp[(int64_t)b * D * K + i];
        u_tok[i] = cand_tok[(int64_t)b * D * K + i];
    }
    __syncwarp();
    rank_candidates(u_lp, u_tok, s_lp, s_tok, D, K, lane);
    __syncwarp();
    uint64_t key[R];
    float nsc[R];
    int32_t npar[R], nsel[R];                           // node: parent, (depth << 5) | rank
#pragma unroll R
    for (int j = 0; j < R; ++j) {
        key[j] = ~0ull;                                 // empty slot: above every packed entry
        nsc[j] = 0.f;
        npar[j] = -1;
        nsel[j] = 0;
    }
    if (lane == 0) key[0] = pack_key(__fadd_rn(0.f, s_lp[0]), 1, 0, 0);
    int F = 1, U = 1;                                   // live entries, slots used
    int n = 1;
    for (; n < T && F > 0; ++n) {
        uint64_t mine = key[0];
#pragma unroll R
        for (int j = 1; j < R; ++j) mine = key[j] < mine ? key[j] : mine;
        const uint32_t hi = __reduce_min_sync(0xffffffffu, (uint32_t)(mine >> 32));
        const uint32_t lo = __reduce_min_sync(0xffffffffu, (uint32_t)(mine >> 32) == hi ? (uint32_t)mine : ~0u);
        const uint64_t best = ((uint64_t)hi << 32) | lo;
        const float bscore = key_score(best);
        const int bdepth = (int)(lo >> 17), bpar = (int)((lo >> 5) & 0xfffu), brank = (int)(lo & 31u);
        const bool sib = brank + 1 < K, child = bdepth < D;
        float ps = 0.f;                                 // the parent's path score
#pragma unroll R
        for (int j = 0; j < R; ++j) {
            const float v = __shfl_sync(0xffffffffu, nsc[j], bpar & 31);
            if (j == (bpar >> 5)) ps = v;
        }
        const uint64_t ksib =
            sib ? pack_key(__fadd_rn(ps, s_lp[(bdepth - 1) * K + brank + 1]), bdepth, bpar, brank + 1) : ~0ull;
        const uint64_t kchild = child ? pack_key(__fadd_rn(bscore, s_lp[bdepth * K]), bdepth + 1, n, 0) : ~0ull;
        const uint64_t refill = sib ? ksib : kchild;
#pragma unroll R
        for (int j = 0; j < R; ++j) {
            if (key[j] == best) key[j] = refill;        // entries are unique: one slot in one lane
            if (sib && child && j == (U >> 5) && lane == (U & 31)) key[j] = kchild;
            if (j == (n >> 5) && lane == (n & 31)) {
                nsc[j] = bscore;
                npar[j] = bpar;
                nsel[j] = (bdepth << 5) | brank;
            }
        }
        U += (sib && child) ? 1 : 0;
        F += (sib ? 1 : 0) + (child ? 1 : 0) - 1;
    }
    const int64_t ob = (int64_t)b * T;
#pragma unroll R
    for (int j = 0; j < R; ++j) {
        const int m = 32 * j + lane;
        if (m >= n) continue;                           // n: nodes joined (all T of them when the shape allows)
        const int dm = nsel[j] >> 5;
        parent[ob + m] = npar[j];
        tok[ob + m] = m == 0 ? (root_tok ? root_tok[b] : -1) : s_tok[(dm - 1) * K + (nsel[j] & 31)];
        if (depth) depth[ob + m] = dm;
        if (score) score[ob + m] = nsc[j];
    }
}

template <int R>
kdt_status launch_build_reg(const int32_t *cand_tok, const float *cand_lp, int B, int D, int K, int N,
                            const int32_t *root_tok, int32_t *parent, int32_t *tok, int32_t *depth, float *score,
                            cudaStream_t stream) {
    const size_t smem = (size_t)D * K * 16;             // ranked and unranked lists: at most 32 KB
    tree_build_reg_kernel<R><<<B, 32, smem, stream>>>(cand_tok, cand_lp, D, K, N, root_tok, parent, tok, depth, score);
    return cudaGetLastError() == cudaSuccess ? KDT_OK : KDT_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kdt

using namespace kdt;

extern "C" {

kdt_status kdt_tree_build(const int32_t *cand_tok, const float *cand_lp, int B, int D, int K, int N,
                          const int32_t *root_tok, int32_t *parent, int32_t *tok, int32_t *depth, float *score,
                          cudaStream_t stream) {
    if (B < 0 || D < 1 || D > kMaxBuildDepth || K < 1 || K > kMaxBuildK || N < 1 || N > kMaxBuildN)
        return KDT_ERR_BAD_SHAPE;
    int64_t avail = 0, level = 1;                      // nodes below the root: K + K^2 + ... + K^D
    for (int d = 0; d < D && avail < N; ++d) {
        level *= K;
        avail += level;
    }
    if (avail < N) return KDT_ERR_BAD_SHAPE;
    if (B == 0) return KDT_OK;
    if (!cand_tok || !cand_lp || !parent || !tok) return KDT_ERR_NULL_ARG;
    if (N + 1 <= 32) return launch_build_reg<1>(cand_tok, cand_lp, B, D, K, N, root_tok, parent, tok, depth, score, stream);
    if (N + 1 <= 64) return launch_build_reg<2>(cand_tok, cand_lp, B, D, K, N, root_tok, parent, tok, depth, score, stream);
    if (N + 1 <= 128)
        return launch_build_reg<4>(cand_tok, cand_lp, B, D, K, N, root_tok, parent, tok, depth, score, stream);
    const size_t smem = build_smem_bytes(D, K, N);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(tree_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return KDT_ERR_CUDA;
    tree_build_kernel<<<B, 32, smem, stream>>>(cand_tok, cand_lp, D, K, N, root_tok, parent, tok, depth, score);
    return cudaGetLastError() == cudaSuccess ? KDT_OK : KDT_ERR_CUDA;
}

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
    RopeFreqs f;
    for (int j = 0; j < a->D_r / 2; ++j) f.w[j] = pow(a->base, (-2.0 * (double)j) / (double)a->D_r);
    // 16-byte vectors when every half-row starts on a 16-byte boundary, else one pair a thread
    const int esz = a->dtype == KDT_F32 ? 4 : 2, V = 16 / esz;
    const bool vec = (a->D_r / 2) % V == 0 && (!a->q || (aligned16(a->q) && (a->q_row_stride * esz) % 16 == 0)) &&
                     (!a->k_pe || aligned16(a->k_pe));
    const int threads = 128;
    const dim3 grid(a->B * a->T);
    if (a->dtype == KDT_F32) {
        float *q = static_cast<float *>(a->q), *k = static_cast<float *>(a->k_pe);
        if (vec)
            rope_neox_kernel<float, 4><<<grid, threads, 0, stream>>>(q, a->q_row_stride, a->H, k, a->kv_row_stride,
                                                                     a->prefix_len, a->pos, a->T, a->D_r, f);
        else
            rope_neox_kernel<float, 1><<<grid, threads, 0, stream>>>(q, a->q_row_stride, a->H, k, a->kv_row_stride,
                                                                     a->prefix_len, a->pos, a->T, a->D_r, f);
    } else {
        __nv_bfloat16 *q = static_cast<__nv_bfloat16 *>(a->q), *k = static_cast<__nv_bfloat16 *>(a->k_pe);
        if (vec)
            rope_neox_kernel<__nv_bfloat16, 8><<<grid, threads, 0, stream>>>(
                q, a->q_row_stride, a->H, k, a->kv_row_stride, a->prefix_len, a->pos, a->T, a->D_r, f);
        else
            rope_neox_kernel<__nv_bfloat16, 1><<<grid, threads, 0, stream>>>(
                q, a->q_row_stride, a->H, k, a->kv_row_stride, a->prefix_len, a->pos, a->T, a->D_r, f);
    }
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
    if (((int64_t)D_c * esz + (int64_t)D_r * esz) > kCompactSmem) return KDT_ERR_BAD_SHAPE;
    kv_compact_kernel<<<B, 256, 0, stream>>>(static_cast<uint4 *>(c_kv), static_cast<uint4 *>(k_pe),
                                             D_c * esz / 16, D_r * esz / 16, kv_row_stride, prefix_len, acc_nodes,
                                             n_acc, T, update_prefix ? 1 : 0);
    return cudaGetLastError() == cudaSuccess ? KDT_OK : KDT_ERR_CUDA;
}

}  // extern "C"
