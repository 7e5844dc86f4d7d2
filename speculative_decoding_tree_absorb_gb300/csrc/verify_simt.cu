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
// Design (differs from the pages' one-block-per-(b,h,i) kernel): a CTA owns 64
// consecutive rows of one sequence -- all heads of a few tree queries -- so each
// cache row it stages in shared memory serves 64 query rows instead of one.
// Scores for a 64x64 (rows x keys) block are a register-tiled SIMT product (each
// of 256 threads owns a 4x4 sub-tile); P.V accumulates a 64x512 fp32 output tile
// (4 rows x 32 columns per thread). No atomics: every output element has one owner.
// Split-KV: blockIdx.y takes a contiguous range of key blocks; with more than one
// split the CTA writes a normalised partial (o_s, lse_s) that K2 merges.
#include "kdt_internal.cuh"

#include <math.h>

namespace kdt {
namespace {

constexpr int kRows = kSimtRows;       // 64 query rows per CTA
constexpr int kKeys = kSimtKeys;       // 64 keys per block
constexpr int kThreads = 256;
constexpr int kDChunk = 32;            // reduction-dim chunk staged per step
constexpr int kVKeys = 16;             // keys per staged slice of V
constexpr int kPad = 4;

struct __align__(16) SimtSmem {
    float qs[kDChunk][kRows + kPad];   // Q chunk, transposed: qs[d][row]
    float ks[kDChunk][kKeys + kPad];   // K chunk, transposed: ks[d][key]
    float ps[kRows][kKeys + kPad];     // softmax numerators of the block
    float vs[kVKeys][kDc];             // slice of V = c_kv rows
};

__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[2 * k] = __uint_as_float(w[k] << 16);
        v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads, 1) verify_simt_kernel(const VerifyParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SimtSmem &sm = *reinterpret_cast<SimtSmem *>(smem_raw);

    const int tid = threadIdx.x;
    const int tx = tid & 15;          // key group (S) / column group (O)
    const int ty = tid >> 4;          // row group: rows ty*4 .. ty*4+3
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

    // query index of each of this thread's 4 rows (for the tree mask)
    int qidx[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) qidx[i] = min(r0 + ty * 4 + i, rows_seq - 1) / p.H;

    float o[4][32];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 32; ++c) o[i][c] = 0.f;
    float m2[4], lpart[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) { m2[i] = -INFINITY; lpart[i] = 0.f; }

    const int64_t q_row0 = (int64_t)b * rows_seq + r0;
    const int64_t kv_row0 = (int64_t)b * p.L;

    for (int kb = kb0; kb < kb1; ++kb) {
        const int k0 = kb * kKeys;
        // ---------------- S = Q K^T for 64 rows x 64 keys --------------------
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

        for (int dc = 0; dc < kDqk / kDChunk; ++dc) {
            {
                const int lr = tid >> 2, d8 = (tid & 3) * 8;
                const int dglob = dc * kDChunk + d8;
                float v[8];
                // Q rows beyond the sequence's T*H rows read as zero
                if (r0 + lr < rows_seq) {
                    if (dglob < kDc) load8(q_nope + (q_row0 + lr) * p.q_nope_stride + dglob, v);
                    else load8(q_pe + (q_row0 + lr) * p.q_pe_stride + (dglob - kDc), v);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = 0.f;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) sm.qs[d8 + e][lr] = v[e];
                // keys at or beyond key_end (padding, other splits) read as zero
                const int key = k0 + lr;
                if (key < key_end) {
                    if (dglob < kDc) load8(c_kv + (kv_row0 + key) * kDc + dglob, v);
                    else load8(k_pe + (kv_row0 + key) * kDr + (dglob - kDc), v);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = 0.f;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) sm.ks[d8 + e][lr] = v[e];
            }
            __syncthreads();
#pragma unroll
            for (int d = 0; d < kDChunk; ++d) {
                const float4 a = *reinterpret_cast<const float4 *>(&sm.qs[d][ty * 4]);
                const float4 k = *reinterpret_cast<const float4 *>(&sm.ks[d][tx * 4]);
                const float av[4] = {a.x, a.y, a.z, a.w};
                const float kvv[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], kvv[j], acc[i][j]);
            }
            __syncthreads();
        }

        // ---------------- mask, online softmax --------------------------------
        float alpha[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float s[4];
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int key = k0 + tx * 4 + j;
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
            alpha[i] = (mnew == -INFINITY) ? 1.f : exp2f(m2[i] - mnew);
            float rs = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float pj = (mnew == -INFINITY) ? 0.f : exp2f(s[j] - mnew);
                sm.ps[ty * 4 + i][tx * 4 + j] = pj;
                rs += pj;
            }
            lpart[i] = lpart[i] * alpha[i] + rs;
            m2[i] = mnew;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int c = 0; c < 32; ++c) o[i][c] *= alpha[i];

        // ---------------- O += P V ------------------------------------------------
        for (int vc = 0; vc < kKeys / kVKeys; ++vc) {
            __syncthreads();   // ps written / previous slice consumed
            {
                const int lk = tid >> 4, d0 = (tid & 15) * 32;
                const int key = k0 + vc * kVKeys + lk;
                float v[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (key < key_end) load8(c_kv + (kv_row0 + key) * kDc + d0 + q * 8, v);
                    else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = 0.f;
                    }
                    *reinterpret_cast<float4 *>(&sm.vs[lk][d0 + q * 8]) = make_float4(v[0], v[1], v[2], v[3]);
                    *reinterpret_cast<float4 *>(&sm.vs[lk][d0 + q * 8 + 4]) = make_float4(v[4], v[5], v[6], v[7]);
                }
            }
            __syncthreads();
#pragma unroll 4
            for (int kk = 0; kk < kVKeys; ++kk) {
                float pr[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) pr[i] = sm.ps[ty * 4 + i][vc * kVKeys + kk];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 v = *reinterpret_cast<const float4 *>(&sm.vs[kk][c * 64 + tx * 4]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        o[i][c * 4 + 0] = fmaf(pr[i], v.x, o[i][c * 4 + 0]);
                        o[i][c * 4 + 1] = fmaf(pr[i], v.y, o[i][c * 4 + 1]);
                        o[i][c * 4 + 2] = fmaf(pr[i], v.z, o[i][c * 4 + 2]);
                        o[i][c * 4 + 3] = fmaf(pr[i], v.w, o[i][c * 4 + 3]);
                    }
                }
            }
        }
        __syncthreads();
    }

    // ---------------- epilogue: o = O / l, lse = ln2 * (m2 + log2 l) -------------
    const bool partial = p.num_splits > 1;
    float *obase = partial ? p.part_o + (int64_t)split * p.rows_total * kDc : p.out;
    float *lbase = partial ? p.part_lse + (int64_t)split * p.rows_total : p.lse;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float l = lpart[i];
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        const int r = r0 + ty * 4 + i;
        if (r >= rows_seq) continue;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int64_t grow = (int64_t)b * rows_seq + r;
        float *orow = obase + grow * kDc;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 v = make_float4(o[i][c * 4] * inv, o[i][c * 4 + 1] * inv, o[i][c * 4 + 2] * inv,
                                         o[i][c * 4 + 3] * inv);
            *reinterpret_cast<float4 *>(orow + c * 64 + tx * 4) = v;
        }
        if (tx == 0 && lbase) {
            lbase[grow] = (l > 0.f) ? 0.6931471805599453f * (m2[i] + log2f(l)) : -INFINITY;
        }
    }
}

}  // namespace

cudaError_t launch_verify_simt(const VerifyParams &p, kdt_dtype dt, cudaStream_t s) {
    const int rows_seq = p.T * p.H;
    const dim3 grid((rows_seq + kRows - 1) / kRows, p.num_splits, p.B);
    const size_t smem = sizeof(SimtSmem);
    cudaError_t e;
    if (dt == KDT_F32) {
        e = cudaFuncSetAttribute(verify_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        verify_simt_kernel<float><<<grid, kThreads, smem, s>>>(p);
    } else {
        e = cudaFuncSetAttribute(verify_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        verify_simt_kernel<__nv_bfloat16><<<grid, kThreads, smem, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace kdt
