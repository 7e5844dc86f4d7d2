// Internal declarations shared by the translation units of libkdt.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kdt.h"
#include "kdt_testing.h"

namespace kdt {

constexpr int kDc = 512;   // latent width of the MLA cache
constexpr int kDr = 64;    // rope width
constexpr int kDqk = kDc + kDr;

// err <- min(err, v) treating 0 as "no error yet" (v >= 1): the first offending entry
// of a malformed tree, whatever order the threads find them in.
__device__ __forceinline__ void record_error(int32_t *err, int32_t v) {
    if (!err) return;
    int32_t old = *reinterpret_cast<volatile int32_t *>(err);
    while (old == 0 || v < old) {
        int32_t seen = atomicCAS(err, old, v);
        if (seen == old) break;
        old = seen;
    }
}
constexpr int kMaxSplits = 32;
constexpr int kMaxT = 4096;

// Everything an attention kernel needs, already validated on the host.
struct VerifyParams {
    int B, T, H, W;            // W = ceil(T/32) visibility words per query
    int64_t L;                 // cache rows per sequence
    int max_kv = 0;            // the caller's bound on prefix_len[b] + T
    const void *q_nope, *q_pe, *c_kv, *k_pe;
    int64_t q_nope_stride, q_pe_stride;   // elements between consecutive (b,i,h) query rows
    const int32_t *prefix_len;
    const uint32_t *vis;       // [B,T,W]
    float scale_log2;          // scale * log2(e): scores are kept in base-2 units
    float *out, *lse;          // final outputs (used when num_splits == 1)
    float *part_o, *part_lse;  // [num_splits, rows_total, 512] / [num_splits, rows_total]
    int num_splits;
    int blocks_per_split;      // key blocks (of the kernel's block size) per split
    int64_t rows_total;        // B*T*H
    int32_t *err;              // caller error word (tensor-core path: negative = pipeline timeout)
    // Tensor-core path: the resident clusters the work is split across; part_o/part_lse
    // then hold [2 * tc_clusters][256] partial states (unused when tc_clusters == 1).
    int tc_clusters;
    // SIMT 64-row tile: the CTAs the (row tile, key block) work is split across; with more
    // than one, part_o/part_lse hold [2 * simt_ctas][64] piece states.
    int simt_ctas = 0;
    // Tensor path: the kernel may start while the visibility kernel this call launched just
    // before it still runs (programmatic dependent launch); it waits for that kernel only
    // before its first read of the bits. Set only when the previous kernel of the stream is
    // that visibility kernel: the kernel reads its other inputs before any wait.
    bool overlap_vis = false;
    int64_t *tc_sched = nullptr;   // tensor path with tc_clusters > 1: the work split's cut points,
                                   // written by the kernel for the merge pass (kTcSchedWords int64)
    // Tensor-core path, test hooks only: wait limit in ns (0 = the default 200 ms) and an
    // arrival to withhold (0 = none, 1 = the first item's Q-ready arrivals).
    uint64_t wait_ns = 0;
    int fault = 0;
};

// K0: parent -> packed ancestor bits.
cudaError_t launch_build_visibility(const int32_t *parent, int B, int T, uint32_t *vis, int32_t *err,
                                    cudaStream_t s);

// K3: SIMT verify (fp32 arithmetic, fp32 or bf16 inputs), with 64-row tiles (512 threads)
// or, for small shapes, 16-row tiles (128 threads) spread over more CTAs.
constexpr int kSimtRows = 64;
constexpr int kSimtSmallRows = 16;
constexpr int kSimtKeys = 64;          // keys per block of the 16-row tile
constexpr int kSimtKeysTm = 128;       // keys per block of the 64-row tile
cudaError_t launch_verify_simt(const VerifyParams &p, kdt_dtype dt, int rows_per_cta, cudaStream_t s);
// Shapes with max_kv_len <= kSimtOneKeys: one pass a CTA of 1, 2 or 4 rows, the visibility
// built in the kernel from `parent` (or read from p.vis when parent is NULL); no workspace.
constexpr int kSimtOneKeys = 64;
// Rows a CTA of the one-pass kernel takes: the fewest of 1, 2 or 4 whose grid the device
// holds at once (every CTA loads its sequence's whole key block, so more and shorter CTAs
// pay only within one wave); 4 when none fits.
int simt_one_rows(kdt_dtype dt, int64_t B, int64_t rows_seq);
// check_all: one CTA validates every parent entry and writes the error word (no clearing
// needed); else the caller clears the word first. kSimtOneCheckAll bounds B * T for it.
constexpr int kSimtOneCheckAll = 1024;
cudaError_t launch_verify_simt_one(const VerifyParams &p, kdt_dtype dt, const int32_t *parent, bool check_all,
                                   int rows_per_cta, cudaStream_t s);
// Merges the piece states the 64-row SIMT tile left (when simt_ctas > 1).
cudaError_t launch_merge_simt_pieces(const VerifyParams &p, cudaStream_t s);

// K1: tcgen05 verify (bf16 inputs): one 4-CTA cluster (two CTA pairs) per resident slot,
// each taking an equal share of the (256-row unit, 128-key block) work; launch_verify_tc
// also merges the units cut by the split.
int tc_rows_per_unit();   // query rows of one work unit (256)
int tc_max_clusters();    // 4-CTA clusters resident at once on the current device (<= 48)
int tc_keys_per_block();
constexpr int kTcSchedWords = 2 + 48 + 1;   // R, boundary cost, cut points of up to 48 clusters
cudaError_t launch_verify_tc(const VerifyParams &p, cudaStream_t s);

// K2: merge the split partials into out/lse.
cudaError_t launch_merge_splits(const float *part_o, const float *part_lse, int num_splits, int64_t rows,
                                float *out, float *lse, cudaStream_t s);

// Public two-state merge.
cudaError_t launch_merge_two(const float *o_a, const float *lse_a, const float *o_b, const float *lse_b,
                             int64_t rows, int D, float *o, float *lse, cudaStream_t s);

// K4: per-head value up-projection v[r, h, :D_v] = o[r, h, :512] . w_vc[h] (bf16 weights,
// D_v 64 or 128), persistent tcgen05 tiles; err (may be NULL) gets a negative code if
// an internal wait expired.
cudaError_t launch_vc_proj(const float *o, const void *w_vc, int R, int H, int Dv, float *v, int32_t *err,
                           cudaStream_t s);

// Per-device SM count (cached).
int sm_count();

// kdt_verify_attn with the device-memory checks selectable: the caller's tensors
// (check_tensors) and the workspace (check_workspace) must be device memory of the current
// device. Entry points whose buffers are already known to be (the host pipeline's chunks
// inside its checked device buffer, the no-allocation entry's library array) skip them.
// `hooks` (may be NULL) carries the tensor-core kernel's test hooks.
struct TestHooks {
    uint64_t wait_ns;
    int fault;
};
kdt_status verify_attn_checked(const kdt_verify_args *a, void *workspace, size_t ws_bytes, cudaStream_t stream,
                               bool check_tensors, bool check_workspace, const TestHooks *hooks = nullptr);

}  // namespace kdt
