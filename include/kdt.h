/*
 * kdt.h -- C ABI of libkdt.so: DDTree tree-verify MLA-absorb attention with
 * visibility masking, for NVIDIA GB300 (sm_103a).
 *
 * The method (page "The Verify-Attn Kernel: A Single File Write That Completed a
 * Critical Piece of the DDTree Engine", section "The Design Journey: From Concept
 * to CUDA"; page "The Moment of Truth: Validating a Custom CUDA Attention Kernel
 * for Speculative Decoding", sections "Context" and "The Design Journey: From
 * Theory to Silicon"): for every sequence b, draft-tree query i and head h,
 *
 *   s_j = scale * ( q_nope[b,i,h,:512] . c_kv[b,j,:512] + q_pe[b,i,h,:64] . k_pe[b,j,:64] )
 *
 * over the visible keys j -- the shared prefix j < prefix_len[b], plus tree node i
 * itself and its ancestors (node t at cache row prefix_len[b] + t) -- then
 *
 *   out[b,i,h,:] = sum_j softmax(s)_j * c_kv[b,j,:]      (the latent; the w_vc
 *                                                          up-projection stays outside)
 *   lse[b,i,h]   = ln sum_j exp(s_j)                      (natural log, scaled scores)
 *
 * The per-row lse is what merges this result with attention computed elsewhere
 * over other keys (section "Design Decisions and Trade-Offs" of the first page:
 * long prefix by another kernel, tree tail by this one, combined by log-sum-exp).
 *
 * Conventions for every entry point:
 *  - All tensor arguments are caller-owned DEVICE pointers, row-major and
 *    contiguous, 16-byte aligned, with no aliasing between inputs and outputs
 *    (kdt_verify_attn_host alone takes host tensors).
 *  - Calls are asynchronous on `stream` (0 = legacy default stream). Argument
 *    checks run on the host before any launch and never synchronise. A launch
 *    failure is returned as KDT_ERR_CUDA; faults inside a kernel surface at the
 *    caller's next synchronisation.
 *  - The library allocates no memory: scratch space is the caller's `workspace`
 *    (kdt_verify_attn_noalloc, at the end, uses a fixed array inside the library
 *    instead; kdt_verify_attn_host creates and releases its events). Its global
 *    state: that fixed device array (KDT_NOALLOC_SCRATCH_BYTES on every GPU that
 *    loads the library) and per-device caches of the SM count, of how many
 *    tensor-core clusters are resident at once, and of the array's device address.
 *    Concurrent calls are safe given distinct workspaces.
 *  - One GPU per call: kdt_verify_attn's tensors (and its workspace) must be device
 *    memory of the device current on the calling thread -- not host, managed or
 *    another GPU's memory reached through unified addressing -- else the call
 *    returns KDT_ERR_NOT_DEVICE before any launch. The tensor-core kernel loads key
 *    tiles with cluster-multicast TMA, which this library issues only over the
 *    memory of the GPU the call runs on.
 *  - Errors found in the DATA on the device (a malformed tree) are reported
 *    through a caller-provided device word `err` (0 = ok, else 1 + the flat index
 *    b*T + i of the first offending parent entry), never by a trap.
 */
#ifndef KDT_H
#define KDT_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDT_OK = 0,
    KDT_ERR_NULL_ARG = 1,     /* a required pointer is NULL, or both/neither of parent and vis */
    KDT_ERR_BAD_SHAPE = 2,    /* sizes out of range or inconsistent (B, T, H, strides, kv bounds) */
    KDT_ERR_UNSUPPORTED = 3,  /* valid but not implemented here (D_c != 512, D_r != 64, impl) */
    KDT_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than kdt_verify_attn_workspace_size() */
    KDT_ERR_CUDA = 5,         /* a CUDA runtime call or kernel launch failed */
    KDT_ERR_NOT_DEVICE = 6    /* a tensor is not device memory of the current device */
} kdt_status;

/* Static, never-NULL English name of a status. */
const char *kdt_status_str(kdt_status s);

/* Library version: major * 10000 + minor * 100 + patch. */
int kdt_version(void);

typedef enum { KDT_F32 = 0, KDT_BF16 = 1 } kdt_dtype;

/* Kernel family. AUTO picks by shape and dtype: small problems -- B*T*H * max_kv_len at
 * most 2^18 for bf16 inputs, 2^19 for fp32 -- go to SIMT_SMALL, the SIMT kernel on 16-row
 * tiles with one 64-key block per split, spread over many CTAs (the tensor-core kernel's
 * pipeline has a fixed latency of tens of microseconds); otherwise bf16 inputs use the
 * tcgen05 tensor-core kernel and fp32 inputs the SIMT kernel on 64-row tiles (which
 * computes in fp32; the tensor path would round inputs). kdt_verify_attn_plan reports the
 * choice. Both SIMT forms are valid for both dtypes. */
typedef enum { KDT_IMPL_AUTO = 0, KDT_IMPL_SIMT = 1, KDT_IMPL_TCGEN05 = 2, KDT_IMPL_SIMT_SMALL = 3 } kdt_impl;

/*
 * kdt_build_visibility -- draft-tree parent array -> packed ancestor bits.
 *
 * The mask comes from the tree (page "The Moment of Truth ...", section
 * "Context"): tree key t is visible to query i iff t == i or t is an ancestor of i
 * ("The Verify-Attn Kernel ...", sections "The Design Journey" and "Assumptions
 * and the Path Forward").
 *
 *   parent  device int32 [B,T]; parent[b,0] is normally -1 (the root). Requires
 *           -1 <= parent[b,i] < i (topological order; several roots allowed).
 *   vis     device uint32 [B,T,W], W = ceil(T/32): bit (t % 32) of word t / 32 of
 *           vis[b,i] is set iff t == i or t is an ancestor of i. Bits >= T are 0.
 *   err     device int32, may be NULL. Zeroed, then set to 1 + (b*T + i) of the
 *           first parent entry outside [-1, i); rows reached through such an entry
 *           stop at it. If NULL, malformed entries are silently cut the same way.
 * Errors: KDT_ERR_NULL_ARG (parent or vis NULL), KDT_ERR_BAD_SHAPE (B < 0, T < 1,
 * T > 4096), KDT_ERR_CUDA.
 */
kdt_status kdt_build_visibility(const int32_t *parent, int B, int T, uint32_t *vis, int32_t *err,
                                cudaStream_t stream);

/* Arguments of kdt_verify_attn. Sizes: B >= 0 sequences, 1 <= T <= 4096 tree
 * queries per sequence, 1 <= H <= 1024 heads. */
typedef struct {
    int B, T, H;
    int D_c;                /* latent width, must be 512 */
    int D_r;                /* rope width, must be 64 */
    kdt_dtype dtype;        /* element type of q_nope, q_pe, c_kv, k_pe (all the same) */
    const void *q_nope;     /* [B,T,H,512] absorbed query (q_nope . w_kc done by the caller) */
    const void *q_pe;       /* [B,T,H,64] rotated rope query */
    const void *c_kv;       /* [B,L,512] latent cache; row j of sequence b at c_kv + (b*L + j)*512 */
    const void *k_pe;       /* [B,L,64]  rope keys, same row indexing */
    int64_t kv_row_stride;  /* L: rows per sequence in c_kv/k_pe, >= max_kv_len */
    const int32_t *prefix_len; /* device [B]: shared-prefix length; tree node t at row prefix_len[b]+t */
    int max_kv_len;         /* host bound: >= max_b prefix_len[b] + T (sizes the grid, no sync) */
    const int32_t *parent;  /* device [B,T] parent array, or NULL */
    const uint32_t *vis;    /* device [B,T,ceil(T/32)] packed visibility bits, or NULL */
    float scale;            /* score scale, e.g. 1/sqrt(192) */
    float *out;             /* device fp32 [B,T,H,512] */
    float *lse;             /* device fp32 [B,T,H], or NULL */
    int32_t *err;           /* device int32 error word, or NULL: 0, or with `parent` 1 + the
                               index b*T + i of the first malformed entry, or a negative
                               code if an internal wait for a copy or pipeline stage gave up */
    int impl;               /* kdt_impl */
    int num_splits;         /* 0 = choose automatically. SIMT_SMALL: KV splits per 16-row
                               tile (at most 32), merged by log-sum-exp. SIMT (64-row tiles):
                               the number of CTAs its (64-row tile, 128-key block) pairs are
                               cut into equal contiguous shares for (at most one per pair;
                               automatic: one per SM). Tensor-core kernel: the number of
                               persistent 4-CTA clusters its (256-row unit, 128-key block)
                               work is cut into equal shares for (at most those resident at
                               once). With either share split, the tiles or units a share
                               boundary cuts are merged by log-sum-exp. */
    int64_t q_nope_row_stride; /* elements between consecutive (b,i,h) rows of q_nope; 0 = 512
                                  (contiguous). Lets the kernels read a combined [.., 512 + 64]
                                  query buffer where it lies (stride 576, q_pe = q_nope + 512)
                                  instead of a split copy. Else >= 512, a multiple of 8. */
    int64_t q_pe_row_stride;   /* the same for q_pe; 0 = 64, else >= 64, a multiple of 8 */
} kdt_verify_args;

/*
 * kdt_verify_attn -- tree-verify MLA-absorb attention (the definition at the top).
 *
 * Exactly one of `parent` and `vis` must be non-NULL. With `parent`, the bits are
 * first built into the workspace as by kdt_build_visibility (and `err` reports a
 * malformed tree). With `vis`, the caller's bits are used as given: they need not
 * come from a tree, and a row whose visible set is empty (no prefix, no bit set)
 * gets out = 0 and lse = -inf.
 * Rows of c_kv/k_pe at or beyond prefix_len[b] + T never affect the result, whatever
 * they hold (NaN included); rows below max_kv_len may be read (the one-pass small-shape
 * kernel copies a sequence's first max_kv_len rows before it knows prefix_len[b]).
 * Inputs are all fp32 or all bf16; out and lse are fp32.
 * `workspace` must hold kdt_verify_attn_workspace_size(a) bytes (256-byte aligned;
 * may be NULL when that size is 0). Its contents need no initialisation.
 * Errors: KDT_ERR_NULL_ARG, KDT_ERR_BAD_SHAPE (including prefix bound violations
 * detectable on the host: max_kv_len > kv_row_stride, max_kv_len < T),
 * KDT_ERR_UNSUPPORTED (D_c != 512, D_r != 64, unknown impl, TCGEN05 with fp32),
 * KDT_ERR_WORKSPACE, KDT_ERR_NOT_DEVICE (a tensor or the workspace is not device
 * memory of the current device), KDT_ERR_CUDA. prefix_len values are device data: the
 * caller guarantees prefix_len[b] + T <= max_kv_len.
 */
kdt_status kdt_verify_attn(const kdt_verify_args *a, void *workspace, size_t ws_bytes,
                           cudaStream_t stream);

/* Bytes of workspace kdt_verify_attn needs for these arguments (0 possible).
 * Depends only on host-side fields (sizes, dtype, impl, num_splits, which of
 * parent/vis is given). Returns 0 for arguments kdt_verify_attn would reject. */
size_t kdt_verify_attn_workspace_size(const kdt_verify_args *a);

/* What kdt_verify_attn will launch for these arguments. */
typedef struct {
    int impl;               /* the kdt_impl chosen (never KDT_IMPL_AUTO) */
    int num_splits;         /* splits, CTAs or clusters actually used (see kdt_verify_args) */
    int num_launches;       /* kernels launched per call */
    int ctas;               /* CTAs of the main attention kernel */
    size_t workspace_bytes;
} kdt_plan;

kdt_status kdt_verify_attn_plan(const kdt_verify_args *a, kdt_plan *plan);

/*
 * kdt_verify_attn_host -- kdt_verify_attn on HOST buffers, the copies pipelined with
 * the compute.
 *
 * Same arguments and results as kdt_verify_attn, except that q_nope, q_pe, c_kv,
 * k_pe, prefix_len, parent (or vis), out and lse are HOST pointers; `err`, when
 * given, stays a DEVICE word with the same meaning (flat index over the whole
 * batch). Host rows must be contiguous (both row strides 0) and every host tensor
 * 16-byte aligned. For the copies to overlap the host buffers must be page-locked
 * (cudaHostAlloc, cudaHostRegister, a pinned torch tensor); pageable buffers give
 * the same results with the copies serialised.
 *
 * The B sequences are cut into n_chunks chunks of B / n_chunks whole sequences
 * (n_chunks must divide B; 0 = 4, else 2, else 1). Every chunk's inputs are copied
 * into `dev_buf` on stream_in (one copy per tensor); chunk c's attention (with its
 * visibility bits when parent is given) runs on `stream` once its inputs landed; its
 * out and lse are copied back on stream_out right behind it. So the copy of chunk c+1
 * in, the compute of chunk c and the copy of chunk c-1 out overlap, and the host link
 * sets the pace. The chunks' results are those of kdt_verify_attn called on each
 * chunk: they agree with one call over the whole batch within the path's tolerance
 * (the work split differs), not bit for bit.
 *
 *   dev_buf     device scratch of kdt_verify_attn_host_buffer_size(a, n_chunks)
 *               bytes, 256-byte aligned, no initialisation needed: every chunk's
 *               inputs and outputs, one error word per chunk, one verify workspace.
 *   stream      carries the compute; the call is complete -- out and lse written
 *               on the host -- once `stream` reaches the point after the call
 *               (synchronise it, or an event recorded on it, before reading out).
 *               The copies in wait for the work queued on `stream` before the call.
 *   stream_in, stream_out
 *               two more streams, distinct from each other and from `stream`. They
 *               should be non-blocking (cudaStreamNonBlocking) and `stream` not the
 *               legacy default stream with blocking streams, or the copies and the
 *               compute serialise (the results are the same).
 * The library creates two events per chunk plus two per call and releases them
 * before it returns (CUDA frees an event destroyed while pending once it completes).
 * Errors: those of kdt_verify_attn; KDT_ERR_BAD_SHAPE also for an n_chunks that
 * does not divide B, a nonzero row stride, or two equal streams; KDT_ERR_WORKSPACE
 * for a missing, short or misaligned dev_buf; KDT_ERR_NOT_DEVICE when dev_buf or
 * `err` is not device memory of the current device.
 */
kdt_status kdt_verify_attn_host(const kdt_verify_args *a, int n_chunks, void *dev_buf, size_t dev_bytes,
                                cudaStream_t stream, cudaStream_t stream_in, cudaStream_t stream_out);

/* Bytes of dev_buf kdt_verify_attn_host needs for these (host-pointer) arguments and
 * chunk count; 0 for arguments it would reject (and for B = 0). */
size_t kdt_verify_attn_host_buffer_size(const kdt_verify_args *a, int n_chunks);

/*
 * kdt_merge_attn_states -- combine two attention results over DISJOINT key sets
 * (e.g. a long prefix done elsewhere and the tree tail done here; section "Design
 * Decisions and Trade-Offs" of "The Verify-Attn Kernel ..."):
 *   M = max(lse_a, lse_b), w = exp(lse - M),
 *   o = (w_a o_a + w_b o_b) / (w_a + w_b),  lse = M + ln(w_a + w_b);
 * both -inf gives o = 0, lse = -inf.
 *   o_a, o_b, o    device fp32 [rows, D]; lse_a, lse_b, lse  device fp32 [rows].
 *   D a multiple of 4, 4 <= D <= 4096. `o`/`lse` may alias o_a/lse_a (in place).
 * Errors: KDT_ERR_NULL_ARG, KDT_ERR_BAD_SHAPE, KDT_ERR_CUDA.
 */
kdt_status kdt_merge_attn_states(const float *o_a, const float *lse_a, const float *o_b,
                                 const float *lse_b, int64_t rows, int D, float *o, float *lse,
                                 cudaStream_t stream);

/*
 * kdt_vc_up_proj -- per-head value up-projection of the latent attention output. The
 * verify kernel stops at the latent, and each head's value weights are applied by a
 * separate GEMM after it (page "The Verify-Attn Kernel ...", section "Design Decisions
 * and Trade-Offs"):
 *
 *   v[r, h, n] = sum_{d < D_c} o[r, h, d] * w_vc[h, d, n]        r < R, h < H, n < D_v
 *
 *   o      device fp32 [R, H, D_c]: e.g. kdt_verify_attn's `out` with R = B*T rows
 *   w_vc   device [H, D_c, D_v] in w_dtype (bf16)
 *   v      device fp32 [R, H, D_v], written whole; must not overlap o or w_vc
 *   err    device int32, may be NULL: zeroed, then a negative code if an internal
 *          pipeline wait expired (the kernel then returns early; v is incomplete)
 * Sizes: D_c = 512, D_v 64 or 128, 1 <= H <= 1024, R >= 0, R*H <= 2^31.
 * Arithmetic: each o element is split into two bf16 parts whose sum is o to within
 * 2^-16 |o|; both are multiplied by the bf16 weights on the tensor cores with fp32
 * accumulation, so the result meets the fp32 path's bound (1e-4 absolute + 1e-4
 * relative) against the exact product.
 * Errors: KDT_ERR_BAD_SHAPE (sizes, 16-byte alignment of o, w_vc and v),
 * KDT_ERR_UNSUPPORTED (D_c, D_v, w_dtype other than KDT_BF16), KDT_ERR_NULL_ARG,
 * KDT_ERR_NOT_DEVICE (a tensor not in device memory of the current device; its weights
 * and rows are read through TMA tensor maps), KDT_ERR_CUDA.
 */
kdt_status kdt_vc_up_proj(const float *o, const void *w_vc, kdt_dtype w_dtype, int R, int H, int D_c, int D_v,
                          float *v, int32_t *err, cudaStream_t stream);

/*
 * kdt_verify_attn_noalloc -- kdt_verify_attn without a caller workspace.
 *
 * The method's pages have no counterpart to this entry point; it exists for
 * callers that cannot allocate device memory when they call the library: a
 * serving engine that reserved nearly all HBM for its KV-cache pool at start-up
 * (a later cudaMalloc fails, or would fragment the pool), a plugin inside a host
 * framework whose allocator it may not call, or a latency-critical loop that cannot
 * afford the implicit device synchronisation of cudaMalloc/cudaFree.
 *
 * Same arguments, results and errors as kdt_verify_attn, but the scratch space
 * (packed visibility bits built from `parent`, split-KV partials) lives in a fixed
 * device array of KDT_NOALLOC_SCRATCH_BYTES inside libkdt.so, present on every GPU
 * that loads the library until the process exits. Nothing is allocated: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *  - Size limit: 64 MiB, enough for the partial states of the tensor-core path and of
 *    the 64-row SIMT path on any GPU they support. If the call needs more scratch, a
 *    SIMT_SMALL call's automatic split count (num_splits == 0) is lowered until the
 *    partials fit;
 *    if the call still does not fit, or an explicit num_splits does not fit, it
 *    returns KDT_ERR_WORKSPACE and launches nothing.
 *  - Set-up: the first call made on a device (with that device current) looks up
 *    the array's device address with cudaGetSymbolAddress and keeps it for that
 *    device; make that first call before any stream capture on that device. A
 *    cudaDeviceReset destroys the array with the context: the kept address then
 *    dangles, so do not call this entry point again in a process after resetting
 *    a device it was used on.
 *  - Sharing: every call on a device uses the same array and it keeps the last
 *    call's contents. The kernels overwrite every scratch byte they read, so no
 *    clearing is needed, but calls whose work overlaps on the GPU (other streams,
 *    other host threads) race on the array: order them on one stream or serialise
 *    them.
 */
#define KDT_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

kdt_status kdt_verify_attn_noalloc(const kdt_verify_args *a, cudaStream_t stream);

/* ------------------------------------------------------------------------------
 * The steps next to verify in a DDTree step: rotary embedding of the tree's rope
 * parts before it, the greedy accept walk and the cache compaction after it.
 * ------------------------------------------------------------------------------ */

/*
 * kdt_tree_build -- best-first draft tree on the device (page "The Architecture of an
 * Inference Engine ...", section "The Context": the tree builder constructs the draft
 * tree on the GPU instead of with a per-request CPU heap).
 * For every depth d = 1..D ahead of the root the drafter gives K candidates,
 * cand_tok[b,d-1,:] with log-probabilities cand_lp[b,d-1,:], the same below every node of
 * depth d-1. A node's score is the float32 sum of the log-probabilities on its path (the
 * root's is 0). The tree grows N times by the best node not yet in it whose parent is:
 * higher score, then lower depth, then lower parent index, then lower candidate rank
 * (a depth's candidates ranked by log-probability, highest first, ties by position; NaN
 * counts as -inf). Nodes are numbered in the order they join, the root 0, so the output
 * is in topological order and feeds kdt_build_visibility / kdt_verify_attn directly.
 *   cand_tok  device int32 [B,D,K];  cand_lp  device float32 [B,D,K]
 *   root_tok  device int32 [B] or NULL: tok[b,0] (else -1)
 *   parent, tok  device int32 [B,N+1] out; depth (int32) and score (float32) [B,N+1]
 *            out, each may be NULL
 * Sizes: 1 <= D <= 64, 1 <= K <= 32, 1 <= N <= 4095 and N <= K + K^2 + ... + K^D.
 * Errors: KDT_ERR_NULL_ARG, KDT_ERR_BAD_SHAPE, KDT_ERR_CUDA.
 */
kdt_status kdt_tree_build(const int32_t *cand_tok, const float *cand_lp, int B, int D, int K, int N,
                          const int32_t *root_tok, int32_t *parent, int32_t *tok, int32_t *depth, float *score,
                          cudaStream_t stream);

/* Arguments of kdt_rope_neox. */
typedef struct {
    int B, T, H;            /* sequences, tree nodes per sequence (1..4096), heads (1..1024) */
    int D_r;                /* rope width: even, 2..256 */
    kdt_dtype dtype;        /* element type of q and k_pe */
    void *q;                /* device, or NULL: the rope part of query row (b,i,h) is the D_r
                               elements at q + ((b*T + i)*H + h) * q_row_stride; rotated in place.
                               Point it at the rope slice of a combined [.., D_c + D_r] query
                               buffer to rotate that buffer where it lies. */
    int64_t q_row_stride;   /* elements between consecutive (b,i,h) rows, >= D_r */
    void *k_pe;             /* device [B, L, D_r], or NULL: rows prefix_len[b] + i (the tree's
                               new key rows) rotated in place; rows outside [0, L) are skipped */
    int64_t kv_row_stride;  /* L, >= T (used with k_pe) */
    const int32_t *prefix_len; /* device [B] (used with k_pe) */
    const int32_t *pos;     /* device [B,T]: rotary position of tree node i (normally
                               prefix_len[b] + depth(i), the root at depth 0) */
    double base;            /* angle base (theta), > 0, e.g. 10000 */
} kdt_rope_args;

/*
 * kdt_rope_neox -- NeoX rotary embedding in place (page "The Query-Split Kernel: A
 * Pivotal Edit ...", sections "The Reasoning Chain" -- rope applied in place on the rope
 * portion of the query buffer -- and "Input Knowledge" -- NeoX variant, float64 angles).
 * For a vector x of width d at position p and j < d/2: a_j = p * base^(-2j/d) in float64,
 * c_j and s_j its cosine and sine rounded to float32, then in float32
 *   (x_j, x_{j+d/2}) <- (x_j c_j - x_{j+d/2} s_j,  x_{j+d/2} c_j + x_j s_j),
 * each product and sum rounded to nearest on its own (no fused multiply-add), the
 * results rounded to nearest (even) to the element type. Every head of node (b,i) and
 * its key row use pos[b,i].
 * Errors: KDT_ERR_NULL_ARG (pos NULL, both q and k_pe NULL, k_pe without prefix_len),
 * KDT_ERR_BAD_SHAPE, KDT_ERR_UNSUPPORTED (dtype), KDT_ERR_CUDA.
 */
kdt_status kdt_rope_neox(const kdt_rope_args *a, cudaStream_t stream);

/*
 * kdt_tree_accept -- greedy walk of a verified draft tree (page "The Moment of Truth
 * ...", section "Context": the accept kernel walks the tree greedily to decide which
 * draft tokens are accepted). Node 0 is the root; from it, move to the child c of the
 * current node with tok[c] == target[current] (the lowest index if several), until no
 * child matches.
 *   parent   device int32 [B,T], -1 <= parent[b,i] < i (as for kdt_build_visibility)
 *   tok      device int32 [B,T]: node i's draft token (tok[b,0] unused)
 *   target   device int32 [B,T]: the target model's greedy next token after node i
 *   acc_nodes device int32 [B,T] out: the accepted path (node indices from the root),
 *            then -1
 *   n_acc    device int32 [B] out: path length, >= 1 (the root always stays)
 *   bonus    device int32 [B] out: target[last node of the path], the token the
 *            target model adds after the accepted ones
 *   err      device int32, may be NULL: zeroed, then 1 + (b*T + i) of the first parent
 *            entry outside [-1, i); such entries are skipped.
 * Errors: KDT_ERR_NULL_ARG, KDT_ERR_BAD_SHAPE (B < 0, T < 1, T > 4096), KDT_ERR_CUDA.
 */
kdt_status kdt_tree_accept(const int32_t *parent, const int32_t *tok, const int32_t *target, int B, int T,
                           int32_t *acc_nodes, int32_t *n_acc, int32_t *bonus, int32_t *err,
                           cudaStream_t stream);

/*
 * kdt_kv_compact -- drop the unaccepted branches from the cache (page "The Architecture
 * of an Inference Engine ...", sections "The Context" and "Input Knowledge Required").
 * The tree's rows sit at cache rows prefix_len[b] + t; the k-th node of the accepted
 * path moves to row prefix_len[b] + k of both c_kv [B,L,D_c] and k_pe [B,L,D_r], in
 * place. With update_prefix != 0, prefix_len[b] += n_acc[b] afterwards. Rows past the
 * new length keep what they held. Path entries that are not increasing tree indices, or
 * that point past row L, are not copied.
 * D_c and D_r times the element size must be multiples of 16 bytes; c_kv and k_pe
 * 16-byte aligned. Errors: KDT_ERR_NULL_ARG, KDT_ERR_BAD_SHAPE, KDT_ERR_UNSUPPORTED,
 * KDT_ERR_CUDA.
 */
kdt_status kdt_kv_compact(void *c_kv, void *k_pe, kdt_dtype dtype, int D_c, int D_r, int B, int T,
                          int64_t kv_row_stride, int32_t *prefix_len, const int32_t *acc_nodes,
                          const int32_t *n_acc, int update_prefix, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDT_H */
