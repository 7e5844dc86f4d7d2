// C ABI of libkdt.so: argument checks, planning (kernel family, KV splits,
// workspace layout) and launches. See include/kdt.h for the contract.
#include "kdt_internal.cuh"

#include <atomic>
#include <initializer_list>
#include <math.h>
#include <vector>

namespace kdt {

int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
    const int slot = dev & 63;
    int v = cached[slot].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        cached[slot].store(v, std::memory_order_relaxed);
    }
    return v;
}

namespace {

constexpr size_t kAlign = 256;

// Problems with at most this many (query row x cache row) pairs go to the SIMT kernel on
// 16-row tiles when the caller leaves the choice to the library: the crossovers measured
// on GB300 (device time, L2 flushed) against the tensor-core kernel for bf16 inputs (about
// 0.6 GFLOP; below it the 16-row SIMT kernel took 0.45-0.8 of the tensor kernel's time) and
// against the 64-row SIMT kernel for fp32 inputs (about 1.1 GFLOP; 0.1-0.8 of its time).
constexpr int64_t kSmallShapeWorkBf16 = (int64_t)1 << 18;
constexpr int64_t kSmallShapeWorkF32 = (int64_t)1 << 19;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every tensor a verify call touches must be device memory of the current device. The
// tensor-core kernel encodes TMA tensor maps over c_kv, k_pe and q_pe and loads key tiles
// with cluster multicast; those are issued here over this GPU's own memory only, never
// over host, managed or another GPU's memory reached through unified addressing.
// NULL entries are skipped. KDT_ERR_CUDA if the query itself fails.
kdt_status check_on_current_device(std::initializer_list<const void *> ptrs) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return KDT_ERR_CUDA;
    }
    for (const void *p : ptrs) {
        if (!p) continue;
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
            cudaGetLastError();
            return KDT_ERR_CUDA;
        }
        if (at.type != cudaMemoryTypeDevice || at.device != dev) return KDT_ERR_NOT_DEVICE;
    }
    return KDT_OK;
}

struct Plan;
int unit_rows_of(const Plan &p);

struct Plan {
    int impl = KDT_IMPL_SIMT;
    int splits = 1;
    int tc_clusters = 1;                   // tensor path: resident clusters the work is split across
    int simt_ctas = 0;                     // SIMT 64-row tile: CTAs the work is split across
    bool one_pass = false;                 // SIMT_SMALL with every sequence in one 64-key block
    int one_rows = 4;                      // one-pass kernel: query rows a CTA
    int blocks_per_split = 1;
    int ctas = 0;
    int launches = 0;
    size_t vis_off = 0, vis_bytes = 0;
    size_t po_off = 0, po_bytes = 0;
    size_t pl_off = 0, pl_bytes = 0;
    size_t sched_off = 0;                  // tensor path with pieces: the work split's cut points
    size_t ws_bytes = 0;
};

int unit_rows_of(const Plan &p) { return p.impl == KDT_IMPL_SIMT_SMALL ? kSimtSmallRows : kSimtRows; }

kdt_status check_args(const kdt_verify_args *a) {
    if (!a) return KDT_ERR_NULL_ARG;
    if (a->B < 0 || a->B > 65535 || a->T < 1 || a->T > kMaxT || a->H < 1 || a->H > 1024)
        return KDT_ERR_BAD_SHAPE;
    if (a->D_c != kDc || a->D_r != kDr) return KDT_ERR_UNSUPPORTED;
    if (a->dtype != KDT_F32 && a->dtype != KDT_BF16) return KDT_ERR_UNSUPPORTED;
    if (a->impl != KDT_IMPL_AUTO && a->impl != KDT_IMPL_SIMT && a->impl != KDT_IMPL_TCGEN05 &&
        a->impl != KDT_IMPL_SIMT_SMALL)
        return KDT_ERR_UNSUPPORTED;
    if (a->num_splits < 0) return KDT_ERR_BAD_SHAPE;
    if (a->B == 0) return KDT_OK;
    if (!a->q_nope || !a->q_pe || !a->c_kv || !a->k_pe || !a->prefix_len || !a->out) return KDT_ERR_NULL_ARG;
    if ((a->parent == nullptr) == (a->vis == nullptr)) return KDT_ERR_NULL_ARG;
    if (a->max_kv_len < a->T || (int64_t)a->max_kv_len > a->kv_row_stride) return KDT_ERR_BAD_SHAPE;
    if (!aligned16(a->q_nope) || !aligned16(a->q_pe) || !aligned16(a->c_kv) || !aligned16(a->k_pe) ||
        !aligned16(a->out) || (reinterpret_cast<uintptr_t>(a->lse) & 3u))
        return KDT_ERR_BAD_SHAPE;
    if (!(a->scale == a->scale) || isinf(a->scale)) return KDT_ERR_BAD_SHAPE;
    if ((a->q_nope_row_stride && (a->q_nope_row_stride < kDc || a->q_nope_row_stride % 8)) ||
        (a->q_pe_row_stride && (a->q_pe_row_stride < kDr || a->q_pe_row_stride % 8)))
        return KDT_ERR_BAD_SHAPE;
    return KDT_OK;
}

// Pure function of host-side fields: kernel family, splits, workspace layout.
kdt_status make_plan(const kdt_verify_args *a, Plan *pl) {
    kdt_status st = check_args(a);
    if (st != KDT_OK) return st;
    Plan p;
    if (a->B == 0) {
        *pl = p;
        return KDT_OK;
    }
    const int64_t rows_seq = (int64_t)a->T * a->H;
    const int64_t rows_total = rows_seq * a->B;
    // Kernel family: small problems go to the SIMT kernel on 16-row tiles (the tensor-core
    // kernel's pipeline has a fixed latency of tens of microseconds, the 64-row SIMT tile
    // puts a whole 64 x 64 block on one SM); otherwise bf16 inputs go to the tensor-core
    // kernel and fp32 inputs stay on the SIMT kernel (the tensor path would round them).
    const bool small =
        rows_total * a->max_kv_len <= (a->dtype == KDT_BF16 ? kSmallShapeWorkBf16 : kSmallShapeWorkF32);
    int impl = a->impl;
    if (impl == KDT_IMPL_AUTO)
        impl = small ? KDT_IMPL_SIMT_SMALL : (a->dtype == KDT_BF16 ? KDT_IMPL_TCGEN05 : KDT_IMPL_SIMT);
    const bool tc = impl == KDT_IMPL_TCGEN05;
    if (tc && a->dtype != KDT_BF16) return KDT_ERR_UNSUPPORTED;
    if (tc && (rows_total >= ((int64_t)1 << 31) || a->kv_row_stride >= ((int64_t)1 << 31)))
        return KDT_ERR_BAD_SHAPE;
    p.impl = impl;
    const bool simt_small = impl == KDT_IMPL_SIMT_SMALL;
    const int unit_rows = tc ? tc_rows_per_unit() : (simt_small ? kSimtSmallRows : kSimtRows);
    const int unit_keys = tc ? tc_keys_per_block() : (simt_small ? kSimtKeys : kSimtKeysTm);
    const int unit_tiles = (int)((rows_seq + unit_rows - 1) / unit_rows);   // work units per sequence
    const int nblk = (a->max_kv_len + unit_keys - 1) / unit_keys;
    const int64_t base = (int64_t)unit_tiles * a->B;
    if (tc) {
        // Persistent 4-CTA clusters, each taking an equal share of all units' key blocks
        // (the split adapts on the device to the actual prefix lengths): one per resident
        // slot, or the caller's num_splits of them (at most the resident ones).
        const int resident = tc_max_clusters();
        p.tc_clusters = a->num_splits > 0 && a->num_splits < resident ? a->num_splits : resident;
        p.splits = p.tc_clusters;
        p.blocks_per_split = nblk;
        p.ctas = 4 * p.tc_clusters;
    } else if (!simt_small) {
        // SIMT 64-row tile: one CTA per SM, each taking an equal contiguous share of all
        // (row tile, key block) pairs (the split adapts on the device to the actual prefix
        // lengths), or the caller's num_splits CTAs; never more CTAs than pairs
        const int64_t pairs = base * nblk;
        int64_t C = a->num_splits > 0 ? a->num_splits : sm_count();
        if (C > pairs) C = pairs;
        if (C < 1) C = 1;
        p.simt_ctas = (int)C;
        p.splits = p.simt_ctas;
        p.blocks_per_split = nblk;
        p.ctas = p.simt_ctas;
    } else if (a->max_kv_len <= kSimtOneKeys) {
        // every sequence is one block: the one-pass kernel, 1, 2 or 4 rows a CTA, visibility
        // built in the kernel (no visibility launch, no workspace)
        p.one_pass = true;
        p.one_rows = simt_one_rows(a->dtype, a->B, rows_seq);
        p.ctas = (int)(((rows_seq + p.one_rows - 1) / p.one_rows) * a->B);
    } else {
        // SIMT 16-row tile: one 64-key block per split unless the caller fixed the splits
        int splits;
        if (a->num_splits > 0) {
            splits = a->num_splits;
        } else {
            splits = nblk;                  // one 64-key block per split: short chains, many CTAs
        }
        if (splits > kMaxSplits) splits = kMaxSplits;
        if (splits > nblk) splits = nblk;
        p.blocks_per_split = (nblk + splits - 1) / splits;
        p.splits = (nblk + p.blocks_per_split - 1) / p.blocks_per_split;
        p.ctas = (int)(base * p.splits);
    }
    size_t off = 0;
    if (a->parent && !p.one_pass) {
        const int W = (a->T + 31) / 32;
        p.vis_off = off;
        p.vis_bytes = (size_t)a->B * a->T * W * sizeof(uint32_t);
        off = align_up(off + p.vis_bytes);
    }
    const bool tc_pieces = tc && p.tc_clusters > 1;
    const bool simt_pieces = impl == KDT_IMPL_SIMT && p.simt_ctas > 1;
    if (simt_pieces) {
        // [2 * CTAs][64] piece states
        const int64_t prow = (int64_t)2 * p.simt_ctas * unit_rows;
        p.po_off = off;
        p.po_bytes = (size_t)prow * kDc * sizeof(float);
        off = align_up(off + p.po_bytes);
        p.pl_off = off;
        p.pl_bytes = (size_t)prow * sizeof(float);
        off = align_up(off + p.pl_bytes);
    } else if (p.splits > 1 || tc_pieces) {
        // SIMT: [splits][rows_total]; tensor path: [2 * clusters][256] piece states
        const int64_t prow = tc_pieces ? (int64_t)2 * p.tc_clusters * unit_rows : rows_total;
        const int ns = tc_pieces ? 1 : p.splits;
        p.po_off = off;
        p.po_bytes = (size_t)ns * prow * kDc * sizeof(float);
        off = align_up(off + p.po_bytes);
        p.pl_off = off;
        p.pl_bytes = (size_t)ns * prow * sizeof(float);
        off = align_up(off + p.pl_bytes);
        if (tc_pieces) {
            p.sched_off = off;
            off = align_up(off + kTcSchedWords * sizeof(int64_t));
        }
    }
    p.ws_bytes = off;
    p.launches = ((a->parent && !p.one_pass) ? 1 : 0) + 1 + ((p.splits > 1 || tc_pieces) ? 1 : 0);   // SIMT pieces: splits > 1 too
    *pl = p;
    return KDT_OK;
}

// ---------------------------------------------------------------- host entry --
// Device buffer of kdt_verify_attn_host: for every chunk of nb sequences its inputs, its
// out/lse, then one error word per chunk and one verify workspace the chunks share (their
// computes run in order on one stream). Every region starts on a 256-byte boundary.
struct HostLayout {
    int chunks = 0, nb = 0;
    size_t b_qn = 0, b_qp = 0, b_kv = 0, b_kp = 0, b_pre = 0, b_tree = 0, b_out = 0, b_lse = 0;
    size_t o_qn = 0, o_qp = 0, o_kv = 0, o_kp = 0, o_pre = 0, o_tree = 0, o_out = 0, o_lse = 0;
    size_t chunk = 0, errs_off = 0, ws_off = 0, ws_bytes = 0, total = 0;
};

// Chunk c's arguments: the caller's, with B = nb and every tensor in the device buffer.
kdt_verify_args chunk_args(const kdt_verify_args *a, const HostLayout &L, unsigned char *base, int c) {
    unsigned char *ch = base + (size_t)c * L.chunk;
    kdt_verify_args d = *a;
    d.B = L.nb;
    d.q_nope = ch + L.o_qn;
    d.q_pe = ch + L.o_qp;
    d.c_kv = ch + L.o_kv;
    d.k_pe = ch + L.o_kp;
    d.prefix_len = reinterpret_cast<const int32_t *>(ch + L.o_pre);
    d.parent = a->parent ? reinterpret_cast<const int32_t *>(ch + L.o_tree) : nullptr;
    d.vis = a->vis ? reinterpret_cast<const uint32_t *>(ch + L.o_tree) : nullptr;
    d.out = reinterpret_cast<float *>(ch + L.o_out);
    d.lse = a->lse ? reinterpret_cast<float *>(ch + L.o_lse) : nullptr;
    d.err = a->err ? reinterpret_cast<int32_t *>(base + L.errs_off) + c : nullptr;
    return d;
}

kdt_status host_layout(const kdt_verify_args *a, int n_chunks, HostLayout *L) {
    kdt_status st = check_args(a);
    if (st != KDT_OK) return st;
    if (a->q_nope_row_stride || a->q_pe_row_stride) return KDT_ERR_BAD_SHAPE;   // host rows are contiguous
    HostLayout l;
    if (a->B == 0) {
        *L = l;
        return KDT_OK;
    }
    l.chunks = n_chunks ? n_chunks : (a->B % 4 == 0 ? 4 : (a->B % 2 == 0 ? 2 : 1));
    if (l.chunks < 1 || a->B % l.chunks) return KDT_ERR_BAD_SHAPE;
    l.nb = a->B / l.chunks;
    const size_t elt = a->dtype == KDT_BF16 ? 2 : 4, nb = (size_t)l.nb, rows = nb * a->T * a->H;
    const size_t W = (size_t)(a->T + 31) / 32;
    l.b_qn = rows * kDc * elt;
    l.b_qp = rows * kDr * elt;
    l.b_kv = nb * (size_t)a->kv_row_stride * kDc * elt;
    l.b_kp = nb * (size_t)a->kv_row_stride * kDr * elt;
    l.b_pre = nb * sizeof(int32_t);
    l.b_tree = a->parent ? nb * a->T * sizeof(int32_t) : nb * a->T * W * sizeof(uint32_t);
    l.b_out = rows * kDc * sizeof(float);
    l.b_lse = a->lse ? rows * sizeof(float) : 0;
    size_t off = 0;
    for (auto [o, b] : {std::pair<size_t *, size_t>{&l.o_qn, l.b_qn}, {&l.o_qp, l.b_qp}, {&l.o_kv, l.b_kv},
                        {&l.o_kp, l.b_kp}, {&l.o_pre, l.b_pre}, {&l.o_tree, l.b_tree}, {&l.o_out, l.b_out},
                        {&l.o_lse, l.b_lse}}) {
        *o = off;
        off = align_up(off + b);
    }
    l.chunk = off;
    l.errs_off = (size_t)l.chunks * l.chunk;
    l.ws_off = align_up(l.errs_off + (size_t)l.chunks * sizeof(int32_t));
    // the workspace of one chunk's call (any base gives the same size)
    kdt_verify_args d = chunk_args(a, l, reinterpret_cast<unsigned char *>(kAlign), 0);
    Plan p;
    if ((st = make_plan(&d, &p)) != KDT_OK) return st;
    l.ws_bytes = p.ws_bytes;
    l.total = l.ws_off + l.ws_bytes;
    *L = l;
    return KDT_OK;
}

// err = the first chunk's nonzero word, shifted to the flat index of the whole batch
__global__ void combine_chunk_errors(const int32_t *chunk_err, int chunks, int64_t rows_per_chunk, int32_t *err) {
    int32_t e = 0;
    for (int c = 0; c < chunks && e == 0; ++c)
        if (chunk_err[c]) e = (int32_t)(chunk_err[c] + c * rows_per_chunk);
    *err = e;
}

}  // namespace
}  // namespace kdt

using namespace kdt;

extern "C" {

const char *kdt_status_str(kdt_status s) {
    switch (s) {
        case KDT_OK: return "ok";
        case KDT_ERR_NULL_ARG: return "null argument";
        case KDT_ERR_BAD_SHAPE: return "bad shape or layout";
        case KDT_ERR_UNSUPPORTED: return "unsupported configuration";
        case KDT_ERR_WORKSPACE: return "workspace missing or too small";
        case KDT_ERR_CUDA: return "CUDA error";
        case KDT_ERR_NOT_DEVICE: return "tensor not in device memory of the current device";
    }
    return "unknown status";
}

int kdt_version(void) { return 100; }

kdt_status kdt_build_visibility(const int32_t *parent, int B, int T, uint32_t *vis, int32_t *err,
                                cudaStream_t stream) {
    if (B < 0 || B > 65535 || T < 1 || T > kMaxT) return KDT_ERR_BAD_SHAPE;
    if (B > 0 && (!parent || !vis)) return KDT_ERR_NULL_ARG;
    return launch_build_visibility(parent, B, T, vis, err, stream) == cudaSuccess ? KDT_OK : KDT_ERR_CUDA;
}

size_t kdt_verify_attn_workspace_size(const kdt_verify_args *a) {
    Plan p;
    if (make_plan(a, &p) != KDT_OK) return 0;
    return p.ws_bytes;
}

kdt_status kdt_verify_attn_plan(const kdt_verify_args *a, kdt_plan *out) {
    if (!out) return KDT_ERR_NULL_ARG;
    Plan p;
    kdt_status st = make_plan(a, &p);
    if (st != KDT_OK) return st;
    out->impl = p.impl;
    out->num_splits = p.splits;
    out->num_launches = p.launches;
    out->ctas = p.ctas;
    out->workspace_bytes = p.ws_bytes;
    return KDT_OK;
}

kdt_status kdt_verify_attn(const kdt_verify_args *a, void *workspace, size_t ws_bytes, cudaStream_t stream) {
    return kdt::verify_attn_checked(a, workspace, ws_bytes, stream, true, true);
}

}  // extern "C"

namespace kdt {

kdt_status verify_attn_checked(const kdt_verify_args *a, void *workspace, size_t ws_bytes, cudaStream_t stream,
                               bool check_tensors, bool check_workspace, const TestHooks *hooks) {
    Plan p;
    kdt_status st = make_plan(a, &p);
    if (st != KDT_OK) return st;
    if (a->B == 0) return KDT_OK;
    if (p.ws_bytes > 0 && (!workspace || ws_bytes < p.ws_bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return KDT_ERR_WORKSPACE;
    if (check_tensors &&
        (st = check_on_current_device({a->q_nope, a->q_pe, a->c_kv, a->k_pe, a->prefix_len, a->parent, a->vis,
                                       a->out, a->lse, a->err})) != KDT_OK)
        return st;
    if (check_workspace && p.ws_bytes > 0 && (st = check_on_current_device({workspace})) != KDT_OK) return st;
    unsigned char *ws = static_cast<unsigned char *>(workspace);

    VerifyParams vp;
    vp.B = a->B;
    vp.T = a->T;
    vp.H = a->H;
    vp.W = (a->T + 31) / 32;
    vp.L = a->kv_row_stride;
    vp.max_kv = a->max_kv_len;
    vp.q_nope = a->q_nope;
    vp.q_pe = a->q_pe;
    vp.q_nope_stride = a->q_nope_row_stride ? a->q_nope_row_stride : kDc;
    vp.q_pe_stride = a->q_pe_row_stride ? a->q_pe_row_stride : kDr;
    vp.c_kv = a->c_kv;
    vp.k_pe = a->k_pe;
    vp.prefix_len = a->prefix_len;
    vp.scale_log2 = a->scale * 1.4426950408889634f;
    vp.out = a->out;
    vp.lse = a->lse;
    vp.num_splits = p.splits;
    vp.blocks_per_split = p.blocks_per_split;
    vp.rows_total = (int64_t)a->B * a->T * a->H;
    const bool partials = p.splits > 1 || (p.impl == KDT_IMPL_TCGEN05 && p.tc_clusters > 1);   // SIMT: splits = CTAs
    vp.part_o = partials ? reinterpret_cast<float *>(ws + p.po_off) : nullptr;
    vp.part_lse = partials ? reinterpret_cast<float *>(ws + p.pl_off) : nullptr;
    vp.err = a->err;
    vp.tc_clusters = p.tc_clusters;
    vp.simt_ctas = p.simt_ctas;
    if (p.impl == KDT_IMPL_SIMT) vp.num_splits = 1;   // pieces, not uniform splits
    vp.tc_sched = (p.impl == KDT_IMPL_TCGEN05 && p.tc_clusters > 1) ? reinterpret_cast<int64_t *>(ws + p.sched_off)
                                                                    : nullptr;
    if (hooks) {
        vp.wait_ns = hooks->wait_ns;
        vp.fault = hooks->fault;
    }

    if (p.one_pass) {
        vp.vis = a->vis;
        const bool check_all = (int64_t)a->B * a->T <= kSimtOneCheckAll;
        if (a->err && !check_all && cudaMemsetAsync(a->err, 0, sizeof(int32_t), stream) != cudaSuccess)
            return KDT_ERR_CUDA;
        return launch_verify_simt_one(vp, a->dtype, a->parent, check_all, p.one_rows, stream) == cudaSuccess
                   ? KDT_OK
                   : KDT_ERR_CUDA;
    }
    if (a->parent) {
        uint32_t *vis = reinterpret_cast<uint32_t *>(ws + p.vis_off);
        if (launch_build_visibility(a->parent, a->B, a->T, vis, a->err, stream) != cudaSuccess) return KDT_ERR_CUDA;
        vp.vis = vis;
        vp.overlap_vis = true;
    } else {
        vp.vis = a->vis;
        if (a->err && cudaMemsetAsync(a->err, 0, sizeof(int32_t), stream) != cudaSuccess) return KDT_ERR_CUDA;
    }
    const cudaError_t e = p.impl == KDT_IMPL_TCGEN05 ? launch_verify_tc(vp, stream)
                                                     : launch_verify_simt(vp, a->dtype, unit_rows_of(p), stream);
    if (e != cudaSuccess) return KDT_ERR_CUDA;
    if (p.impl == KDT_IMPL_SIMT_SMALL && p.splits > 1) {
        if (launch_merge_splits(vp.part_o, vp.part_lse, p.splits, vp.rows_total, a->out, a->lse, stream) !=
            cudaSuccess)
            return KDT_ERR_CUDA;
    }
    if (p.impl == KDT_IMPL_SIMT && p.simt_ctas > 1) {
        if (launch_merge_simt_pieces(vp, stream) != cudaSuccess) return KDT_ERR_CUDA;
    }
    return KDT_OK;
}

}  // namespace kdt

extern "C" {

kdt_status kdt_test_verify_attn_wait_expiry(const kdt_verify_args *a, void *workspace, size_t ws_bytes,
                                            uint32_t wait_us, cudaStream_t stream) {
    Plan p;
    kdt_status st = make_plan(a, &p);
    if (st != KDT_OK) return st;
    if (p.impl != KDT_IMPL_TCGEN05 || wait_us < 100 || wait_us > 1000000) return KDT_ERR_UNSUPPORTED;
    const TestHooks hooks{(uint64_t)wait_us * 1000ull, 1};
    return verify_attn_checked(a, workspace, ws_bytes, stream, true, true, &hooks);
}

size_t kdt_verify_attn_host_buffer_size(const kdt_verify_args *a, int n_chunks) {
    HostLayout L;
    return host_layout(a, n_chunks, &L) == KDT_OK ? L.total : 0;
}

kdt_status kdt_verify_attn_host(const kdt_verify_args *a, int n_chunks, void *dev_buf, size_t dev_bytes,
                                cudaStream_t stream, cudaStream_t stream_in, cudaStream_t stream_out) {
    HostLayout L;
    kdt_status st = host_layout(a, n_chunks, &L);
    if (st != KDT_OK) return st;
    if (a->B == 0) return KDT_OK;
    if (stream == stream_in || stream == stream_out || stream_in == stream_out) return KDT_ERR_BAD_SHAPE;
    if (!dev_buf || dev_bytes < L.total || (reinterpret_cast<uintptr_t>(dev_buf) & (kAlign - 1)))
        return KDT_ERR_WORKSPACE;
    // every chunk's device tensors and workspace lie inside dev_buf, checked once here
    if ((st = check_on_current_device({dev_buf, a->err})) != KDT_OK) return st;
    unsigned char *base = static_cast<unsigned char *>(dev_buf);
    const int C = L.chunks;
    std::vector<cudaEvent_t> ev(2 * (size_t)C + 2, nullptr);      // start, end, copied in [C], computed [C]
    auto release = [&]() {
        for (cudaEvent_t e : ev)
            if (e) cudaEventDestroy(e);                            // freed once the event completes
    };
    for (cudaEvent_t &e : ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            e = nullptr;
            release();
            return KDT_ERR_CUDA;
        }
    cudaEvent_t ev_start = ev[0], ev_end = ev[1];
    cudaEvent_t *ev_in = &ev[2], *ev_comp = &ev[2 + C];
    bool ok = true;
    // the copies in and out follow the work queued on `stream` before this call
    ok = ok && cudaEventRecord(ev_start, stream) == cudaSuccess &&
         cudaStreamWaitEvent(stream_in, ev_start, 0) == cudaSuccess &&
         cudaStreamWaitEvent(stream_out, ev_start, 0) == cudaSuccess;
    // every chunk's inputs, one copy per tensor, queued first
    for (int c = 0; c < C && ok; ++c) {
        unsigned char *ch = base + (size_t)c * L.chunk;
        const struct {
            size_t off;
            const void *src;
            size_t bytes;
        } in[6] = {{L.o_qn, a->q_nope, L.b_qn}, {L.o_qp, a->q_pe, L.b_qp}, {L.o_kv, a->c_kv, L.b_kv},
                   {L.o_kp, a->k_pe, L.b_kp}, {L.o_pre, a->prefix_len, L.b_pre},
                   {L.o_tree, a->parent ? (const void *)a->parent : (const void *)a->vis, L.b_tree}};
        for (const auto &t : in)
            ok = ok && cudaMemcpyAsync(ch + t.off, static_cast<const unsigned char *>(t.src) + (size_t)c * t.bytes,
                                       t.bytes, cudaMemcpyHostToDevice, stream_in) == cudaSuccess;
        ok = ok && cudaEventRecord(ev_in[c], stream_in) == cudaSuccess;
    }
    // each chunk's compute, with its copy out queued right behind it
    for (int c = 0; c < C && ok; ++c) {
        const kdt_verify_args d = chunk_args(a, L, base, c);
        ok = cudaStreamWaitEvent(stream, ev_in[c], 0) == cudaSuccess;
        if (ok && (st = verify_attn_checked(&d, base + L.ws_off, L.ws_bytes, stream, false, false)) != KDT_OK)
            break;
        ok = ok && cudaEventRecord(ev_comp[c], stream) == cudaSuccess &&
             cudaStreamWaitEvent(stream_out, ev_comp[c], 0) == cudaSuccess &&
             cudaMemcpyAsync(static_cast<unsigned char *>(static_cast<void *>(a->out)) + (size_t)c * L.b_out, d.out,
                             L.b_out, cudaMemcpyDeviceToHost, stream_out) == cudaSuccess;
        if (ok && a->lse)
            ok = cudaMemcpyAsync(reinterpret_cast<unsigned char *>(a->lse) + (size_t)c * L.b_lse, d.lse, L.b_lse,
                                 cudaMemcpyDeviceToHost, stream_out) == cudaSuccess;
    }
    if (st == KDT_OK && ok && a->err) {
        combine_chunk_errors<<<1, 1, 0, stream>>>(reinterpret_cast<const int32_t *>(base + L.errs_off), C,
                                                  (int64_t)L.nb * a->T, a->err);
        ok = cudaGetLastError() == cudaSuccess;
    }
    // the call is complete on `stream` once the last copy out has landed
    ok = ok && cudaEventRecord(ev_end, stream_out) == cudaSuccess && cudaStreamWaitEvent(stream, ev_end, 0) == cudaSuccess;
    release();
    if (st != KDT_OK) return st;
    return ok ? KDT_OK : KDT_ERR_CUDA;
}

kdt_status kdt_vc_up_proj(const float *o, const void *w_vc, kdt_dtype w_dtype, int R, int H, int D_c, int D_v,
                          float *v, int32_t *err, cudaStream_t stream) {
    if (R < 0 || H < 1 || H > 1024 || (int64_t)R * H > ((int64_t)1 << 31)) return KDT_ERR_BAD_SHAPE;
    if (D_c != kDc || (D_v != 64 && D_v != 128) || w_dtype != KDT_BF16) return KDT_ERR_UNSUPPORTED;
    if (R == 0) return KDT_OK;
    if (!o || !w_vc || !v) return KDT_ERR_NULL_ARG;
    if (!aligned16(o) || !aligned16(w_vc) || !aligned16(v) || (reinterpret_cast<uintptr_t>(err) & 3u))
        return KDT_ERR_BAD_SHAPE;
    kdt_status st = check_on_current_device({o, w_vc, v, err});
    if (st != KDT_OK) return st;
    if (err && cudaMemsetAsync(err, 0, sizeof(int32_t), stream) != cudaSuccess) return KDT_ERR_CUDA;
    return launch_vc_proj(o, w_vc, R, H, D_v, v, err, stream) == cudaSuccess ? KDT_OK : KDT_ERR_CUDA;
}

kdt_status kdt_merge_attn_states(const float *o_a, const float *lse_a, const float *o_b, const float *lse_b,
                                 int64_t rows, int D, float *o, float *lse, cudaStream_t stream) {
    if (rows < 0 || D < 4 || D > 4096 || (D & 3)) return KDT_ERR_BAD_SHAPE;
    if (rows == 0) return KDT_OK;
    if (!o_a || !lse_a || !o_b || !lse_b || !o || !lse) return KDT_ERR_NULL_ARG;
    if (!aligned16(o_a) || !aligned16(o_b) || !aligned16(o)) return KDT_ERR_BAD_SHAPE;
    if (rows > (int64_t)1 << 34) return KDT_ERR_BAD_SHAPE;
    return launch_merge_two(o_a, lse_a, o_b, lse_b, rows, D, o, lse, stream) == cudaSuccess ? KDT_OK
                                                                                               : KDT_ERR_CUDA;
}

}  // extern "C"
