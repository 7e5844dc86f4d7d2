// kdt_verify_attn_noalloc: the verify-attn entry point for callers that cannot
// allocate device memory.
//
// Some callers cannot hand the library a workspace: a serving engine that
// reserved nearly all HBM for its KV-cache pool at start-up (a later cudaMalloc
// fails, or would fragment the pool), a plugin running inside a host framework
// whose allocator it is not allowed to call, or a latency-critical loop where the
// implicit device synchronisation of cudaMalloc/cudaFree is not acceptable. For
// them this file keeps the scratch space in a fixed device array that is part of
// the library image: it exists on every GPU that loads libkdt.so and stays there
// until the process exits.
//
// The array is shared by every call on a device and keeps whatever the last call
// left in it. The kernels fully overwrite every scratch byte they later read (the
// visibility words and the split partials), so nothing has to be cleared between
// calls -- but two calls whose work overlaps on the GPU (different streams, or
// different host threads without ordering) race on the array and may corrupt each
// other's results.
#include "kdt_internal.cuh"

#include <atomic>

namespace {

// Fixed scratch: KDT_NOALLOC_SCRATCH_BYTES (64 MiB) per device, 256-byte aligned.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDT_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch, looked up once per device (on the first call
// made with that device current). In host code the symbol names a host-side stand-in,
// not device memory, so it is never passed to a kernel directly. A cudaDeviceReset
// frees the array with its context and leaves the kept address dangling; the header
// tells callers not to use this entry point on a device after resetting it.
std::atomic<void *> g_scratch_ptr[64];

kdt_status scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KDT_ERR_CUDA;
    void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KDT_ERR_CUDA;
        g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return KDT_OK;
}

}  // namespace

extern "C" {

kdt_status kdt_verify_attn_noalloc(const kdt_verify_args *a, cudaStream_t stream) {
    if (!a) return KDT_ERR_NULL_ARG;
    kdt_verify_args args = *a;
    size_t need = kdt_verify_attn_workspace_size(&args);
    if (need == 0) return kdt_verify_attn(&args, nullptr, 0, stream);   // no scratch, or arguments it rejects
    if (need > KDT_NOALLOC_SCRATCH_BYTES && args.num_splits == 0) {
        // automatic split count: use fewer KV splits until the partials fit
        kdt_plan p;
        kdt_status st = kdt_verify_attn_plan(&args, &p);
        if (st != KDT_OK) return st;
        for (int s = p.num_splits - 1; s >= 1 && need > KDT_NOALLOC_SCRATCH_BYTES; --s) {
            args.num_splits = s;
            need = kdt_verify_attn_workspace_size(&args);
        }
    }
    if (need > KDT_NOALLOC_SCRATCH_BYTES) return KDT_ERR_WORKSPACE;   // larger than the fixed scratch
    void *scratch = nullptr;
    kdt_status st = scratch_for_current_device(&scratch);
    if (st != KDT_OK) return st;
    // the caller's tensors are checked like kdt_verify_attn's; the scratch is this
    // device's copy of the library array
    return kdt::verify_attn_checked(&args, scratch, KDT_NOALLOC_SCRATCH_BYTES, stream, true, false);
}

}  // extern "C"
