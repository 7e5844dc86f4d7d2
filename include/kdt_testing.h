/*
 * kdt_testing.h -- test hooks of libkdt.so. Not part of the stable API: these entry
 * points exist so that a test can drive failure paths that correct inputs never reach.
 */
#ifndef KDT_TESTING_H
#define KDT_TESTING_H

#include "kdt.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * kdt_test_verify_attn_wait_expiry -- kdt_verify_attn on the tensor-core kernel with
 * one hand-off deliberately left incomplete: the first work item's "query rows are in
 * tensor memory" arrivals are withheld, and every pipeline wait gives up after
 * `wait_us` microseconds instead of the normal 200 ms. The kernel must then record a
 * negative code in `err` (the number says which wait expired first), release every
 * waiting warp, let its in-flight copies and MMAs finish, free its tensor memory and
 * return; the CUDA context stays usable and the next normal call is unaffected. `out`
 * and `lse` are left incomplete.
 *   a, workspace, ws_bytes, stream: as for kdt_verify_attn; `a` must select the
 *           tensor-core kernel (bf16 inputs, impl AUTO or TCGEN05) and should carry an
 *           `err` word.
 *   wait_us 100 .. 1000000.
 * Errors: those of kdt_verify_attn; KDT_ERR_UNSUPPORTED for the SIMT kernel or a
 * wait_us out of range.
 */
kdt_status kdt_test_verify_attn_wait_expiry(const kdt_verify_args *a, void *workspace, size_t ws_bytes,
                                            uint32_t wait_us, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDT_TESTING_H */
