/*
 * idx_diag.h -- diagnostics beside the C ABI of idx.h: a probe of the FP8
 * tensor-core rate that the scoring's roofline is measured against, and a
 * test hook for the device-timeout path.  Neither is part of the index chain
 * of "sgl-amd-mono-upstream PR 18"; the pages have no counterpart to them.
 * Same conventions as idx.h (device pointers owned by the caller, nothing
 * allocated, asynchronous on `stream`).
 */
#ifndef IDX_DIAG_H
#define IDX_DIAG_H

#include "idx.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * idx_probe_fp8_mma -- the FP8 (E4M3 x E4M3 -> f32) tcgen05 MMA rate of this
 * device.  One CTA per SM issues n_mma back-to-back M = 128 x N = n_cols x
 * K = 32 MMAs (the shape the scoring issues, at n_cols = 256) from shared
 * memory into tensor memory and waits for them; CTA i writes the elapsed wall
 * time in ns to out_ns[i] and SM clocks to out_clk[i] (0 if its wait gave up).
 * The device's rate is 2 * 128 * n_cols * 32 * n_mma * SMs / max_i out_ns[i].
 *
 *  n_mma    8 .. 2^22
 *  n_cols   16 .. 256, a multiple of 16
 *  out_ns, out_clk  device arrays of at least n_out >= SM-count entries
 *
 * Errors: IDX_ERR_ARG, IDX_ERR_UNSUPPORTED (not sm_103), IDX_ERR_CUDA.
 */
idx_status idx_probe_fp8_mma(int n_mma, int n_cols, unsigned long long *out_ns,
                             unsigned long long *out_clk, int n_out, void *stream);

/*
 * idx_test_set_wait_limit -- TEST ONLY.  For scoring launches made later by
 * the calling host thread: every wait of the scoring kernel gives up after
 * wait_ns of wall time instead of 2 s (0 restores 2 s), and with
 * drop_query_handoff != 0 the kernel's epilogue never signals that the query
 * operand is written, so that the MMA issuer's and the epilogue's waits on it
 * run out.  The kernel then stops every role, waits for its own copies and
 * MMAs in flight, releases its tensor memory and records IDX_ERR_TIMEOUT in
 * the workspace status word (read by idx_check_status); the launch's scores
 * are undefined.  Call idx_test_set_wait_limit(0, 0) to return to normal
 * operation.  Always IDX_OK.
 */
idx_status idx_test_set_wait_limit(unsigned long long wait_ns, int drop_query_handoff);

#ifdef __cplusplus
}
#endif

#endif /* IDX_DIAG_H */
