/*
 * gbattn_test.h - test hooks of libgbattn.so.
 *
 * Not part of the attention API and not a step of the method: these entry
 * points let a test drive the library's failure paths on a real GPU without
 * faulting or hanging it. Every wait inside the kernels is bounded; when one
 * runs out, the kernel records GBATTN_ERR_TIMEOUT in its device error word,
 * lets the copies it started land, frees its tensor memory and returns, so
 * the CUDA context stays usable and gbattn_last_device_error() reports the
 * timeout.
 */
#ifndef GBATTN_TEST_H
#define GBATTN_TEST_H

#include "gbattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gbattn_test_fwd_stalled - the bf16 tensor-core forward of attn_fwd (no
 * mask, B x H heads of Sq queries over Sk keys, Dqk = Dv = D) launched with
 * two changes: every mbarrier wait gives up after wait_ns nanoseconds
 * (instead of 2 s), and the producer never loads the K tile of each CTA's
 * first key tile, so the MMA thread's wait for it runs out.
 *   q [B, H, Sq, D], k / v [B, H, Sk, D] bf16, o [B, H, Sq, D] bf16 and
 *   lse [B, H, Sq] fp32: caller-owned device memory, 16-byte aligned (lse 4).
 *   D in {32, 64, 128}; 1 <= wait_ns <= 2e9.
 * O and LSE are left unwritten (their contents are undefined afterwards).
 * Returns GBATTN_OK once the launch is queued (the timeout itself is read
 * back with gbattn_last_device_error, which also clears it), or the
 * argument codes of attn_fwd.
 */
int gbattn_test_fwd_stalled(int B, int H, int Sq, int Sk, int D, const void* q, const void* k, const void* v,
                            void* o, float* lse, unsigned long long wait_ns, gbattn_stream stream);

/*
 * gbattn_test_bwd_stalled - the bf16 tensor-core backward of attn_bwd (no
 * mask, B x H heads of S queries over S keys, Dqk = Dv = D, the one-CTA
 * dK/dV kernel unless gbattn_set_dkdv_cta_pair selected the pair) launched
 * with two changes: every mbarrier wait gives up after wait_ns nanoseconds,
 * the producer of each dK/dV CTA never loads the dO tile of its first query
 * tile, and the producer of each dQ CTA never loads the K tile of its first
 * key tile, so both kernels' MMA issuers' waits run out.
 *   q, k, v, o, dout [B, H, S, D] bf16, lse [B, H, S] fp32 (as attn_fwd wrote
 *   it), dq / dk / dv [B, H, S, D] bf16, workspace of at least
 *   attn_bwd_workspace_bytes(GBATTN_BF16, B, H, S, S, D, D) bytes: caller-owned
 *   device memory, 16-byte aligned. D in {32, 64, 128}; 1 <= wait_ns <= 2e9.
 * dQ, dK and dV are left undefined. Returns GBATTN_OK once the launches are
 * queued (the timeout is read back with gbattn_last_device_error, which also
 * clears it), or the argument codes of attn_bwd.
 */
int gbattn_test_bwd_stalled(int B, int H, int S, int D, const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv, void* workspace,
                            size_t workspace_bytes, unsigned long long wait_ns, gbattn_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_TEST_H */
