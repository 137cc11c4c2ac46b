/* gdn.h -- C ABI of the Gated DeltaNet scan in libmoe.so (sm_103a).
 *
 * Source: "Perplexity open-sources Lily" -- "three workload shapes" (30 of the
 * model's 40 layers are Gated DeltaNet layers, a fixed-size recurrence) and
 * "Prefill" (a scan that keeps the recurrent state in GPU registers, +5.6 %
 * at 2K tokens).  The pages do not print the recurrence; this is the gated
 * delta rule as its authors publish it ("Gated Delta Networks", Yang, Kautz
 * and Hatamizadeh, 2024), per value head h and token t, state S [dk][dv]:
 *
 *   S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *   o_t = S_t^T q_t
 *
 * Value head h reads query/key head h / (Hv / Hk).  Normalising or scaling q
 * and k, and computing alpha and beta from the layer's projections, happen
 * before the scan.  Arithmetic: fp32 state and sums; o rounded once to bf16.
 *
 * Conventions as in moe.h: *_d pointers are device pointers, bf16 tensors are
 * raw 16-bit patterns, checks run on the host before anything is enqueued,
 * nothing is allocated or synchronised, launch failures return MOE_ERR_CUDA.
 */
#ifndef GDN_H
#define GDN_H
#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One sequence of T tokens through the scan, on `stream` (a cudaStream_t,
 * NULL for the default stream).
 *   q_d, k_d   bf16 [T][Hk][dk]        queries and keys (read)
 *   v_d        bf16 [T][Hv][dv]        values (read)
 *   alpha_d    fp32 [T][Hv]            decay, in (0, 1] (read)
 *   beta_d     fp32 [T][Hv]            write strength, in [0, 1] (read)
 *   state_d    fp32 [Hv][dk][dv]       state before token 0 on entry, after
 *                                      token T-1 on return (read and written)
 *   o_d        bf16 [T][Hv][dv]        outputs (written)
 * Supported: dk == 128, dv a positive multiple of 32, Hk >= 1, Hv a multiple
 * of Hk.  T == 0 returns MOE_OK with nothing enqueued.
 * Errors: MOE_ERR_INVALID_ARGUMENT (null pointer with T > 0, T < 0, Hk < 1,
 * Hv not a multiple of Hk, o_d overlapping an input), MOE_ERR_UNSUPPORTED
 * (dk, dv), MOE_ERR_MISALIGNED (any pointer not 16-byte aligned), MOE_ERR_CUDA.
 * The buffers are the caller's; the call only reads and writes them. */
moe_status gdn_scan(const void *q_d, const void *k_d, const void *v_d, const float *alpha_d, const float *beta_d,
                    float *state_d, void *o_d, int T, int Hk, int Hv, int dk, int dv, void *stream);

#ifdef __cplusplus
}
#endif
#endif
