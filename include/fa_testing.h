/*
 * fa_testing.h — entry points of the TESTING build of the library only
 * (libfa_gb300_testing.so, compiled with -DFA_TESTING). The product library
 * libfa_gb300.so does not export them.
 *
 * They exist for the validation steps of the dataflow page's section 4.1
 * (layer 2: compare the per-block running max and sum with the reference)
 * and for testing the bounded barrier waits without faulting a GPU.
 */
#ifndef FA_TESTING_H_
#define FA_TESTING_H_

#ifdef __cplusplus
extern "C" {
#endif

/*
 * fa_fwd with instrumentation. Arguments up to `stream` are those of fa_fwd.
 *  inject:       0 = none; 1 = the TMA producer skips the V load of the first
 *                key tile, so the MMA warp's wait on it runs out (fp16/bf16
 *                kernel only). The kernel then records FA_ERR_DEVICE_TIMEOUT,
 *                drains its own copies and MMAs, frees TMEM and exits.
 *  stats_trace:  NULL, or a device array [B*H*N, ceil(N/128), 2] of fp32 that
 *                receives, after every key tile, the row's reference max in
 *                natural-log units and its running denominator (fp16/bf16 only).
 *  timeline:     NULL, or a device array [8, 16, 64] of uint64 receiving clock64
 *                stamps of pipeline events of the first 8 CTAs (fp16/bf16 only).
 *  wait_limit_cycles: > 0 overrides the barrier wait limit for this call.
 */
int fa_fwd_testing(const void *Q, const void *K, const void *V, void *O, float *LSE,
                   int B, int H, int N, int d, float scale, int dtype, void *stream,
                   int inject, float *stats_trace, unsigned long long *timeline,
                   long long wait_limit_cycles);

/* "Where" code of the first timeout recorded in the status word (0 = none;
 * not cleared by this call). */
unsigned int fa_testing_last_timeout_where(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_TESTING_H_ */
