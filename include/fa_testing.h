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
 *  timeline:     NULL, or a device array [8, 32, 64] of uint64 receiving clock64
 *                stamps of pipeline events of the first 8 CTAs (fp16/bf16 only).
 *  wait_limit_cycles: > 0 overrides the barrier wait limit for this call.
 */
int fa_fwd_testing(const void *Q, const void *K, const void *V, void *O, float *LSE,
                   int B, int H, int N, int d, float scale, int dtype, void *stream,
                   int inject, float *stats_trace, unsigned long long *timeline,
                   long long wait_limit_cycles);

/*
 * fa_bwd with instrumentation. Arguments up to `stream` are those of fa_bwd.
 *  inject:       0 = none; 1 = the TMA producer skips the dO load of the first
 *                Q tile, so the MMA warp's wait on it runs out; the kernel then
 *                records FA_ERR_DEVICE_TIMEOUT, drains, frees TMEM and exits.
 *  timeline:     NULL, or a device array [8, 32, 64] of uint64 receiving clock64
 *                stamps of pipeline events of the first 8 CTAs of the main kernel.
 *  wait_limit_cycles: > 0 overrides the barrier wait limit for this call.
 */
int fa_bwd_testing(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *LSE,
                   void *dQ, void *dK, void *dV, int B, int H, int N, int d, float scale, int dtype,
                   void *workspace, unsigned long long workspace_bytes, void *stream,
                   int inject, unsigned long long *timeline, long long wait_limit_cycles);

/*
 * fa_fwd with the two test-only controls the parity gates need. Arguments up
 * to `stream` are those of fa_fwd (fp16/bf16 only for the first control).
 *  O_f32:  NULL, or a device fp32 array [B,H,N,d] (16-byte aligned) that
 *          receives O normalised by l but NOT rounded to the input type; O is
 *          then not written and may be NULL. This isolates the fp32
 *          accumulation (S, P.V, l) from the rounding of the stored output,
 *          which for bf16 outputs of |O| ~ 4 alone exceeds 1e-2 (the accuracy
 *          threshold of the dataflow page, section 4.1). fp16/bf16 and no
 *          mask, unsplit; otherwise FA_ERR_UNSUPPORTED.
 *  rescale_threshold_log2: the lazy-rescale threshold in log2 units; < 0
 *          takes the built-in 15; 0 rescales O whenever a row's max grows
 *          (the dataflow page, section 2.3). Must lie in [0, 64] otherwise
 *          (FA_ERR_SCALE). Ignored by fp32 inputs, whose rescale is eager.
 *  stats_trace: as in fa_fwd_testing (NULL for none).
 * Errors: those of fa_fwd, returned before any launch.
 */
int fa_fwd_debug(const void *Q, const void *K, const void *V, void *O, float *LSE,
                 int B, int H, int N, int d, float scale, int dtype, void *stream,
                 float *O_f32, float rescale_threshold_log2, float *stats_trace);

/*
 * on != 0: every entry point of this library returns FA_OK after its argument
 * and device checks, before anything is enqueued (0 restores normal calls).
 * Lets argument-error tests pass placeholder addresses safely: a validation
 * check that regressed shows up as FA_OK instead of the expected error code,
 * never as a kernel launched on memory that does not exist.
 */
void fa_testing_set_dry_run(int on);

/* "Where" code of the first timeout recorded in the status word (0 = none;
 * not cleared by this call). */
unsigned int fa_testing_last_timeout_where(void);

/*
 * The streamed tail's partition as the persistent kernel walks it (host
 * copy of the device arithmetic, see fa_fwd_stream_plan): piece q (0 = the
 * one holding the range's first tile) of range c among `ctas` over `tiles`
 * tail tiles of n tiles per unit. Returns 1 and out[0..3] = (tail unit,
 * first tile, end tile, part slot; slot -1 = whole unit), or 0 when the
 * range has no piece q. With q = -1 it returns 1 and out[0..1] = (c_lo,
 * c_hi), the ranges that hold tiles of tail unit c (the merge's view).
 * Requires tiles >= 1, 1 <= ctas, tiles * ctas < 2^31, n >= 1; returns -1
 * for arguments outside that (out untouched).
 */
int fa_testing_stream_piece(int tiles, int ctas, int n, int c, int q, int *out);

/*
 * The key tile CTA `cta` of the backward's main kernels takes (host copy of
 * the device arithmetic): out[0] = b*h, out[1] = key tile (128 keys each at
 * every d). Without the causal mask a head's
 * key tiles come in a row; with it, longest first within windows of heads
 * whose Q, dO and fp32 dQ accumulator (8 N d bytes per head) fit 64 MiB.
 * Requires B, H, N >= 1, d in {64, 128, 256}, 0 <= cta < B*H*ceil(N/128)
 * < 2^31; returns 1, or -1 for arguments outside that (out untouched).
 */
int fa_testing_bwd_tile(int B, int H, int N, int d, int causal, int cta, int *out);

/*
 * The work unit the one-CTA-per-unit forward kernels give unit number `unit`
 * of an unsplit launch over every unit (host copy of the device arithmetic):
 * out[0] = b*h, out[1] = Q block (256 rows at d = 64 / 128, 128 at d = 256).
 * Unmasked, a head's Q blocks come in a row; causal, longest first within
 * windows of heads whose K and V (4 N d bytes per head) fit 64 MiB, or,
 * when every unit fits on the device's num_sms SMs at once (num_sms > 0),
 * longest first within each head. Requires B, H, N >= 1, d in {64, 128,
 * 256}, num_sms >= 0, 0 <= unit < B*H*(Q blocks) < 2^31; returns 1, or -1
 * for arguments outside that (out untouched).
 */
int fa_testing_fwd_unit(int B, int H, int N, int d, int causal, int num_sms, int unit, int *out);

#ifdef __cplusplus
}
#endif

#endif /* FA_TESTING_H_ */
