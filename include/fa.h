/*
 * fa.h — C ABI of the GB300 (sm_103a) FlashAttention forward library.
 *
 * The operation (MUSA SDK programming guide, "FlashAttention 优化": the
 * standard attention formula under "计算流程", computed by the tiled
 * online-softmax algorithm under "FlashAttention 完整算法", formula steps 1-4):
 *
 *     for every batch b < B and head h < H, and query row i < N:
 *         s_ij   = scale * sum_k Q[b,h,i,k] * K[b,h,j,k]          (j < N)
 *         O[b,h,i,:] = sum_j softmax_j(s_i.) * V[b,h,j,:]
 *         LSE[b,h,i] = ln sum_j exp(s_ij)
 *
 * Non-causal, no mask. S and P are never written to memory. LSE is the
 * per-row logsumexp that a backward pass by recomputation needs (the Triton
 * page, "反向传播要不要自己写": keep the row statistics, recompute P).
 *
 * Ownership: the caller owns every buffer. The library allocates no device
 * memory per call; it keeps one process-lifetime device status word per GPU
 * (a __device__ variable of the module) and nothing else.
 *
 * Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 * fa_fwd only enqueues work and never synchronises.
 *
 * Devices: sm_103 (GB300) only; other devices get FA_ERR_ARCH.
 */
#ifndef FA_H_
#define FA_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of Q, K, V and O. */
typedef enum { FA_F32 = 0, FA_F16 = 1, FA_BF16 = 2 } fa_dtype;

/* Return codes. Every entry point returns one of these. */
typedef enum {
    FA_OK = 0,
    FA_ERR_NULL = 1,           /* a required pointer is NULL                         */
    FA_ERR_DTYPE = 2,          /* dtype is not one of fa_dtype                       */
    FA_ERR_SHAPE = 3,          /* B, H or N < 1, or B*H*N*d overflows 2^40 elements  */
    FA_ERR_HEADDIM = 4,        /* d is not 64 or 128 (or 256, 16-bit types only)     */
    FA_ERR_ALIGN = 5,          /* a base pointer is not 16-byte aligned              */
    FA_ERR_CUDA = 6,           /* a CUDA runtime/driver call failed (launch, query)  */
    FA_ERR_DEVICE_TIMEOUT = 7, /* a kernel gave up waiting on a pipeline barrier     */
    FA_ERR_ARCH = 8,           /* the current device is not sm_103                   */
    FA_ERR_SCALE = 9,          /* scale is not finite and > 0                        */
    FA_ERR_WORKSPACE = 10,     /* split-KV workspace NULL, misaligned or too small   */
    FA_ERR_SCRATCH_LIMIT = 11, /* shape needs more than the built-in scratch         */
    FA_ERR_UNSUPPORTED = 12,   /* the entry point does not take this dtype           */
    FA_ERR_DEVICE_SMEM = 13    /* a kernel found its shared memory misaligned        */
} fa_status;

/*
 * Forward pass.
 *
 * Q, K, V, O: device pointers to [B, H, N, d] row-major contiguous arrays of
 *             `dtype` (the last index d is contiguous, then N, then H, then B).
 *             O has the same dtype as Q. O must not alias Q, K or V.
 * LSE:        device pointer to a [B, H, N] contiguous fp32 array: natural-log
 *             logsumexp of each scaled score row, ln sum_j exp(scale * q_i.k_j).
 * d:          64 or 128; 256 for FA_F16 / FA_BF16 (a kernel with one 128-row Q
 *             tile per CTA and 64-key K/V tiles: the MUSA guide's block-size
 *             table shrinks the key block as d grows).
 * scale:      multiplies q.k before the softmax (1/sqrt(d) is the usual value);
 *             must be finite and > 0.
 * dtype:      FA_F32, FA_F16 or FA_BF16. For FA_F16/FA_BF16 both matrix
 *             products run on the tensor cores with fp32 accumulation and P is
 *             rounded to `dtype` before P.V; for FA_F32 they run as three
 *             TF32 products (hi*hi + hi*lo + lo*hi) with fp32 accumulation.
 * stream:     cudaStream_t to enqueue on.
 *
 * Errors: argument errors return before anything is enqueued (FA_ERR_NULL,
 * FA_ERR_DTYPE, FA_ERR_SHAPE, FA_ERR_HEADDIM, FA_ERR_ALIGN, FA_ERR_SCALE,
 * FA_ERR_ARCH). A failed launch returns FA_ERR_CUDA. A kernel that times out
 * on an internal barrier records FA_ERR_DEVICE_TIMEOUT in the device status
 * word, drains its own asynchronous copies, frees its tensor memory and
 * returns; read it with fa_get_device_status.
 */
int fa_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
           int B, int H, int N, int d, float scale, int dtype, void *stream);

/*
 * Masked forward pass. The Triton page masks scores with -inf where keys must
 * not be seen ("FlashAttention + Triton", section 4.3: boundary masks; section
 * 5.1: padded variable-length batches, where a row can be fully masked).
 *   causal:    0 or 1. 1: query row i sees keys j <= i only.
 *   seqlens_k: NULL, or a DEVICE array of B int32 key lengths: row i of batch
 *              b sees keys j < seqlens_k[b] only (values are clamped to
 *              [0, N]). Padded keys may hold anything (their scores are
 *              replaced by -inf); padded values must be finite (they are
 *              multiplied by zero weights).
 * A row with no key to see (seqlens_k[b] == 0) gets O = 0 and LSE = -inf.
 * Other arguments and errors: as fa_fwd (causal outside {0, 1}: FA_ERR_SHAPE).
 */
int fa_fwd_ex(const void *Q, const void *K, const void *V, void *O, float *LSE,
              int B, int H, int N, int d, float scale, int dtype,
              int causal, const int *seqlens_k, void *stream);

/*
 * Split-KV forward pass: the same result as fa_fwd, computed by splitting the
 * keys of every (batch, head) into `num_splits` contiguous ranges (whole K/V
 * tiles: multiples of 128 keys, of 64 at d = 256) that run as separate work
 * units, then merging the per-range
 * results with the block merge of the Triton page ("FlashAttention + Triton",
 * section 2.3: m_new = max(m_old, m_block), l and O rescaled by exp(m - m_new)),
 * written in LSE form: LSE = log sum_r exp(LSE_r), O = sum_r exp(LSE_r - LSE) O_r.
 * It raises the number of work units when B*H*ceil(N/q) (q = 256 Q rows per
 * unit; 128 at d = 256) is small against the number of SMs (long sequences,
 * few heads).
 *
 * Arguments up to `dtype` are those of fa_fwd.
 * num_splits: >= 1 explicit (ranges of whole K/V tiles, so at most
 *             ceil(N/128), ceil(N/64) at d = 256; a count that does not divide the tiles evenly
 *             gives ceil(tiles / ceil(tiles / num_splits)) ranges); 0 = chosen from the
 *             shape and the device's SM count (fa_fwd_splitkv_num_splits)
 *             by a cost model, which can also pick the tail plan: when the
 *             B*H*ceil(N/q) work units end in a partial last wave of SMs,
 *             the full waves run unsplit and only the last wave's units are
 *             split (as many ways as fit in one wave) and merged; that is
 *             three launches (full waves, split tail, merge of its rows).
 *             For unmasked d = 128 inputs with N a multiple of 256 and at
 *             most 4096 the automatic count may instead stream the tail: the persistent
 *             kernel runs the full rounds of Q blocks whole and cuts the K/V
 *             tiles of the units left over into one contiguous range per
 *             SM; units a range boundary cuts are computed in pieces and
 *             merged (two launches; fa_fwd_stream_plan).
 * workspace:  device memory owned by the caller, 256-byte aligned, at least
 *             fa_fwd_splitkv_workspace_size(...) bytes; holds the per-range
 *             fp32 O and LSE of the split rows only (all B*H*N rows, or under
 *             the tail plan the rows of the last wave's units). Unused (may be
 *             NULL) when the effective split count is 1, and for FA_F32
 *             inputs, which always run unsplit. Under the streamed tail it
 *             holds the pieces' fp32 O and LSE (two 256-row slots per SM
 *             that shares the tail); its size is then the larger of that
 *             and what the key-range plan of the same arguments needs, so
 *             that masked calls (fa_fwd_splitkv_ex, which always take the
 *             key-range plan) fit the same workspace.
 * Errors: those of fa_fwd, plus FA_ERR_WORKSPACE. Two or three launches are
 * enqueued on `stream` (fa_fwd_splitkv_launches); nothing is synchronised.
 */
int fa_fwd_splitkv(const void *Q, const void *K, const void *V, void *O, float *LSE,
                   int B, int H, int N, int d, float scale, int dtype,
                   int num_splits, void *workspace, unsigned long long workspace_bytes, void *stream);

/*
 * Masked split-KV forward pass: fa_fwd_ex's masks with fa_fwd_splitkv's key
 * ranges. This is the padded variable-length batch of the Triton page
 * ("FlashAttention + Triton", section 5.1), typically few heads with long
 * sequences, where splitting the keys gives the SMs enough work units. Each
 * (unit, key range) sees the keys of its range that the masks leave it; a
 * range it sees none of contributes O = 0, LSE = -inf and the merge ignores
 * it; a row that no range sees (seqlens_k[b] == 0) gets O = 0, LSE = -inf.
 *   causal, seqlens_k: as fa_fwd_ex (seqlens_k: NULL or a device int32 [B]).
 *   num_splits, workspace, workspace_bytes: as fa_fwd_splitkv; the plan and
 *              the workspace size do not depend on the masks
 *              (fa_fwd_splitkv_workspace_size applies).
 * Errors: those of fa_fwd_ex and fa_fwd_splitkv.
 */
int fa_fwd_splitkv_ex(const void *Q, const void *K, const void *V, void *O, float *LSE,
                      int B, int H, int N, int d, float scale, int dtype, int causal, const int *seqlens_k,
                      int num_splits, void *workspace, unsigned long long workspace_bytes, void *stream);

/* The effective split count fa_fwd_splitkv uses for num_splits = 0 on the
 * current device (>= 1: key ranges of each split unit after clamping to whole
 * K/V tiles; 1 = unsplit), or a negative fa_status on error. Under the
 * tail plan only the units of the last wave are split this many ways. */
int fa_fwd_splitkv_num_splits(int B, int H, int N, int d);

/* Kernel launches fa_fwd_splitkv enqueues for this shape and split count on
 * the current device, for FA_F16 / FA_BF16 inputs: 1 (unsplit), 2 (every
 * unit split, then the merge) or 3 (the tail plan: full waves, the split
 * tail, the merge of its rows); a negative fa_status on error. */
int fa_fwd_splitkv_launches(int B, int H, int N, int d, int num_splits);

/*
 * The split-KV plan fa_fwd_splitkv follows for FA_F16 / FA_BF16 inputs of
 * this shape on a device with `num_sms` SMs, computed on the host (no device
 * is touched; a caller can size workspaces for a device it has not opened).
 * With num_sms = the current device's SM count it agrees with
 * fa_fwd_splitkv_num_splits, fa_fwd_splitkv_launches and
 * fa_fwd_splitkv_workspace_size.
 *
 * Work units are the B*H*ceil(N/q) (batch*head, q-row Q block) pairs, q = 256
 * (128 at d = 256); K/V tiles hold 128 keys (64 at d = 256).
 * Outputs (all written on success):
 *   splits           key ranges of each split unit after clamping to whole
 *                    K/V tiles (1: nothing is split); under the streamed
 *                    tail the most pieces one unit is cut into;
 *   first_split_unit index of the first split unit: 0 when every unit is
 *                    split, B*H*ceil(N/q) when none is, in between under the
 *                    tail plan (the units of the last, partial wave of SMs)
 *                    and the streamed tail (its first unit);
 *   launches         kernel launches enqueued: 1, 2 or 3 (the streamed
 *                    tail: 2);
 *   workspace_bytes  the workspace fa_fwd_splitkv needs (0: none).
 * Errors: FA_ERR_NULL (an output pointer is NULL), FA_ERR_SHAPE (B, H, N or
 * num_sms < 1, num_splits < 0, B*H >= 2^31), FA_ERR_HEADDIM (d not 64, 128 or
 * 256).
 */
int fa_fwd_splitkv_plan(int B, int H, int N, int d, int num_splits, int num_sms, int *splits,
                        long long *first_split_unit, int *launches, unsigned long long *workspace_bytes);

/*
 * The streamed tail of fa_fwd_splitkv's automatic plan (num_splits = 0) for
 * unmasked FA_F16 / FA_BF16 inputs of this shape on a device with `num_sms`
 * SMs, computed on the host. The persistent d = 128 kernel hands out Q blocks
 * (units of 256 rows of one (b, h), numbered head by head) whole in rounds of
 * num_sms until `unit0`; the `tiles` K/V tiles (128 keys) of units unit0 ..
 * B*H*N/256 - 1, laid end to end, are then cut into `ctas` contiguous ranges,
 * range c = [floor(c * tiles / ctas), floor((c + 1) * tiles / ctas)) taken by
 * SM c. A unit that a range boundary cuts is computed in pieces, each written
 * as normalised fp32 O and LSE, and a merge pass combines them (the block
 * merge in LSE form, as fa_fwd_splitkv). The tail is streamed when the cost
 * model expects it to shorten the pass: the units then end in a partial last
 * round (B*H*N/256 not a multiple of num_sms) long enough to pay for the merge.
 * Outputs (all written on success): ctas = 0 when the plan does not stream
 * the tail (other d, N not a multiple of 256 or above 4096, or it does not
 * pay; unit0 = tiles = 0 then); else 1 <= ctas <= num_sms, unit0 a multiple of num_sms.
 * Errors: FA_ERR_NULL (an output pointer is NULL), FA_ERR_SHAPE (B, H, N or
 * num_sms < 1, B*H >= 2^31), FA_ERR_HEADDIM (d not 64, 128 or 256).
 */
int fa_fwd_stream_plan(int B, int H, int N, int d, int num_sms, int *unit0, int *tiles, int *ctas);

/* Workspace bytes fa_fwd_splitkv needs for this shape and split count on the
 * current device (num_splits = 0: the automatic plan, which depends on the
 * SM count); 0 when no workspace is needed or on error. */
unsigned long long fa_fwd_splitkv_workspace_size(int B, int H, int N, int d, int num_splits);

/*
 * fa_fwd_splitkv without a caller workspace, for callers that cannot allocate
 * device memory: code running under an allocation-free policy after start-up
 * (real-time or safety-certified pipelines, plugins that a host framework
 * forbids to call cudaMalloc, allocators that must not be re-entered), where a
 * cudaMalloc/cudaFree would also synchronise the device in the middle of the
 * work. The pages have no counterpart for it; it is a library addition.
 *
 * The per-range partial results live in a scratch array that is part of the
 * library itself (a __device__ array of FA_NOALLOC_SCRATCH_BYTES = 32 MiB,
 * present on every GPU that loads the library until the process exits). This
 * entry point calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments: as fa_fwd_splitkv, without workspace. Shapes whose split-KV
 * workspace (fa_fwd_splitkv_workspace_size for the effective split count)
 * exceeds the scratch size return FA_ERR_SCRATCH_LIMIT before anything is
 * enqueued; with an effective split count of 1 the scratch is not used.
 * The first call on each device looks up the scratch array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. All calls share the one array and it keeps the
 * last call's contents; nothing in it needs to start at zero (each call writes
 * every byte it reads). Calls that can overlap on the GPU (other streams,
 * other host threads) race on the array: serialise them, e.g. on one stream.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32ull << 20)
int fa_fwd_splitkv_noalloc(const void *Q, const void *K, const void *V, void *O, float *LSE,
                           int B, int H, int N, int d, float scale, int dtype,
                           int num_splits, void *stream);

/*
 * Backward pass by recomputation (the MUSA guide's fourth core principle,
 * "重计算（Recompute）换存储"; the Triton page, sections 2.4 and 4.4: the
 * forward pass keeps only O and the row statistics, the backward pass rebuilds
 * P from Q, K and them, then applies the chain rule). For every (b, h), with
 * s_ij = scale * q_i.k_j, P_ij = exp(s_ij - LSE_i) and D_i = sum_c dO_ic O_ic:
 *
 *     dV_j = sum_i P_ij dO_i
 *     dQ_i = scale * sum_j P_ij (dO_i.v_j - D_i) k_j
 *     dK_j = scale * sum_i P_ij (dO_i.v_j - D_i) q_i
 *
 * the gradients of sum(dO * O) for O = softmax(scale Q K^T) V (non-causal, no
 * mask). P and dS are never written to memory.
 *
 * Q, K, V, O, dO: device pointers to [B, H, N, d] contiguous arrays of
 *             `dtype`; O and LSE are fa_fwd's outputs for these Q, K, V and
 *             scale (LSE as fa_fwd writes it, [B, H, N] fp32).
 * dQ, dK, dV: device pointers to [B, H, N, d] arrays of `dtype` that receive
 *             the gradients; they must not alias any input.
 * dtype:      FA_F16 or FA_BF16 (FA_F32: FA_ERR_UNSUPPORTED). Products run on
 *             the tensor cores with fp32 accumulation; P and dS*scale are
 *             rounded to `dtype` before they enter a product; dQ is
 *             accumulated in fp32 and rounded once at the end.
 * d:          64, 128 or 256. At d = 256 the pass runs two main kernels (dV,
 *             then dK with the dQ contributions: dK and dV do not fit the
 *             tensor memory together) with 64-row Q tiles; S^T is computed
 *             in both.
 * workspace:  device memory owned by the caller, 256-byte aligned, at least
 *             fa_bwd_workspace_size(B, H, N, d) bytes: the fp32 dQ
 *             accumulator and two fp32 values per row. Its contents need not
 *             be initialised; they are overwritten.
 * Other arguments: as fa_fwd.
 * Errors: those of fa_fwd (checked before anything is enqueued), plus
 * FA_ERR_WORKSPACE and FA_ERR_UNSUPPORTED. Three launches are enqueued on
 * `stream` (row statistics, main pass, dQ rounding; four at d = 256);
 * nothing is synchronised.
 */
int fa_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *LSE,
           void *dQ, void *dK, void *dV, int B, int H, int N, int d, float scale, int dtype,
           void *workspace, unsigned long long workspace_bytes, void *stream);

/*
 * One part of attention over a key set split across parts (devices, for
 * context parallelism): all Nq queries against these Nk keys. The Triton
 * page's block merge (section 2.3) combines such parts exactly: each part
 * keeps its own normalised output and logsumexp, and fa_merge folds them.
 *   Q:        [B, H, Nq, d] device array, FA_F16 or FA_BF16.
 *   K, V:     [B, H, Nk, d] device arrays of the same dtype (this part's keys).
 *   O_part:   [B, H, Nq, d] fp32 device array (caller-owned): this part's
 *             softmax(scale Q K^T) V over its own keys.
 *   LSE_part: [B, H, Nq] fp32 device array: this part's row logsumexp.
 * No mask. Errors: as fa_fwd (FA_F32 -> FA_ERR_UNSUPPORTED; d must be 64, 128
 * or 256; Nq, Nk >= 1). One launch on `stream`; nothing is synchronised.
 */
int fa_fwd_partial(const void *Q, const void *K, const void *V, float *O_part, float *LSE_part,
                   int B, int H, int Nq, int Nk, int d, float scale, int dtype, void *stream);

/*
 * Merge of num_parts results over disjoint key sets (the Triton page, section
 * 2.3, in LSE form): LSE = m + ln sum_p exp(LSE_p - m) with m = max_p LSE_p,
 * O = sum_p exp(LSE_p - LSE) O_p, rounded to `dtype` once.
 *   O_parts:   [num_parts, B, H, N, d] fp32 device array (parts contiguous,
 *              16-byte aligned), e.g. gathered outputs of fa_fwd_partial.
 *   LSE_parts: [num_parts, B, H, N] fp32 device array.
 *   O:         [B, H, N, d] device array of `dtype` (FA_F16 or FA_BF16).
 *   LSE:       [B, H, N] fp32 device array.
 * A part with LSE = -inf contributes nothing; a row whose parts are all -inf
 * gets O = 0 and LSE = -inf. d must be 64, 128 or 256. Errors: as fa_fwd
 * (FA_F32 -> FA_ERR_UNSUPPORTED). One launch on `stream`.
 */
int fa_merge(const float *O_parts, const float *LSE_parts, int num_parts, void *O, float *LSE,
             int B, int H, int N, int d, int dtype, void *stream);

/* Workspace bytes fa_bwd needs for this shape (0 for invalid arguments). */
unsigned long long fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Masked backward pass: the gradients of the masked forward pass (fa_fwd_ex)
 * with the same masks. A masked score is -inf in the forward pass, so its
 * P_ij and dS_ij are exactly 0 ("FlashAttention + Triton", sections 4.3 and
 * 5.1, the masks; the backward of section 4.4 then sums over the seen keys
 * only): keys a row does not see add nothing to its dQ, keys no row sees
 * (j >= seqlens_k[b]) get dK = dV = 0, and a row with no key to see
 * (LSE = -inf) gets dQ = 0.
 *   causal:    0 or 1, as fa_fwd_ex. With 1, key tiles skip the query tiles
 *              before them, so the pass does about half the work.
 *   seqlens_k: NULL or a DEVICE array of B int32 key lengths, as fa_fwd_ex
 *              (clamped to [0, N]). Padded keys and values must be finite:
 *              both enter products with zero weights.
 * O and LSE must be the outputs of fa_fwd_ex with the same masks. Other
 * arguments, workspace and errors: as fa_bwd (causal outside {0, 1}:
 * FA_ERR_SHAPE).
 */
int fa_bwd_ex(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *LSE,
              void *dQ, void *dK, void *dV, int B, int H, int N, int d, float scale, int dtype, int causal,
              const int *seqlens_k, void *workspace, unsigned long long workspace_bytes, void *stream);

/*
 * Synchronises `stream`, then returns and clears the status word that kernels
 * of this library on the current device write when they give up on a wait:
 * FA_OK, FA_ERR_DEVICE_TIMEOUT, FA_ERR_DEVICE_SMEM (a kernel found its shared
 * memory misaligned and did no work), or FA_ERR_CUDA if the synchronisation or
 * the read failed.
 */
int fa_get_device_status(void *stream);

/* Static English text for a status code (never NULL). */
const char *fa_strerror(int status);

/* Library ABI version: 100 * major + minor. */
int fa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
