/*
 * moe.h -- C ABI of libmoe.so, a GB300 (sm_103a) MoE expert layer.
 *
 * The layer, as the sources describe it:
 *   - "Mixture of Experts in transformers", MoE basics: a router picks k of
 *     the E experts for every token; "pluggable expert backends": the
 *     grouped_mm backend sorts tokens by expert id and runs one grouped GEMM;
 *   - "Hugging Face Transformers: MoE and FP8 kernel optimisation"
 *     (transformers PR #45621), section 1: fine-grained FP8 entries
 *     (fp8_act_quant / per_token_cast_to_fp8, grouped_fp8_matmul); section 2:
 *     sentinel slots are excluded from the expert histogram (sorted last)
 *     instead of being clamped onto the last expert, and offsets[-1] is the
 *     number of live rows; section 3: outputs of sentinel rows must be
 *     written, not left uninitialised;
 *   - "LlamaFactory Triton fused MoE kernel" (LlamaFactory PR #10481),
 *     section 1: moe_scatter -> group_gemm_same_nk (fc1) -> silu(gate) * up
 *     -> group_gemm_same_nk (fc2) -> moe_gather.
 *
 * Notation: T tokens, E experts, k picks per token, H hidden size, I expert
 * intermediate size, R = T*k routed slots.  A slot is the flat index
 * f = t*k + j.  The sentinel expert id is E.  L = offsets[E] live rows.
 * bf16 tensors are passed as raw 16-bit storage (void*), e4m3 (OCP FP8
 * E4M3FN) tensors as uint8_t*.
 *
 * Conventions for every entry point:
 *   - Ownership: every pointer is caller-owned.  Unless stated otherwise a
 *     pointer is DEVICE memory (or managed memory) of the current device and
 *     must be 16-byte aligned; row-major layouts are dense (no padding).
 *   - Asynchrony: work is enqueued on `stream` (NULL = legacy default
 *     stream); the functions do not synchronise, allocate or free device
 *     memory, except moe_get_device_error (which synchronises the stream) and
 *     moe_forward with MOE_FWD_HOST_IO (which enqueues host<->device copies).
 *   - Devices: the library looks up, once per device, the device addresses
 *     of its own device variables (the error word below, and the static
 *     array of moe_route_sort_noalloc) and keeps them for the life of the
 *     process; a cudaDeviceReset of a device makes them stale.
 *   - Errors: host-side argument checks run before any launch and return
 *     MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_WORKSPACE with
 *     nothing enqueued; a failed launch returns MOE_ERR_CUDA.  Conditions
 *     that only the device can see (an offsets array that is not a monotone
 *     prefix starting at 0 and ending at or below M_cap, or a pipeline wait
 *     that ran out of time) make the kernel skip the unsafe work and record a
 *     code in a per-device error word, read and cleared by
 *     moe_get_device_error.  There is no CPU fallback.
 *   - Determinism: every result is bit-reproducible from run to run (no
 *     floating-point atomics; fixed reduction orders).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1

typedef struct CUstream_st* moe_stream_t; /* the same handle as cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* a NULL/misaligned pointer or an out-of-range size */
    MOE_ERR_UNSUPPORTED = 2,  /* a valid request this build does not implement */
    MOE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
    MOE_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    MOE_ERR_DEVICE_CHECK = 5, /* (moe_get_device_error) a kernel rejected its device-side input */
    MOE_ERR_TIMEOUT = 6       /* (moe_get_device_error) a pipeline wait gave up */
} moe_status_t;

/* device error codes, as returned by moe_get_device_error */
#define MOE_DEVERR_NONE 0
#define MOE_DEVERR_OFFSETS 1 /* offsets[0] != 0, decreasing, or offsets[E] > M_cap */
#define MOE_DEVERR_TIMEOUT 2 /* an mbarrier wait inside a GEMM exceeded its time limit */
#define MOE_DEVERR_ROUTE 3   /* an expert id outside [0, E] reached the sort */

typedef enum {
    MOE_BF16 = 0,          /* bf16 operands, fp32 accumulation */
    MOE_FP8_E4M3_B128 = 1  /* e4m3 operands; activations scaled per row per 128
                              columns, weights per 128x128 block; fp32 scales */
} moe_dtype_t;

typedef enum {
    MOE_EPI_STORE = 0,            /* C = A*B^T, stored bf16 [M_cap, N] */
    MOE_EPI_SWIGLU = 1,           /* h = silu(C[:, :N/2]) * C[:, N/2:], bf16 [M_cap, N/2] */
    MOE_EPI_SWIGLU_QUANT_FP8 = 2  /* h rounded to bf16, then quantised like
                                     moe_act_quant_fp8: e4m3 [M_cap, N/2] plus
                                     scales [N/256, M_cap] */
} moe_epilogue_t;

int moe_abi_version(void);
const char* moe_status_string(moe_status_t status);

/*
 * moe_get_device_error: synchronise `stream`, then read and clear the error
 * word of the current device.  *code receives a MOE_DEVERR_* value.  Returns
 * MOE_OK when the word was clear, MOE_ERR_DEVICE_CHECK or MOE_ERR_TIMEOUT
 * when it was set, MOE_ERR_CUDA if the synchronisation failed.
 */
moe_status_t moe_get_device_error(int32_t* code /* host */, moe_stream_t stream);

/*
 * moe_selftest_wait_timeout: diagnostic of the failure path.  Launches one
 * thread that waits on an mbarrier nothing ever arrives on, bounded by
 * limit_ns (1 ns .. 2 s) exactly like the waits inside the GEMM pipeline; the
 * wait gives up and records MOE_DEVERR_TIMEOUT in the device error word, and
 * the context stays usable.  Returns MOE_ERR_INVALID_ARG for a limit outside
 * the range.
 */
moe_status_t moe_selftest_wait_timeout(uint64_t limit_ns, moe_stream_t stream);

/*
 * moe_route_sort -- top-k routing, sentinel marking and the stable sort by
 * expert id ("MoE basics" and "pluggable expert backends" of "Mixture of
 * Experts in transformers"; section 2 of the transformers MoE/FP8 write-up).
 *
 * logits       fp32 [T, E] or NULL.  When given, l' = logits + expert_bias
 *              (one fp32 add per element, none without a bias) picks the k
 *              largest l' per token, ties to the lower expert id, slot j = the
 *              j-th pick, and topk_w[t, j] = softmax over the k picks
 *              (renormalize != 0) or the full softmax over E evaluated at the
 *              pick (renormalize == 0).  topk_ids/topk_w are then outputs.
 *              -0 and +0 tie.  A NaN l' is never picked: a token with fewer
 *              than k other values gets an invalid pick, which is recorded as
 *              MOE_DEVERR_ROUTE, written to topk_ids as E and sorted as a
 *              sentinel.
 *              When NULL, topk_ids is an input (ids in [0, E]; E = sentinel)
 *              and topk_w is not touched (may be NULL).  An input id outside
 *              [0, E] is recorded as MOE_DEVERR_ROUTE and overwritten with E
 *              (so the sort, moe_combine and topk_ids agree that the slot is
 *              a sentinel).
 * expert_bias  fp32 [E] or NULL.
 * sentinel_mask uint8 [T*k] or NULL: slots with a nonzero byte get id E.
 * topk_ids     int32 [T, k].   topk_w  fp32 [T, k].
 * sorted_rows  int32 [R] out: the slots ordered by (id, slot); sentinels last.
 * row_pos      int32 [R] out: inverse of sorted_rows.
 * offsets      int32 [E+1] out: offsets[0] = 0, offsets[e+1] - offsets[e] =
 *              number of slots with id e; the sentinel bin is left out, so
 *              offsets[E] = L.
 * ws           device scratch of moe_route_sort_workspace_size(T, E, k) bytes.
 * Limits: 1 <= E <= 256, 1 <= k <= min(E, 32), T >= 1, T*k < 2^31.
 */
size_t moe_route_sort_workspace_size(int T, int E, int k);
moe_status_t moe_route_sort(const float* logits, const float* expert_bias,
                            const uint8_t* sentinel_mask, int32_t* topk_ids, float* topk_w,
                            int T, int E, int k, int renormalize, int32_t* sorted_rows,
                            int32_t* row_pos, int32_t* offsets, void* ws, size_t ws_bytes,
                            moe_stream_t stream);

/*
 * moe_route_sort_noalloc -- moe_route_sort without caller workspace.  The
 * sources have no counterpart: this entry point exists for callers that
 * cannot allocate device memory themselves, such as a plug-in running inside
 * a serving engine that reserves and owns the whole device memory pool, or a
 * latency-critical path where an allocation call (which may synchronise the
 * device) is not allowed.
 *
 * Same arguments, results and limits as moe_route_sort, minus ws/ws_bytes.
 * The per-sort-block histogram lives in a static device array of 256 KiB
 * inside libmoe.so (present on every GPU that loads the library, until the
 * process exits).  It holds blocks * (E + 1) 32-bit counters, where
 * blocks = ceil(T / floor(1024 / k)); a request that needs more returns
 * MOE_ERR_WORKSPACE with nothing enqueued (for example E = 256 allows up to
 * 255 blocks, about 261 thousand slots at k = 8).
 * The call allocates and frees nothing.  On its first call on a device that
 * uses the array it looks up the array's device address (cudaGetSymbolAddress,
 * with that device current); make that first call before any stream capture.
 * The address is kept for the life of the process: a cudaDeviceReset of that
 * device makes it stale, so do not reset a device this library has run on.
 * Small batches, which one CTA routes and sorts in shared memory, do not use
 * the array (nor the size limit above): those with T*k <= 1024 and
 * ceil(T/32) * v <= 4, where v = 1, 2 or 4 for E up to 32, 64 or 128.  A
 * batch with E > 128 always uses the array.  Each call clears the counters it
 * uses on `stream` before use.  All calls share the one array: calls whose
 * work overlaps on the GPU (different streams without ordering between them)
 * race on it and give wrong results.
 */
moe_status_t moe_route_sort_noalloc(const float* logits, const float* expert_bias,
                                    const uint8_t* sentinel_mask, int32_t* topk_ids,
                                    float* topk_w, int T, int E, int k, int renormalize,
                                    int32_t* sorted_rows, int32_t* row_pos, int32_t* offsets,
                                    moe_stream_t stream);

/*
 * moe_ep_local_ids -- the router side of expert parallelism ("Mixture of
 * Experts in transformers", section on expert parallelism: the stacked
 * expert weights are sharded on their first dimension, and the router's
 * global expert ids are remapped to each rank's local ids, the picks of other
 * ranks' experts being masked; the ranks' partial outputs are then summed by
 * an all-reduce).  For the rank holding global experts [first_expert,
 * first_expert + E_local):
 *   local_ids[f] = topk_ids[f] - first_expert  if that expert is local,
 *                  E_local (the local sentinel) otherwise,
 * for every slot f < T*k.  The global sentinel E_global maps to E_local; an id
 * outside [0, E_global] is recorded as MOE_DEVERR_ROUTE and maps to E_local.
 * local_ids then feeds moe_route_sort (logits NULL, E = E_local) or
 * moe_forward (logits NULL, topk_ids = local_ids, topk_w = the global
 * weights, the rank's own W1/W2 slices, E = E_local); summing the ranks'
 * outputs gives the unsharded layer (the combine is linear in the experts).
 * topk_ids and local_ids int32 [T, k] (device; they may be the same buffer).
 * Limits: 1 <= E_global <= 256, E_local >= 1, 0 <= first_expert,
 * first_expert + E_local <= E_global, T*k < 2^31.
 */
moe_status_t moe_ep_local_ids(const int32_t* topk_ids, int T, int k, int E_global, int first_expert,
                              int E_local, int32_t* local_ids, moe_stream_t stream);

/*
 * moe_act_quant_fp8 -- per-token activation quantisation (fp8_act_quant /
 * per_token_cast_to_fp8 of section 1 of the transformers MoE/FP8 write-up).
 * For row m and 128-column group g: s = amax(|x[m, g*128 : g*128+128]|) / 448
 * (fp32, IEEE division; 1.0 when the group is all zeros) and
 * q = e4m3_rn_satfinite(x / s) (IEEE fp32 division, then one rounding to
 * nearest-even e4m3, saturating at +-448).
 * x bf16 [M, K]; q uint8 [M, K]; scales fp32 [M, K/128] (row-major).
 * Limits: M >= 1, K a positive multiple of 128.
 * These scales are token-major, while moe_grouped_gemm reads its A scales
 * group-major ([K/128, M_cap]): quantised tokens reach the GEMM through
 * moe_permute, which moves each row's scales into that layout.
 */
moe_status_t moe_act_quant_fp8(const void* x, int M, int K, uint8_t* q, float* scales,
                               moe_stream_t stream);

/*
 * moe_weight_quant_fp8 -- offline weight preparation for the FP8 layer: e4m3
 * weights with one fp32 scale per 128x128 block (the fine-grained FP8 weight
 * format of section 1 of the transformers MoE/FP8 write-up).  Same scale and
 * rounding rule as moe_act_quant_fp8, over blocks.
 * w bf16 [E, N, K]; q uint8 [E, N, K]; scales fp32 [E, ceil(N/128), K/128].
 * Limits: E, N >= 1, K a positive multiple of 128.
 */
moe_status_t moe_weight_quant_fp8(const void* w, int E, int N, int K, uint8_t* q, float* scales,
                                  moe_stream_t stream);

/*
 * moe_permute -- scatter of token rows into expert order (moe_scatter of
 * the LlamaFactory write-up): xp[p] = x[sorted_rows[p] / k] for p < L =
 * offsets[E]; rows p >= L are not written.
 * MOE_BF16: x bf16 [T, H], xp bf16 [M_cap, H]; scales unused (NULL).
 * MOE_FP8_E4M3_B128: x uint8 [T, H] with x_scales fp32 [T, H/128] (as written
 *   by moe_act_quant_fp8); xp uint8 [M_cap, H] and xp_scales fp32
 *   [H/128, M_cap] -- group-major, so that a GEMM reads the scales of
 *   consecutive rows contiguously.
 * offsets int32 [E+1] as written by moe_route_sort (read on the device only).
 * Limits: H a positive multiple of 8 (bf16) or 128 (FP8); R = T*k <= M_cap.
 */
moe_status_t moe_permute(moe_dtype_t dtype, const void* x, const float* x_scales, int T, int H,
                         int k, const int32_t* sorted_rows, const int32_t* offsets, int E,
                         int M_cap, void* xp, float* xp_scales, moe_stream_t stream);

/*
 * moe_grouped_gemm -- one GEMM per expert over its rows of the permuted
 * buffer (group_gemm_same_nk of the LlamaFactory write-up, grouped_fp8_matmul
 * of the transformers MoE/FP8 write-up).  For every expert e and row p in
 * [offsets[e], offsets[e+1]):  C[p, n] = sum_c A[p, c] * B[e, n, c].
 * Rows p >= offsets[E] (sentinel rows) are written as zeros (bf16 0; for the
 * quantising epilogue q = 0 and scale 1.0) and never read for arithmetic.
 * The tile schedule is derived on the device from offsets; no tile is issued
 * for sentinel rows.
 *
 * A        bf16 [M_cap, K], or e4m3 [M_cap, K] with A_scales fp32 [K/128, M_cap]
 * B        bf16 [E, N, K], or e4m3 [E, N, K] with B_scales fp32 [E, ceil(N/128), K/128]
 *          (B_scales need only be 4-byte aligned, so that a run of experts
 *          sliced out of a larger stack can be passed as it is)
 * offsets  int32 [E+1] (device).
 * epilogue MOE_EPI_STORE:  C bf16 [M_cap, N]
 *          MOE_EPI_SWIGLU: rows [0, N/2) of B[e] are the gate, [N/2, N) the
 *            up projection; C = h bf16 [M_cap, N/2]
 *          MOE_EPI_SWIGLU_QUANT_FP8 (FP8 only): C = e4m3 [M_cap, N/2],
 *            C_scales fp32 [N/256, M_cap]
 * Limits: 1 <= E <= 256; K a multiple of 8 (bf16) or 128 (FP8); N a multiple
 *   of 8 (STORE) or of 16 (SWIGLU, so that N/2 is a multiple of 8); FP8 also
 *   needs N (STORE) or N/2 (SWIGLU) a multiple of 128.
 */
moe_status_t moe_grouped_gemm(moe_dtype_t dtype, const void* A, const float* A_scales,
                              const void* B, const float* B_scales, const int32_t* offsets,
                              int E, int M_cap, int N, int K, moe_epilogue_t epilogue, void* C,
                              float* C_scales, moe_stream_t stream);

/*
 * moe_grouped_gemm_gather -- moe_grouped_gemm with the scatter of the
 * LlamaFactory write-up (section 1) folded into the A operand: row p of A is
 * x[sorted_rows[p] / k], read straight from token order, so no permuted copy
 * of the activations is written.  Same arithmetic, tile order and results as
 * moe_permute followed by moe_grouped_gemm, bit for bit.
 *
 * x            bf16 [T, K], or e4m3 [T, K] with x_scales fp32 [T, K/128]
 *              (row-major, as moe_act_quant_fp8 writes them)
 * sorted_rows  int32 [T*k] as written by moe_route_sort (device)
 * B, B_scales, offsets, E, M_cap, N, K, epilogue, C, C_scales: as in
 *              moe_grouped_gemm (C has M_cap rows in permuted order).
 * Limits: those of moe_grouped_gemm, plus K * element size a multiple of 128
 *   bytes (MOE_ERR_UNSUPPORTED otherwise: rows are fetched in whole 128-byte
 *   k-blocks), offsets[E] <= T*k (checked on the device: MOE_DEVERR_OFFSETS,
 *   nothing is computed) and every sorted_rows[p], p < offsets[E], in [0, T*k)
 *   (MOE_DEVERR_ROUTE; that row of C is not meaningful, the others are
 *   unaffected).
 */
moe_status_t moe_grouped_gemm_gather(moe_dtype_t dtype, const void* x, const float* x_scales, int T,
                                     int k, const int32_t* sorted_rows, const void* B,
                                     const float* B_scales, const int32_t* offsets, int E,
                                     int M_cap, int N, int K, moe_epilogue_t epilogue, void* C,
                                     float* C_scales, moe_stream_t stream);

/*
 * moe_grouped_gemm_combine -- the down grouped GEMM with the weighted combine
 * folded into its epilogue (the fused pipeline of section 1 of the
 * LlamaFactory write-up: group_gemm_same_nk (fc2) -> moe_gather), bf16 only.
 * Computes Y2 = moe_grouped_gemm(h, W2, MOE_EPI_STORE) and, in the same
 * kernel, out = moe_combine(Y2, topk_ids, topk_w, row_pos) -- bit for bit the
 * two-call results.  After a CTA has stored its rows of a tile, each row's
 * token bumps a counter per (token, 128-feature block); the CTA that stores
 * the last of a token's live slots for a block sums that token's rows of the
 * block, in slot order, with moe_combine's arithmetic.  Tokens whose slots
 * are all sentinels get zero rows.  Y2 is still written (its rows are the
 * inputs of the sums); only the separate combine launch is saved.
 * h bf16 [M_cap, I]; W2 bf16 [E, H, I]; offsets [E+1]; topk_ids int32 [T, k]
 * and topk_w fp32 [T, k] as given to moe_combine; sorted_rows, row_pos int32
 * [T*k] from moe_route_sort; Y2 bf16 [M_cap, H]; out bf16 [T, H];
 * ws: moe_grouped_gemm_combine_workspace_size(T, H) bytes of counters,
 * cleared by the call.  Limits: those of moe_grouped_gemm (bf16, store) and
 * moe_combine; T*k <= M_cap.
 */
size_t moe_grouped_gemm_combine_workspace_size(int T, int H);
moe_status_t moe_grouped_gemm_combine(const void* h, const void* W2, const int32_t* offsets, int E, int M_cap,
                                      int H, int I, const int32_t* topk_ids, const float* topk_w,
                                      const int32_t* sorted_rows, const int32_t* row_pos, int T, int k, void* Y2,
                                      void* out, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Gradients of the bf16 grouped GEMM C[p, n] = sum_c A[p, c] * B[e, n, c]
 * (rows p of expert e; moe_grouped_gemm with MOE_EPI_STORE), for training
 * ("Mixture of Experts in transformers": MoE training on grouped GEMMs;
 * section 3 of the transformers MoE/FP8 write-up: the gradients of sentinel
 * rows must be written, as zeros, not left uninitialised).  bf16 in and out,
 * fp32 accumulation; offsets as in moe_grouped_gemm (device).  No host
 * synchronisation.
 *
 * moe_grouped_gemm_dgrad:  dA[p, c] = sum_n dC[p, n] * B[e, n, c] for p <
 *   offsets[E]; rows p >= offsets[E] of dA are zeros (dC's are never read).
 *   dC bf16 [M_cap, N]; B bf16 [E, N, K]; dA bf16 [M_cap, K].  B is read in
 *   place (its K features contiguous, an MN-major operand of the tensor
 *   cores): moe_grouped_gemm_dgrad_workspace_size returns 0 and ws may be
 *   NULL.
 * moe_grouped_gemm_wgrad:  dB[e, n, c] = sum over p in [offsets[e],
 *   offsets[e+1]) of dC[p, n] * A[p, c]; an expert without rows gets zeros;
 *   rows p >= offsets[E] of A and dC are never read.
 *   A bf16 [M_cap, K]; dC bf16 [M_cap, N]; dB bf16 [E, N, K].
 *   A and dC are read in place.  Workspace:
 *   moe_grouped_gemm_wgrad_workspace_size(E, M_cap, N, K) bytes, 128 (N + K) E:
 *   each expert's last cnt mod 64 rows of dC and A, zero-padded to 64 rows.
 * Limits: 1 <= E <= 256, N and K positive multiples of 8; offsets not a
 *   monotone prefix from 0 to at most M_cap: MOE_DEVERR_OFFSETS, nothing
 *   computed.  Missing or small workspace: MOE_ERR_WORKSPACE.
 */
size_t moe_grouped_gemm_dgrad_workspace_size(int E, int N, int K);
moe_status_t moe_grouped_gemm_dgrad(const void* dC, const void* B, const int32_t* offsets, int E,
                                    int M_cap, int N, int K, void* dA, void* ws, size_t ws_bytes,
                                    moe_stream_t stream);
size_t moe_grouped_gemm_wgrad_workspace_size(int E, int M_cap, int N, int K);
moe_status_t moe_grouped_gemm_wgrad(const void* A, const void* dC, const int32_t* offsets, int E,
                                    int M_cap, int N, int K, void* dB, void* ws, size_t ws_bytes,
                                    moe_stream_t stream);

/*
 * moe_batched_matmul -- the batched expert backend ("Mixture of Experts in
 * transformers", pluggable expert backends: batched_mm; batched_fp8_matmul
 * in section 1 of the transformers MoE/FP8 write-up): every routed (token,
 * expert) product on its own, without weighting or a sum over the picks:
 *   out[t*k + j, n] = sum_c x[t, c] * W[e, n, c],   e = topk_ids[t, j] < E,
 * with fp32 accumulation (FP8: the block-scaled sum of moe_grouped_gemm),
 * stored bf16; a sentinel slot (id E) gets a zero row.  Computed by sorting
 * the slots by expert and running one grouped GEMM (each expert's weights
 * are read once per call), then gathering the product rows back into slot
 * order; the results equal moe_permute + moe_grouped_gemm's rows bit for bit.
 * x        bf16 [T, K], or e4m3 [T, K] with x_scales fp32 [T, K/128]
 *          (row-major, as moe_act_quant_fp8 writes them)
 * topk_ids int32 [T, k] (device; read only -- an id outside [0, E] is
 *          recorded as MOE_DEVERR_ROUTE and its row is zero)
 * W        bf16 [E, N, K], or e4m3 with W_scales fp32 [E, N/128, K/128]
 * out      bf16 [T*k, N]
 * ws       moe_batched_matmul_workspace_size(dtype, T, K, k, E, N) bytes
 * Limits: 1 <= E <= 256, 1 <= k <= min(E, 32), T*k < 2^31; bf16: N, K
 *   multiples of 8; FP8: N and K multiples of 128.
 */
size_t moe_batched_matmul_workspace_size(moe_dtype_t dtype, int T, int K, int k, int E, int N);
moe_status_t moe_batched_matmul(moe_dtype_t dtype, const void* x, const float* x_scales, int T, int K,
                                const int32_t* topk_ids, int k, const void* W, const float* W_scales, int E,
                                int N, void* out, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_swiglu -- standalone silu(gate) * up (LlamaFactory write-up, section
 * 1): h[p, n] = g / (1 + exp(-g)) * Y1[p, I + n] with g = Y1[p, n], for
 * p < offsets[E]; rows p >= offsets[E] of h are written as zeros.
 * Y1 bf16 [M_cap, 2I]; h bf16 [M_cap, I].  Limits: I a multiple of 8.
 */
moe_status_t moe_swiglu(const void* Y1, const int32_t* offsets, int E, int M_cap, int I, void* h,
                        moe_stream_t stream);

/*
 * moe_combine -- routing-weighted gather back to token order (moe_gather of
 * the LlamaFactory write-up; the partial-output sum of expert parallelism in
 * "Mixture of Experts in transformers"):
 *   out[t, :] = sum over j = 0..k-1 with topk_ids[t, j] != E of
 *               topk_w[t, j] * Y2[row_pos[t*k + j], :]
 * accumulated in fp32 in j order, stored bf16.  A token whose slots are all
 * sentinels gets a zero row.
 * Y2 bf16 [M_cap, H]; topk_ids int32 [T, k]; topk_w fp32 [T, k];
 * row_pos int32 [T*k]; out bf16 [T, H].  Limits: H a multiple of 8.
 */
moe_status_t moe_combine(const void* Y2, const int32_t* topk_ids, const float* topk_w,
                         const int32_t* row_pos, int T, int k, int H, int E, void* out,
                         moe_stream_t stream);

/* moe_forward flags */
#define MOE_FWD_HOST_IO 1u /* x, logits and out are HOST pointers (pinned memory
                              recommended).  x and logits are staged through
                              the workspace with cudaMemcpyAsync: x on a
                              second stream owned by the library (one per
                              device, created on the first such call), so the
                              routing on `stream` overlaps its copy; `stream`
                              waits for it before x is read.  A pinned `out`
                              is written in place by the combine kernel
                              (unless MOE_FWD_STAGED_OUT); pageable `out`
                              gets a staged copy back.  The
                              results equal the device-buffer call's bit for
                              bit.  The kernels of host-I/O calls on one
                              device run in call order: each call's first
                              kernel waits for the previous call's last one,
                              even on another stream (its copies do not), so a
                              caller alternating two streams overlaps one
                              batch's copies with its neighbours' kernels
                              without those kernels sharing the SMs.  Calls
                              made under stream capture take the library's
                              copy stream into the capture and are not
                              chained. */
#define MOE_FWD_GATHER 2u  /* fold the scatter into the gate_up GEMM
                              (moe_grouped_gemm_gather instead of moe_permute
                              + moe_grouped_gemm): same results, bit for bit,
                              and no permuted copy of x (R*H*element-size
                              bytes less workspace), but slower on GB300 (the
                              GEMM fetches its rows four at a time, for every
                              column tile).  Ignored when H * element size is
                              not a multiple of 128. */
#define MOE_FWD_FUSED_COMBINE 4u /* bf16: fold the weighted combine into the
                              down GEMM (moe_grouped_gemm_combine instead of
                              moe_grouped_gemm + moe_combine): same results,
                              bit for bit.  Ignored for FP8. */
#define MOE_FWD_STAGED_OUT 8u /* with MOE_FWD_HOST_IO: a pinned `out` is
                              also written through the workspace and copied
                              back with cudaMemcpyAsync on `stream` (the copy
                              engine instead of the combine kernel writing
                              host memory over the host link).  Slower for a
                              single call; faster for callers that overlap
                              batches on several streams, where the kernel
                              writing host memory would hold SMs the other
                              batch's kernels need.  Same results, bit for
                              bit.  Ignored without MOE_FWD_HOST_IO. */

/*
 * moe_forward -- the whole expert layer on one stream, in the order of the
 * LlamaFactory pipeline: route + sort, [quantise x], permute, grouped GEMM
 * gate_up with the SwiGLU (and, for FP8, the quantisation of h) fused into
 * its epilogue, grouped GEMM down (sentinel rows zero), weighted combine.
 * With MOE_FWD_GATHER the permute is folded into the gate_up GEMM.  No host
 * synchronisation; offsets never leave the device.
 */
typedef struct {
    moe_dtype_t dtype;
    int T, E, k, H, I;
    int renormalize;              /* as in moe_route_sort */
    unsigned flags;               /* MOE_FWD_* */
    const float* logits;          /* [T, E] or NULL (then topk_ids/topk_w are inputs) */
    const float* expert_bias;     /* [E] or NULL (device) */
    const uint8_t* sentinel_mask; /* [T*k] or NULL (device) */
    int32_t* topk_ids;            /* [T, k] (device); NULL: held in the workspace (needs logits) */
    float* topk_w;                /* [T, k] (device); NULL likewise */
    const void* x;                /* bf16 [T, H] */
    const void* W1;               /* bf16 or e4m3 [E, 2I, H] (device) */
    const float* W1_scales;       /* FP8: [E, 2I/128, H/128] (device; 4-byte aligned) */
    const void* W2;               /* bf16 or e4m3 [E, H, I] (device) */
    const float* W2_scales;       /* FP8: [E, ceil(H/128), I/128] (device; 4-byte aligned) */
    void* out;                    /* bf16 [T, H] */
} moe_forward_args;

/* Bytes of device workspace moe_forward needs for these arguments (0 on
 * invalid arguments). */
size_t moe_forward_workspace_size(const moe_forward_args* args);
moe_status_t moe_forward(const moe_forward_args* args, void* ws, size_t ws_bytes,
                         moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
