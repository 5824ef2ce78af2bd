/*
 * ncp_attn.h: C ABI of the GB300 (sm_103a) BF16 attention leaf.
 *
 * The operations are those of the page "Audit SGLang interfaces and refresh
 * validated kernel solutions":
 *   - attn_dense_fwd: definitions/dense_attention/noncausal_dense_attention_
 *     h32_d128.json and noncausal_dense_attention_h32_d64.json, field
 *     "reference": O = softmax(Q K^T * D^-0.5) V, no mask, FP32 accumulation,
 *     BF16 output.
 *   - attn_prefix_fwd: definitions/block_causal_attention/prefix_cached_block_
 *     causal_h32_d128.json, field "reference": Q attends with full visibility
 *     to keys cat(K_prefix, K_current) and values cat(V_prefix, V_current)
 *     (prefix tokens first), scale D^-0.5.  No concatenated copy is made.
 *
 * Common conventions
 *   Layout:     every tensor is a contiguous [B, N, H, D] bf16 array (token-
 *               major, head, then head dim), the layout of the definitions'
 *               "inputs" fields.
 *   Memory:     all tensor pointers are DEVICE pointers owned by the caller on
 *               the current CUDA device.  Inputs are read only; `out` is fully
 *               overwritten and must not overlap any input.  The library
 *               allocates no device memory per call.  When the work does not
 *               fill the last round of SMs, the tail is cut into key-range
 *               pieces on separate SMs whose partial results are merged
 *               through a split workspace: 2 x SMs slots of 2 x 128 x
 *               (128 + 4) floats plus 2 x SMs 64-bit counters (about 41 MB
 *               on a 152-SM GPU).  Workspaces form a pool of at most 4 per
 *               device, each allocated by the first call that needs it and
 *               kept until the process exits (at most about 165 MB per
 *               device, whatever streams come and go).  A call takes the
 *               workspace its stream used last, else one whose previous
 *               launch has finished, else a new one while the pool has room;
 *               when all are busy on other streams it runs without splitting
 *               (the same result up to rounding order; every call that splits
 *               gives bit-identical output for the same inputs).  Calls in
 *               flight at once never share a workspace.  Each launch tags its
 *               counters with a fresh epoch, so a launch that gave up on a
 *               bounded wait leaves nothing that affects the next one.
 *   Graphs:     a call made while its stream is being captured into a CUDA
 *               graph allocates nothing and queries nothing: it uses the
 *               workspace that stream used last (make one eager call on the
 *               capture stream first; otherwise it runs without splitting),
 *               claims it for good (no other stream takes it afterwards) and
 *               captures a clear of its counters before the kernel.  The
 *               graph's replays must not run at the same time as other work
 *               that uses that workspace: eager calls on the capture stream,
 *               or replays of other graphs captured on it.
 *   Reset:      the library keeps per-device state (workspaces, kernel
 *               attributes, the address of the static scratch of
 *               attn_dense_fwd_noalloc).  cudaDeviceReset invalidates it: do
 *               not call the library after resetting a device in the same
 *               process.
 *   Alignment:  every pointer must be 16-byte aligned (tensor-memory-access
 *               descriptors require it).
 *   Head dim:   D must be 64 or 128; H >= 1 (the definitions fix H = 32, any
 *               H is accepted).  The scale is fixed to D^-0.5 (the definitions
 *               expose no scale argument).
 *   Streams:    work is enqueued on `stream` (0 = legacy default stream); the
 *               calls return without synchronising.
 *   Errors:     argument errors return a negative attn_status and launch
 *               nothing.  A launch failure returns ATTN_ERR_CUDA.  Every wait
 *               inside the kernels is bounded; a wait that gives up records a
 *               device status that attn_device_status() returns as
 *               ATTN_ERR_TIMEOUT.
 */
#ifndef NCP_ATTN_H
#define NCP_ATTN_H

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = -1,     /* a required pointer is NULL */
    ATTN_ERR_SHAPE = -2,    /* a size is out of range (B, N, Nq, Nc, H < 1; Np < 0; too large) */
    ATTN_ERR_HEADDIM = -3,  /* D is not 64 or 128 */
    ATTN_ERR_ALIGN = -4,    /* a pointer is not 16-byte aligned */
    ATTN_ERR_ALIAS = -5,    /* out overlaps an input */
    ATTN_ERR_CUDA = -6,     /* a CUDA runtime/driver call failed */
    ATTN_ERR_TIMEOUT = -7   /* a bounded in-kernel wait gave up (see attn_device_status) */
} attn_status;

/*
 * Dense non-causal self-attention.
 *   q, k, v: [B, N, H, D] bf16, device, read only.
 *   out:     [B, N, H, D] bf16, device, written.
 * Returns ATTN_OK or a negative attn_status.
 */
int attn_dense_fwd(const void *q, const void *k, const void *v, void *out,
                   int B, int N, int H, int D, cudaStream_t stream);

/*
 * Dense non-causal cross attention: the same definitions as attn_dense_fwd,
 * whose description allows it ("self attention uses Nq=Nk; cross attention
 * allows unequal lengths").
 *   q:    [B, Nq, H, D] bf16, device, read only.
 *   k, v: [B, Nk, H, D] bf16, device, read only.
 *   out:  [B, Nq, H, D] bf16, device, written.
 * Nq, Nk >= 1.  When the (b, h, 256-query) work units are fewer than the
 * SMs, each unit's keys are cut into pieces on separate SMs and merged (the
 * split workspace, see "Memory" above), so short-query, long-context calls
 * still fill the GPU.  Returns ATTN_OK or a negative attn_status.
 */
int attn_dense_cross_fwd(const void *q, const void *k, const void *v, void *out,
                         int B, int Nq, int Nk, int H, int D, cudaStream_t stream);

/*
 * Prefix-cached full-visibility attention.
 *   q:      [B, Nq, H, D]
 *   kp, vp: [B, Np, H, D]  cached prefix keys/values (may be NULL when Np == 0)
 *   kc, vc: [B, Nc, H, D]  current keys/values
 *   out:    [B, Nq, H, D]
 * Each query attends to all Np + Nc keys, prefix first.  The definition
 * requires Np >= 1 and Nc == Nq; this entry also accepts Np == 0 (dense
 * attention over the current keys) and Nc != Nq (cross attention).
 */
int attn_prefix_fwd(const void *q, const void *kp, const void *vp, const void *kc,
                    const void *vc, void *out, int B, int Nq, int Np, int Nc, int H, int D,
                    cudaStream_t stream);

/*
 * Block-causal self-attention with image segments: the definition
 * definitions/block_causal_attention/prefix_cached_block_causal_h32_d128_
 * prefix0.json, field "reference" (the empty-prefix specialisation of the
 * prefix-cached form).  Query i sees key j iff j <= i (text and different
 * images are causal), or image_ids[i] == image_ids[j] >= 0 (tokens of one
 * image see each other).  Scale D^-0.5.
 *   q, k, v:   [B, N, H, D] bf16, device, read only.
 *   image_ids: [N] int32, device, read only, shared by the batch; -1 marks a
 *              text token, non-negative values name images.  Any ids give the
 *              exact definition; ids that form contiguous, distinct image
 *              blocks (the definition's engine segment list) let whole key
 *              tiles be skipped.  Must be 16-byte aligned.
 *   out:       [B, N, H, D] bf16, device, written; must not overlap an input.
 * N <= 131072 (the per-CTA tile table lives in shared memory).  Returns
 * ATTN_OK or a negative attn_status (ATTN_ERR_SHAPE for N too large).
 */
int attn_block_causal_fwd(const void *q, const void *k, const void *v, const int *image_ids,
                          void *out, int B, int N, int H, int D, cudaStream_t stream);

/*
 * Masked prefix-cached attention: the earlier form of the definition
 * definitions/block_causal_attention/prefix_cached_block_causal_h32_d128.json
 * (field "reference" before the audit made every key visible).  Keys and
 * values are cat(K_prefix, K_current) / cat(V_prefix, V_current); query i
 * sits at position Np + i and sees key position j iff (j <= Np + i, or
 * image_ids[Np + i] == image_ids[j] >= 0) and key_valid[b, j].  Scores are
 * scaled by sm_scale (the old form's runtime scale).  Operand order is the
 * old definition's: Q, K_current, V_current, K_prefix, V_prefix, image_ids,
 * key_valid, sm_scale.
 *   q, kc, vc:  [B, Nq, H, D] bf16, device, read only (Nc == Nq).
 *   kp, vp:     [B, Np, H, D] bf16, device, read only (may be NULL when Np == 0).
 *   image_ids:  [Np + Nq] int32, device, 16-byte aligned; -1 = text.
 *   key_valid:  [B, Np + Nq] bytes (bool), device; 0 hides a key; NULL = all valid.
 *   sm_scale:   finite, > 0.
 *   out:        [B, Nq, H, D] bf16, device, written.
 * Np + Nq <= 131072.  The definition requires every query to see at least
 * one key; a row that sees none comes out as NaN.  Returns ATTN_OK or a
 * negative attn_status (ATTN_ERR_SHAPE also for a bad sm_scale).
 */
int attn_masked_prefix_fwd(const void *q, const void *kc, const void *vc, const void *kp,
                           const void *vp, const int *image_ids, const unsigned char *key_valid,
                           float sm_scale, void *out, int B, int Nq, int Np, int H, int D,
                           cudaStream_t stream);

/*
 * attn_dense_fwd without any allocation, for callers that cannot call
 * cudaMalloc: an engine whose memory pool already owns the device memory, a
 * plugin that is handed only its input and output buffers, or a latency-bound
 * loop that cannot afford an allocation's implicit device synchronisation.
 * The pages define no such call; it is a deployment variant of the dense form.
 *
 * Same arguments, result and errors as attn_dense_fwd.  The split workspace
 * (partial rows of key-range pieces and their arrival counters) lives in one
 * static device array of 43.3 MB (320 slots and 320 counters, enough for a
 * GPU with up to 160 SMs at D <= 128) that every GPU loading this library
 * holds until the process exits; no cudaMalloc, no cudaFree.  A call whose
 * schedule needs more than that (only on a GPU with more than 160 SMs)
 * returns ATTN_ERR_SHAPE and launches nothing.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Every call clears the counters on `stream`, then uses the array: calls
 * that overlap on the GPU (other streams, other host threads) race on it and
 * must be serialised by the caller.
 */
int attn_dense_fwd_noalloc(const void *q, const void *k, const void *v, void *out,
                           int B, int N, int H, int D, cudaStream_t stream);

/* Static, human-readable name of a status code (never NULL). */
const char *attn_status_string(int status);

/*
 * Synchronises `stream`, then returns ATTN_ERR_TIMEOUT if any kernel of this
 * library recorded a bounded-wait failure since the previous call (and clears
 * the record), ATTN_OK otherwise, or ATTN_ERR_CUDA if the synchronisation
 * fails.  If `info` is not NULL it receives the first failure's site code
 * (bits 0-7: wait site, bits 8-31: block index), or 0.
 */
int attn_device_status(cudaStream_t stream, unsigned int *info);

/*
 * Test hook.  mode 0: normal operation.  mode 1: in block 0 of the next
 * launches, the loader skips the value tile of the second key/value tile, so
 * the matrix-multiply role's wait for it runs out (needs at least two key
 * tiles).  wait_limit_us sets the bound of every in-kernel wait (0 restores
 * the default of 2 s).  Returns ATTN_OK, or ATTN_ERR_SHAPE for an unknown
 * mode.  Host-side setting, applies to subsequent launches of this process.
 */
int attn_debug_set_fault(int mode, unsigned int wait_limit_us);

/*
 * Test hook: y[i] = 2^x[i] for i < n through one of the two exponential paths
 * of the softmax: mode 0 the FMA-pipe polynomial (Cody-Waite reduction and a
 * minimax cubic, relative error <= 1.02e-4 for -126 <= x <= 127, exactly 0 for
 * x <= -127), mode 1 the hardware ex2.approx unit.  x and y are device
 * pointers to n floats (caller-owned); enqueued on `stream`.  Returns ATTN_OK,
 * ATTN_ERR_NULL, ATTN_ERR_SHAPE (n < 0, bad mode) or ATTN_ERR_CUDA.
 */
int attn_debug_exp2(const float *x, float *y, long long n, int mode, cudaStream_t stream);

/*
 * Test hook: the work schedule of a launch, computed on the host without a
 * GPU.  masked = 0: the dense family (dense, cross, prefix-cached) with
 * n_key_tiles key tiles of 128 (image_ids and Np ignored).  masked = 1: the
 * block-causal and masked prefix forms, Np prefix positions then Nq current
 * ones, image_ids a host array of Np + Nq ids (caller-owned; the key tiles
 * are counted from Np and Nq, n_key_tiles is ignored).  A launch over B
 * batches, Nq queries and H heads on a GPU with `sms` SMs runs *grid_out
 * persistent CTAs; each item of each CTA is one row of 12 ints:
 *   cta, n (the CTA's n-th item), b, h, q0 (first query row of the unit's
 *   pair of 128-row tiles), two (the second tile has rows), t_begin, t_end
 *   (key tiles [t_begin, t_end); masked forms visit only some of them), tail
 *   (-1: a whole unit, else its tail unit), piece, pieces (this piece's index
 *   and the tail unit's piece count), slot0 (workspace slot of the tail
 *   unit's piece 0).
 * Rows go to `rows` (caller-owned host memory, cap rows of 12 ints);
 * *n_rows receives the item count, *slots_out the workspace slots used.
 * Returns ATTN_OK, ATTN_ERR_NULL, or ATTN_ERR_SHAPE (a size out of range, or
 * more than cap items: then only cap rows are written).
 */
int attn_debug_schedule(int B, int Nq, int H, int n_key_tiles, int sms, int masked,
                        const int *image_ids, int Np, int *rows, int cap, int *n_rows,
                        int *grid_out, int *slots_out);

#ifdef __cplusplus
}
#endif

#endif /* NCP_ATTN_H */
