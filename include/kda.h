/*
 * kda.h - C ABI of the GB300 (sm_103a) Kimi Delta Attention (KDA) hot path.
 *
 * Four operations, each an asynchronous launch on a caller-given CUDA stream:
 *
 *   kda_state_gather    per-request recurrent state gather from a paged cache
 *   kda_prefill_varlen  chunkwise (C = 64) gated delta-rule prefill over a
 *                       cu_seqlens varlen batch
 *   kda_state_scatter   final-state scatter back to cache rows
 *   kda_decode_step     one-token recurrent decode step on cache rows
 *
 * Conventions shared by every entry point
 *   - Every data pointer is a DEVICE pointer unless stated otherwise; the
 *     caller owns every buffer.  The library keeps no pointer or buffer of
 *     the caller's after a call returns, allocates no device memory and never
 *     synchronises the host with the device.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued on it and nothing else, with one exception:
 *     the segmented prefill of one long sequence (kda_prefill_varlen) also
 *     enqueues on a stream of the library's own, ordered after `stream` and
 *     joined back into it by events, so work enqueued on `stream` after the
 *     call still sees every result.
 *   - All argument checks run on the host, on metadata only, before anything
 *     is launched.  A failed check returns a negative kda_status and launches
 *     nothing.  KDA_ERR_CUDA means the launch itself failed (for example no
 *     device, or an unsupported architecture); its message is available from
 *     kda_last_cuda_error_string().
 *   - Device-side index VALUES are never checked on the host (that would need
 *     a device-to-host copy); the kernels treat out-of-range indices as the
 *     contract below says.
 *   - Floating point: states and gates are fp32; q/k/v/o are bf16 or fp32.
 *     bf16 results are rounded to nearest, ties to even.
 *
 * State layout.  A recurrent state S of one head is a K x V matrix.  Cache
 * rows and packed states store it transposed, as [V][K] (element (v, k) is
 * S[k][v]), with the heads outermost: one row is [H][V][K], H*V*K elements
 * ("payload").  Consecutive cache rows are `row_stride` elements apart,
 * row_stride >= payload; the gap between a row's payload and the next row is
 * never read or written.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_NULL = -1,        /* a required pointer is NULL                       */
    KDA_ERR_DTYPE = -2,       /* unknown or unsupported element / index type      */
    KDA_ERR_LAYOUT = -3,      /* cache layout: n_rows <= 0, row_stride < payload  */
    KDA_ERR_SHAPE = -4,       /* a size is negative / zero where it must not be   */
    KDA_ERR_RANGE = -5,       /* a size is beyond what the kernels address        */
    KDA_ERR_WORKSPACE = -6,   /* workspace missing, too small or misaligned       */
    KDA_ERR_CUDA = -7,        /* the CUDA launch failed                           */
    KDA_ERR_UNSUPPORTED = -8, /* head size / combination not built                */
    KDA_ERR_ALIGN = -9        /* a pointer is not aligned to its element size     */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;
typedef enum { KDA_I32 = 0, KDA_I64 = 1 } kda_itype;

/* A paged recurrent-state cache [n_rows, h, v, k] with a row stride.
 * `data` points at element 0 of row 0 (any storage offset already applied).
 * Layout rule of the "vllm-ascend KDA state copy" page, section "Automatic
 * dispatch": dtype fp32 or bf16, four dimensions, n_rows > 0, the inner
 * [h, v, k] block dense, stride(0) >= payload (pages do not overlap). */
typedef struct {
    void *data;
    int32_t dtype;      /* kda_dtype */
    int32_t reserved;   /* must be 0 */
    int64_t n_rows;
    int64_t h, v, k;
    int64_t row_stride; /* in elements */
} kda_cache;

/* ------------------------------------------------------------------------
 * kda_state_gather
 *
 * packed[s] = cache[idx[s]]   when 0 <= idx[s] < n_rows and
 *                             (flags == NULL or flags[s] != 0)
 * packed[s] = 0               otherwise.
 * Defined by the "vllm-ascend KDA state copy" page, section "Numeric
 * contract / Gather side": invalid or negative indices and flag=false rows
 * yield zeros, flags=None gathers every valid row, duplicate indices are
 * legal, and the packed output is written completely.
 *
 *   cache     cache descriptor (host pointer to the struct; data on device)
 *   idx       [selected] device indices, int32 or int64 (`idx_type`); int32
 *             indices are read as int32 (no conversion) and every address is
 *             formed in 64-bit arithmetic, so rows more than 4 GiB apart
 *             resolve ("Memory and addressing").
 *   selected  number of rows; 0 returns KDA_OK and launches nothing.
 *   flags     [selected] device bytes (bool), or NULL.
 *   packed    [selected, h, v, k] device, contiguous, cache dtype.  Must not
 *             overlap the cache.
 * ---------------------------------------------------------------------- */
int kda_state_gather(const kda_cache *cache, const void *idx, int32_t idx_type,
                     int64_t selected, const uint8_t *flags, void *packed, void *stream);

/* ------------------------------------------------------------------------
 * kda_state_scatter
 *
 * cache[idx[s]] = convert(packed[s]) for every s with 0 <= idx[s] < n_rows;
 * other s are skipped.  Defined by the same page, "Numeric contract /
 * Scatter side": invalid targets are skipped, initial-state flags play no
 * part, and the final state is converted to the cache dtype before it is
 * written ("Memory and addressing").  Gap elements and rows not selected
 * are never touched.
 *
 *   packed        [selected, h, v, k] device, contiguous, `packed_dtype`
 *                 (fp32 or bf16; fp32 -> bf16 rounds to nearest even,
 *                 bf16 -> fp32 is exact).
 *   Preconditions (not checked, no host sync): valid targets are unique;
 *   packed does not overlap the cache; no concurrent writer.
 * ---------------------------------------------------------------------- */
int kda_state_scatter(const kda_cache *cache, const void *idx, int32_t idx_type,
                      int64_t selected, const void *packed, int32_t packed_dtype, void *stream);

/* ------------------------------------------------------------------------
 * kda_prefill_workspace_size
 *
 * Bytes of device workspace kda_prefill_varlen needs for a batch of
 * `num_seqs` sequences totalling `total_tokens` tokens, `h` heads and head
 * sizes dk, dv.  The size depends only on these numbers (an upper bound on
 * the chunk count is used), never on device data.  Returns 0 for an
 * unsupported combination.
 * ---------------------------------------------------------------------- */
size_t kda_prefill_workspace_size(int64_t total_tokens, int64_t num_seqs, int32_t h, int32_t dk,
                                  int32_t dv);

/* ------------------------------------------------------------------------
 * kda_prefill_workspace_size_compact
 *
 * The smallest workspace kda_prefill_varlen (and _timed, _cached) accepts
 * for the batch with inputs of `io_dtype`.  For bf16 at dk == dv == 128 it is
 * a few kilobytes (a header and the chunk table): a call given less than
 * kda_prefill_workspace_size(...) bytes runs the fused kernel, which keeps
 * every per-chunk intermediate on chip (one persistent CTA per SM runs the
 * chunk preparation and the state pass of its (sequence, head) items
 * together) instead of the two-kernel form, whose per-chunk records (74,240 B
 * per chunk and head) pass through the workspace.  The results agree within
 * the same tolerances; the two-kernel form is the faster one on this GPU
 * (the fused kernel keeps one chunk's preparation in flight per SM), so it is
 * taken whenever the workspace holds the records.  Other dtypes and head
 * sizes: the same value as kda_prefill_workspace_size.  0 for an unsupported
 * combination.
 * ---------------------------------------------------------------------- */
size_t kda_prefill_workspace_size_compact(int64_t total_tokens, int64_t num_seqs, int32_t h,
                                          int32_t dk, int32_t dv, int32_t io_dtype);

/* ------------------------------------------------------------------------
 * kda_prefill_varlen
 *
 * For every sequence b (tokens cu_seqlens[b] .. cu_seqlens[b+1]-1) and head:
 *   S <- init_state[b] (zeros when init_state == NULL)
 *   for each token t in order:
 *     q_t, k_t <- L2-normalised (x / sqrt(sum x^2 + 1e-6)) when qk_l2norm
 *     S   <- (I - beta_t k_t k_t^T) Diag(exp g_t) S + beta_t k_t v_t^T
 *     o_t <- scale * S^T q_t
 *   final_state[b] <- S
 * The recurrence is the one of the "KDA's challenges for AI infra" page,
 * section 1.1; the kernels evaluate it chunkwise, 64 tokens at a time, in
 * the order of the "Support Kimi-K3 on NPU" report's extend listing
 * (l2norm -> chunk table -> in-chunk gate cumsum -> gated K K^T and Q K^T ->
 * triangular solve -> W, U -> inter-chunk state pass -> output).  Chunks
 * restart at every sequence start.
 *
 *   q, k        [total_tokens, h, dk] device, `io_dtype` (bf16 or fp32)
 *   v           [total_tokens, h, dv] device, `io_dtype`
 *   g           [total_tokens, h, dk] device fp32, per-channel log-decay.
 *               Any decay (g <= 0, however strong: a factor e^{G_i - G_j}
 *               below fp32's range is zero, as it is in exact arithmetic to
 *               within that range).  The kernels split exponentials through
 *               16-token block midpoints while every channel's partial sums
 *               stay within 44 nats of them (the pages' gate
 *               -softplus(N(0,1)) stays within about 15) and evaluate each
 *               factor from its own exponent difference in the chunks where
 *               they do not (slower, exact).  g > 0 (growth) is accepted; a
 *               growing state amplifies the rounding of the bf16 tensor-core
 *               operands, so the outputs keep the tolerance of decaying gates
 *               only while growth stays slow.
 *   beta        [total_tokens, h] device fp32
 *   cu_seqlens  [num_seqs + 1] device int32, cu_seqlens[0] = 0, non-
 *               decreasing, cu_seqlens[num_seqs] = total_tokens (precondition,
 *               not checked).  Empty sequences are allowed: their final state
 *               equals their initial state.
 *   num_seqs    >= 1;  total_tokens >= 0 (0: final = init, no output).
 *   h, dk, dv   heads and head sizes; built: dk == dv in {32, 64, 128}.
 *   scale       output scale (the report's listing uses dk^-0.5).
 *   qk_l2norm   1: normalise q and k; 0: use them as given.
 *   init_state  [num_seqs, h, dv, dk] device, `init_dtype` (fp32 / bf16),
 *               or NULL for zero initial states.
 *   final_state [num_seqs, h, dv, dk] device fp32, or NULL (not written).
 *   out         [total_tokens, h, dv] device, `io_dtype`; must not overlap
 *               any input (unlike the report's listing, which reuses v's
 *               buffer, the output is a separate buffer here).
 *   workspace   device scratch of at least kda_prefill_workspace_size(...)
 *               bytes (the two-kernel form), or, for bf16 at head size 128,
 *               of at least kda_prefill_workspace_size_compact(...) bytes
 *               (the fused kernel, when ws_bytes is below the former);
 *               256-byte aligned; its contents on entry do not matter.
 *   Calls on one workspace must not overlap in time.
 * Segmented prefill.  One sequence (num_seqs == 1) at head size 128, bf16,
 * with at least 512 chunks and at most half as many heads as the GPU has SMs,
 * given the full workspace, runs in segments of 256 chunks: the state pass of
 * a segment runs on a second stream (the device's highest priority, created by
 * the library on the first such call on each device and kept until the process
 * exits; make that first call outside stream capture) while the next segment's
 * chunks are prepared on `stream`.  The results are bit-identical with the
 * unsegmented form.  Calls from several host threads are serialised while
 * they enqueue.
 * Errors, checked on the host before anything is launched: KDA_ERR_DTYPE;
 * KDA_ERR_SHAPE (num_seqs < 1, total_tokens < 0, h, dk or dv < 1);
 * KDA_ERR_UNSUPPORTED (head sizes); KDA_ERR_RANGE (total_tokens >= 2^31,
 * num_seqs >= 2^30, h > 65535, chunk bound x h >= 2^31 or num_seqs x h x 8
 * >= 2^31: the kernels' one-dimensional grids); KDA_ERR_NULL; KDA_ERR_ALIGN
 * (16-byte aligned tensors, 4-byte aligned beta and cu_seqlens);
 * KDA_ERR_WORKSPACE (256-byte alignment, size).  KDA_ERR_CUDA when a launch
 * fails.
 * ---------------------------------------------------------------------- */
int kda_prefill_varlen(const void *q, const void *k, const void *v, int32_t io_dtype,
                       const float *g, const float *beta, const int32_t *cu_seqlens,
                       int64_t num_seqs, int64_t total_tokens, int32_t h, int32_t dk, int32_t dv,
                       float scale, int32_t qk_l2norm, const void *init_state, int32_t init_dtype,
                       float *final_state, void *out, void *workspace, size_t ws_bytes,
                       void *stream);

/* ------------------------------------------------------------------------
 * kda_prefill_varlen_timed
 *
 * kda_prefill_varlen, launching the same kernels, that also records four
 * caller-created CUDA events (cudaEvent_t passed as void*, host array
 * `events`) on `stream`: events[0] before the chunk-table kernel, events[1]
 * before the chunk-preparation kernel, events[2] before the state-pass
 * kernel, events[3] after it.  For measuring each kernel's device time.  In
 * the segmented prefill the state passes overlap the preparation: events[2]
 * follows the last segment's preparation and events[3] the last state pass.
 * events == NULL returns KDA_ERR_NULL; a NULL entry leaves its boundary
 * unrecorded (each record costs a few microseconds of stream time).
 * ---------------------------------------------------------------------- */
int kda_prefill_varlen_timed(const void *q, const void *k, const void *v, int32_t io_dtype,
                             const float *g, const float *beta, const int32_t *cu_seqlens,
                             int64_t num_seqs, int64_t total_tokens, int32_t h, int32_t dk,
                             int32_t dv, float scale, int32_t qk_l2norm, const void *init_state,
                             int32_t init_dtype, float *final_state, void *out, void *workspace,
                             size_t ws_bytes, void *stream, void *const *events);

/* ------------------------------------------------------------------------
 * kda_prefill_varlen_cached
 *
 * kda_prefill_varlen with its initial and final states in the state cache,
 * the fused form named in the "Support Kimi-K3 on NPU" report's extend
 * listing (the state pass takes the cache and the per-sequence cache indices
 * directly, step 3), plus optional chunk-boundary checkpoints - the states
 * the same listing returns on request for state tracking and the recurrent
 * checkpoints the infra page's vLLM section (8.2.4) writes during prefill.
 * Equivalent to, and bit-identical with, the unfused composition
 *   kda_state_gather(cache, idx_in, flags) -> kda_prefill_varlen ->
 *   kda_state_scatter(cache, idx_out)
 * without the two packed round trips:
 *   initial state of b = cache row idx_in[b] (upcast to fp32) when
 *       0 <= idx_in[b] < n_rows and (flags == NULL or flags[b] != 0),
 *       else zeros (the gather rule);
 *   final state of b   -> cache row idx_out[b], cast to the cache dtype
 *       (fp32 -> bf16 rounds to nearest even), when idx_out != NULL and
 *       0 <= idx_out[b] < n_rows (the scatter rule); other rows untouched;
 *       and -> final_state[b] (fp32, packed) when final_state != NULL.
 *   checkpoints: when checkpoints != NULL, the state after the first
 *       m * ckpt_every tokens of sequence b, for m = 1 .. len_b / ckpt_every
 *       (the final state too when len_b is a multiple), goes to slot
 *       first_b + m - 1, first_b = sum over b' < b of len_b' / ckpt_every,
 *       cast to ckpt_dtype.  ckpt_every is a multiple of 64 (checkpoints sit
 *       on chunk boundaries).  Slots >= ckpt_slots are not written;
 *       kda_prefill_checkpoint_count gives the number needed.
 *
 *   cache       [n_rows, h, dv, dk] rows with row_stride, cache->h == h,
 *               ->v == dv, ->k == dk; data and row stride 16-byte aligned.
 *   idx_in      [num_seqs] device, idx_type; required.
 *   flags       [num_seqs] device uint8, or NULL (all set).
 *   idx_out     [num_seqs] device, idx_type, or NULL (no write-back).
 *   final_state [num_seqs, h, dv, dk] device fp32, or NULL.
 *   checkpoints [ckpt_slots, h, dv, dk] device, ckpt_dtype, or NULL.
 *   Other arguments as kda_prefill_varlen (same workspace size).
 *   Preconditions (not checked, no host sync): valid idx_out rows are
 *   unique; no row is read as an initial state by one sequence and written
 *   by another (idx_in[b] == idx_out[b], an in-place update, is fine).
 *   Errors as kda_prefill_varlen, plus check_cache's layout errors,
 *   KDA_ERR_SHAPE when the cache does not match h, dk, dv or ckpt_every is
 *   not a positive multiple of 64, KDA_ERR_ALIGN for misaligned rows.
 * ---------------------------------------------------------------------- */
int kda_prefill_varlen_cached(const void *q, const void *k, const void *v, int32_t io_dtype,
                              const float *g, const float *beta, const int32_t *cu_seqlens,
                              int64_t num_seqs, int64_t total_tokens, int32_t h, int32_t dk,
                              int32_t dv, float scale, int32_t qk_l2norm, const kda_cache *cache,
                              const void *idx_in, const uint8_t *flags, const void *idx_out,
                              int32_t idx_type, float *final_state, void *checkpoints,
                              int32_t ckpt_dtype, int32_t ckpt_every, int64_t ckpt_slots, void *out,
                              void *workspace, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * kda_prefill_checkpoint_count
 *
 * Host helper: checkpoint slots kda_prefill_varlen_cached writes for the
 * sequences of a HOST copy of cu_seqlens, sum over b of len_b / ckpt_every.
 * Returns -1 for a NULL pointer, num_seqs < 1, a decreasing cu_seqlens or a
 * ckpt_every that is not a positive multiple of 64.
 * ---------------------------------------------------------------------- */
int64_t kda_prefill_checkpoint_count(const int32_t *cu_seqlens_host, int64_t num_seqs,
                                     int32_t ckpt_every);

/* ------------------------------------------------------------------------
 * kda_prefill_varlen_noalloc
 *
 * The reference pages have no counterpart to this entry point; it exists for
 * callers that cannot allocate device memory - a host program that links
 * only this library and has no device allocator, or a serving runtime that
 * fixes its device memory at start-up and allows no allocation (cudaMalloc
 * may synchronise the device and fail under fragmentation) on the request
 * path.
 *
 * Same computation, arguments and results as kda_prefill_varlen, without the
 * workspace: the kernels use a fixed array of KDA_NOALLOC_SCRATCH_BYTES bytes
 * of device memory owned by the library (held by every GPU that loads the
 * library until the process exits).  The call allocates nothing.
 *   - A batch whose kda_prefill_workspace_size_compact(...) exceeds
 *     KDA_NOALLOC_SCRATCH_BYTES is rejected with KDA_ERR_WORKSPACE and
 *     nothing is launched.  With bf16 at head size 128 that is never the
 *     case in practice (the compact workspace is the chunk table: a batch
 *     larger than the array holds records for, about 53 chunks of 64 tokens
 *     at h = 32, runs the fused kernel); with fp32, or head size 32 or 64,
 *     the records must fit (at h = 32, dk = dv = 128, fp32: about 53 chunks,
 *     e.g. one 3,300-token sequence).
 *   - The first call on a device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *     KDA_ERR_CUDA if the lookup fails.
 *   - Every call shares the one array: calls that overlap on the GPU (other
 *     streams, or other threads without ordering) race and corrupt each
 *     other's results.  Its contents left by the previous call do not matter.
 *   - The caller cannot see the array, so the device status word that
 *     kda_prefill_workspace_status reads from a workspace is read here by
 *     kda_prefill_noalloc_status.  The precondition cu_seqlens[num_seqs] ==
 *     total_tokens also sizes the array's records: a call that breaks it gets
 *     status 4 and reads no record beyond the array.
 * ---------------------------------------------------------------------- */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)128 << 20)

int kda_prefill_varlen_noalloc(const void *q, const void *k, const void *v, int32_t io_dtype,
                               const float *g, const float *beta, const int32_t *cu_seqlens,
                               int64_t num_seqs, int64_t total_tokens, int32_t h, int32_t dk,
                               int32_t dv, float scale, int32_t qk_l2norm, const void *init_state,
                               int32_t init_dtype, float *final_state, void *out, void *stream);

/* The device status word of the last kda_prefill_varlen_noalloc call on the
 * current device (the codes of kda_prefill_workspace_status), read from the
 * library's fixed array.  Like kda_prefill_workspace_status it copies 4 bytes
 * on `stream` and waits; order it after the prefill call (same stream).  The
 * pages have no counterpart.  KDA_ERR_NULL for a NULL status_out,
 * KDA_ERR_CUDA if the array's address cannot be looked up or the copy fails. */
int kda_prefill_noalloc_status(int32_t *status_out, void *stream);

/* ------------------------------------------------------------------------
 * kda_target_verify
 *
 * Speculative target verification ("KDA's challenges for AI infra", section
 * 6.4, target_verify, and 6.5, verify intermediate state indices): for each
 * request r, L draft tokens run through the recurrence of kda_decode_step
 * from S = cache row idx[r] (zeros for an invalid index); token t's output
 * goes to out[r][t] and the state after token t to row inter_idx[r][t] of
 * the intermediate-state pool (converted to the pool dtype; an invalid slot
 * is not written).  The cache is only read: a caller commits the accepted
 * prefix of n tokens by copying pool row inter_idx[r][n-1] into the cache
 * (kda_state_gather / kda_state_scatter).
 *
 *   q, k, g     [batch, L, h, dk] device (q, k io_dtype; g fp32)
 *   v, out      [batch, L, h, dv] device, io_dtype;  beta [batch, L, h] fp32
 *   cache, pool state caches with ->h == h, ->v == dv, ->k == dk; data and
 *               row strides 16-byte aligned; fp32 or bf16 each
 *   idx         [batch];  inter_idx [batch, L];  idx_type int32 / int64
 *   dk == dv in {32, 64, 128}.  Valid pool slots must be unique and must not
 *   alias cache rows that are read (preconditions, not checked).
 *   batch == 0 validates the metadata and launches nothing.
 * ---------------------------------------------------------------------- */
int kda_target_verify(const void *q, const void *k, const void *v, int32_t io_dtype, const float *g,
                      const float *beta, int64_t batch, int32_t L, int32_t h, int32_t dk, int32_t dv,
                      float scale, int32_t qk_l2norm, const kda_cache *cache, const void *idx,
                      const kda_cache *pool, const void *inter_idx, int32_t idx_type, void *out,
                      void *stream);

/* ------------------------------------------------------------------------
 * kda_conv1d_varlen / kda_conv1d_update
 *
 * The short causal convolution that q, k and v pass before the recurrence,
 * with a convolution state per request ("KDA's challenges for AI infra",
 * sections 6.5 and 8.2.3: causal_conv1d_fn in prefill, causal_conv1d_update
 * in decode; the pages give no formula, the textbook depthwise causal
 * convolution is used).  For channel c of width W (2..4):
 *   y_t[c] = act(bias[c] + sum_{i<W} weight[c][i] * x_{t-(W-1)+i}[c]),
 *   act = identity (activation 0) or SiLU y * sigmoid(y) (activation 1),
 * where inputs before a sequence's first token come from its state: the last
 * W-1 inputs, oldest first (zeros when no state is given).  fp32 arithmetic.
 *
 * kda_conv1d_varlen: over a cu_seqlens varlen batch (the prefill layout).
 *   x, y         [total_tokens, channels] device, io_dtype (fp32 / bf16);
 *                q, k and v may be convolved in one call as one buffer.
 *   cu_seqlens   [num_seqs + 1] device int32 (monotone; precondition).
 *   weight       [channels, W] device fp32 (weight[c][W-1] multiplies the
 *                current token);  bias [channels] device fp32 or NULL.
 *   init_state   [num_seqs, W-1, channels] device, state_dtype, or NULL.
 *   final_state  [num_seqs, W-1, channels] device, state_dtype, or NULL:
 *                each sequence's last W-1 inputs (an empty sequence keeps
 *                its initial state); bf16 rounds to nearest even.
 *   A state cache row [W-1, channels] is a kda_cache with h = 1, v = W-1,
 *   k = channels, so kda_state_gather / kda_state_scatter move conv states
 *   between cache rows and these packed buffers, as for the recurrence.
 * kda_conv1d_update: one token per request on cache rows in place (decode):
 *   x, y [batch, channels]; conv_cache rows [W-1, channels] (h == 1,
 *   v == W-1, k == channels); idx [batch] int32 / int64.  A valid row is
 *   read as the state and replaced by the state after the token; an invalid
 *   index uses zeros and writes nothing.  Valid rows must be unique.
 * channels must be a multiple of 8; all arrays 16-byte aligned (cu_seqlens
 * and indices: their element size).  Errors: KDA_ERR_UNSUPPORTED for W
 * outside 2..4, KDA_ERR_SHAPE for channels % 8 != 0, an unknown activation
 * or a conv cache that does not match W and channels, KDA_ERR_RANGE for
 * channels > 65535 * 1024 or (total_tokens + 15) / 8 * ceil(channels / 1024)
 * > 2^31 - 1 (the kernels' grids); the others as for the calls above.  Nothing is launched on an error; batch == 0 launches nothing.
 * ---------------------------------------------------------------------- */
int kda_conv1d_varlen(const void *x, int32_t io_dtype, const int32_t *cu_seqlens, int64_t num_seqs,
                      int64_t total_tokens, int64_t channels, int32_t width, const float *weight,
                      const float *bias, int32_t activation, const void *init_state, void *final_state,
                      int32_t state_dtype, void *y, void *stream);
int kda_conv1d_update(const void *x, int32_t io_dtype, int64_t batch, int64_t channels, int32_t width,
                      const float *weight, const float *bias, int32_t activation,
                      const kda_cache *conv_cache, const void *idx, int32_t idx_type, void *y,
                      void *stream);

/* ------------------------------------------------------------------------
 * kda_ckpt_store_int8 / kda_ckpt_load_int8
 *
 * INT8 checkpoints of recurrent states, the Int8CheckpointStore of the
 * "KDA's challenges for AI infra" page, section 6.6.2: inactive states are
 * kept as symmetric int8 codes with one fp32 scale per (slot, head, key
 * channel), taken from the max-abs along the value dimension; a cache hit
 * dequantises once into an active slot, which then continues in full
 * precision.  For one layer's pools:
 *
 *   qdata  [n_slots, h, v, k] device int8, contiguous, 16-byte aligned
 *   scale  [n_slots, h, k]    device fp32, contiguous, 16-byte aligned
 *   active the state cache (kda_cache; v == k in {32, 64, 128}; data and
 *          row stride 16-byte aligned)
 *
 * store: for each pair s with 0 <= src_rows[s] < n_rows and
 *   0 <= dst_slots[s] < n_slots, for each head h and key channel k of the
 *   row's [h][v][k] block x (upcast to fp32):
 *     amax = max_v |x[h][v][k]|,  scale[dst][h][k] = amax / 127,
 *     qdata[dst][h][v][k] = round_half_even(x / scale) clamped to
 *     [-127, 127]; a scale below the smallest normal fp32 (amax == 0, or
 *     amax < 127 * 2^-126) is stored as 0 with all codes 0,
 *   each a correctly rounded fp32 operation.  Pairs with an invalid index
 *   are skipped; other slots are not touched.
 * load: for each pair s with 0 <= src_slots[s] < n_slots and
 *   0 <= dst_rows[s] < n_rows:  active[dst][h][v][k] =
 *   qdata[src][h][v][k] * scale[src][h][k] (one fp32 multiply), converted
 *   to the cache dtype (bf16: round to nearest even).  Gaps and other rows
 *   are not touched.
 *   src_*, dst_*  [count] device, idx_type (int32 / int64).
 *   count == 0 validates the metadata and launches nothing.
 *   Preconditions (not checked, no host sync): valid destinations are
 *   unique; the pools do not overlap the cache.
 * ---------------------------------------------------------------------- */
int kda_ckpt_store_int8(const kda_cache *active, const void *src_rows, const void *dst_slots,
                        int32_t idx_type, int64_t count, int8_t *qdata, float *scale, int64_t n_slots,
                        void *stream);
int kda_ckpt_load_int8(const int8_t *qdata, const float *scale, int64_t n_slots,
                       const void *src_slots, const void *dst_rows, int32_t idx_type, int64_t count,
                       const kda_cache *active, void *stream);

/* ------------------------------------------------------------------------
 * kda_decode_step
 *
 * For each request r and head: with row = idx[r],
 *   S   <- cache[row] (upcast to fp32) when 0 <= row < n_rows, else zeros
 *   q, k <- L2-normalised when qk_l2norm
 *   S   <- (I - beta k k^T) Diag(exp g) S + beta k v^T
 *   o   <- scale * S^T q
 *   cache[row] <- S converted to the cache dtype, only when row is valid.
 * One token of the same recurrence (infra page, section 1.1), on cache rows
 * in place - the decode route named on the state-copy page, "Background".
 * An invalid index behaves as gather (zeros) -> step -> scatter (skipped).
 *
 *   q, k, v     [batch, h, dk] / [batch, h, dv] device, `io_dtype`
 *   g           [batch, h, dk] device fp32;  beta [batch, h] device fp32
 *   cache       state cache with cache->h == h, ->k == dk, ->v == dv
 *   idx         [batch] device int32 / int64
 *   out         [batch, h, dv] device, `io_dtype`
 *   Preconditions (not checked): valid indices are unique.
 *   Built: dk == dv in {32, 64, 128}.  batch == 0 launches nothing.
 * ---------------------------------------------------------------------- */
int kda_decode_step(const void *q, const void *k, const void *v, int32_t io_dtype, const float *g,
                    const float *beta, int64_t batch, int32_t h, int32_t dk, int32_t dv,
                    float scale, int32_t qk_l2norm, const kda_cache *cache, const void *idx,
                    int32_t idx_type, void *out, void *stream);

/* Human-readable name of a kda_status value (static string, never NULL). */
const char *kda_status_string(int32_t status);

/* Text of the CUDA error behind the last KDA_ERR_CUDA returned on this host
 * thread (static storage; "no error" if none). */
const char *kda_last_cuda_error_string(void);

/* Reads the device-side status word a prefill call leaves in its workspace:
 * 0 when every internal wait completed, otherwise a non-zero code (1: a
 * record copy awaited by the register state pass did not complete within its
 * bound; 2: a record copy or MMA awaited by the tensor-memory state pass did
 * not; 3: an input tensor copy awaited by the chunk preparation did not; 4:
 * cu_seqlens gave more chunks than total_tokens allows, a broken
 * precondition whose results are undefined, though no record beyond the
 * workspace is read).  A kernel whose wait expires stops waiting, finishes
 * without touching memory it has not been given and releases its tensor
 * memory, so the context stays usable.  This call and
 * kda_prefill_noalloc_status are the ones that synchronise: each copies 4
 * bytes on `stream` and waits. */
int kda_prefill_workspace_status(const void *workspace, int32_t *status_out, void *stream);

/* Diagnostic of the bounded waits above (infra-level failure detection: a
 * hang is reported, never left on the GPU).  Launches one CTA on `stream`
 * that waits, with the same bounded mbarrier wait as the prefill kernels
 * (at most `polls` polls, > 0), on a barrier that receives its arrival
 * (arrive != 0) or never does (arrive == 0), and writes to the device int32
 * *status_dev: 0 when the wait completed, 1 when it expired.  Errors:
 * KDA_ERR_NULL (status_dev NULL), KDA_ERR_RANGE (polls == 0), KDA_ERR_CUDA
 * (launch failure).  Asynchronous; nothing is allocated. */
int kda_selftest_bounded_wait(int32_t *status_dev, uint32_t polls, int32_t arrive, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
