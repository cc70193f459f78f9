// Internal launcher interface between the C ABI (api.cu) and the kernels.
// Launchers assume their arguments were validated by the ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Maps a CUDA result to a kda_status, remembering a failure for
// kda_last_cuda_error_string (api.cu).  For entry points defined outside api.cu.
int record_cuda_status(cudaError_t e);

// Streaming multiprocessors of the current device (cached per device; 152 if unknown).
int64_t sm_count();

struct CacheDesc {
    void *data;
    int32_t dtype;
    int64_t n_rows, h, v, k, row_stride;
};

constexpr int kChunk = 64;  // tokens per chunk (the report's extend listing fixes 64)
// Channels per CTA of the short convolution; the per-sequence and update kernels put these
// channel blocks in the grid's y dimension (at most 65,535 of them).
constexpr int kConvChannelsPerBlock = 1024;

cudaError_t launch_state_gather(const CacheDesc &c, const void *idx, int32_t idx_type, int64_t selected,
                                const uint8_t *flags, void *packed, cudaStream_t st);
cudaError_t launch_state_scatter(const CacheDesc &c, const void *idx, int32_t idx_type, int64_t selected,
                                 const void *packed, int32_t packed_dtype, cudaStream_t st);

struct DecodeArgs {
    const void *q, *k, *v;
    int32_t io_dtype;
    const float *g, *beta;
    int64_t batch;
    int32_t h, d;
    float scale;
    int32_t l2norm;
    CacheDesc cache;
    const void *idx;
    int32_t idx_type;
    void *out;
};
cudaError_t launch_decode_step(const DecodeArgs &a, cudaStream_t st);

// Speculative target verification (head size d = dk = dv in {32, 64, 128}).
struct VerifyArgs {
    const void *q, *k, *v;
    int32_t io_dtype;
    const float *g, *beta;
    int64_t batch;
    int32_t L, h, d;
    float scale;
    int32_t l2norm;
    CacheDesc cache;       // initial states, read only
    const void *idx;       // [batch]
    CacheDesc pool;        // intermediate states
    const void *inter_idx; // [batch, L]
    int32_t idx_type;
    void *out;
};
cudaError_t launch_target_verify(const VerifyArgs &a, cudaStream_t st);

// Short causal convolution (width 2..4, channels a multiple of 8).
struct Conv1dArgs {
    const void *x;
    int32_t io_dtype;
    const int32_t *cu_seqlens;
    int64_t num_seqs, total_tokens, channels;
    int32_t width;
    const float *weight, *bias;
    int32_t activation;
    const void *init_state;
    void *final_state;
    int32_t state_dtype;
    void *y;
};
cudaError_t launch_conv1d_varlen(const Conv1dArgs &a, cudaStream_t st);

struct Conv1dUpdateArgs {
    const void *x;
    int32_t io_dtype;
    int64_t batch, channels;
    int32_t width;
    const float *weight, *bias;
    int32_t activation;
    CacheDesc cache;
    const void *idx;
    int32_t idx_type;
    void *y;
};
cudaError_t launch_conv1d_update(const Conv1dUpdateArgs &a, cudaStream_t st);

// INT8 checkpoints; the cache's head size k (== v) is 32, 64 or 128.
cudaError_t launch_ckpt_store_int8(const CacheDesc &c, const void *src, const void *dst, int32_t idx_type,
                                   int64_t count, int8_t *qdata, float *scale, int64_t n_slots, cudaStream_t st);
cudaError_t launch_ckpt_load_int8(const CacheDesc &c, const int8_t *qdata, const float *scale, int64_t n_slots,
                                  const void *src, const void *dst, int32_t idx_type, int64_t count, cudaStream_t st);

// Prefill workspace: a header (status word), the chunk table, and one record
// per (chunk, head) holding the chunk's W, Q~, K~, A_qk, gamma and U^T.
struct PrefillLayout {
    int64_t n_chunk_max;
    size_t off_chunk_off, off_seq_order, off_chunk_info, off_ckpt_off, off_fix_list, off_records, rec_bytes, total;
    size_t off_seg_state;  // one sequence at head size 128: its state between segments (fp32 [H][V][K]), else 0
    size_t compact;  // bytes the fused kernel needs: the header and the chunk table, no records
};

// Where each sequence's initial state comes from and where its final state and
// checkpoints go.  A state of head h is [V][K] (the cache orientation): element
// (v, k) of the state at base element offset o sits at o + (h * D + v) * D + k.
struct StateEnds {
    const void *init;         // nullable (zeros): packed [B][H][V][K], or cache rows when in_idx is set
    int32_t init_dtype;       // KDA_F32 / KDA_BF16
    const void *in_idx;       // nullable: initial state of sequence b = cache row in_idx[b]
    const uint8_t *in_flags;  // nullable: flags[b] == 0 -> zeros
    int32_t idx_type;         // KDA_I32 / KDA_I64, for in_idx and out_idx
    int64_t n_rows;           // cache rows; an index outside [0, n_rows) means "no row"
    int64_t row_stride;       // elements between cache rows
    float *final_state;       // nullable: packed fp32 [B][H][V][K]
    void *out_cache;          // nullable: final state -> cache row out_idx[b], cast to out_dtype
    int32_t out_dtype;
    const void *out_idx;
    void *ckpt;               // nullable: [ckpt_slots][H][V][K] in ckpt_dtype
    int32_t ckpt_dtype;
    int32_t ckpt_every;       // tokens between checkpoints, a multiple of 64 (0: none)
    int64_t ckpt_slots;       // capacity of ckpt; slots at or beyond it are not written
    const int32_t *ckpt_off;  // [B + 1] first checkpoint slot of each sequence
};

bool prefill_layout(int64_t total_tokens, int64_t num_seqs, int32_t h, int32_t d, PrefillLayout *out);

struct PrefillArgs {
    const void *q, *k, *v;
    int32_t io_dtype;
    const float *g, *beta;
    const int32_t *cu_seqlens;
    int64_t num_seqs, total_tokens;
    int32_t h, d;
    float scale;
    int32_t l2norm;
    StateEnds se;  // ckpt_off is filled in from the workspace
    void *out;
    void *workspace;
    size_t ws_bytes;      // below the layout's total: the compact form (fused kernel)
    void *const *events;  // NULL, or 4 cudaEvent_t (NULL entries skipped) recorded at the kernel boundaries
};
cudaError_t launch_prefill(const PrefillArgs &a, const PrefillLayout &L, cudaStream_t st);

// One CTA that waits, with the bounded mbarrier wait of the kernels, on a barrier
// that gets its arrival (arrive != 0) or never does; *status = 0 or 1 (expired).
cudaError_t launch_bounded_wait_selftest(int32_t *status, uint32_t polls, int32_t arrive, cudaStream_t st);

}  // namespace kda
