// C ABI of the KDA hot path: argument validation on the host (metadata only,
// before any launch) and dispatch to the kernel launchers.
//
// Fail-closed, as the "vllm-ascend KDA state copy" page requires ("Startup
// preparation": bad layouts and metadata are rejected before compile or
// launch; "Numeric contract": an empty selection validates metadata and
// launches nothing).  No call allocates, synchronises or keeps a pointer.
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace {

thread_local cudaError_t t_last_cuda = cudaSuccess;

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return KDA_OK;
    t_last_cuda = e;
    return KDA_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int64_t esize(int32_t dtype) { return dtype == KDA_F32 ? 4 : 2; }

bool valid_dtype(int32_t d) { return d == KDA_F32 || d == KDA_BF16; }

bool valid_itype(int32_t t) { return t == KDA_I32 || t == KDA_I64; }

bool built_head_size(int32_t dk, int32_t dv) { return dk == dv && (dk == 32 || dk == 64 || dk == 128); }

// The prefill has a compact form (the fused kernel, no per-chunk records) for bf16 at head size 128.
bool compact_form(int32_t io_dtype, int32_t dk) { return io_dtype == KDA_BF16 && dk == 128; }

// Layout predicate of the state-copy page ("Automatic dispatch"): fp32/bf16,
// n_rows > 0, positive inner sizes, rows that do not overlap.
int check_cache(const kda_cache *c, kda::CacheDesc *out)
{
    if (c == nullptr || c->data == nullptr) return KDA_ERR_NULL;
    if (!valid_dtype(c->dtype)) return KDA_ERR_DTYPE;
    if (c->reserved != 0) return KDA_ERR_LAYOUT;
    if (c->n_rows <= 0 || c->h <= 0 || c->v <= 0 || c->k <= 0) return KDA_ERR_LAYOUT;
    const int64_t lim = INT64_C(1) << 40;
    if (c->h > lim || c->v > lim || c->k > lim) return KDA_ERR_RANGE;
    const __int128 payload = static_cast<__int128>(c->h) * c->v * c->k;
    if (payload > (INT64_C(1) << 40)) return KDA_ERR_RANGE;
    if (c->row_stride < static_cast<int64_t>(payload)) return KDA_ERR_LAYOUT;
    const __int128 bytes = static_cast<__int128>(c->n_rows) * c->row_stride * esize(c->dtype);
    if (bytes > (static_cast<__int128>(1) << 62)) return KDA_ERR_RANGE;
    if (!aligned(c->data, static_cast<uintptr_t>(esize(c->dtype)))) return KDA_ERR_ALIGN;
    *out = kda::CacheDesc{c->data, c->dtype, c->n_rows, c->h, c->v, c->k, c->row_stride};
    return KDA_OK;
}

int check_index_array(const void *idx, int32_t idx_type)
{
    if (idx == nullptr) return KDA_ERR_NULL;
    if (!aligned(idx, idx_type == KDA_I32 ? 4 : 8)) return KDA_ERR_ALIGN;
    return KDA_OK;
}

}  // namespace

int kda::record_cuda_status(cudaError_t e) { return cuda_status(e); }

extern "C" {

int kda_state_gather(const kda_cache *cache, const void *idx, int32_t idx_type, int64_t selected,
                     const uint8_t *flags, void *packed, void *stream)
{
    kda::CacheDesc c{};
    int rc = check_cache(cache, &c);
    if (rc != KDA_OK) return rc;
    if (!valid_itype(idx_type)) return KDA_ERR_DTYPE;
    if (selected < 0) return KDA_ERR_SHAPE;
    if (selected == 0) return KDA_OK;
    if ((rc = check_index_array(idx, idx_type)) != KDA_OK) return rc;
    if (packed == nullptr) return KDA_ERR_NULL;
    if (!aligned(packed, static_cast<uintptr_t>(esize(c.dtype)))) return KDA_ERR_ALIGN;
    if (static_cast<__int128>(selected) * c.h * c.v * c.k * esize(c.dtype) > (static_cast<__int128>(1) << 62))
        return KDA_ERR_RANGE;
    return cuda_status(kda::launch_state_gather(c, idx, idx_type, selected, flags, packed,
                                                static_cast<cudaStream_t>(stream)));
}

int kda_state_scatter(const kda_cache *cache, const void *idx, int32_t idx_type, int64_t selected,
                      const void *packed, int32_t packed_dtype, void *stream)
{
    kda::CacheDesc c{};
    int rc = check_cache(cache, &c);
    if (rc != KDA_OK) return rc;
    if (!valid_itype(idx_type) || !valid_dtype(packed_dtype)) return KDA_ERR_DTYPE;
    if (selected < 0) return KDA_ERR_SHAPE;
    if (selected == 0) return KDA_OK;
    if ((rc = check_index_array(idx, idx_type)) != KDA_OK) return rc;
    if (packed == nullptr) return KDA_ERR_NULL;
    if (!aligned(packed, static_cast<uintptr_t>(esize(packed_dtype)))) return KDA_ERR_ALIGN;
    if (static_cast<__int128>(selected) * c.h * c.v * c.k * 4 > (static_cast<__int128>(1) << 62))
        return KDA_ERR_RANGE;
    return cuda_status(kda::launch_state_scatter(c, idx, idx_type, selected, packed, packed_dtype,
                                                 static_cast<cudaStream_t>(stream)));
}

size_t kda_prefill_workspace_size(int64_t total_tokens, int64_t num_seqs, int32_t h, int32_t dk, int32_t dv)
{
    if (!built_head_size(dk, dv)) return 0;
    kda::PrefillLayout L{};
    if (!kda::prefill_layout(total_tokens, num_seqs, h, dk, &L)) return 0;
    return L.total;
}

size_t kda_prefill_workspace_size_compact(int64_t total_tokens, int64_t num_seqs, int32_t h, int32_t dk, int32_t dv,
                                          int32_t io_dtype)
{
    if (!built_head_size(dk, dv) || !valid_dtype(io_dtype)) return 0;
    kda::PrefillLayout L{};
    if (!kda::prefill_layout(total_tokens, num_seqs, h, dk, &L)) return 0;
    return compact_form(io_dtype, dk) ? L.compact : L.total;
}

namespace {
// Shared by every prefill entry point; `se` says where states come from and go
// (its cache fields are validated by the caller).
int prefill_impl(const void *q, const void *k, const void *v, int32_t io_dtype, const float *g, const float *beta,
                 const int32_t *cu_seqlens, int64_t num_seqs, int64_t total_tokens, int32_t h, int32_t dk,
                 int32_t dv, float scale, int32_t qk_l2norm, const kda::StateEnds &se, void *out, void *workspace,
                 size_t ws_bytes, void *stream, void *const *events)
{
    if (!valid_dtype(io_dtype)) return KDA_ERR_DTYPE;
    if (se.init != nullptr && !valid_dtype(se.init_dtype)) return KDA_ERR_DTYPE;
    if (num_seqs < 1 || total_tokens < 0 || h < 1 || dk < 1 || dv < 1) return KDA_ERR_SHAPE;
    if (!built_head_size(dk, dv)) return KDA_ERR_UNSUPPORTED;
    if (total_tokens >= (INT64_C(1) << 31) || num_seqs >= (INT64_C(1) << 30) || h > 65535)
        return KDA_ERR_RANGE;
    if (static_cast<__int128>(total_tokens) * h * dk >= (static_cast<__int128>(1) << 62)) return KDA_ERR_RANGE;
    if (cu_seqlens == nullptr || workspace == nullptr) return KDA_ERR_NULL;
    if (total_tokens > 0 && (q == nullptr || k == nullptr || v == nullptr || g == nullptr || beta == nullptr ||
                             out == nullptr))
        return KDA_ERR_NULL;
    const void *vec16[] = {q, k, v, g, out, se.init, se.final_state, se.out_cache, se.ckpt};
    for (const void *p : vec16)
        if (p != nullptr && !aligned(p, 16)) return KDA_ERR_ALIGN;
    if (!aligned(beta, 4) || !aligned(cu_seqlens, 4)) return KDA_ERR_ALIGN;
    kda::PrefillLayout L{};
    if (!kda::prefill_layout(total_tokens, num_seqs, h, dk, &L)) return KDA_ERR_SHAPE;
    if (L.n_chunk_max >= (INT64_C(1) << 31)) return KDA_ERR_RANGE;
    // one-dimensional launch grids: chunk preparation (chunks x heads) and the state pass
    // ((sequence, head) pairs x at most 8 value slices), checked before anything is launched
    if (L.n_chunk_max * h >= (INT64_C(1) << 31) || num_seqs * h * 8 >= (INT64_C(1) << 31)) return KDA_ERR_RANGE;
    if (!aligned(workspace, 256)) return KDA_ERR_WORKSPACE;
    if (ws_bytes < (compact_form(io_dtype, dk) ? L.compact : L.total)) return KDA_ERR_WORKSPACE;
    kda::PrefillArgs a{q, k, v, io_dtype, g, beta, cu_seqlens, num_seqs, total_tokens, h, dk, scale,
                       qk_l2norm ? 1 : 0, se, out, workspace, ws_bytes, events};
    return cuda_status(kda::launch_prefill(a, L, static_cast<cudaStream_t>(stream)));
}

kda::StateEnds packed_ends(const void *init_state, int32_t init_dtype, float *final_state)
{
    kda::StateEnds se{};
    se.init = init_state;
    se.init_dtype = init_dtype;
    se.final_state = final_state;
    return se;
}
}  // namespace

int kda_prefill_varlen(const void *q, const void *k, const void *v, int32_t io_dtype, const float *g,
                       const float *beta, const int32_t *cu_seqlens, int64_t num_seqs, int64_t total_tokens,
                       int32_t h, int32_t dk, int32_t dv, float scale, int32_t qk_l2norm, const void *init_state,
                       int32_t init_dtype, float *final_state, void *out, void *workspace, size_t ws_bytes,
                       void *stream)
{
    return prefill_impl(q, k, v, io_dtype, g, beta, cu_seqlens, num_seqs, total_tokens, h, dk, dv, scale,
                        qk_l2norm, packed_ends(init_state, init_dtype, final_state), out, workspace, ws_bytes,
                        stream, nullptr);
}

int kda_prefill_varlen_timed(const void *q, const void *k, const void *v, int32_t io_dtype, const float *g,
                             const float *beta, const int32_t *cu_seqlens, int64_t num_seqs,
                             int64_t total_tokens, int32_t h, int32_t dk, int32_t dv, float scale,
                             int32_t qk_l2norm, const void *init_state, int32_t init_dtype, float *final_state,
                             void *out, void *workspace, size_t ws_bytes, void *stream, void *const *events)
{
    if (events == nullptr) return KDA_ERR_NULL;  // NULL entries: boundaries left unrecorded
    return prefill_impl(q, k, v, io_dtype, g, beta, cu_seqlens, num_seqs, total_tokens, h, dk, dv, scale,
                        qk_l2norm, packed_ends(init_state, init_dtype, final_state), out, workspace, ws_bytes,
                        stream, events);
}

int kda_prefill_varlen_cached(const void *q, const void *k, const void *v, int32_t io_dtype, const float *g,
                              const float *beta, const int32_t *cu_seqlens, int64_t num_seqs, int64_t total_tokens,
                              int32_t h, int32_t dk, int32_t dv, float scale, int32_t qk_l2norm,
                              const kda_cache *cache, const void *idx_in, const uint8_t *flags,
                              const void *idx_out, int32_t idx_type, float *final_state, void *checkpoints,
                              int32_t ckpt_dtype, int32_t ckpt_every, int64_t ckpt_slots, void *out,
                              void *workspace, size_t ws_bytes, void *stream)
{
    kda::CacheDesc c{};
    int rc = check_cache(cache, &c);
    if (rc != KDA_OK) return rc;
    if (!valid_itype(idx_type)) return KDA_ERR_DTYPE;
    if (c.h != h || c.k != dk || c.v != dv) return KDA_ERR_SHAPE;
    if (!aligned(c.data, 16) || (c.row_stride * esize(c.dtype)) % 16 != 0) return KDA_ERR_ALIGN;
    if ((rc = check_index_array(idx_in, idx_type)) != KDA_OK) return rc;
    if (idx_out != nullptr && (rc = check_index_array(idx_out, idx_type)) != KDA_OK) return rc;
    if (checkpoints != nullptr) {
        if (!valid_dtype(ckpt_dtype)) return KDA_ERR_DTYPE;
        if (ckpt_every <= 0 || ckpt_every % 64 != 0 || ckpt_slots < 0) return KDA_ERR_SHAPE;
    }
    kda::StateEnds se{};
    se.init = c.data;
    se.init_dtype = c.dtype;
    se.in_idx = idx_in;
    se.in_flags = flags;
    se.idx_type = idx_type;
    se.n_rows = c.n_rows;
    se.row_stride = c.row_stride;
    se.final_state = final_state;
    se.out_cache = idx_out != nullptr ? c.data : nullptr;
    se.out_dtype = c.dtype;
    se.out_idx = idx_out;
    se.ckpt = checkpoints;
    se.ckpt_dtype = ckpt_dtype;
    se.ckpt_every = checkpoints != nullptr ? ckpt_every : 0;
    se.ckpt_slots = ckpt_slots;
    return prefill_impl(q, k, v, io_dtype, g, beta, cu_seqlens, num_seqs, total_tokens, h, dk, dv, scale,
                        qk_l2norm, se, out, workspace, ws_bytes, stream, nullptr);
}

int64_t kda_prefill_checkpoint_count(const int32_t *cu_seqlens_host, int64_t num_seqs, int32_t ckpt_every)
{
    if (cu_seqlens_host == nullptr || num_seqs < 1 || ckpt_every <= 0 || ckpt_every % 64 != 0) return -1;
    int64_t n = 0;
    for (int64_t b = 0; b < num_seqs; ++b) {
        const int64_t len = static_cast<int64_t>(cu_seqlens_host[b + 1]) - cu_seqlens_host[b];
        if (len < 0) return -1;
        n += len / ckpt_every;
    }
    return n;
}

int kda_decode_step(const void *q, const void *k, const void *v, int32_t io_dtype, const float *g,
                    const float *beta, int64_t batch, int32_t h, int32_t dk, int32_t dv, float scale,
                    int32_t qk_l2norm, const kda_cache *cache, const void *idx, int32_t idx_type, void *out,
                    void *stream)
{
    kda::CacheDesc c{};
    int rc = check_cache(cache, &c);
    if (rc != KDA_OK) return rc;
    if (!valid_dtype(io_dtype) || !valid_itype(idx_type)) return KDA_ERR_DTYPE;
    if (batch < 0 || h < 1 || dk < 1 || dv < 1) return KDA_ERR_SHAPE;
    if (!built_head_size(dk, dv)) return KDA_ERR_UNSUPPORTED;
    if (c.h != h || c.k != dk || c.v != dv) return KDA_ERR_SHAPE;
    if (batch == 0) return KDA_OK;
    if (batch * static_cast<int64_t>(h) >= (INT64_C(1) << 31)) return KDA_ERR_RANGE;
    if ((rc = check_index_array(idx, idx_type)) != KDA_OK) return rc;
    if (q == nullptr || k == nullptr || v == nullptr || g == nullptr || beta == nullptr || out == nullptr)
        return KDA_ERR_NULL;
    const void *vec16[] = {q, k, v, g, out, c.data};
    for (const void *p : vec16)
        if (!aligned(p, 16)) return KDA_ERR_ALIGN;
    if (!aligned(beta, 4)) return KDA_ERR_ALIGN;
    if ((c.row_stride * esize(c.dtype)) % 16 != 0) return KDA_ERR_ALIGN;
    kda::DecodeArgs a{q, k, v, io_dtype, g, beta, batch, h, dk, scale, qk_l2norm ? 1 : 0, c, idx, idx_type, out};
    return cuda_status(kda::launch_decode_step(a, static_cast<cudaStream_t>(stream)));
}

namespace {
// Shared checks of the INT8 checkpoint calls: a built head size, 16-byte rows,
// aligned index arrays and checkpoint buffers.
int check_ckpt_args(const kda_cache *active, kda::CacheDesc *c, const void *src, const void *dst,
                    int32_t idx_type, int64_t count, const void *qdata, const void *scale, int64_t n_slots)
{
    int rc = check_cache(active, c);
    if (rc != KDA_OK) return rc;
    if (!valid_itype(idx_type)) return KDA_ERR_DTYPE;
    if (count < 0 || n_slots < 0) return KDA_ERR_SHAPE;
    if (!built_head_size(static_cast<int32_t>(c->k), static_cast<int32_t>(c->v))) return KDA_ERR_UNSUPPORTED;
    if (c->h > 65535) return KDA_ERR_RANGE;
    if (count == 0) return KDA_OK;
    if (count * c->h >= (INT64_C(1) << 31)) return KDA_ERR_RANGE;
    if ((rc = check_index_array(src, idx_type)) != KDA_OK) return rc;
    if ((rc = check_index_array(dst, idx_type)) != KDA_OK) return rc;
    if (qdata == nullptr || scale == nullptr) return KDA_ERR_NULL;
    if (!aligned(qdata, 16) || !aligned(scale, 16) || !aligned(c->data, 16)) return KDA_ERR_ALIGN;
    if ((c->row_stride * esize(c->dtype)) % 16 != 0) return KDA_ERR_ALIGN;
    return KDA_OK;
}
}  // namespace

int kda_ckpt_store_int8(const kda_cache *active, const void *src_rows, const void *dst_slots, int32_t idx_type,
                        int64_t count, int8_t *qdata, float *scale, int64_t n_slots, void *stream)
{
    kda::CacheDesc c{};
    const int rc = check_ckpt_args(active, &c, src_rows, dst_slots, idx_type, count, qdata, scale, n_slots);
    if (rc != KDA_OK || count == 0) return rc;
    return cuda_status(kda::launch_ckpt_store_int8(c, src_rows, dst_slots, idx_type, count, qdata, scale, n_slots,
                                                   static_cast<cudaStream_t>(stream)));
}

int kda_ckpt_load_int8(const int8_t *qdata, const float *scale, int64_t n_slots, const void *src_slots,
                       const void *dst_rows, int32_t idx_type, int64_t count, const kda_cache *active, void *stream)
{
    kda::CacheDesc c{};
    const int rc = check_ckpt_args(active, &c, src_slots, dst_rows, idx_type, count, qdata, scale, n_slots);
    if (rc != KDA_OK || count == 0) return rc;
    return cuda_status(kda::launch_ckpt_load_int8(c, qdata, scale, n_slots, src_slots, dst_rows, idx_type, count,
                                                  static_cast<cudaStream_t>(stream)));
}

int kda_target_verify(const void *q, const void *k, const void *v, int32_t io_dtype, const float *g,
                      const float *beta, int64_t batch, int32_t L, int32_t h, int32_t dk, int32_t dv, float scale,
                      int32_t qk_l2norm, const kda_cache *cache, const void *idx, const kda_cache *pool,
                      const void *inter_idx, int32_t idx_type, void *out, void *stream)
{
    kda::CacheDesc c{}, pl{};
    int rc = check_cache(cache, &c);
    if (rc != KDA_OK) return rc;
    if ((rc = check_cache(pool, &pl)) != KDA_OK) return rc;
    if (!valid_dtype(io_dtype) || !valid_itype(idx_type)) return KDA_ERR_DTYPE;
    if (batch < 0 || L < 1 || h < 1 || dk < 1 || dv < 1) return KDA_ERR_SHAPE;
    if (!built_head_size(dk, dv)) return KDA_ERR_UNSUPPORTED;
    if (c.h != h || c.k != dk || c.v != dv || pl.h != h || pl.k != dk || pl.v != dv) return KDA_ERR_SHAPE;
    if (batch == 0) return KDA_OK;
    if (batch * static_cast<int64_t>(h) >= (INT64_C(1) << 31) || L > (1 << 20)) return KDA_ERR_RANGE;
    if ((rc = check_index_array(idx, idx_type)) != KDA_OK) return rc;
    if ((rc = check_index_array(inter_idx, idx_type)) != KDA_OK) return rc;
    if (q == nullptr || k == nullptr || v == nullptr || g == nullptr || beta == nullptr || out == nullptr)
        return KDA_ERR_NULL;
    const void *vec16[] = {q, k, v, g, c.data, pl.data};
    for (const void *p : vec16)
        if (!aligned(p, 16)) return KDA_ERR_ALIGN;
    if (!aligned(beta, 4) || !aligned(out, 4)) return KDA_ERR_ALIGN;
    if ((c.row_stride * esize(c.dtype)) % 16 != 0 || (pl.row_stride * esize(pl.dtype)) % 16 != 0)
        return KDA_ERR_ALIGN;
    kda::VerifyArgs a{q, k, v, io_dtype, g, beta, batch, L, h, dk, scale, qk_l2norm ? 1 : 0, c, idx, pl, inter_idx,
                      idx_type, out};
    return cuda_status(kda::launch_target_verify(a, static_cast<cudaStream_t>(stream)));
}

namespace {
int check_conv_common(const void *x, int32_t io_dtype, int64_t channels, int32_t width, const float *weight,
                      const float *bias, int32_t activation, const void *y)
{
    if (!valid_dtype(io_dtype)) return KDA_ERR_DTYPE;
    if (width < 2 || width > 4 || channels < 1) return KDA_ERR_UNSUPPORTED;
    if (channels % 8 != 0) return KDA_ERR_SHAPE;
    if (activation != 0 && activation != 1) return KDA_ERR_SHAPE;
    // channel blocks sit in the y dimension of the per-sequence and update grids
    if (channels > INT64_C(65535) * kda::kConvChannelsPerBlock) return KDA_ERR_RANGE;
    if (weight == nullptr) return KDA_ERR_NULL;
    const void *vec16[] = {x, weight, bias, y};
    for (const void *p : vec16)
        if (p != nullptr && !aligned(p, 16)) return KDA_ERR_ALIGN;
    return KDA_OK;
}
}  // namespace

int kda_conv1d_varlen(const void *x, int32_t io_dtype, const int32_t *cu_seqlens, int64_t num_seqs,
                      int64_t total_tokens, int64_t channels, int32_t width, const float *weight, const float *bias,
                      int32_t activation, const void *init_state, void *final_state, int32_t state_dtype, void *y,
                      void *stream)
{
    int rc = check_conv_common(x, io_dtype, channels, width, weight, bias, activation, y);
    if (rc != KDA_OK) return rc;
    if ((init_state != nullptr || final_state != nullptr) && !valid_dtype(state_dtype)) return KDA_ERR_DTYPE;
    if (num_seqs < 1 || total_tokens < 0) return KDA_ERR_SHAPE;
    if (num_seqs >= (INT64_C(1) << 30) || total_tokens >= (INT64_C(1) << 36)) return KDA_ERR_RANGE;
    if ((total_tokens + 15) / 16 >= (INT64_C(1) << 31)) return KDA_ERR_RANGE;
    // one-dimensional grid of (token block, channel block) pairs, token blocks of 8 or more tokens
    const int64_t cblocks = (channels + kda::kConvChannelsPerBlock - 1) / kda::kConvChannelsPerBlock;
    if ((total_tokens + 15) / 8 * cblocks > INT64_C(0x7fffffff)) return KDA_ERR_RANGE;
    if (cu_seqlens == nullptr) return KDA_ERR_NULL;
    if (total_tokens > 0 && (x == nullptr || y == nullptr)) return KDA_ERR_NULL;
    if (!aligned(cu_seqlens, 4)) return KDA_ERR_ALIGN;
    const void *st16[] = {init_state, final_state};
    for (const void *p : st16)
        if (p != nullptr && !aligned(p, 16)) return KDA_ERR_ALIGN;
    kda::Conv1dArgs a{x, io_dtype, cu_seqlens, num_seqs, total_tokens, channels, width, weight, bias, activation,
                      init_state, final_state, state_dtype, y};
    return cuda_status(kda::launch_conv1d_varlen(a, static_cast<cudaStream_t>(stream)));
}

int kda_conv1d_update(const void *x, int32_t io_dtype, int64_t batch, int64_t channels, int32_t width,
                      const float *weight, const float *bias, int32_t activation, const kda_cache *conv_cache,
                      const void *idx, int32_t idx_type, void *y, void *stream)
{
    kda::CacheDesc c{};
    int rc = check_cache(conv_cache, &c);
    if (rc != KDA_OK) return rc;
    if ((rc = check_conv_common(x, io_dtype, channels, width, weight, bias, activation, y)) != KDA_OK) return rc;
    if (!valid_itype(idx_type)) return KDA_ERR_DTYPE;
    if (c.h != 1 || c.v != width - 1 || c.k != channels) return KDA_ERR_SHAPE;
    if (batch < 0) return KDA_ERR_SHAPE;
    if (batch == 0) return KDA_OK;
    if (batch >= (INT64_C(1) << 31)) return KDA_ERR_RANGE;
    if ((rc = check_index_array(idx, idx_type)) != KDA_OK) return rc;
    if (x == nullptr || y == nullptr) return KDA_ERR_NULL;
    if (!aligned(c.data, 16) || (c.row_stride * esize(c.dtype)) % 16 != 0) return KDA_ERR_ALIGN;
    kda::Conv1dUpdateArgs a{x, io_dtype, batch, channels, width, weight, bias, activation, c, idx, idx_type, y};
    return cuda_status(kda::launch_conv1d_update(a, static_cast<cudaStream_t>(stream)));
}

const char *kda_status_string(int32_t status)
{
    switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_NULL: return "KDA_ERR_NULL: a required pointer is NULL";
    case KDA_ERR_DTYPE: return "KDA_ERR_DTYPE: unknown or unsupported element or index type";
    case KDA_ERR_LAYOUT: return "KDA_ERR_LAYOUT: invalid cache layout (n_rows, sizes or row stride)";
    case KDA_ERR_SHAPE: return "KDA_ERR_SHAPE: invalid size or shape";
    case KDA_ERR_RANGE: return "KDA_ERR_RANGE: size beyond the supported range";
    case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE: workspace missing, too small or misaligned";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA launch failed";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: head size combination not built";
    case KDA_ERR_ALIGN: return "KDA_ERR_ALIGN: pointer or stride misaligned";
    default: return "unknown kda_status";
    }
}

const char *kda_last_cuda_error_string(void) { return cudaGetErrorString(t_last_cuda); }

int kda_selftest_bounded_wait(int32_t *status_dev, uint32_t polls, int32_t arrive, void *stream)
{
    if (status_dev == nullptr) return KDA_ERR_NULL;
    if (polls == 0) return KDA_ERR_RANGE;
    return cuda_status(kda::launch_bounded_wait_selftest(status_dev, polls, arrive, static_cast<cudaStream_t>(stream)));
}

int kda_prefill_workspace_status(const void *workspace, int32_t *status_out, void *stream)
{
    if (workspace == nullptr || status_out == nullptr) return KDA_ERR_NULL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(status_out, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return cuda_status(e);
}

}  // extern "C"
