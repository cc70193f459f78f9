// Definitions shared by the prefill kernels: the per-(chunk, head) workspace
// record written by the chunk-preparation kernel and read by the state pass,
// and small load/store helpers.
#pragma once

#include <cuda.h>

#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace prefill {

constexpr int C = kChunk;  // 64 tokens per chunk

// Byte offset of bf16 element (r, c) of a [ROWS][D] tile.  D >= 64: the
// canonical 128-byte-swizzle layout of the tensor cores - 64-column slabs of
// ROWS rows x 128 bytes, 16-byte chunks XOR-permuted by r % 8 - which serves as
// a K-major operand when the long side is K and as an MN-major one when it is
// N.  D == 32: 64-byte rows with the 64-byte permutation.
template <int D, int ROWS> __device__ __forceinline__ uint32_t tile_off(int r, int c)
{
    if constexpr (D >= 64) return static_cast<uint32_t>((c >> 6) * (ROWS * 128)) + swz_off<128>(r, c & 63);
    else return swz_off<64>(r, c);
}
template <int D> __host__ __device__ constexpr int tile_row_bytes() { return D >= 64 ? 128 : 64; }

// One record per (chunk, head).  bf16 tiles use tile_off (A_qk and U^T: 128-
// byte rows) so the state pass can bulk-copy a record verbatim into shared
// memory and use it directly as tensor-core operands.  W and Q~ are the rows
// 0..63 and 64..127 of one [128][D] tile, so that a single operand of 128 rows
// (or N = 128) takes both.
template <int D> struct Rec {
    static constexpr int TILE = C * D * 2;            // bf16 [64][D]
    static constexpr int WQ = 0;                      // [W; Q~] [128][D]  (Q~ = scale q e^G)
    static constexpr int KT = 2 * TILE;               // K~      [64][D]  (k e^{G_last - G})
    static constexpr int AQK = 3 * TILE;              // A_qk    [64][64] (scaled, causal)
    static constexpr int GAMMA = AQK + C * C * 2;     // e^G_last [D] fp32
    static constexpr int UT = GAMMA + D * 4;          // U^T     [D][64]
    static constexpr int BYTES = UT + D * C * 2;
    static_assert(UT % 128 == 0 && BYTES % 128 == 0, "record alignment");
    // byte offsets of W[r][c] and Q~[r][c]
    static __device__ __forceinline__ uint32_t w_at(int r, int c) { return WQ + tile_off<D, 2 * C>(r, c); }
    static __device__ __forceinline__ uint32_t qt_at(int r, int c) { return WQ + tile_off<D, 2 * C>(C + r, c); }
};

inline int rec_bytes_for(int d)
{
    switch (d) {
    case 32: return Rec<32>::BYTES;
    case 64: return Rec<64>::BYTES;
    case 128: return Rec<128>::BYTES;
    default: return 0;
    }
}

struct PrepParams {
    const void *q, *k, *v;
    const float *g, *beta;
    const int2 *chunk_info;  // per chunk {first token, length}; length 0 past the last chunk
    int32_t H;
    float scale;
    int32_t l2norm;
    char *records;
    int32_t *status;       // workspace status word (3: a bounded wait of the prep expired)
    int64_t total_tokens;  // rows of q, k, v (host side: the tensor maps' extent)
    int32_t *fix_count;    // (chunk, head) items whose decay the block split cannot take ...
    int32_t *fix_list;     // ... (chunk * H + head), formed by the exact kernel
    int64_t chunk_base;    // first chunk of this launch (CTA i takes chunk chunk_base + i / H)
};

// Tensor maps of the bf16 q, k, v inputs [T][H][D] (3-D: channel, head, token;
// boxes of 64 channels x 1 head x 64 tokens, 128-byte swizzle), encoded on the
// host per call and passed as a __grid_constant__ kernel parameter.
struct PrepMaps {
    CUtensorMap q, k, v;
};

struct PassParams {
    const int32_t *cu;
    const int32_t *chunk_off;
    const int32_t *seq_order;
    int32_t *status;
    const char *records;
    int32_t H;
    StateEnds se;
    void *out;
    // A segment of every sequence's chunks, [seg_lo, seg_hi) (the value-split tensor-memory pass
    // only): a segment after the first starts from seg_state, one before the last ends in it
    // (fp32 [B][H][V][K]); the defaults take whole sequences.
    int32_t seg_lo = 0, seg_hi = 0x7fffffff;
    float *seg_state = nullptr;
};

__device__ __forceinline__ int64_t row_index(const void *idx, int32_t it, int64_t b)
{
    return it == KDA_I64 ? static_cast<const int64_t *>(idx)[b] : static_cast<const int32_t *>(idx)[b];
}

// Base element offset of sequence b's initial state, or -1 for zeros.
__device__ __forceinline__ int64_t init_base(const StateEnds &e, int64_t b, int64_t per_seq)
{
    if (e.init == nullptr) return -1;
    if (e.in_idx == nullptr) return b * per_seq;
    const int64_t r = row_index(e.in_idx, e.idx_type, b);
    if (r < 0 || r >= e.n_rows || (e.in_flags != nullptr && e.in_flags[b] == 0)) return -1;
    return r * e.row_stride;
}

// Base element offset of the cache row that receives sequence b's final state, or -1.
__device__ __forceinline__ int64_t out_base(const StateEnds &e, int64_t b)
{
    if (e.out_cache == nullptr) return -1;
    const int64_t r = row_index(e.out_idx, e.idx_type, b);
    return (r < 0 || r >= e.n_rows) ? -1 : r * e.row_stride;
}

// Checkpoint slot written after chunk c (0-based) of sequence b, or -1.
__device__ __forceinline__ int64_t ckpt_slot(const StateEnds &e, int64_t b, int32_t c, int64_t len)
{
    if (e.ckpt == nullptr || e.ckpt_every <= 0) return -1;
    const int64_t end = static_cast<int64_t>(c + 1) * kChunk;  // tokens done after chunk c
    if (end > len || end % e.ckpt_every != 0) return -1;
    const int64_t s = e.ckpt_off[b] + end / e.ckpt_every - 1;
    return s < e.ckpt_slots ? s : -1;
}

// Four consecutive state elements: load as fp32 / store with the dtype's cast (bf16: RNE).
__device__ __forceinline__ float4 load_state4(const void *base, int32_t dtype, int64_t e)
{
    if (dtype == KDA_F32) return *reinterpret_cast<const float4 *>(static_cast<const float *>(base) + e);
    const uint2 u = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(base) + e);
    return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
}
__device__ __forceinline__ void store_state4(void *base, int32_t dtype, int64_t e, float4 x)
{
    if (dtype == KDA_F32) {
        *reinterpret_cast<float4 *>(static_cast<float *>(base) + e) = x;
    } else {
        *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(base) + e) =
            make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w));
    }
}
__device__ __forceinline__ float2 load_state2(const void *base, int32_t dtype, int64_t e)
{
    if (dtype == KDA_F32) return *reinterpret_cast<const float2 *>(static_cast<const float *>(base) + e);
    const uint32_t u = *reinterpret_cast<const uint32_t *>(static_cast<const uint16_t *>(base) + e);
    return make_float2(bf16_lo(u), bf16_hi(u));
}
__device__ __forceinline__ void store_state2(void *base, int32_t dtype, int64_t e, float2 x)
{
    if (dtype == KDA_F32) *reinterpret_cast<float2 *>(static_cast<float *>(base) + e) = x;
    else *reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(base) + e) = pack_bf16x2(x.x, x.y);
}

// Launches the tensor-memory state pass (D = 128, bf16 output, one CTA per
// (sequence, head)) over `items` = num_seqs x h CTAs.
cudaError_t launch_state_pass_tc(const PassParams &p, int64_t items, cudaStream_t st);
// Value-split form: state_pass_split_slices() CTAs per (sequence, head).
int state_pass_split_slices();
cudaError_t launch_state_pass_split(const PassParams &p, int64_t items, cudaStream_t st);

// Tensor map of a bf16 input [T][H][D]: dims (D, H, T), boxes of 64 channels x 1 head
// x 64 tokens, 128-byte swizzle, zeros outside the tensor (chunk_prep.cu).
bool encode_rows(CUtensorMap *m, const void *base, int64_t T, int32_t H, int D);
// ... of an fp32 input [T][H][D] with boxes of D channels x 1 head x 64 tokens, no swizzle.
bool encode_rows_f32(CUtensorMap *m, const float *base, int64_t T, int32_t H, int D);

// Launches the fused prefill (head size 128, bf16 q, k, v and outputs): one persistent CTA per
// SM (at most one per item) over the num_seqs x h (sequence, head) items in seq_order.
// status[0] receives 5 if a bounded wait expires; *item_counter must be zero.
cudaError_t launch_prefill_fused(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                 const int32_t *cu, const int32_t *seq_order, int32_t *status, int32_t *item_counter,
                                 int64_t num_seqs, int64_t total_tokens, int32_t h, float scale, int32_t l2norm,
                                 const StateEnds &se, void *out, cudaStream_t st);

// Launches the chunk-preparation kernel over n_chunk_max x h CTAs (heads fastest).
cudaError_t launch_chunk_prep(int d, int32_t io_dtype, const PrepParams &p, int64_t n_chunk_max, int32_t h,
                              cudaStream_t st);

// N consecutive io elements as fp32 (N = 1, 2 or 4; pointer aligned to N elements).
template <typename IO, int N> __device__ __forceinline__ void load_slice(const IO *p, float x[N])
{
    if constexpr (sizeof(IO) == 4) {
        if constexpr (N == 4) {
            const float4 a = *reinterpret_cast<const float4 *>(p);
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        } else if constexpr (N == 2) {
            const float2 a = *reinterpret_cast<const float2 *>(p);
            x[0] = a.x; x[1] = a.y;
        } else {
            x[0] = *reinterpret_cast<const float *>(p);
        }
    } else {
        if constexpr (N == 4) {
            const uint2 a = *reinterpret_cast<const uint2 *>(p);
            x[0] = bf16_lo(a.x); x[1] = bf16_hi(a.x); x[2] = bf16_lo(a.y); x[3] = bf16_hi(a.y);
        } else if constexpr (N == 2) {
            const uint32_t a = *reinterpret_cast<const uint32_t *>(p);
            x[0] = bf16_lo(a); x[1] = bf16_hi(a);
        } else {
            x[0] = bf16_bits_to_f32(*reinterpret_cast<const uint16_t *>(p));
        }
    }
}

// Store N (1, 2 or 4) consecutive values as bf16 at byte offset `off` of `base`.
template <int N> __device__ __forceinline__ void store_bf16(char *base, uint32_t off, const float x[N])
{
    if constexpr (N == 4) {
        *reinterpret_cast<uint2 *>(base + off) = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
    } else if constexpr (N == 2) {
        *reinterpret_cast<uint32_t *>(base + off) = pack_bf16x2(x[0], x[1]);
    } else {
        *reinterpret_cast<uint16_t *>(base + off) = f32_to_bf16_bits(x[0]);
    }
}

}  // namespace prefill
}  // namespace kda
