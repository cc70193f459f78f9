// Definitions shared by the prefill kernels: the per-(chunk, head) workspace
// record written by the chunk-preparation kernel and read by the state pass,
// and small load/store helpers.
#pragma once

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
// memory and use it directly as tensor-core operands.
template <int D> struct Rec {
    static constexpr int TILE = C * D * 2;            // bf16 [64][D]
    static constexpr int W = 0;                       // W       [64][D]
    static constexpr int QT = TILE;                   // Q~      [64][D]  (scale q e^G)
    static constexpr int KT = 2 * TILE;               // K~      [64][D]  (k e^{G_last - G})
    static constexpr int AQK = 3 * TILE;              // A_qk    [64][64] (scaled, causal)
    static constexpr int GAMMA = AQK + C * C * 2;     // e^G_last [D] fp32
    static constexpr int UT = GAMMA + D * 4;          // U^T     [D][64]
    static constexpr int BYTES = UT + D * C * 2;
    static_assert(UT % 128 == 0 && BYTES % 128 == 0, "record alignment");
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
};

struct PassParams {
    const int32_t *cu;
    const int32_t *chunk_off;
    const int32_t *seq_order;
    int32_t *status;
    const char *records;
    int32_t H;
    const void *init;
    int32_t init_dtype;
    float *final_state;
    void *out;
};

// Launches the tensor-memory state pass (D = 128, bf16 output, one CTA per
// (sequence, head)) over `items` = num_seqs x h CTAs.
cudaError_t launch_state_pass_tc(const PassParams &p, int64_t items, cudaStream_t st);

// Launches the chunk-preparation kernel over n_chunk_max x h CTAs.
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
