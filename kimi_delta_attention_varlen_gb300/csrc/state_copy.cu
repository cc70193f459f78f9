// State gather / scatter between a paged [N, H, V, K] cache and packed rows.
//
// Contract: "vllm-ascend KDA state copy" page, section "Numeric contract".
//   gather:  packed[s] = cache[idx[s]] if 0 <= idx[s] < N and flag, else 0
//   scatter: cache[idx[s]] = convert(packed[s]) if 0 <= idx[s] < N
// Every row address is formed as int64(idx) * row_stride, so int32 indices
// and rows more than 4 GiB apart resolve ("Memory and addressing").
//
// Layout on the GPU: one CTA copies one tile of one selected row; the grid is
// (tiles per row, selected rows).  Row validity is evaluated once per thread
// from the same two words, so it is uniform across the CTA (no divergence).
// Payload bytes move as 16-byte vectors with non-allocating loads and
// streaming stores; layouts that are not 16-byte aligned take the scalar
// kernels instead.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kVecPerThread = 4;  // 16-byte vectors in flight per thread
constexpr int kMaxGridY = 65535;

template <typename IdxT>
__device__ __forceinline__ bool row_valid(const IdxT *idx, const uint8_t *flags, int64_t s,
                                          int64_t n_rows, int64_t *row)
{
    const int64_t r = static_cast<int64_t>(idx[s]);
    *row = r;
    return r >= 0 && r < n_rows && (flags == nullptr || flags[s] != 0);
}

// Bitwise row copy in 16-byte vectors.  GATHER: cache -> packed (zeros for
// invalid rows).  !GATHER: packed -> cache (same dtype), invalid rows skipped.
template <typename IdxT, bool GATHER>
__global__ void __launch_bounds__(kCopyThreads)
copy_rows_v16(uint4 *__restrict__ cache, int64_t n_rows, int64_t stride_v16, int64_t payload_v16,
              const IdxT *__restrict__ idx, const uint8_t *__restrict__ flags, int64_t selected,
              uint4 *__restrict__ packed)
{
    const int64_t v0 = static_cast<int64_t>(blockIdx.x) * (kCopyThreads * kVecPerThread) + threadIdx.x;
    for (int64_t s = blockIdx.y; s < selected; s += gridDim.y) {
        int64_t row;
        const bool valid = row_valid(idx, GATHER ? flags : nullptr, s, n_rows, &row);
        if (!GATHER && !valid) continue;
        uint4 *crow = cache + (valid ? row : 0) * stride_v16;
        uint4 *prow = packed + s * payload_v16;
        uint4 buf[kVecPerThread];
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const int64_t v = v0 + u * kCopyThreads;
            buf[u] = make_uint4(0u, 0u, 0u, 0u);
            if (v < payload_v16 && valid) buf[u] = ld_nc_v4(GATHER ? crow + v : prow + v);
        }
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const int64_t v = v0 + u * kCopyThreads;
            if (v < payload_v16) st_cs_v4(GATHER ? prow + v : crow + v, buf[u]);
        }
    }
}

// Scatter with conversion, 8 elements per unit: fp32 -> bf16 (RNE) or
// bf16 -> fp32 (exact).  Requires 16-byte aligned bases / strides.
template <typename IdxT, typename SrcT, typename DstT>
__global__ void __launch_bounds__(kCopyThreads)
scatter_cast_v(DstT *__restrict__ cache, int64_t n_rows, int64_t row_stride, int64_t payload,
               const IdxT *__restrict__ idx, int64_t selected, const SrcT *__restrict__ packed)
{
    const int64_t units = payload / 8;
    const int64_t u0 = static_cast<int64_t>(blockIdx.x) * (kCopyThreads * kVecPerThread) + threadIdx.x;
    for (int64_t s = blockIdx.y; s < selected; s += gridDim.y) {
        int64_t row;
        if (!row_valid(idx, static_cast<const uint8_t *>(nullptr), s, n_rows, &row)) continue;
        DstT *crow = cache + row * row_stride;
        const SrcT *prow = packed + s * payload;
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const int64_t unit = u0 + u * kCopyThreads;
            if (unit >= units) continue;
            if constexpr (sizeof(SrcT) == 4) {  // fp32 -> bf16
                const uint4 a = ld_nc_v4(prow + unit * 8);
                const uint4 b = ld_nc_v4(prow + unit * 8 + 4);
                uint4 o;
                o.x = pack_bf16x2(__uint_as_float(a.x), __uint_as_float(a.y));
                o.y = pack_bf16x2(__uint_as_float(a.z), __uint_as_float(a.w));
                o.z = pack_bf16x2(__uint_as_float(b.x), __uint_as_float(b.y));
                o.w = pack_bf16x2(__uint_as_float(b.z), __uint_as_float(b.w));
                st_cs_v4(crow + unit * 8, o);
            } else {  // bf16 -> fp32
                const uint4 a = ld_nc_v4(prow + unit * 8);
                uint4 lo, hi;
                lo.x = __float_as_uint(bf16_lo(a.x));
                lo.y = __float_as_uint(bf16_hi(a.x));
                lo.z = __float_as_uint(bf16_lo(a.y));
                lo.w = __float_as_uint(bf16_hi(a.y));
                hi.x = __float_as_uint(bf16_lo(a.z));
                hi.y = __float_as_uint(bf16_hi(a.z));
                hi.z = __float_as_uint(bf16_lo(a.w));
                hi.w = __float_as_uint(bf16_hi(a.w));
                st_cs_v4(crow + unit * 8, lo);
                st_cs_v4(crow + unit * 8 + 4, hi);
            }
        }
    }
}

template <typename T> __device__ __forceinline__ float elem_to_f32(T x);
template <> __device__ __forceinline__ float elem_to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float elem_to_f32<uint16_t>(uint16_t x) { return bf16_bits_to_f32(x); }
template <typename T> __device__ __forceinline__ T f32_to_elem(float x);
template <> __device__ __forceinline__ float f32_to_elem<float>(float x) { return x; }
template <> __device__ __forceinline__ uint16_t f32_to_elem<uint16_t>(float x) { return f32_to_bf16_bits(x); }

// Element-wise kernels for layouts that are not 16-byte aligned.
template <typename IdxT, typename T>
__global__ void __launch_bounds__(kCopyThreads)
gather_scalar(const T *__restrict__ cache, int64_t n_rows, int64_t row_stride, int64_t payload,
              const IdxT *__restrict__ idx, const uint8_t *__restrict__ flags, int64_t selected,
              T *__restrict__ packed)
{
    const int64_t e = static_cast<int64_t>(blockIdx.x) * kCopyThreads + threadIdx.x;
    if (e >= payload) return;
    for (int64_t s = blockIdx.y; s < selected; s += gridDim.y) {
        int64_t row;
        const bool valid = row_valid(idx, flags, s, n_rows, &row);
        packed[s * payload + e] = valid ? cache[row * row_stride + e] : T(0);
    }
}

template <typename IdxT, typename SrcT, typename DstT>
__global__ void __launch_bounds__(kCopyThreads)
scatter_scalar(DstT *__restrict__ cache, int64_t n_rows, int64_t row_stride, int64_t payload,
               const IdxT *__restrict__ idx, int64_t selected, const SrcT *__restrict__ packed)
{
    const int64_t e = static_cast<int64_t>(blockIdx.x) * kCopyThreads + threadIdx.x;
    if (e >= payload) return;
    for (int64_t s = blockIdx.y; s < selected; s += gridDim.y) {
        int64_t row;
        if (!row_valid(idx, static_cast<const uint8_t *>(nullptr), s, n_rows, &row)) continue;
        const SrcT x = packed[s * payload + e];
        if constexpr (sizeof(SrcT) == sizeof(DstT)) cache[row * row_stride + e] = x;
        else cache[row * row_stride + e] = f32_to_elem<DstT>(elem_to_f32<SrcT>(x));
    }
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline dim3 copy_grid(int64_t work_per_row, int64_t per_cta, int64_t selected)
{
    const int64_t gx = (work_per_row + per_cta - 1) / per_cta;
    const int64_t gy = selected < kMaxGridY ? selected : kMaxGridY;
    return dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1);
}

template <typename IdxT>
cudaError_t gather_typed(const CacheDesc &c, const IdxT *idx, int64_t selected, const uint8_t *flags,
                         void *packed, cudaStream_t st)
{
    const int64_t es = c.dtype == KDA_F32 ? 4 : 2;
    const int64_t payload = c.h * c.v * c.k;
    if (aligned16(c.data) && aligned16(packed) && (c.row_stride * es) % 16 == 0 && (payload * es) % 16 == 0) {
        const int64_t pv = payload * es / 16;
        const dim3 grid = copy_grid(pv, kCopyThreads * kVecPerThread, selected);
        copy_rows_v16<IdxT, true><<<grid, kCopyThreads, 0, st>>>(
            static_cast<uint4 *>(c.data), c.n_rows, c.row_stride * es / 16, pv, idx, flags, selected,
            static_cast<uint4 *>(packed));
    } else {
        const dim3 grid = copy_grid(payload, kCopyThreads, selected);
        if (c.dtype == KDA_F32)
            gather_scalar<IdxT, float><<<grid, kCopyThreads, 0, st>>>(
                static_cast<const float *>(c.data), c.n_rows, c.row_stride, payload, idx, flags, selected,
                static_cast<float *>(packed));
        else
            gather_scalar<IdxT, uint16_t><<<grid, kCopyThreads, 0, st>>>(
                static_cast<const uint16_t *>(c.data), c.n_rows, c.row_stride, payload, idx, flags,
                selected, static_cast<uint16_t *>(packed));
    }
    return cudaGetLastError();
}

template <typename IdxT>
cudaError_t scatter_typed(const CacheDesc &c, const IdxT *idx, int64_t selected, const void *packed,
                          int32_t packed_dtype, cudaStream_t st)
{
    const int64_t es = c.dtype == KDA_F32 ? 4 : 2;
    const int64_t ps = packed_dtype == KDA_F32 ? 4 : 2;
    const int64_t payload = c.h * c.v * c.k;
    const bool vec = aligned16(c.data) && aligned16(packed) && (c.row_stride * es) % 16 == 0 &&
                     payload % 8 == 0;
    if (vec && packed_dtype == c.dtype) {
        const int64_t pv = payload * es / 16;
        const dim3 grid = copy_grid(pv, kCopyThreads * kVecPerThread, selected);
        copy_rows_v16<IdxT, false><<<grid, kCopyThreads, 0, st>>>(
            static_cast<uint4 *>(c.data), c.n_rows, c.row_stride * es / 16, pv, idx, nullptr, selected,
            static_cast<uint4 *>(const_cast<void *>(packed)));
    } else if (vec) {
        const dim3 grid = copy_grid(payload / 8, kCopyThreads * kVecPerThread, selected);
        if (packed_dtype == KDA_F32)
            scatter_cast_v<IdxT, float, uint16_t><<<grid, kCopyThreads, 0, st>>>(
                static_cast<uint16_t *>(c.data), c.n_rows, c.row_stride, payload, idx, selected,
                static_cast<const float *>(packed));
        else
            scatter_cast_v<IdxT, uint16_t, float><<<grid, kCopyThreads, 0, st>>>(
                static_cast<float *>(c.data), c.n_rows, c.row_stride, payload, idx, selected,
                static_cast<const uint16_t *>(packed));
    } else {
        const dim3 grid = copy_grid(payload, kCopyThreads, selected);
        if (c.dtype == KDA_F32 && ps == 4)
            scatter_scalar<IdxT, float, float><<<grid, kCopyThreads, 0, st>>>(
                static_cast<float *>(c.data), c.n_rows, c.row_stride, payload, idx, selected,
                static_cast<const float *>(packed));
        else if (c.dtype == KDA_F32)
            scatter_scalar<IdxT, uint16_t, float><<<grid, kCopyThreads, 0, st>>>(
                static_cast<float *>(c.data), c.n_rows, c.row_stride, payload, idx, selected,
                static_cast<const uint16_t *>(packed));
        else if (ps == 4)
            scatter_scalar<IdxT, float, uint16_t><<<grid, kCopyThreads, 0, st>>>(
                static_cast<uint16_t *>(c.data), c.n_rows, c.row_stride, payload, idx, selected,
                static_cast<const float *>(packed));
        else
            scatter_scalar<IdxT, uint16_t, uint16_t><<<grid, kCopyThreads, 0, st>>>(
                static_cast<uint16_t *>(c.data), c.n_rows, c.row_stride, payload, idx, selected,
                static_cast<const uint16_t *>(packed));
    }
    (void)ps;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_state_gather(const CacheDesc &c, const void *idx, int32_t idx_type, int64_t selected,
                                const uint8_t *flags, void *packed, cudaStream_t st)
{
    if (idx_type == KDA_I32)
        return gather_typed(c, static_cast<const int32_t *>(idx), selected, flags, packed, st);
    return gather_typed(c, static_cast<const int64_t *>(idx), selected, flags, packed, st);
}

cudaError_t launch_state_scatter(const CacheDesc &c, const void *idx, int32_t idx_type, int64_t selected,
                                 const void *packed, int32_t packed_dtype, cudaStream_t st)
{
    if (idx_type == KDA_I32)
        return scatter_typed(c, static_cast<const int32_t *>(idx), selected, packed, packed_dtype, st);
    return scatter_typed(c, static_cast<const int64_t *>(idx), selected, packed, packed_dtype, st);
}

}  // namespace kda
