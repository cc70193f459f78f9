// INT8 checkpoints of recurrent states (the "KDA's challenges for AI infra"
// page, section 6.6.2, Int8CheckpointStore): quantise active state rows into
// checkpoint slots and dequantise them back.
//
// Per (slot, head, key channel k) one fp32 scale from the max-abs over the
// value dimension: scale = amax / 127, code = round_half_even(x / scale)
// clamped to [-127, 127]; a scale below the smallest normal fp32 (an all-zero
// column, or every |x| < 127 * 2^-126) is stored as 0 with codes 0; loading writes
// code * scale in the active row's dtype.  Codes are decided with correctly
// rounded fp32 division and a round-to-nearest-even conversion.
//
// Both kernels are HBM-bound copies of [V][K] state blocks (fp32 64 KB or
// bf16 32 KB at V = K = 128) and their 16 KB of codes.  Store: one CTA per
// (pair, head, key-column slice) stages its slice in shared memory with
// 16-byte asynchronous copies (one HBM read) for the column max and the codes.
// Load: one CTA per (pair, head) streams codes in and rows out with coalesced
// accesses.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 256;

template <typename IdxT> __device__ __forceinline__ int64_t idx_at(const void *p, int64_t s)
{
    return static_cast<int64_t>(static_cast<const IdxT *>(p)[s]);
}

// Codes of four values of one row (columns with scales sc, reciprocals rc),
// packed little-endian: round_half_even(x / sc) with x / sc the correctly
// rounded fp32 quotient.  x * (1 / sc) lies within a few ulps (< 1e-4 for
// |x / sc| <= 128) of the exact quotient, so it rounds to the same integer
// unless it is within that distance of a half-integer; only there the
// quotient itself is formed.  No clamp is needed: |x| <= amax, so the
// quotient is at most 127 (1 + 2^-22) in magnitude and rounds into
// [-127, 127].  A zero scale has rc = 0 and gives code 0.
__device__ __forceinline__ uint32_t quantize4(const float x[4], const float sc[4], const float rc[4])
{
    float y[4];
    bool near = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        y[e] = __fmul_rn(x[e], rc[e]);
        near |= fabsf(y[e] - rintf(y[e])) > 0.499f;  // y - rint(y) is exact, in [-0.5, 0.5]
    }
    if (near) {  // rare: within 1e-3 of a half-integer
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (fabsf(y[e] - rintf(y[e])) > 0.499f) y[e] = __fdiv_rn(x[e], sc[e]);
    }
    int q[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) q[e] = __float2int_rn(y[e]);  // ties to even
    return __byte_perm(__byte_perm(q[0], q[1], 0x0040), __byte_perm(q[2], q[3], 0x0040), 0x5410);
}

// Store geometry: a [ROWS][COLS] slice of a state block, THREADS threads, each
// holding 4 consecutive columns of NR rows spaced RPP apart.
template <int ROWS, int COLS, int THREADS> struct Geo {
    static constexpr int K4 = COLS / 4;                                    // 4-column groups per row
    static constexpr int RPP = THREADS / K4 < ROWS ? THREADS / K4 : ROWS;  // rows per pass of the CTA
    static constexpr int NR = ROWS / RPP;                                  // rows per thread
    static constexpr int ACTIVE = RPP * K4;                                // threads holding rows
    static_assert(NR * RPP == ROWS && K4 <= 32 && ACTIVE % 32 == 0, "geometry");
};

// Column slices per block and threads per CTA of the store.  The max-abs runs over
// the value rows of each key column, so column slices are independent: a CTA takes
// one [V][K / NS] slice, which keeps more, smaller slices in flight per SM (fp32
// blocks at K = 128: two 32 KB halves, six CTAs per SM; bf16 blocks stay whole).
template <int D, typename ElemT> struct StoreCfg {
    static constexpr int NS = D >= 128 && sizeof(ElemT) == 4 ? 2 : 1;
    static constexpr int THREADS = 256;
};

// One CTA per (pair, head, column slice): the slice streams into shared memory
// (16-byte asynchronous copies; one HBM read), then the column max-abs and the
// codes are computed from there.
template <int D, typename ElemT, typename IdxT>
__global__ void __launch_bounds__(StoreCfg<D, ElemT>::THREADS)
ckpt_store_kernel(const ElemT *__restrict__ active, int64_t n_rows, int64_t row_stride, int32_t H,
                  const void *__restrict__ src, const void *__restrict__ dst, int64_t n_slots,
                  int8_t *__restrict__ qdata, float *__restrict__ scale)
{
    constexpr int NS = StoreCfg<D, ElemT>::NS, THREADS = StoreCfg<D, ElemT>::THREADS, DS = D / NS;
    constexpr int ES = static_cast<int>(sizeof(ElemT));
    using G = Geo<D, DS, THREADS>;
    constexpr int RB = DS * ES;        // bytes of one slice row
    constexpr int BLK = D * RB;        // bytes of one [V][DS] slice
    extern __shared__ __align__(16) char smem[];
    float(*part)[DS] = reinterpret_cast<float(*)[DS]>(smem + BLK);  // [warps][DS] column maxima
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sl = static_cast<int>(blockIdx.x % NS);
    const int64_t ph = blockIdx.x / NS;
    const int64_t pair = ph / H;
    const int h = static_cast<int>(ph % H);
    const int64_t r = idx_at<IdxT>(src, pair), c = idx_at<IdxT>(dst, pair);
    if (r < 0 || r >= n_rows || c < 0 || c >= n_slots) return;  // uniform over the CTA
    const char *blk = reinterpret_cast<const char *>(active + r * row_stride + static_cast<int64_t>(h) * D * D +
                                                     sl * DS);
#pragma unroll 4
    for (int e = tid; e < BLK / 16; e += THREADS) {
        const int v = e / (RB / 16), ch = e % (RB / 16);
        cp_async16(smem_u32(smem + v * RB + 16 * ch), blk + static_cast<int64_t>(v) * D * ES + 16 * ch, 16u);
    }
    cp_async_wait_all();
    __syncthreads();

    const int cg = tid % G::K4, r0 = tid / G::K4;
    const bool act = tid < G::ACTIVE;  // (all threads unless the block has fewer rows)
    auto load4 = [&](int v, float x[4]) {
        const char *p = smem + v * RB + 4 * cg * ES;
        if constexpr (ES == 4) {
            const float4 a = *reinterpret_cast<const float4 *>(p);
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        } else {
            const uint2 a = *reinterpret_cast<const uint2 *>(p);
            x[0] = bf16_lo(a.x); x[1] = bf16_hi(a.x); x[2] = bf16_lo(a.y); x[3] = bf16_hi(a.y);
        }
    };
    float m[4] = {0.f, 0.f, 0.f, 0.f};
    if (act) {
#pragma unroll
        for (int j = 0; j < G::NR; ++j) {
            float x[4];
            load4(r0 + G::RPP * j, x);
#pragma unroll
            for (int e = 0; e < 4; ++e) m[e] = fmaxf(m[e], fabsf(x[e]));
        }
    }
    // column max-abs: lanes of this warp holding the same columns, then the warps
#pragma unroll
    for (int o = G::K4; o < 32; o <<= 1)
#pragma unroll
        for (int e = 0; e < 4; ++e) m[e] = fmaxf(m[e], __shfl_xor_sync(0xffffffffu, m[e], o));
    if (lane < G::K4) *reinterpret_cast<float4 *>(&part[warp][4 * cg]) = make_float4(m[0], m[1], m[2], m[3]);
    __syncthreads();
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w) {
        const float4 a = *reinterpret_cast<const float4 *>(&part[w][4 * cg]);
        m[0] = fmaxf(m[0], a.x); m[1] = fmaxf(m[1], a.y); m[2] = fmaxf(m[2], a.z); m[3] = fmaxf(m[3], a.w);
    }
    float sc[4], rc[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        sc[e] = __fdiv_rn(m[e], 127.f);
        if (sc[e] < 1.17549435e-38f) sc[e] = 0.f;  // subnormal scales are stored as 0 (codes 0)
        rc[e] = sc[e] > 0.f ? __frcp_rn(sc[e]) : 0.f;
    }
    const int64_t sbase = (c * H + h) * static_cast<int64_t>(D);
    const int col = sl * DS + 4 * cg;  // first key column of this thread
    if (r0 == 0) *reinterpret_cast<float4 *>(scale + sbase + col) = make_float4(sc[0], sc[1], sc[2], sc[3]);
    if (!act) return;
    int8_t *qb = qdata + sbase * D;
#pragma unroll
    for (int j = 0; j < G::NR; ++j) {
        const int v = r0 + G::RPP * j;
        float x[4];
        load4(v, x);
        *reinterpret_cast<uint32_t *>(qb + static_cast<int64_t>(v) * D + col) = quantize4(x, sc, rc);
    }
}

template <int D, typename ElemT, typename IdxT>
__global__ void __launch_bounds__(kThreads)
ckpt_load_kernel(const int8_t *__restrict__ qdata, const float *__restrict__ scale, int64_t n_slots,
                 const void *__restrict__ src, const void *__restrict__ dst, ElemT *__restrict__ active,
                 int64_t n_rows, int64_t row_stride, int32_t H)
{
    const int64_t pair = blockIdx.x / H;
    const int h = static_cast<int>(blockIdx.x % H);
    const int64_t c = idx_at<IdxT>(src, pair), r = idx_at<IdxT>(dst, pair);
    if (c < 0 || c >= n_slots || r < 0 || r >= n_rows) return;  // uniform over the CTA
    const int64_t sbase = (c * H + h) * static_cast<int64_t>(D);
    const int8_t *qb = qdata + sbase * D;
    const float *sb = scale + sbase;
    ElemT *out = active + r * row_stride + static_cast<int64_t>(h) * D * D;
    // four codes per thread and step: consecutive threads cover consecutive 16 (fp32) or
    // 8 (bf16) output bytes, so every store instruction writes one contiguous span.  A thread's
    // key columns are the same at every step (kThreads is a multiple of D / 4), so its four
    // scales are loaded once.
    constexpr int CH = D * D / 4;
    static_assert(kThreads % (D / 4) == 0, "fixed columns per thread");
    const uint32_t *qb4 = reinterpret_cast<const uint32_t *>(qb);
    const float4 s4 = __ldg(reinterpret_cast<const float4 *>(sb + (4 * static_cast<int>(threadIdx.x)) % D));
#pragma unroll 8
    for (int e = threadIdx.x; e < CH; e += kThreads) {
        const uint32_t w = __ldg(qb4 + e);
        const float y0 = __fmul_rn(static_cast<float>(static_cast<int8_t>(w & 0xffu)), s4.x);
        const float y1 = __fmul_rn(static_cast<float>(static_cast<int8_t>((w >> 8) & 0xffu)), s4.y);
        const float y2 = __fmul_rn(static_cast<float>(static_cast<int8_t>((w >> 16) & 0xffu)), s4.z);
        const float y3 = __fmul_rn(static_cast<float>(static_cast<int8_t>(w >> 24)), s4.w);
        if constexpr (sizeof(ElemT) == 4) {
            reinterpret_cast<float4 *>(out)[e] = make_float4(y0, y1, y2, y3);
        } else {
            reinterpret_cast<uint2 *>(out)[e] = make_uint2(pack_bf16x2(y0, y1), pack_bf16x2(y2, y3));
        }
    }
}

template <int D, typename ElemT, typename IdxT>
cudaError_t store_typed(const CacheDesc &c, const void *src, const void *dst, int64_t count, int8_t *qdata,
                        float *scale, int64_t n_slots, cudaStream_t st)
{
    using Cfg = StoreCfg<D, ElemT>;
    const int64_t blocks = count * c.h * Cfg::NS;
    constexpr int smem = D * (D / Cfg::NS) * static_cast<int>(sizeof(ElemT)) + (Cfg::THREADS / 32) * (D / Cfg::NS) * 4;
    auto kern = ckpt_store_kernel<D, ElemT, IdxT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(blocks), Cfg::THREADS, smem, st>>>(
        static_cast<const ElemT *>(c.data), c.n_rows, c.row_stride, static_cast<int32_t>(c.h), src, dst, n_slots,
        qdata, scale);
    return cudaGetLastError();
}

template <int D, typename ElemT, typename IdxT>
cudaError_t load_typed(const CacheDesc &c, const int8_t *qdata, const float *scale, int64_t n_slots,
                       const void *src, const void *dst, int64_t count, cudaStream_t st)
{
    const int64_t blocks = count * c.h;
    ckpt_load_kernel<D, ElemT, IdxT><<<static_cast<unsigned>(blocks), kThreads, 0, st>>>(
        qdata, scale, n_slots, src, dst, static_cast<ElemT *>(c.data), c.n_rows, c.row_stride,
        static_cast<int32_t>(c.h));
    return cudaGetLastError();
}

template <int D, typename IdxT>
cudaError_t store_d(const CacheDesc &c, const void *src, const void *dst, int64_t count, int8_t *q, float *s,
                    int64_t n_slots, cudaStream_t st)
{
    return c.dtype == KDA_F32 ? store_typed<D, float, IdxT>(c, src, dst, count, q, s, n_slots, st)
                              : store_typed<D, uint16_t, IdxT>(c, src, dst, count, q, s, n_slots, st);
}

template <int D, typename IdxT>
cudaError_t load_d(const CacheDesc &c, const int8_t *q, const float *s, int64_t n_slots, const void *src,
                   const void *dst, int64_t count, cudaStream_t st)
{
    return c.dtype == KDA_F32 ? load_typed<D, float, IdxT>(c, q, s, n_slots, src, dst, count, st)
                              : load_typed<D, uint16_t, IdxT>(c, q, s, n_slots, src, dst, count, st);
}

}  // namespace

cudaError_t launch_ckpt_store_int8(const CacheDesc &c, const void *src, const void *dst, int32_t idx_type,
                                   int64_t count, int8_t *qdata, float *scale, int64_t n_slots, cudaStream_t st)
{
    const bool i64 = idx_type == KDA_I64;
    switch (c.k) {
    case 32: return i64 ? store_d<32, int64_t>(c, src, dst, count, qdata, scale, n_slots, st)
                        : store_d<32, int32_t>(c, src, dst, count, qdata, scale, n_slots, st);
    case 64: return i64 ? store_d<64, int64_t>(c, src, dst, count, qdata, scale, n_slots, st)
                        : store_d<64, int32_t>(c, src, dst, count, qdata, scale, n_slots, st);
    default: return i64 ? store_d<128, int64_t>(c, src, dst, count, qdata, scale, n_slots, st)
                        : store_d<128, int32_t>(c, src, dst, count, qdata, scale, n_slots, st);
    }
}

cudaError_t launch_ckpt_load_int8(const CacheDesc &c, const int8_t *qdata, const float *scale, int64_t n_slots,
                                  const void *src, const void *dst, int32_t idx_type, int64_t count, cudaStream_t st)
{
    const bool i64 = idx_type == KDA_I64;
    switch (c.k) {
    case 32: return i64 ? load_d<32, int64_t>(c, qdata, scale, n_slots, src, dst, count, st)
                        : load_d<32, int32_t>(c, qdata, scale, n_slots, src, dst, count, st);
    case 64: return i64 ? load_d<64, int64_t>(c, qdata, scale, n_slots, src, dst, count, st)
                        : load_d<64, int32_t>(c, qdata, scale, n_slots, src, dst, count, st);
    default: return i64 ? load_d<128, int64_t>(c, qdata, scale, n_slots, src, dst, count, st)
                        : load_d<128, int32_t>(c, qdata, scale, n_slots, src, dst, count, st);
    }
}

}  // namespace kda
