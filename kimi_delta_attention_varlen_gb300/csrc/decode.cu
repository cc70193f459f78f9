// One-token recurrent decode step on cache rows, in place.
//
// Per (request r, head h):  S <- cache[idx[r]] (zeros for an invalid index),
//   S <- (I - beta k k^T) Diag(exp g) S + beta k v^T,  o = scale * S^T q,
//   cache[idx[r]] <- S (cache dtype) when the index is valid.
// The recurrence is the one of the "KDA's challenges for AI infra" page,
// section 1.1; decode on cache rows by index is the route the state-copy page
// names in its "Background" section.
//
// The cache stores S transposed: row v of a head's [V][K] block is column v
// of S.  Column v evolves on its own:
//   a_v = sum_k k_k e^{g_k} S[k][v],  b_v = sum_k q_k e^{g_k} S[k][v]
//   u_v = beta (v_v - a_v)
//   S'[k][v] = e^{g_k} S[k][v] + k_k u_v,   o_v = scale (b_v + (q.k) u_v)
// so one pass over the state suffices: read row, two dot products, write row.
//
// GPU mapping: one CTA (128 threads) per (request, head).  D/8 lanes share a
// state row, each holding 8 channels (one 16-byte bf16 vector); a CTA covers
// 128/(D/8) rows per pass and keeps NR rows per thread in flight.  The kernel
// is bound by HBM: 2 * D * D * sizeof(cache) bytes per (request, head).
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kDecodeThreads = 128;

__device__ __forceinline__ void load8(const float *p, float x[8])
{
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float x[8])
{
    const uint4 a = *reinterpret_cast<const uint4 *>(p);
    x[0] = bf16_lo(a.x); x[1] = bf16_hi(a.x); x[2] = bf16_lo(a.y); x[3] = bf16_hi(a.y);
    x[4] = bf16_lo(a.z); x[5] = bf16_hi(a.z); x[6] = bf16_lo(a.w); x[7] = bf16_hi(a.w);
}

__device__ __forceinline__ void store8(float *p, const float x[8])
{
    st_cs_v4(p, make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                           __float_as_uint(x[3])));
    st_cs_v4(p + 4, make_uint4(__float_as_uint(x[4]), __float_as_uint(x[5]), __float_as_uint(x[6]),
                               __float_as_uint(x[7])));
}

__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float x[8])
{
    st_cs_v4(p, make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                           pack_bf16x2(x[6], x[7])));
}

template <int LPR> __device__ __forceinline__ float group_sum(float x)
{
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <int D, typename IO, typename CT, typename IdxT>
__global__ void __launch_bounds__(kDecodeThreads)
decode_kernel(const IO *__restrict__ q, const IO *__restrict__ k, const IO *__restrict__ v,
              const float *__restrict__ g, const float *__restrict__ beta, int32_t H, float scale,
              int32_t l2norm, CT *__restrict__ cache, int64_t n_rows, int64_t row_stride,
              const IdxT *__restrict__ idx, IO *__restrict__ out)
{
    constexpr int LPR = D / 8;                     // lanes per state row
    constexpr int RPP = kDecodeThreads / LPR;      // rows per pass
    constexpr int PASSES = D / RPP;
    constexpr int NR = PASSES >= 4 ? 4 : PASSES;   // rows in flight per thread
    static_assert(PASSES % NR == 0, "row batching");

    __shared__ float s_out[D];

    const int64_t item = blockIdx.x;
    const int64_t r = item / H;
    const int h = static_cast<int>(item % H);
    const int lr = threadIdx.x % LPR;   // lane within the row group
    const int rip = threadIdx.x / LPR;  // row within the pass
    const int c0 = lr * 8;
    const int64_t tok = r * H + h;

    float qv[8], kv[8], gv[8];
    load8(q + tok * D + c0, qv);
    load8(k + tok * D + c0, kv);
    load8(g + tok * D + c0, gv);
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        sq += qv[c] * qv[c];
        sk += kv[c] * kv[c];
    }
    sq = group_sum<LPR>(sq);
    sk = group_sum<LPR>(sk);
    const float rq = l2norm ? rsqrtf(sq + 1e-6f) : 1.f;
    const float rk = l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
    float ke[8], qe[8], eg[8], kh[8];
    float qk = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float qh = qv[c] * rq;
        kh[c] = kv[c] * rk;
        eg[c] = expf(gv[c]);
        ke[c] = kh[c] * eg[c];
        qe[c] = qh * eg[c];
        qk += qh * kh[c];
    }
    qk = group_sum<LPR>(qk);
    const float bt = beta[tok];

    const int64_t row = static_cast<int64_t>(idx[r]);
    const bool valid = row >= 0 && row < n_rows;
    CT *srow = cache + (valid ? row : 0) * row_stride + static_cast<int64_t>(h) * D * D;
    const IO *vrow = v + tok * D;

#pragma unroll 1
    for (int p0 = 0; p0 < PASSES; p0 += NR) {
        float s[NR][8];
#pragma unroll
        for (int j = 0; j < NR; ++j) {
            const int vi = (p0 + j) * RPP + rip;
            if (valid) {
                load8(srow + vi * D + c0, s[j]);
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c) s[j][c] = 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < NR; ++j) {
            const int vi = (p0 + j) * RPP + rip;
            float a = 0.f, b = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                a += ke[c] * s[j][c];
                b += qe[c] * s[j][c];
            }
            a = group_sum<LPR>(a);
            b = group_sum<LPR>(b);
            const float vv = load_as_f32(vrow + vi);
            const float u = bt * (vv - a);
            if (valid) {
                float sn[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) sn[c] = eg[c] * s[j][c] + kh[c] * u;
                store8(srow + vi * D + c0, sn);
            }
            if (lr == 0) s_out[vi] = scale * (b + qk * u);
        }
    }
    __syncthreads();
    for (int vi = threadIdx.x; vi < D; vi += kDecodeThreads) out[tok * D + vi] = from_f32<IO>(s_out[vi]);
}

template <int D, typename IO, typename CT>
cudaError_t decode_launch_idx(const DecodeArgs &a, cudaStream_t st)
{
    const int64_t items = a.batch * a.h;
    const dim3 grid(static_cast<unsigned>(items));
    const IO *q = static_cast<const IO *>(a.q);
    const IO *k = static_cast<const IO *>(a.k);
    const IO *v = static_cast<const IO *>(a.v);
    CT *cache = static_cast<CT *>(a.cache.data);
    IO *out = static_cast<IO *>(a.out);
    if (a.idx_type == KDA_I32)
        decode_kernel<D, IO, CT, int32_t><<<grid, kDecodeThreads, 0, st>>>(
            q, k, v, a.g, a.beta, a.h, a.scale, a.l2norm, cache, a.cache.n_rows, a.cache.row_stride,
            static_cast<const int32_t *>(a.idx), out);
    else
        decode_kernel<D, IO, CT, int64_t><<<grid, kDecodeThreads, 0, st>>>(
            q, k, v, a.g, a.beta, a.h, a.scale, a.l2norm, cache, a.cache.n_rows, a.cache.row_stride,
            static_cast<const int64_t *>(a.idx), out);
    return cudaGetLastError();
}

template <int D>
cudaError_t decode_launch_d(const DecodeArgs &a, cudaStream_t st)
{
    if (a.io_dtype == KDA_BF16) {
        if (a.cache.dtype == KDA_BF16) return decode_launch_idx<D, __nv_bfloat16, __nv_bfloat16>(a, st);
        return decode_launch_idx<D, __nv_bfloat16, float>(a, st);
    }
    if (a.cache.dtype == KDA_BF16) return decode_launch_idx<D, float, __nv_bfloat16>(a, st);
    return decode_launch_idx<D, float, float>(a, st);
}

}  // namespace

cudaError_t launch_decode_step(const DecodeArgs &a, cudaStream_t st)
{
    switch (a.d) {
    case 32: return decode_launch_d<32>(a, st);
    case 64: return decode_launch_d<64>(a, st);
    default: return decode_launch_d<128>(a, st);
    }
}

}  // namespace kda
