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
// GPU mapping: persistent CTAs (up to 256 threads) over the (request, head)
// items.  D/8 lanes share a state row, each holding 8 channels (one 16-byte
// bf16 vector).  Every thread copies its own slices of the next item's state
// into its own shared-memory slots (cp.async, two stages) and holds the next
// item's token inputs in registers, so the state read of one item overlaps
// the work on the previous one without a block barrier.  The kernel is bound
// by HBM: 2 * D * D * sizeof(cache) bytes per (request, head).
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {


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

// Threads per CTA: one 16-byte state slice (8 channels) per lane, up to 256 lanes.
template <int D> __host__ __device__ constexpr int decode_threads() { return D * D / 8 < 256 ? D * D / 8 : 256; }

// Per-item inputs of one lane, loaded one item ahead.
template <int D, typename IO, int ROWS> struct ItemIn {
    float q[8], k[8], g[8], v[ROWS], beta;
    int64_t row;
};

template <int D, typename IO, typename CT, typename IdxT>
__global__ void __launch_bounds__(decode_threads<D>())
decode_kernel(const IO *__restrict__ q, const IO *__restrict__ k, const IO *__restrict__ v,
              const float *__restrict__ g, const float *__restrict__ beta, int32_t H, float scale,
              int32_t l2norm, CT *__restrict__ cache, int64_t n_rows, int64_t row_stride,
              const IdxT *__restrict__ idx, IO *__restrict__ out, int64_t items)
{
    constexpr int THREADS = decode_threads<D>();
    constexpr int LPR = D / 8;              // lanes per state row
    constexpr int RPP = THREADS / LPR;      // rows per pass
    constexpr int ROWS = D / RPP;           // rows per thread
    constexpr int V16 = 8 * static_cast<int>(sizeof(CT)) / 16;  // 16-byte pieces per slice
    extern __shared__ __align__(16) uint4 slots[];  // [2 stages][ROWS][V16][THREADS]

    const int tid = threadIdx.x;
    const int lr = tid % LPR, rip = tid / LPR, c0 = lr * 8;

    auto fetch_inputs = [&](int64_t it, ItemIn<D, IO, ROWS> &in) {
        const int64_t r = it / H, tok = it;
        load8(q + tok * D + c0, in.q);
        load8(k + tok * D + c0, in.k);
        load8(g + tok * D + c0, in.g);
#pragma unroll
        for (int j = 0; j < ROWS; ++j) in.v[j] = load_as_f32(v + tok * D + j * RPP + rip);
        in.beta = beta[tok];
        const int64_t row = static_cast<int64_t>(idx[r]);
        in.row = (row >= 0 && row < n_rows) ? row : -1;
    };
    // Copies this thread's slices of item `it` into stage `s` (nothing for an invalid row).
    auto fetch_state = [&](int64_t it, int64_t row, int s) {
        if (row >= 0) {
            const CT *src = cache + row * row_stride + static_cast<int64_t>(it % H) * D * D;
#pragma unroll
            for (int j = 0; j < ROWS; ++j)
#pragma unroll
                for (int w = 0; w < V16; ++w)
                    cp_async16(smem_u32(&slots[((s * ROWS + j) * V16 + w) * THREADS + tid]),
                               src + (j * RPP + rip) * D + c0 + w * (16 / sizeof(CT)), 16u);
        }
        asm volatile("cp.async.commit_group;\n" ::: "memory");
    };

    int64_t it = blockIdx.x;
    if (it >= items) return;
    ItemIn<D, IO, ROWS> cur, nxt;
    fetch_inputs(it, cur);
    fetch_state(it, cur.row, 0);
    for (int s = 0; it < items; it += gridDim.x, s ^= 1) {
        const int64_t it2 = it + gridDim.x;
        if (it2 < items) {
            fetch_inputs(it2, nxt);
            fetch_state(it2, nxt.row, s ^ 1);
        } else {
            asm volatile("cp.async.commit_group;\n" ::: "memory");
        }
        asm volatile("cp.async.wait_group 1;\n" ::: "memory");  // this item's slices have landed

        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            sq += cur.q[c] * cur.q[c];
            sk += cur.k[c] * cur.k[c];
        }
        sq = group_sum<LPR>(sq);
        sk = group_sum<LPR>(sk);
        const float rq = l2norm ? rsqrtf(sq + 1e-6f) : 1.f;
        const float rk = l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
        float ke[8], qe[8], eg[8], kh[8];
        float qk = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float qh = cur.q[c] * rq;
            kh[c] = cur.k[c] * rk;
            eg[c] = ex2_approx(cur.g[c] * 1.4426950408889634f);  // e^g
            ke[c] = kh[c] * eg[c];
            qe[c] = qh * eg[c];
            qk += qh * kh[c];
        }
        qk = group_sum<LPR>(qk);
        const bool valid = cur.row >= 0;
        CT *dst = cache + (valid ? cur.row : 0) * row_stride + static_cast<int64_t>(it % H) * D * D;
        if constexpr (2 * ROWS == LPR) {
            // the 2 ROWS dot products reduced over the LPR lanes of a row by a transposed
            // butterfly: lane g of the group ends with value g (a of row g / 2 for even g, b for
            // odd g); u of each row is broadcast from its lane; the state slices are read from
            // shared memory again for the update instead of being held across the reduction
            auto slice = [&](int j, float st[8]) {
                if (valid) {
                    if constexpr (V16 == 1) {
                        const uint4 a = slots[((s * ROWS + j) * V16) * THREADS + tid];
                        st[0] = bf16_lo(a.x); st[1] = bf16_hi(a.x); st[2] = bf16_lo(a.y); st[3] = bf16_hi(a.y);
                        st[4] = bf16_lo(a.z); st[5] = bf16_hi(a.z); st[6] = bf16_lo(a.w); st[7] = bf16_hi(a.w);
                    } else {
                        const uint4 a = slots[((s * ROWS + j) * V16) * THREADS + tid];
                        const uint4 b = slots[((s * ROWS + j) * V16 + 1) * THREADS + tid];
                        st[0] = __uint_as_float(a.x); st[1] = __uint_as_float(a.y);
                        st[2] = __uint_as_float(a.z); st[3] = __uint_as_float(a.w);
                        st[4] = __uint_as_float(b.x); st[5] = __uint_as_float(b.y);
                        st[6] = __uint_as_float(b.z); st[7] = __uint_as_float(b.w);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c) st[c] = 0.f;
                }
            };
            float vals[2 * ROWS];
#pragma unroll
            for (int j = 0; j < ROWS; ++j) {  // channel pairs through the packed fp32x2 instructions
                float st[8];
                float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
                slice(j, st);
#pragma unroll
                for (int c = 0; c < 8; c += 2) {
                    const float2 s2 = make_float2(st[c], st[c + 1]);
                    a = fma2(make_float2(ke[c], ke[c + 1]), s2, a);
                    b = fma2(make_float2(qe[c], qe[c + 1]), s2, b);
                }
                vals[2 * j] = a.x + a.y;
                vals[2 * j + 1] = b.x + b.y;
            }
            const int lane = tid & 31;
#pragma unroll
            for (int mask = LPR / 2, half = ROWS; mask >= 1; mask >>= 1, half >>= 1) {
                const bool up = (lane & mask) != 0;
#pragma unroll
                for (int i = 0; i < half; ++i) {
                    const float send = up ? vals[i] : vals[i + half];
                    const float kept = up ? vals[i + half] : vals[i];
                    vals[i] = kept + __shfl_xor_sync(0xffffffffu, send, mask);
                }
            }
            const int jr = lr >> 1;
            // cur.v[jr] with jr varying by lane: select from the registers without local memory
            float vj = cur.v[0];
#pragma unroll
            for (int j = 1; j < ROWS; ++j) vj = jr == j ? cur.v[j] : vj;
            const float u_even = cur.beta * (vj - vals[0]);
            const float u_pair = __shfl_sync(0xffffffffu, u_even, lane & ~1);
            if (lr & 1) out[it * D + jr * RPP + rip] = from_f32<IO>(scale * fmaf(qk, u_pair, vals[0]));
            const int gbase = lane & ~(LPR - 1);
#pragma unroll
            for (int j = 0; j < ROWS; ++j) {
                const float u = __shfl_sync(0xffffffffu, u_even, gbase + 2 * j);
                if (valid) {
                    float st[8], sn[8];
                    slice(j, st);
#pragma unroll
                    for (int c = 0; c < 8; c += 2) {  // e^g S + k u: k u rounded, then one fma, per element
                        const float2 r = fma2(make_float2(eg[c], eg[c + 1]), make_float2(st[c], st[c + 1]),
                                              mul2(make_float2(kh[c], kh[c + 1]), make_float2(u, u)));
                        sn[c] = r.x;
                        sn[c + 1] = r.y;
                    }
                    store8(dst + (j * RPP + rip) * D + c0, sn);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < ROWS; ++j) {
                const int vi = j * RPP + rip;
                float st[8];
                if (valid) {
                    if constexpr (V16 == 1) {
                        const uint4 a = slots[((s * ROWS + j) * V16) * THREADS + tid];
                        st[0] = bf16_lo(a.x); st[1] = bf16_hi(a.x); st[2] = bf16_lo(a.y); st[3] = bf16_hi(a.y);
                        st[4] = bf16_lo(a.z); st[5] = bf16_hi(a.z); st[6] = bf16_lo(a.w); st[7] = bf16_hi(a.w);
                    } else {
                        const uint4 a = slots[((s * ROWS + j) * V16) * THREADS + tid];
                        const uint4 b = slots[((s * ROWS + j) * V16 + 1) * THREADS + tid];
                        st[0] = __uint_as_float(a.x); st[1] = __uint_as_float(a.y);
                        st[2] = __uint_as_float(a.z); st[3] = __uint_as_float(a.w);
                        st[4] = __uint_as_float(b.x); st[5] = __uint_as_float(b.y);
                        st[6] = __uint_as_float(b.z); st[7] = __uint_as_float(b.w);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c) st[c] = 0.f;
                }
                float a = 0.f, b = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    a += ke[c] * st[c];
                    b += qe[c] * st[c];
                }
                a = group_sum<LPR>(a);
                b = group_sum<LPR>(b);
                const float u = cur.beta * (cur.v[j] - a);
                if (valid) {
                    float sn[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) sn[c] = eg[c] * st[c] + kh[c] * u;
                    store8(dst + vi * D + c0, sn);
                }
                if (lr == 0) out[it * D + vi] = from_f32<IO>(scale * (b + qk * u));
            }
        }
        cur = nxt;
    }
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

template <int D, typename IO, typename CT, typename IdxT>
cudaError_t decode_launch_typed(const DecodeArgs &a, cudaStream_t st)
{
    constexpr int THREADS = decode_threads<D>();
    constexpr int ROWS = D / (THREADS / (D / 8));
    constexpr int smem = 2 * ROWS * 8 * static_cast<int>(sizeof(CT)) * THREADS;
    const int64_t items = a.batch * a.h;
    auto kern = decode_kernel<D, IO, CT, IdxT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, THREADS, smem)) != cudaSuccess) return e;
    const int64_t resident = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
    const unsigned grid = static_cast<unsigned>(items < resident ? items : resident);
    kern<<<grid, THREADS, smem, st>>>(static_cast<const IO *>(a.q), static_cast<const IO *>(a.k),
                                      static_cast<const IO *>(a.v), a.g, a.beta, a.h, a.scale, a.l2norm,
                                      static_cast<CT *>(a.cache.data), a.cache.n_rows, a.cache.row_stride,
                                      static_cast<const IdxT *>(a.idx), static_cast<IO *>(a.out), items);
    return cudaGetLastError();
}

template <int D, typename IO, typename CT>
cudaError_t decode_launch_idx(const DecodeArgs &a, cudaStream_t st)
{
    return a.idx_type == KDA_I32 ? decode_launch_typed<D, IO, CT, int32_t>(a, st)
                                 : decode_launch_typed<D, IO, CT, int64_t>(a, st);
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
