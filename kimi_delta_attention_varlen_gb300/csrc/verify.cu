// Speculative target verification: L draft tokens per request run through
// the recurrence from the request's cached state; every token's output is
// returned and the state after each token is written to its own slot of an
// intermediate-state pool ("KDA's challenges for AI infra", section 6.4,
// target_verify, and 6.5, verify intermediate state indices).  The cached
// state is only read; committing the accepted prefix is a copy of one slot
// (kda_state_gather / kda_state_scatter).
//
// Per (request, head) and token, as in the decode step (column v of S, row v
// of the cache block, evolves on its own):
//   a_v = sum_k k_k e^{g_k} S[k][v],  b_v = sum_k q_k e^{g_k} S[k][v],
//   u_v = beta (v_v - a_v),  S'[k][v] = e^{g_k} S[k][v] + k_k u_v,
//   o_v = scale (b_v + (q.k) u_v).
// GPU mapping: persistent CTAs over the (request, head) items; D/8 lanes share
// a state row, each holding 8 channels of ROWS rows in registers for all L
// tokens, so the state is read once and each intermediate state is one
// coalesced write.  Each thread copies its own slices of the next item's
// state into shared memory while it computes the current one; the draft
// tokens' inputs are staged in shared memory 8 tokens at a time, and each
// token's factors (norms, q^.k^, e^g, k^ e^g, q^ e^g) are formed once, by one
// row group, for all rows.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

template <int D> __host__ __device__ constexpr int verify_threads() { return D * D / 8 < 256 ? D * D / 8 : 256; }

template <int LPR> __device__ __forceinline__ float group_sum(float x)
{
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ void load8(const void *base, int32_t dtype, int64_t e, float x[8])
{
    if (dtype == KDA_F32) {
        const float4 a = *reinterpret_cast<const float4 *>(static_cast<const float *>(base) + e);
        const float4 b = *(reinterpret_cast<const float4 *>(static_cast<const float *>(base) + e) + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
        const uint4 u = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + e);
        x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
        x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
    }
}

__device__ __forceinline__ void store8_stream(void *base, int32_t dtype, int64_t e, const float x[8])
{
    if (dtype == KDA_F32) {
        float *p = static_cast<float *>(base) + e;
        st_cs_v4(p, make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                               __float_as_uint(x[3])));
        st_cs_v4(p + 4, make_uint4(__float_as_uint(x[4]), __float_as_uint(x[5]), __float_as_uint(x[6]),
                                   __float_as_uint(x[7])));
    } else {
        st_cs_v4(static_cast<uint16_t *>(base) + e,
                 make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                            pack_bf16x2(x[6], x[7])));
    }
}

constexpr int kVT = 8;  // draft tokens staged per group

// S'[k][v] = e^{g_k} S[k][v] + k_k u_v on a lane's 8 channels of one row, as channel
// pairs: k u rounded, then one fused multiply-add, per element as the scalar form.
__device__ __forceinline__ void update_row(float s[8], const float2 e[4], const float2 kn[4], float u)
{
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float2 r = fma2(e[c], make_float2(s[2 * c], s[2 * c + 1]), mul2(kn[c], make_float2(u, u)));
        s[2 * c] = r.x;
        s[2 * c + 1] = r.y;
    }
}

template <int D, typename IO> struct VerifyLayout {
    static constexpr int ROW = D * static_cast<int>(sizeof(IO));
    static constexpr int Q = 0;
    static constexpr int K = Q + kVT * ROW;
    static constexpr int V = K + kVT * ROW;
    static constexpr int G = V + kVT * ROW;
    static constexpr int BETA = G + kVT * D * 4;
    // per-token factors, fp32 [kVT][D] each: e^g, k^ (normalised k), k^ e^g, q^ e^g; then q^.k^ [kVT]
    static constexpr int E = BETA + kVT * 4;
    static constexpr int KN = E + kVT * D * 4;
    static constexpr int KE = KN + kVT * D * 4;
    static constexpr int QE = KE + kVT * D * 4;
    static constexpr int QK = QE + kVT * D * 4;
    static constexpr int BYTES = QK + kVT * 4;
};

// Bytes of the token staging, rounded to 16 (the state slots follow it).
template <int D, typename IO> __host__ __device__ constexpr int verify_stage_bytes() { return (VerifyLayout<D, IO>::BYTES + 15) / 16 * 16; }

// Persistent CTAs over the (request, head) items.  Every thread copies its own slices of the
// next item's state into its own shared-memory slots (cp.async) while it computes the current
// item, so the state read overlaps the work and needs no block barrier; the current item's
// token inputs are staged cooperatively first, so one wait covers both.
template <int D, typename IO, typename IdxT>
__global__ void __launch_bounds__(verify_threads<D>())
verify_kernel(VerifyArgs a)
{
    constexpr int LPR = D / 8;                    // lanes per state row
    constexpr int THREADS = verify_threads<D>();
    constexpr int RPP = THREADS / LPR;            // rows per pass
    constexpr int ROWS = D / RPP;                 // rows per thread
    const int tid = threadIdx.x;
    const int c0 = 8 * (tid % LPR);               // this lane's channels
    const int r0 = tid / LPR;                     // rows r0 + RPP j
    const int64_t H = a.h;
    const int64_t items = a.batch * H;
    int64_t it = blockIdx.x;
    if (it >= items) return;  // (uniform over the CTA)
    const IO *qg = static_cast<const IO *>(a.q);
    const IO *kg = static_cast<const IO *>(a.k);
    const IO *vg = static_cast<const IO *>(a.v);
    IO *og = static_cast<IO *>(a.out);
    const IdxT *inter = static_cast<const IdxT *>(a.inter_idx);
    const int esz = a.cache.dtype == KDA_F32 ? 4 : 2;
    const int v16 = esz / 2;  // 16-byte pieces per 8-channel slice
    // token inputs, staged VT tokens at a time: q, k, v [VT][D] io, g [VT][D] fp32, beta [VT];
    // then the state slots [2 stages][ROWS][v16][THREADS] x 16 bytes
    extern __shared__ __align__(16) char smem[];
    using VL = VerifyLayout<D, IO>;
    IO *sq = reinterpret_cast<IO *>(smem + VL::Q);
    IO *sk = reinterpret_cast<IO *>(smem + VL::K);
    IO *sv = reinterpret_cast<IO *>(smem + VL::V);
    float *sg = reinterpret_cast<float *>(smem + VL::G);
    float *sb = reinterpret_cast<float *>(smem + VL::BETA);
    float *fe = reinterpret_cast<float *>(smem + VL::E);
    float *fkn = reinterpret_cast<float *>(smem + VL::KN);
    float *fke = reinterpret_cast<float *>(smem + VL::KE);
    float *fqe = reinterpret_cast<float *>(smem + VL::QE);
    float *fqk = reinterpret_cast<float *>(smem + VL::QK);
    uint4 *slots = reinterpret_cast<uint4 *>(smem + verify_stage_bytes<D, IO>());
    constexpr int IOCH = D * static_cast<int>(sizeof(IO)) / 16;  // 16-byte chunks of one io row
    constexpr int GCH = D * 4 / 16;                               // ... of one g row

    auto row_of = [&](int64_t item) -> int64_t {
        const int64_t r = static_cast<int64_t>(static_cast<const IdxT *>(a.idx)[item / H]);
        return r >= 0 && r < a.cache.n_rows ? r : -1;
    };
    // this thread's slices of item `item`'s cached state -> stage st (nothing for an invalid row)
    auto prefetch_state = [&](int64_t item, int st) {
        const int64_t row = row_of(item);
        if (row >= 0) {
            const char *src = static_cast<const char *>(a.cache.data) +
                              (row * a.cache.row_stride + (item % H) * D * D) * esz;
#pragma unroll
            for (int j = 0; j < ROWS; ++j)
                for (int w = 0; w < v16; ++w)
                    cp_async16(smem_u32(&slots[((st * ROWS + j) * v16 + w) * THREADS + tid]),
                               src + (static_cast<int64_t>(r0 + RPP * j) * D + c0) * esz + 16 * w, 16u);
        }
        asm volatile("cp.async.commit_group;\n" ::: "memory");
    };
    // the inputs of tokens t0 .. t0 + nt - 1 of request req, head h -> the staging
    auto stage_tokens = [&](int64_t req, int h, int t0, int nt) {
        for (int e = tid; e < nt * (3 * IOCH + GCH); e += THREADS) {
            const int tt = e / (3 * IOCH + GCH), part = e % (3 * IOCH + GCH);
            const int64_t base = ((req * a.L + t0 + tt) * H + h) * D;
            if (part < 3 * IOCH) {
                const int which = part / IOCH, ch = part % IOCH;
                const IO *src = (which == 0 ? qg : which == 1 ? kg : vg) + base;
                IO *dst = (which == 0 ? sq : which == 1 ? sk : sv) + tt * D;
                cp_async16(smem_u32(reinterpret_cast<char *>(dst) + 16 * ch),
                           reinterpret_cast<const char *>(src) + 16 * ch, 16u);
            } else {
                const int ch = part - 3 * IOCH;
                cp_async16(smem_u32(reinterpret_cast<char *>(sg + tt * D) + 16 * ch),
                           reinterpret_cast<const char *>(a.g + base) + 16 * ch, 16u);
            }
        }
        if (tid < nt) sb[tid] = a.beta[(req * a.L + t0 + tid) * H + h];
        asm volatile("cp.async.commit_group;\n" ::: "memory");
    };

    // The factors of staged token tt, computed once by row group tt (its LPR lanes hold all D
    // channels, 8 each, exactly as every row group used them) into shared memory.  Groups past
    // the last token repeat token 0 and store nothing: every lane of a warp takes part in the
    // full-warp shuffles of the group sums.
    static_assert(THREADS / LPR >= kVT, "one row group per staged token");
    auto token_factors = [&](int nt) {
        const bool mine = tid / LPR < nt;
        const int tt = mine ? tid / LPR : 0;
        float qv[8], kv[8], gv[8];
        load8(sq + tt * D, sizeof(IO) == 4 ? KDA_F32 : KDA_BF16, c0, qv);
        load8(sk + tt * D, sizeof(IO) == 4 ? KDA_F32 : KDA_BF16, c0, kv);
        load8(sg + tt * D, KDA_F32, c0, gv);
        // channel pairs (c, c + 1) go through the packed fp32x2 instructions
        float2 sq2 = make_float2(0.f, 0.f), sk2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 8; c += 2) {
            const float2 q2 = make_float2(qv[c], qv[c + 1]), k2 = make_float2(kv[c], kv[c + 1]);
            sq2 = fma2(q2, q2, sq2);
            sk2 = fma2(k2, k2, sk2);
        }
        const float sqs = group_sum<LPR>(sq2.x + sq2.y);
        const float sks = group_sum<LPR>(sk2.x + sk2.y);
        const float nq = a.l2norm ? rsqrtf(sqs + 1e-6f) : 1.f, nk = a.l2norm ? rsqrtf(sks + 1e-6f) : 1.f;
        float2 qk2 = make_float2(0.f, 0.f);
        float e[8], kn[8], ke[8], qe[8];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float2 q2 = mul2(make_float2(qv[2 * c], qv[2 * c + 1]), make_float2(nq, nq));
            const float2 k2 = mul2(make_float2(kv[2 * c], kv[2 * c + 1]), make_float2(nk, nk));
            qk2 = fma2(q2, k2, qk2);
            const float2 e2 = make_float2(ex2_approx(gv[2 * c] * 1.4426950408889634f),  // e^g
                                          ex2_approx(gv[2 * c + 1] * 1.4426950408889634f));
            const float2 ke2 = mul2(k2, e2), qe2 = mul2(q2, e2);
            e[2 * c] = e2.x; e[2 * c + 1] = e2.y;
            kn[2 * c] = k2.x; kn[2 * c + 1] = k2.y;
            ke[2 * c] = ke2.x; ke[2 * c + 1] = ke2.y;
            qe[2 * c] = qe2.x; qe[2 * c + 1] = qe2.y;
        }
        const float qk = group_sum<LPR>(qk2.x + qk2.y);
        if (!mine) return;
        const int o = tt * D + c0;
        *reinterpret_cast<float4 *>(fe + o) = make_float4(e[0], e[1], e[2], e[3]);
        *reinterpret_cast<float4 *>(fe + o + 4) = make_float4(e[4], e[5], e[6], e[7]);
        *reinterpret_cast<float4 *>(fkn + o) = make_float4(kn[0], kn[1], kn[2], kn[3]);
        *reinterpret_cast<float4 *>(fkn + o + 4) = make_float4(kn[4], kn[5], kn[6], kn[7]);
        *reinterpret_cast<float4 *>(fke + o) = make_float4(ke[0], ke[1], ke[2], ke[3]);
        *reinterpret_cast<float4 *>(fke + o + 4) = make_float4(ke[4], ke[5], ke[6], ke[7]);
        *reinterpret_cast<float4 *>(fqe + o) = make_float4(qe[0], qe[1], qe[2], qe[3]);
        *reinterpret_cast<float4 *>(fqe + o + 4) = make_float4(qe[4], qe[5], qe[6], qe[7]);
        if (tid % LPR == 0) fqk[tt] = qk;
    };

    prefetch_state(it, 0);
    for (int st = 0; it < items; it += gridDim.x, st ^= 1) {
        const int64_t req = it / H;
        const int h = static_cast<int>(it % H);
        const int64_t blk = (static_cast<int64_t>(h) * D) * D;  // head block within a cache / pool row
        const bool valid = row_of(it) >= 0;
        __syncthreads();  // the previous item's staged inputs are consumed
        stage_tokens(req, h, 0, a.L < kVT ? a.L : kVT);
        if (it + gridDim.x < items) prefetch_state(it + gridDim.x, st ^ 1);
        else asm volatile("cp.async.commit_group;\n" ::: "memory");
        asm volatile("cp.async.wait_group 1;\n" ::: "memory");  // this item's state and first inputs
        __syncthreads();  // ... including the inputs other threads staged
        token_factors(a.L < kVT ? a.L : kVT);
        __syncthreads();
        float s[ROWS][8];
#pragma unroll
        for (int j = 0; j < ROWS; ++j) {
            if (valid) {
                const uint4 x = slots[((st * ROWS + j) * v16) * THREADS + tid];
                if (v16 == 1) {
                    s[j][0] = bf16_lo(x.x); s[j][1] = bf16_hi(x.x); s[j][2] = bf16_lo(x.y); s[j][3] = bf16_hi(x.y);
                    s[j][4] = bf16_lo(x.z); s[j][5] = bf16_hi(x.z); s[j][6] = bf16_lo(x.w); s[j][7] = bf16_hi(x.w);
                } else {
                    const uint4 y = slots[((st * ROWS + j) * v16 + 1) * THREADS + tid];
                    s[j][0] = __uint_as_float(x.x); s[j][1] = __uint_as_float(x.y);
                    s[j][2] = __uint_as_float(x.z); s[j][3] = __uint_as_float(x.w);
                    s[j][4] = __uint_as_float(y.x); s[j][5] = __uint_as_float(y.y);
                    s[j][6] = __uint_as_float(y.z); s[j][7] = __uint_as_float(y.w);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c) s[j][c] = 0.f;
            }
        }
        for (int t0 = 0; t0 < a.L; t0 += kVT) {
            const int nt = a.L - t0 < kVT ? a.L - t0 : kVT;
            if (t0 > 0) {  // later groups of more than kVT draft tokens
                __syncthreads();
                stage_tokens(req, h, t0, nt);
                cp_async_wait_all();
                __syncthreads();
                token_factors(nt);
                __syncthreads();
            }
            for (int tt = 0; tt < nt; ++tt) {
            const int64_t tok = req * a.L + t0 + tt;
            const int64_t base = (tok * H + h) * D;
            float vv[ROWS];
#pragma unroll
            for (int j = 0; j < ROWS; ++j) vv[j] = load_as_f32(sv + tt * D + r0 + RPP * j);
            const float bt = sb[tt];
            float2 e[4], ke[4], qe[4], kn[4];
            {
                const int o = tt * D + c0;
#pragma unroll
                for (int h4 = 0; h4 < 2; ++h4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(fe + o + 4 * h4);
                    const float4 b4 = *reinterpret_cast<const float4 *>(fkn + o + 4 * h4);
                    const float4 c4 = *reinterpret_cast<const float4 *>(fke + o + 4 * h4);
                    const float4 d4 = *reinterpret_cast<const float4 *>(fqe + o + 4 * h4);
                    e[2 * h4] = make_float2(a4.x, a4.y); e[2 * h4 + 1] = make_float2(a4.z, a4.w);
                    kn[2 * h4] = make_float2(b4.x, b4.y); kn[2 * h4 + 1] = make_float2(b4.z, b4.w);
                    ke[2 * h4] = make_float2(c4.x, c4.y); ke[2 * h4 + 1] = make_float2(c4.z, c4.w);
                    qe[2 * h4] = make_float2(d4.x, d4.y); qe[2 * h4 + 1] = make_float2(d4.z, d4.w);
                }
            }
            const float qk = fqk[tt];
            const int64_t slot = static_cast<int64_t>(inter[tok]);
            const bool keep = slot >= 0 && slot < a.pool.n_rows;
            if constexpr (2 * ROWS == LPR) {
                // the 2 ROWS dot products of this thread's rows, reduced over the row's LPR
                // lanes by a transposed butterfly: lane g of the group ends with value g
                // (a of row g / 2 for even g, b for odd g)
                float vals[2 * ROWS];
#pragma unroll
                for (int j = 0; j < ROWS; ++j) {
                    float2 ak = make_float2(0.f, 0.f), bq = make_float2(0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float2 s2 = make_float2(s[j][2 * c], s[j][2 * c + 1]);
                        ak = fma2(ke[c], s2, ak);
                        bq = fma2(qe[c], s2, bq);
                    }
                    vals[2 * j] = ak.x + ak.y;
                    vals[2 * j + 1] = bq.x + bq.y;
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
                const int g = tid % LPR, jr = g >> 1;
                const float u_even = bt * (load_as_f32(sv + tt * D + r0 + RPP * jr) - vals[0]);  // even lanes: u
                const float u_pair = __shfl_sync(0xffffffffu, u_even, lane & ~1);
                if (g & 1) og[base + r0 + RPP * jr] = from_f32<IO>(a.scale * fmaf(qk, u_pair, vals[0]));
                const int gbase = lane & ~(LPR - 1);
#pragma unroll
                for (int j = 0; j < ROWS; ++j) {
                    const float u = __shfl_sync(0xffffffffu, u_even, gbase + 2 * j);
                    update_row(s[j], e, kn, u);
                    if (keep)
                        store8_stream(a.pool.data, a.pool.dtype,
                                      slot * a.pool.row_stride + blk + (r0 + RPP * j) * D + c0, s[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < ROWS; ++j) {
                    float2 ak2 = make_float2(0.f, 0.f), bq2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float2 s2 = make_float2(s[j][2 * c], s[j][2 * c + 1]);
                        ak2 = fma2(ke[c], s2, ak2);
                        bq2 = fma2(qe[c], s2, bq2);
                    }
                    const float ak = group_sum<LPR>(ak2.x + ak2.y);
                    const float bq = group_sum<LPR>(bq2.x + bq2.y);
                    const float u = bt * (vv[j] - ak);
                    update_row(s[j], e, kn, u);
                    if (tid % LPR == 0) og[base + r0 + RPP * j] = from_f32<IO>(a.scale * fmaf(qk, u, bq));
                    if (keep)
                        store8_stream(a.pool.data, a.pool.dtype,
                                      slot * a.pool.row_stride + blk + (r0 + RPP * j) * D + c0, s[j]);
                }
            }
            }
        }
    }
}

template <int D, typename IO, typename IdxT> cudaError_t launch_typed(const VerifyArgs &a, cudaStream_t st)
{
    constexpr int THREADS = verify_threads<D>();
    constexpr int ROWS = D / (THREADS / (D / 8));
    const int v16 = a.cache.dtype == KDA_F32 ? 2 : 1;
    const int smem = verify_stage_bytes<D, IO>() + 2 * ROWS * v16 * THREADS * 16;
    auto kern = verify_kernel<D, IO, IdxT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, THREADS, smem)) != cudaSuccess) return e;
    const int64_t items = a.batch * a.h;
    const int64_t resident = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
    kern<<<static_cast<unsigned>(items < resident ? items : resident), THREADS, smem, st>>>(a);
    return cudaGetLastError();
}

template <int D> cudaError_t launch_d(const VerifyArgs &a, cudaStream_t st)
{
    const bool bf = a.io_dtype == KDA_BF16, i64 = a.idx_type == KDA_I64;
    if (bf)
        return i64 ? launch_typed<D, __nv_bfloat16, int64_t>(a, st) : launch_typed<D, __nv_bfloat16, int32_t>(a, st);
    return i64 ? launch_typed<D, float, int64_t>(a, st) : launch_typed<D, float, int32_t>(a, st);
}

}  // namespace

cudaError_t launch_target_verify(const VerifyArgs &a, cudaStream_t st)
{
    switch (a.d) {
    case 32: return launch_d<32>(a, st);
    case 64: return launch_d<64>(a, st);
    default: return launch_d<128>(a, st);
    }
}

}  // namespace kda
