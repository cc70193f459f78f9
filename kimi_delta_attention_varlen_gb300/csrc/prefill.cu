// Chunkwise (C = 64) gated delta-rule prefill over a cu_seqlens varlen batch.
//
// The method: the recurrence S_t = (I - beta_t k_t k_t^T) Diag(e^{g_t}) S_{t-1}
// + beta_t k_t v_t^T, o_t = scale * S_t^T q_t ("KDA's challenges for AI infra"
// page, section 1.1) is affine in S, so a chunk of tokens composes into one
// affine map (section 1.3).  The "Support Kimi-K3 on NPU" report's extend
// listing evaluates it in this order, which the kernels follow:
//   l2norm(q, k) -> chunk table -> in-chunk cumsum of g -> gated K K^T and
//   Q K^T -> T = (I + A_kk)^-1 -> W, U -> inter-chunk state pass -> output.
//
// With G the in-chunk cumulative gate (per channel), for one chunk and head:
//   A_kk[i,j] = beta_i sum_c k_ic k_jc e^{G_ic - G_jc}       (i > j)
//   A_qk[i,j] = scale  sum_c q_ic k_jc e^{G_ic - G_jc}       (i >= j)
//   T = (I + A_kk)^-1,  W = T diag(beta) (K * e^G),  U = T diag(beta) V
//   V_new = U - W S,   O = (scale Q * e^G) S + A_qk V_new
//   S    <- Diag(e^{G_last}) S + (K * e^{G_last - G})^T V_new
//
// Kernels (all on the caller's stream):
//   1. chunk_table_kernel   one CTA: chunk offsets per sequence (prefix sum of
//                           ceil(len/64)) and a longest-first sequence order.
//   2. chunk_prep_kernel    one CTA per (chunk, head), fully parallel: every
//                           quantity above that does not depend on S, written
//                           to the workspace as one record per (chunk, head).
//   3. state_pass_kernel    one CTA per (sequence, head, value slice): walks the
//                           sequence's chunks in order with S in registers
//                           (fp32 accumulators), double-buffering the records
//                           into shared memory with bulk async copies.
// All products run on the tensor cores (bf16 operands, fp32 accumulation).
//
// Exponent ranges.  Factors e^{G_i - G_j} are split through a reference row:
// off-diagonal 16x16 blocks use the block midpoints, e^{G_i - G_j} =
// P_i F_IJ R_j with P_i = e^{G_i - G_mI}, F_IJ = e^{G_mI - G_mJ} <= 1 and
// R_j = e^{G_mJ - G_j}; each of P and R spans at most 8 tokens of decay, so
// the products stay in fp32/bf16 range while that decay is above -80.  All
// inter-chunk factors (e^G, e^{G_last - G}, e^{G_last}) are <= 1 for g <= 0.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int C = kChunk;
constexpr uint32_t kWaitLimit = 1u << 22;  // bounded mbarrier polls
constexpr int kPrepThreads = 256;

// ------------------------------------------------------------ record ------
// One record per (chunk, head).  bf16 tiles are swizzled (see swz_off) so the
// state pass can bulk-copy a record verbatim into shared memory.
template <int D> struct Rec {
    static constexpr int RB = 2 * D;                  // row bytes of [64][D] tiles
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

// ---------------------------------------------------------- chunk table ---

__global__ void __launch_bounds__(1024)
chunk_table_kernel(const int32_t *__restrict__ cu, int64_t B, int32_t *__restrict__ chunk_off,
                   int32_t *__restrict__ seq_order, int32_t *__restrict__ status)
{
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        carry = 0;
        *status = 0;
    }
    __syncthreads();
    for (int64_t base = 0; base < B; base += 1024) {
        const int64_t b = base + tid;
        int32_t n = 0;
        if (b < B) {
            const int32_t len = cu[b + 1] - cu[b];
            n = len > 0 ? (len + C - 1) / C : 0;
        }
        int32_t x = n;  // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int32_t w = warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_tot[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int32_t before = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + x - n;
        if (b < B) chunk_off[b] = before;
        __syncthreads();
        if (tid == 1023) carry = before + n;
        __syncthreads();
    }
    if (tid == 0) chunk_off[B] = carry;
    // Longest sequences first, so their serial chunk chains start early.
    if (B <= 4096) {
        for (int64_t b = tid; b < B; b += 1024) {
            const int32_t lb = cu[b + 1] - cu[b];
            int32_t rank = 0;
            for (int64_t o = 0; o < B; ++o) {
                const int32_t lo = cu[o + 1] - cu[o];
                rank += (lo > lb) || (lo == lb && o < b);
            }
            seq_order[rank] = static_cast<int32_t>(b);
        }
    } else {
        for (int64_t b = tid; b < B; b += 1024) seq_order[b] = static_cast<int32_t>(b);
    }
}

// ----------------------------------------------------------- chunk prep ---

template <int D> struct PrepSmem {
    static constexpr int TILE = C * D * 2;
    static constexpr int AS = 68;                                    // fp32 row stride of A, T
    static constexpr int GREG = (C * D * 4 > 2 * C * AS * 4) ? C * D * 4 : 2 * C * AS * 4;
    static constexpr int G = 0;                                      // fp32 G [64][D]; later A, T fp32
    static constexpr int KP = ((GREG + 127) / 128) * 128;            // k P      (later W)
    static constexpr int QP = KP + TILE;                             // q P      (later U^T)
    static constexpr int KR = QP + TILE;                             // k R
    static constexpr int KE = KR + TILE;                             // beta k e^G
    static constexpr int VB = KE + TILE;                             // beta v
    static constexpr int AQK = VB + TILE;                            // A_qk bf16 [64][64]
    static constexpr int TB = AQK + C * C * 2;                       // T bf16 [64][64]
    static constexpr int TAB = TB + C * C * 2;                       // L[4][D] Z[4][D] F[16][D]
    static constexpr int BETA = TAB + 24 * D * 4;                    // beta [64]
    static constexpr int XS = BETA + C * 4;                          // solve scratch 8 x [16][16]
    static constexpr int BYTES = XS + 8 * 16 * 16 * 4;
};

template <typename IO, int N> __device__ __forceinline__ void load_slice(const IO *p, float x[N]);
template <> __device__ __forceinline__ void load_slice<float, 4>(const float *p, float x[4])
{
    const float4 a = *reinterpret_cast<const float4 *>(p);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
}
template <> __device__ __forceinline__ void load_slice<float, 2>(const float *p, float x[2])
{
    const float2 a = *reinterpret_cast<const float2 *>(p);
    x[0] = a.x; x[1] = a.y;
}
template <> __device__ __forceinline__ void load_slice<float, 1>(const float *p, float x[1]) { x[0] = *p; }
template <>
__device__ __forceinline__ void load_slice<__nv_bfloat16, 4>(const __nv_bfloat16 *p, float x[4])
{
    const uint2 a = *reinterpret_cast<const uint2 *>(p);
    x[0] = bf16_lo(a.x); x[1] = bf16_hi(a.x); x[2] = bf16_lo(a.y); x[3] = bf16_hi(a.y);
}
template <>
__device__ __forceinline__ void load_slice<__nv_bfloat16, 2>(const __nv_bfloat16 *p, float x[2])
{
    const uint32_t a = *reinterpret_cast<const uint32_t *>(p);
    x[0] = bf16_lo(a); x[1] = bf16_hi(a);
}
template <>
__device__ __forceinline__ void load_slice<__nv_bfloat16, 1>(const __nv_bfloat16 *p, float x[1])
{
    x[0] = __bfloat162float(*p);
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

struct PrepParams {
    const void *q, *k, *v;
    const float *g, *beta;
    const int32_t *cu;
    const int32_t *chunk_off;
    int64_t B;
    int32_t H;
    float scale;
    int32_t l2norm;
    char *records;
};

template <int D, typename IO>
__global__ void __launch_bounds__(kPrepThreads)
chunk_prep_kernel(PrepParams p)
{
    using SM = PrepSmem<D>;
    using R = Rec<D>;
    constexpr int RB = R::RB;
    constexpr int CPL = D / 32;  // channels per lane in the row pass
    extern __shared__ __align__(1024) char smem[];
    __shared__ int32_t s_seq[3];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gid = lane >> 2, tig = lane & 3, mi = lane >> 3, ri = lane & 7;
    const int64_t chunk = blockIdx.x;
    const int h = blockIdx.y;
    const int32_t n_chunks = p.chunk_off[p.B];
    if (chunk >= n_chunks) return;

    if (tid == 0) {  // sequence owning this chunk: chunk_off[b] <= chunk < chunk_off[b + 1]
        int64_t lo = 0, hi = p.B;  // count of b in [1, B] with chunk_off[b] <= chunk
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) / 2;
            if (p.chunk_off[mid] <= chunk) lo = mid;
            else hi = mid - 1;
        }
        const int64_t b = lo;
        const int32_t t0 = p.cu[b] + static_cast<int32_t>(chunk - p.chunk_off[b]) * C;
        const int32_t left = p.cu[b + 1] - t0;
        s_seq[0] = t0;
        s_seq[1] = left < C ? left : C;
    }
    __syncthreads();
    const int64_t t0 = s_seq[0];
    const int len = s_seq[1];
    const int64_t H = p.H;
    char *rec = p.records + (chunk * H + h) * static_cast<int64_t>(R::BYTES);

    float *sG = reinterpret_cast<float *>(smem + SM::G);
    float *sBeta = reinterpret_cast<float *>(smem + SM::BETA);
    float *sL = reinterpret_cast<float *>(smem + SM::TAB);
    float *sZ = sL + 4 * D;
    float *sF = sZ + 4 * D;  // sF[(I * 4 + J) * D + c]

    // ---- 1. gate rows and beta; in-chunk cumulative sum of g per channel ----
    for (int e = tid; e < C * (D / 4); e += kPrepThreads) {
        const int i = e / (D / 4), c4 = e % (D / 4);
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < len) val = *reinterpret_cast<const float4 *>(p.g + ((t0 + i) * H + h) * D + c4 * 4);
        *reinterpret_cast<float4 *>(sG + i * D + c4 * 4) = val;
    }
    if (tid < C) sBeta[tid] = tid < len ? p.beta[(t0 + tid) * H + h] : 0.f;
    __syncthreads();
    {
        constexpr int SEG = kPrepThreads / D, RPS = C / SEG;
        const int c = tid % D, sg = tid / D;
        float acc = 0.f;
        for (int i = sg * RPS; i < (sg + 1) * RPS; ++i) {
            acc += sG[i * D + c];
            sG[i * D + c] = acc;
        }
        __syncthreads();
        float off = 0.f;
        for (int s2 = 0; s2 < sg; ++s2) off += sG[((s2 + 1) * RPS - 1) * D + c];
        __syncthreads();
        if (sg > 0)
            for (int i = sg * RPS; i < (sg + 1) * RPS; ++i) sG[i * D + c] += off;
        __syncthreads();
    }
    // per-channel tables at the 16-row block midpoints m_I = 16 I + 8
    for (int c = tid; c < D; c += kPrepThreads) {
        const float gl = sG[(C - 1) * D + c];
        float gm[4];
#pragma unroll
        for (int I = 0; I < 4; ++I) gm[I] = sG[(16 * I + 8) * D + c];
#pragma unroll
        for (int I = 0; I < 4; ++I) {
            sL[I * D + c] = expf(gm[I]);       // e^{G_mI}          <= 1
            sZ[I * D + c] = expf(gl - gm[I]);  // e^{G_last - G_mI} <= 1
#pragma unroll
            for (int J = 0; J < 4; ++J) sF[(I * 4 + J) * D + c] = J < I ? expf(gm[I] - gm[J]) : 1.f;
        }
        reinterpret_cast<float *>(rec + R::GAMMA)[c] = expf(gl);
    }
    __syncthreads();

    // ---- 2. row pass: normalise q, k; build the bf16 operand tiles ----
    {
        const int cb = lane * CPL;
        const IO *qg = static_cast<const IO *>(p.q);
        const IO *kg = static_cast<const IO *>(p.k);
        const IO *vg = static_cast<const IO *>(p.v);
        for (int i = warp; i < C; i += kPrepThreads / 32) {
            float qv[CPL], kv[CPL], vv[CPL];
            if (i < len) {
                const int64_t off = ((t0 + i) * H + h) * D + cb;
                load_slice<IO, CPL>(qg + off, qv);
                load_slice<IO, CPL>(kg + off, kv);
                load_slice<IO, CPL>(vg + off, vv);
            } else {
#pragma unroll
                for (int c = 0; c < CPL; ++c) qv[c] = kv[c] = vv[c] = 0.f;
            }
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                sq += qv[c] * qv[c];
                sk += kv[c] * kv[c];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            const float rq = p.l2norm ? rsqrtf(sq + 1e-6f) : 1.f;
            const float rk = p.l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
            const int I = i >> 4, m = 16 * I + 8;
            const float bt = sBeta[i];
            float kp[CPL], qp[CPL], kr[CPL], ke[CPL], qt[CPL], kt[CPL], vb[CPL];
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int ch = cb + c;
                const float gi = sG[i * D + ch], gmid = sG[m * D + ch];
                const float P = __expf(gi - gmid);
                const float Rr = __expf(gmid - gi);
                const float qh = qv[c] * rq, kh = kv[c] * rk;
                kp[c] = kh * P;
                qp[c] = qh * P;
                kr[c] = kh * Rr;
                ke[c] = bt * kh * P * sL[I * D + ch];
                qt[c] = p.scale * qh * P * sL[I * D + ch];
                kt[c] = kh * Rr * sZ[I * D + ch];
                vb[c] = bt * vv[c];
            }
            const uint32_t o = swz_off<RB>(i, cb);
            store_bf16<CPL>(smem + SM::KP, o, kp);
            store_bf16<CPL>(smem + SM::QP, o, qp);
            store_bf16<CPL>(smem + SM::KR, o, kr);
            store_bf16<CPL>(smem + SM::KE, o, ke);
            store_bf16<CPL>(smem + SM::VB, o, vb);
            store_bf16<CPL>(rec + R::QT, o, qt);
            store_bf16<CPL>(rec + R::KT, o, kt);
        }
    }
    __syncthreads();

    // ---- 3. gated Gram products: warps 0-3 A_kk, warps 4-7 A_qk ----
    float *sA = reinterpret_cast<float *>(smem + SM::G);  // fp32 [64][AS]
    float *sT = sA + C * SM::AS;                           // fp32 [64][AS]
    {
        const int I = warp & 3;
        const bool is_qk = warp >= 4;
        const char *src = smem + (is_qk ? SM::QP : SM::KP);
        for (int J = 0; J < 4; ++J) {
            float acc[2][4] = {};
            if (J <= I) {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    uint32_t a[4], b[4];
                    ldmatrix_x4(a, smem_u32(src + swz_off<RB>(16 * I + ri + 8 * (mi & 1), 16 * ks + 8 * (mi >> 1))));
                    if (J < I) {  // a <- a * F_IJ over the fragment's four channels
                        const float *f = sF + (I * 4 + J) * D + 16 * ks + 2 * tig;
                        const float f0 = f[0], f1 = f[1], f2 = f[8], f3 = f[9];
                        a[0] = pack_bf16x2(bf16_lo(a[0]) * f0, bf16_hi(a[0]) * f1);
                        a[1] = pack_bf16x2(bf16_lo(a[1]) * f0, bf16_hi(a[1]) * f1);
                        a[2] = pack_bf16x2(bf16_lo(a[2]) * f2, bf16_hi(a[2]) * f3);
                        a[3] = pack_bf16x2(bf16_lo(a[3]) * f2, bf16_hi(a[3]) * f3);
                    }
                    ldmatrix_x4(b, smem_u32(smem + SM::KR +
                                            swz_off<RB>(16 * J + ri + 8 * (mi >> 1), 16 * ks + 8 * (mi & 1))));
                    mma_bf16(acc[0], a, b[0], b[1]);
                    mma_bf16(acc[1], a, b[2], b[3]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int i = 16 * I + gid + 8 * hr;
                    const int j = 16 * J + 8 * nt + 2 * tig;
                    const float x0 = acc[nt][2 * hr], x1 = acc[nt][2 * hr + 1];
                    if (!is_qk) {
                        const float bi = sBeta[i];
                        sA[i * SM::AS + j] = j < i ? x0 * bi : 0.f;
                        sA[i * SM::AS + j + 1] = j + 1 < i ? x1 * bi : 0.f;
                    } else {
                        const float y0 = j <= i ? x0 * p.scale : 0.f;
                        const float y1 = j + 1 <= i ? x1 * p.scale : 0.f;
                        *reinterpret_cast<uint32_t *>(smem + SM::AQK + swz_off<128>(i, j)) = pack_bf16x2(y0, y1);
                    }
                }
            }
        }
    }
    __syncthreads();

    // ---- 4. T = (I + A_kk)^-1, blocked by 16 (fp32) ----
    if (warp < 4 && lane < 16) {  // diagonal blocks: forward substitution, lane = column
        const int I = warp, j = lane;
        const float *A = sA + 16 * I * SM::AS + 16 * I;
        float tcol[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = i == j ? 1.f : 0.f;
#pragma unroll
            for (int kk = 0; kk < i; ++kk) acc -= A[i * SM::AS + kk] * tcol[kk];
            tcol[i] = acc;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) sT[(16 * I + i) * SM::AS + 16 * I + j] = tcol[i];
    }
    __syncthreads();
    for (int d = 1; d < 4; ++d) {  // off-diagonal blocks by sub-diagonal
        if (warp < 4 - d) {
            const int J = warp, I = warp + d;
            const int r = lane >> 1, c0 = (lane & 1) * 8;
            float *xs = reinterpret_cast<float *>(smem + SM::XS) + warp * 256;
            float x[8] = {};
            for (int Kb = J; Kb < I; ++Kb) {
#pragma unroll 4
                for (int m = 0; m < 16; ++m) {
                    const float a = sA[(16 * I + r) * SM::AS + 16 * Kb + m];
                    const float *t = sT + (16 * Kb + m) * SM::AS + 16 * J + c0;
#pragma unroll
                    for (int c = 0; c < 8; ++c) x[c] += a * t[c];
                }
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) xs[r * 16 + c0 + c] = x[c];
            __syncwarp();
            float y[8] = {};
#pragma unroll 4
            for (int m = 0; m < 16; ++m) {
                const float t = sT[(16 * I + r) * SM::AS + 16 * I + m];
#pragma unroll
                for (int c = 0; c < 8; ++c) y[c] += t * xs[m * 16 + c0 + c];
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) sT[(16 * I + r) * SM::AS + 16 * J + c0 + c] = -y[c];
        }
        __syncthreads();
    }
    for (int e = tid; e < C * (C / 2); e += kPrepThreads) {  // T -> bf16, zero above block diagonal
        const int i = e / (C / 2), j = 2 * (e % (C / 2));
        const bool keep = (j >> 4) <= (i >> 4);
        const float t0v = keep ? sT[i * SM::AS + j] : 0.f;
        const float t1v = keep ? sT[i * SM::AS + j + 1] : 0.f;
        *reinterpret_cast<uint32_t *>(smem + SM::TB + swz_off<128>(i, j)) = pack_bf16x2(t0v, t1v);
    }
    __syncthreads();

    // ---- 5. W = T (beta K e^G) (warps 0-3), U = T (beta V) (warps 4-7) ----
    {
        const int I = warp & 3;
        const bool is_u = warp >= 4;
        const char *bsrc = smem + (is_u ? SM::VB : SM::KE);
        float acc[D / 8][4] = {};
        for (int ks = 0; ks <= I; ++ks) {  // T is lower triangular
            uint32_t a[4];
            ldmatrix_x4(a, smem_u32(smem + SM::TB + swz_off<128>(16 * I + ri + 8 * (mi & 1), 16 * ks + 8 * (mi >> 1))));
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t b[4];
                ldmatrix_x4_trans(b, smem_u32(bsrc + swz_off<RB>(16 * ks + ri + 8 * (mi & 1), 16 * np + 8 * (mi >> 1))));
                mma_bf16(acc[2 * np], a, b[0], b[1]);
                mma_bf16(acc[2 * np + 1], a, b[2], b[3]);
            }
        }
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int i = 16 * I + gid + 8 * hr;
                const int c = 8 * n + 2 * tig;
                if (!is_u) {
                    *reinterpret_cast<uint32_t *>(smem + SM::KP + swz_off<RB>(i, c)) =
                        pack_bf16x2(acc[n][2 * hr], acc[n][2 * hr + 1]);
                } else {  // U^T [D][64]
                    *reinterpret_cast<uint16_t *>(smem + SM::QP + swz_off<128>(c, i)) = f32_to_bf16_bits(acc[n][2 * hr]);
                    *reinterpret_cast<uint16_t *>(smem + SM::QP + swz_off<128>(c + 1, i)) =
                        f32_to_bf16_bits(acc[n][2 * hr + 1]);
                }
            }
        }
    }
    __syncthreads();

    // ---- 6. copy W, A_qk, U^T out to the record ----
    {
        const uint4 *sw = reinterpret_cast<const uint4 *>(smem + SM::KP);
        const uint4 *sq = reinterpret_cast<const uint4 *>(smem + SM::AQK);
        const uint4 *su = reinterpret_cast<const uint4 *>(smem + SM::QP);
        uint4 *gw = reinterpret_cast<uint4 *>(rec + R::W);
        uint4 *gq = reinterpret_cast<uint4 *>(rec + R::AQK);
        uint4 *gu = reinterpret_cast<uint4 *>(rec + R::UT);
        for (int e = tid; e < R::TILE / 16; e += kPrepThreads) gw[e] = sw[e];
        for (int e = tid; e < C * C * 2 / 16; e += kPrepThreads) gq[e] = sq[e];
        for (int e = tid; e < D * C * 2 / 16; e += kPrepThreads) gu[e] = su[e];
    }
}

// ----------------------------------------------------------- state pass ---

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

template <int D, typename IO, int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
state_pass_kernel(PassParams p)
{
    using R = Rec<D>;
    constexpr int RB = R::RB;
    constexpr int VT = 16 * WARPS;          // value columns per CTA
    constexpr int NSPLIT = D / VT;
    constexpr int HEAD = R::UT;             // W, Q~, K~, A_qk, gamma
    constexpr int UT_BYTES = VT * C * 2;    // this CTA's rows of U^T
    constexpr int STAGE = HEAD + UT_BYTES;
    static_assert(NSPLIT * VT == D, "value split");
    extern __shared__ __align__(1024) char smem[];
    __shared__ __align__(8) uint64_t bars[2];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gid = lane >> 2, tig = lane & 3, mi = lane >> 3, ri = lane & 7;
    const int64_t H = p.H;
    const int64_t item = blockIdx.x;
    const int vs = static_cast<int>(item % NSPLIT);
    const int h = static_cast<int>((item / NSPLIT) % H);
    const int64_t b = p.seq_order[item / (NSPLIT * H)];
    const int32_t c_begin = p.chunk_off[b], n_chunks = p.chunk_off[b + 1] - c_begin;
    const int64_t tok_begin = p.cu[b], tok_end = p.cu[b + 1];
    const int vl0 = 16 * warp;              // first value column of this warp within the CTA
    const int vg0 = vs * VT + vl0;          // ... within the head
    IO *sO = reinterpret_cast<IO *>(smem + 2 * STAGE) + warp * (C * 16);

    // S^T accumulator fragments: s[n][e] = S^T(v = vg0 + gid + 8 (e >> 1), k = 8 n + 2 tig + (e & 1))
    float s[D / 8][4];
    {
        const int64_t base = ((b * H + h) * D) * D;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int64_t e = base + static_cast<int64_t>(vg0 + gid + 8 * hr) * D + 8 * n + 2 * tig;
                float x0 = 0.f, x1 = 0.f;
                if (p.init != nullptr) {
                    if (p.init_dtype == KDA_F32) {
                        const float2 t = *reinterpret_cast<const float2 *>(static_cast<const float *>(p.init) + e);
                        x0 = t.x;
                        x1 = t.y;
                    } else {
                        const uint32_t t = *reinterpret_cast<const uint32_t *>(static_cast<const uint16_t *>(p.init) + e);
                        x0 = bf16_lo(t);
                        x1 = bf16_hi(t);
                    }
                }
                s[n][2 * hr] = x0;
                s[n][2 * hr + 1] = x1;
            }
        }
    }

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int32_t i, int st) {
        const char *rec = p.records + (static_cast<int64_t>(c_begin + i) * H + h) * R::BYTES;
        char *dst = smem + st * STAGE;
        mbar_arrive_expect_tx(&bars[st], STAGE);
        bulk_g2s(dst, rec, HEAD, &bars[st]);
        bulk_g2s(dst + HEAD, rec + R::UT + vs * UT_BYTES, UT_BYTES, &bars[st]);
    };
    if (tid == 0) {
        if (n_chunks > 0) issue(0, 0);
        if (n_chunks > 1) issue(1, 1);
    }

    IO *out = static_cast<IO *>(p.out);
    bool gave_up = false;  // after one expired wait, stop waiting (the status word reports it)
    for (int32_t i = 0; i < n_chunks; ++i) {
        const int st = i & 1;
        if (!gave_up && !mbar_wait(&bars[st], (i >> 1) & 1, kWaitLimit)) {
            gave_up = true;
            if (lane == 0) atomicExch(p.status, 1);
        }
        const char *sb = smem + st * STAGE;
        const int64_t t0 = tok_begin + static_cast<int64_t>(i) * C;
        const int len = static_cast<int>(tok_end - t0 < C ? tok_end - t0 : C);

        // (1) S^T as bf16 A fragments (M = 16 value rows, K = key channels)
        uint32_t sa[D / 16][4];
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            sa[ks][0] = pack_bf16x2(s[2 * ks][0], s[2 * ks][1]);
            sa[ks][1] = pack_bf16x2(s[2 * ks][2], s[2 * ks][3]);
            sa[ks][2] = pack_bf16x2(s[2 * ks + 1][0], s[2 * ks + 1][1]);
            sa[ks][3] = pack_bf16x2(s[2 * ks + 1][2], s[2 * ks + 1][3]);
        }
        // (2) X^T = S^T W^T and Y^T = S^T Q~^T   (N = 64 chunk rows)
        float x[8][4] = {}, y[8][4] = {};
#pragma unroll
        for (int np = 0; np < 4; ++np) {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t o = swz_off<RB>(16 * np + ri + 8 * (mi >> 1), 16 * ks + 8 * (mi & 1));
                uint32_t bw[4], bq[4];
                ldmatrix_x4(bw, smem_u32(sb + R::W + o));
                ldmatrix_x4(bq, smem_u32(sb + R::QT + o));
                mma_bf16(x[2 * np], sa[ks], bw[0], bw[1]);
                mma_bf16(x[2 * np + 1], sa[ks], bw[2], bw[3]);
                mma_bf16(y[2 * np], sa[ks], bq[0], bq[1]);
                mma_bf16(y[2 * np + 1], sa[ks], bq[2], bq[3]);
            }
        }
        // (3) V_new^T = U^T - X^T, as bf16 A fragments (K = chunk rows)
        uint32_t va[4][4];
        {
            const char *ut = sb + HEAD;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const uint32_t u0 = *reinterpret_cast<const uint32_t *>(ut + swz_off<128>(vl0 + gid, 8 * n + 2 * tig));
                const uint32_t u1 = *reinterpret_cast<const uint32_t *>(ut + swz_off<128>(vl0 + gid + 8, 8 * n + 2 * tig));
                x[n][0] = bf16_lo(u0) - x[n][0];
                x[n][1] = bf16_hi(u0) - x[n][1];
                x[n][2] = bf16_lo(u1) - x[n][2];
                x[n][3] = bf16_hi(u1) - x[n][3];
            }
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                va[ks][0] = pack_bf16x2(x[2 * ks][0], x[2 * ks][1]);
                va[ks][1] = pack_bf16x2(x[2 * ks][2], x[2 * ks][3]);
                va[ks][2] = pack_bf16x2(x[2 * ks + 1][0], x[2 * ks + 1][1]);
                va[ks][3] = pack_bf16x2(x[2 * ks + 1][2], x[2 * ks + 1][3]);
            }
        }
        // (4) O^T = Y^T + V_new^T A_qk^T   (A_qk causal: chunk row t needs s <= t)
#pragma unroll
        for (int tp = 0; tp < 4; ++tp) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                if (ks <= tp) {
                    uint32_t ba[4];
                    ldmatrix_x4(ba, smem_u32(sb + R::AQK + swz_off<128>(16 * tp + ri + 8 * (mi >> 1), 16 * ks + 8 * (mi & 1))));
                    mma_bf16(y[2 * tp], va[ks], ba[0], ba[1]);
                    mma_bf16(y[2 * tp + 1], va[ks], ba[2], ba[3]);
                }
            }
        }
        // (5) output rows through a per-warp staging tile [64][16]
#pragma unroll
        for (int n = 0; n < 8; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = 8 * n + 2 * tig + (e & 1);
                const int vl = gid + 8 * (e >> 1);
                sO[t * 16 + vl] = from_f32<IO>(y[n][e]);
            }
        }
        __syncwarp();
        {
            constexpr int PARTS = 16 * static_cast<int>(sizeof(IO)) / 16;  // uint4 per staged row
            const uint4 *src = reinterpret_cast<const uint4 *>(sO);
            for (int e = lane; e < C * PARTS; e += 32) {
                const int t = e / PARTS, part = e % PARTS;
                if (t < len) {
                    IO *dst = out + ((t0 + t) * H + h) * D + vg0;
                    reinterpret_cast<uint4 *>(dst)[part] = src[e];
                }
            }
        }
        __syncwarp();
        // (6) S^T <- S^T Diag(gamma) + V_new^T K~
        {
            const float *gam = reinterpret_cast<const float *>(sb + R::GAMMA);
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                const float2 gm = *reinterpret_cast<const float2 *>(gam + 8 * n + 2 * tig);
                s[n][0] *= gm.x;
                s[n][1] *= gm.y;
                s[n][2] *= gm.x;
                s[n][3] *= gm.y;
            }
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t bk[4];
                    ldmatrix_x4_trans(bk, smem_u32(sb + R::KT + swz_off<RB>(16 * ks + ri + 8 * (mi & 1), 16 * np + 8 * (mi >> 1))));
                    mma_bf16(s[2 * np], va[ks], bk[0], bk[1]);
                    mma_bf16(s[2 * np + 1], va[ks], bk[2], bk[3]);
                }
            }
        }
        __syncthreads();  // every warp is done with this stage
        if (tid == 0 && i + 2 < n_chunks) issue(i + 2, st);
    }

    if (p.final_state != nullptr) {
        const int64_t base = ((b * H + h) * D) * D;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int64_t e = base + static_cast<int64_t>(vg0 + gid + 8 * hr) * D + 8 * n + 2 * tig;
                *reinterpret_cast<float2 *>(p.final_state + e) = make_float2(s[n][2 * hr], s[n][2 * hr + 1]);
            }
        }
    }
}

template <int D> int rec_bytes() { return Rec<D>::BYTES; }

int rec_bytes_for(int d)
{
    switch (d) {
    case 32: return rec_bytes<32>();
    case 64: return rec_bytes<64>();
    case 128: return rec_bytes<128>();
    default: return 0;
    }
}

template <int D, typename IO, int WARPS>
cudaError_t launch_pass(const PassParams &pp, int64_t items, cudaStream_t st)
{
    constexpr int VT = 16 * WARPS;
    constexpr int STAGE = Rec<D>::UT + VT * C * 2;
    const int smem = 2 * STAGE + WARPS * C * 16 * static_cast<int>(sizeof(IO));
    auto kern = state_pass_kernel<D, IO, WARPS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(items * (D / VT)), WARPS * 32, smem, st>>>(pp);
    return cudaGetLastError();
}

template <int D, typename IO>
cudaError_t launch_typed(const PrefillArgs &a, const PrefillLayout &L, cudaStream_t st)
{
    char *ws = static_cast<char *>(a.workspace);
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    int32_t *chunk_off = reinterpret_cast<int32_t *>(ws + L.off_chunk_off);
    int32_t *seq_order = reinterpret_cast<int32_t *>(ws + L.off_seq_order);
    char *records = ws + L.off_records;

    auto mark = [&](int i) -> cudaError_t {
        return a.events ? cudaEventRecord(static_cast<cudaEvent_t>(a.events[i]), st) : cudaSuccess;
    };
    cudaError_t e = mark(0);
    if (e != cudaSuccess) return e;
    chunk_table_kernel<<<1, 1024, 0, st>>>(a.cu_seqlens, a.num_seqs, chunk_off, seq_order, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if ((e = mark(1)) != cudaSuccess) return e;

    if (L.n_chunk_max > 0) {
        PrepParams pp{a.q, a.k, a.v, a.g, a.beta, a.cu_seqlens, chunk_off, a.num_seqs, a.h, a.scale, a.l2norm, records};
        auto kern = chunk_prep_kernel<D, IO>;
        constexpr int smem = PrepSmem<D>::BYTES;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        kern<<<dim3(static_cast<unsigned>(L.n_chunk_max), static_cast<unsigned>(a.h)), kPrepThreads, smem, st>>>(pp);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }

    if ((e = mark(2)) != cudaSuccess) return e;
    PassParams sp{a.cu_seqlens, chunk_off, seq_order, status, records, a.h, a.init_state, a.init_dtype,
                  a.final_state, a.out};
    // Enough CTAs to cover the SMs: split the value columns when there are few
    // (sequence, head) pairs.  Columns of S evolve independently.
    const int64_t items = a.num_seqs * a.h;
    int warps = D / 16;
    while (warps > 1 && items * (D / (16 * warps)) < 120) warps /= 2;
    if constexpr (D == 128) {
        if (warps == 8) e = launch_pass<D, IO, 8>(sp, items, st);
        else if (warps == 4) e = launch_pass<D, IO, 4>(sp, items, st);
        else if (warps == 2) e = launch_pass<D, IO, 2>(sp, items, st);
        else e = launch_pass<D, IO, 1>(sp, items, st);
    } else if constexpr (D == 64) {
        if (warps == 4) e = launch_pass<D, IO, 4>(sp, items, st);
        else if (warps == 2) e = launch_pass<D, IO, 2>(sp, items, st);
        else e = launch_pass<D, IO, 1>(sp, items, st);
    } else {
        if (warps == 2) e = launch_pass<D, IO, 2>(sp, items, st);
        else e = launch_pass<D, IO, 1>(sp, items, st);
    }
    if (e != cudaSuccess) return e;
    return mark(3);
}

}  // namespace

bool prefill_layout(int64_t total_tokens, int64_t num_seqs, int32_t h, int32_t d, PrefillLayout *out)
{
    const int rb = rec_bytes_for(d);
    if (rb == 0 || total_tokens < 0 || num_seqs < 1 || h < 1) return false;
    auto up = [](size_t x, size_t a) { return (x + a - 1) / a * a; };
    PrefillLayout L{};
    L.n_chunk_max = (total_tokens + (C - 1) * num_seqs) / C;  // >= sum of ceil(len / C)
    L.rec_bytes = static_cast<size_t>(rb);
    L.off_chunk_off = 256;
    L.off_seq_order = up(L.off_chunk_off + 4 * static_cast<size_t>(num_seqs + 1), 256);
    L.off_records = up(L.off_seq_order + 4 * static_cast<size_t>(num_seqs), 1024);
    L.total = L.off_records + static_cast<size_t>(L.n_chunk_max) * static_cast<size_t>(h) * L.rec_bytes;
    *out = L;
    return true;
}

cudaError_t launch_prefill(const PrefillArgs &a, const PrefillLayout &L, cudaStream_t st)
{
    const bool bf = a.io_dtype == KDA_BF16;
    switch (a.d) {
    case 32: return bf ? launch_typed<32, __nv_bfloat16>(a, L, st) : launch_typed<32, float>(a, L, st);
    case 64: return bf ? launch_typed<64, __nv_bfloat16>(a, L, st) : launch_typed<64, float>(a, L, st);
    default: return bf ? launch_typed<128, __nv_bfloat16>(a, L, st) : launch_typed<128, float>(a, L, st);
    }
}

}  // namespace kda
