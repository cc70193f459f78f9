// Chunk preparation: every quantity of one (chunk, head) that does not depend
// on the recurrent state, written to the workspace as one record.
//
// Order of the "Support Kimi-K3 on NPU" report's extend listing, restated:
//   q, k L2-normalised per token; G = in-chunk cumulative sum of g;
//   A_kk[i,j] = beta_i sum_c k_ic k_jc e^{G_ic - G_jc}   (i > j)
//   A_qk[i,j] = scale  sum_c q_ic k_jc e^{G_ic - G_jc}   (i >= j)
//   T = (I + A_kk)^-1;  W = T diag(beta) (K * e^G);  U = T diag(beta) V
// plus the state-pass operands Q~ = scale q e^G, K~ = k e^{G_last - G} and
// gamma = e^{G_last}.
//
// GPU mapping: one CTA (8 warps) per (chunk, head), two CTAs per SM.  All
// global loads of the chunk are issued up front into registers (q/k/v rows
// per warp, g columns per cumsum thread), so one memory latency covers the
// whole chunk and the co-resident CTA's compute hides it.  The gated Gram
// products and W, U run on the tensor cores (bf16 operands, fp32 accumulate);
// the triangular solve is blocked by 16 and stays in fp32.
//
// Exponents: e^{G_i - G_j} = P_i F_IJ R_j with P_i = e^{G_i - G_mI},
// R_j = e^{G_mJ - G_j} (m = midpoint of the 16-row block) and F_IJ =
// e^{G_mI - G_mJ} <= 1 applied to the A fragments; P and R each span at most 8
// tokens of decay.  beta is folded into T (T' = T diag(beta)) and e^G = P L_I
// (L_I = e^{G_mI}) is applied to the k P tile's B fragments, so neither
// beta V nor beta k e^G needs a tile of its own.
#include <type_traits>

#include "prefill_common.cuh"

namespace kda {
namespace prefill {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int D> struct PrepSmem {
    static constexpr int TILE = C * D * 2;                 // bf16 [64][D]
    static constexpr int AS = 68;                          // fp32 row stride of A and T
    static constexpr int GREG0 = C * D * 4 > 2 * C * AS * 4 ? C * D * 4 : 2 * C * AS * 4;
    static constexpr int GREG = (GREG0 + 127) / 128 * 128;
    static constexpr int G = 0;          // G fp32 [64][D] -> A, T fp32 [64][AS] -> T' bf16 [64][64]
    static constexpr int KP = GREG;      // k P: Gram A operand, W's B operand
    static constexpr int QP = KP + TILE; // q P: Gram A operand -> U^T staging [D][64]
    static constexpr int KR = QP + TILE; // k R: Gram B operand -> solve scratch -> W staging
    static constexpr int VS = KR + TILE; // v (bf16): U's B operand
    static constexpr int TAB = VS + TILE;                  // L[4][D], Z[4][D], F[6][D] fp32
    static constexpr int BETA = TAB + 14 * D * 4;          // beta [64]
    static constexpr int TOT = BETA + C * 4;               // cumsum segment totals
    static constexpr int BYTES = TOT + kThreads * 4;
    static_assert(C * C * 2 <= GREG, "T' fits the G region");
};

// CPL io elements of one row, kept packed in registers until used.
template <typename IO, int N> struct Slice {
    static constexpr int BYTES = N * static_cast<int>(sizeof(IO));
    static constexpr int WORDS = BYTES < 4 ? 1 : BYTES / 4;
    uint32_t w[WORDS];
    __device__ __forceinline__ void load(const IO *p)
    {
        if constexpr (BYTES == 16) {
            const uint4 a = *reinterpret_cast<const uint4 *>(p);
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        } else if constexpr (BYTES == 8) {
            const uint2 a = *reinterpret_cast<const uint2 *>(p);
            w[0] = a.x; w[1] = a.y;
        } else if constexpr (BYTES == 4) {
            w[0] = *reinterpret_cast<const uint32_t *>(p);
        } else {
            w[0] = *reinterpret_cast<const uint16_t *>(p);
        }
    }
    __device__ __forceinline__ void zero()
    {
#pragma unroll
        for (int i = 0; i < WORDS; ++i) w[i] = 0u;
    }
    __device__ __forceinline__ void get(float x[N]) const
    {
        if constexpr (sizeof(IO) == 4) {
#pragma unroll
            for (int i = 0; i < N; ++i) x[i] = __uint_as_float(w[i]);
        } else if constexpr (N == 1) {
            x[0] = bf16_lo(w[0]);
        } else {
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                x[2 * i] = bf16_lo(w[i]);
                x[2 * i + 1] = bf16_hi(w[i]);
            }
        }
    }
};

__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t u, float f0, float f1)
{
    return pack_bf16x2(bf16_lo(u) * f0, bf16_hi(u) * f1);
}

// Slot of the factor F_IJ (J < I) in the F table.
__device__ __forceinline__ int fslot(int I, int J) { return I * (I - 1) / 2 + J; }

template <int D, typename IO>
__global__ void __launch_bounds__(kThreads, 2)
chunk_prep_kernel(PrepParams p)
{
    using SM = PrepSmem<D>;
    using R = Rec<D>;
    constexpr int RB = R::RB;
    constexpr int CPL = D / 32;                 // channels per lane in the row pass
    constexpr int ROWS = C / kWarps;            // rows per warp
    constexpr int PRE = (sizeof(IO) == 2 || CPL < 4) ? ROWS : ROWS / 2;  // rows loaded per batch
    constexpr int SEG = kThreads / D;           // cumsum segments per channel
    constexpr int RPS = C / SEG;                // rows per segment
    extern __shared__ __align__(1024) char smem[];
    __shared__ int32_t s_seq[2];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gid = lane >> 2, tig = lane & 3, mi = lane >> 3, ri = lane & 7;
    const int64_t chunk = blockIdx.x;
    const int h = blockIdx.y;
    if (chunk >= p.chunk_off[p.B]) return;
    if (tid == 0) {  // the sequence b with chunk_off[b] <= chunk < chunk_off[b + 1]
        int64_t lo = 0, hi = p.B;
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) / 2;
            if (p.chunk_off[mid] <= chunk) lo = mid;
            else hi = mid - 1;
        }
        const int32_t t0 = p.cu[lo] + static_cast<int32_t>(chunk - p.chunk_off[lo]) * C;
        const int32_t left = p.cu[lo + 1] - t0;
        s_seq[0] = t0;
        s_seq[1] = left < C ? left : C;
    }
    __syncthreads();
    const int64_t t0 = s_seq[0];
    const int len = s_seq[1];
    const int64_t H = p.H;
    char *rec = p.records + (chunk * H + h) * static_cast<int64_t>(R::BYTES);

    float *sG = reinterpret_cast<float *>(smem + SM::G);
    float *sL = reinterpret_cast<float *>(smem + SM::TAB);
    float *sZ = sL + 4 * D;
    float *sF = sZ + 4 * D;
    float *sBeta = reinterpret_cast<float *>(smem + SM::BETA);
    float *sTot = reinterpret_cast<float *>(smem + SM::TOT);

    // ---- 1. issue every load of the chunk: q/k/v rows (per warp), g columns (per thread) ----
    const IO *qg = static_cast<const IO *>(p.q);
    const IO *kg = static_cast<const IO *>(p.k);
    const IO *vg = static_cast<const IO *>(p.v);
    const int cb = lane * CPL;
    Slice<IO, CPL> rq[PRE], rk[PRE], rv[PRE];
    auto load_rows = [&](int j0) {
#pragma unroll
        for (int j = 0; j < PRE; ++j) {
            const int i = warp + kWarps * (j0 + j);
            if (i < len) {
                const int64_t off = ((t0 + i) * H + h) * D + cb;
                rq[j].load(qg + off);
                rk[j].load(kg + off);
                rv[j].load(vg + off);
            } else {
                rq[j].zero();
                rk[j].zero();
                rv[j].zero();
            }
        }
    };
    load_rows(0);
    const int gc = tid % D, gs = tid / D;
    float gr[RPS];
#pragma unroll
    for (int r = 0; r < RPS; ++r) {
        const int i = gs * RPS + r;
        gr[r] = i < len ? p.g[((t0 + i) * H + h) * D + gc] : 0.f;
    }
    if (tid < C) sBeta[tid] = tid < len ? p.beta[(t0 + tid) * H + h] : 0.f;
    // in-chunk cumulative sum of g, per channel: registers, then segment offsets
#pragma unroll
    for (int r = 1; r < RPS; ++r) gr[r] += gr[r - 1];
    sTot[gs * D + gc] = gr[RPS - 1];
    __syncthreads();
    {
        float off = 0.f;
        for (int s2 = 0; s2 < gs; ++s2) off += sTot[s2 * D + gc];
#pragma unroll
        for (int r = 0; r < RPS; ++r) sG[(gs * RPS + r) * D + gc] = gr[r] + off;
    }
    __syncthreads();
    // per-channel factors at the block midpoints m_I = 16 I + 8
    if (tid < D) {
        const int c = tid;
        const float gl = sG[(C - 1) * D + c];
        float gm[4];
#pragma unroll
        for (int I = 0; I < 4; ++I) gm[I] = sG[(16 * I + 8) * D + c];
#pragma unroll
        for (int I = 0; I < 4; ++I) {
            sL[I * D + c] = expf(gm[I]);       // e^{G_mI}          <= 1
            sZ[I * D + c] = expf(gl - gm[I]);  // e^{G_last - G_mI} <= 1
#pragma unroll
            for (int J = 0; J < I; ++J) sF[fslot(I, J) * D + c] = expf(gm[I] - gm[J]);
        }
        reinterpret_cast<float *>(rec + R::GAMMA)[c] = expf(gl);
    }
    __syncthreads();

    // ---- 2. row pass: normalise q, k; operand tiles in shared memory; Q~, K~ to the record ----
#pragma unroll 1
    for (int j0 = 0; j0 < ROWS; j0 += PRE) {
        if (j0 > 0) load_rows(j0);
#pragma unroll
        for (int j = 0; j < PRE; ++j) {
            const int i = warp + kWarps * (j0 + j);
            float qv[CPL], kv[CPL], vv[CPL];
            rq[j].get(qv);
            rk[j].get(kv);
            rv[j].get(vv);
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
            const float nq = p.l2norm ? rsqrtf(sq + 1e-6f) : 1.f;
            const float nk = p.l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
            const int I = i >> 4, m = 16 * I + 8;
            float kp[CPL], qp[CPL], kr[CPL], qt[CPL], kt[CPL];
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int ch = cb + c;
                const float gi = sG[i * D + ch], gmid = sG[m * D + ch];
                const float P = __expf(gi - gmid);
                const float Rr = __expf(gmid - gi);
                const float qh = qv[c] * nq, kh = kv[c] * nk;
                kp[c] = kh * P;
                qp[c] = qh * P;
                kr[c] = kh * Rr;
                qt[c] = p.scale * qh * P * sL[I * D + ch];
                kt[c] = kh * Rr * sZ[I * D + ch];
            }
            const uint32_t o = swz_off<RB>(i, cb);
            store_bf16<CPL>(smem + SM::KP, o, kp);
            store_bf16<CPL>(smem + SM::QP, o, qp);
            store_bf16<CPL>(smem + SM::KR, o, kr);
            store_bf16<CPL>(smem + SM::VS, o, vv);
            store_bf16<CPL>(rec + R::QT, o, qt);
            store_bf16<CPL>(rec + R::KT, o, kt);
        }
    }
    __syncthreads();

    // ---- 3. gated Gram products, 20 (matrix, I, J) block pairs over 8 warps ----
    float *sA = reinterpret_cast<float *>(smem + SM::G);  // A_kk fp32 [64][AS]
    float *sT = sA + C * SM::AS;                           // T fp32 [64][AS]
    for (int pr = warp; pr < 20; pr += kWarps) {
        const bool is_qk = pr >= 10;
        const int li = pr % 10;                            // lower-triangle block index
        const int I = li >= 6 ? 3 : li >= 3 ? 2 : li >= 1 ? 1 : 0;
        const int J = li - I * (I + 1) / 2;
        const char *src = smem + (is_qk ? SM::QP : SM::KP);
        float acc[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t a[4], b[4];
            ldmatrix_x4(a, smem_u32(src + swz_off<RB>(16 * I + ri + 8 * (mi & 1), 16 * ks + 8 * (mi >> 1))));
            if (J < I) {  // a <- a * F_IJ on the fragment's four channels
                const float *f = sF + fslot(I, J) * D + 16 * ks + 2 * tig;
                const float f0 = f[0], f1 = f[1], f2 = f[8], f3 = f[9];
                a[0] = scale_bf16x2(a[0], f0, f1);
                a[1] = scale_bf16x2(a[1], f0, f1);
                a[2] = scale_bf16x2(a[2], f2, f3);
                a[3] = scale_bf16x2(a[3], f2, f3);
            }
            ldmatrix_x4(b, smem_u32(smem + SM::KR + swz_off<RB>(16 * J + ri + 8 * (mi >> 1), 16 * ks + 8 * (mi & 1))));
            mma_bf16(acc[0], a, b[0], b[1]);
            mma_bf16(acc[1], a, b[2], b[3]);
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
                    *reinterpret_cast<uint32_t *>(rec + R::AQK + swz_off<128>(i, j)) = pack_bf16x2(y0, y1);
                }
            }
        }
    }
    __syncthreads();

    // ---- 4. T = (I + A_kk)^-1, blocked by 16, fp32 ----
    if (warp < 4 && lane < 16) {  // diagonal blocks: forward substitution, one column per lane
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
    float *sX = reinterpret_cast<float *>(smem + SM::KR);  // [3][16][16] scratch
    for (int d = 1; d < 4; ++d) {  // blocks (J + d, J), all threads: X = sum_K A_IK T_KJ, then T_IJ = -T_II X
        const int nb = 4 - d;
        for (int o = tid; o < nb * 256; o += kThreads) {
            const int J = o >> 8, I = J + d, r = (o >> 4) & 15, c = o & 15;
            float x = 0.f;
            for (int Kb = J; Kb < I; ++Kb) {
                const float *a = sA + (16 * I + r) * SM::AS + 16 * Kb;
                const float *t = sT + (16 * Kb) * SM::AS + 16 * J + c;
#pragma unroll
                for (int m = 0; m < 16; ++m) x += a[m] * t[m * SM::AS];
            }
            sX[o] = x;
        }
        __syncthreads();
        for (int o = tid; o < nb * 256; o += kThreads) {
            const int J = o >> 8, I = J + d, r = (o >> 4) & 15, c = o & 15;
            const float *t = sT + (16 * I + r) * SM::AS + 16 * I;
            const float *x = sX + (J << 8) + c;
            float y = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) y += t[m] * x[m * 16];
            sT[(16 * I + r) * SM::AS + 16 * J + c] = -y;
        }
        __syncthreads();
    }
    // T' = T diag(beta) as bf16 (the A operand of W and U), zero above the block diagonal
    for (int e = tid; e < C * (C / 2); e += kThreads) {
        const int i = e / (C / 2), j = 2 * (e % (C / 2));
        const bool keep = (j >> 4) <= (i >> 4);
        const float t0v = keep ? sT[i * SM::AS + j] * sBeta[j] : 0.f;
        const float t1v = keep ? sT[i * SM::AS + j + 1] * sBeta[j + 1] : 0.f;
        *reinterpret_cast<uint32_t *>(smem + SM::G + swz_off<128>(i, j)) = pack_bf16x2(t0v, t1v);
    }
    __syncthreads();

    // ---- 5. W = T' (K e^G) (warps 0-3, e^G = P L on the B fragments), U = T' V (warps 4-7) ----
    {
        const int I = warp & 3;
        const bool is_u = warp >= 4;
        const char *bsrc = smem + (is_u ? SM::VS : SM::KP);
        float acc[D / 8][4] = {};
        for (int ks = 0; ks <= I; ++ks) {  // T' is block lower triangular
            uint32_t a[4];
            ldmatrix_x4(a, smem_u32(smem + SM::G + swz_off<128>(16 * I + ri + 8 * (mi & 1), 16 * ks + 8 * (mi >> 1))));
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t b[4];
                ldmatrix_x4_trans(b, smem_u32(bsrc + swz_off<RB>(16 * ks + ri + 8 * (mi & 1), 16 * np + 8 * (mi >> 1))));
                if (!is_u) {  // row block ks of k P times L_ks, per channel
                    const float f0 = sL[ks * D + 16 * np + gid], f1 = sL[ks * D + 16 * np + 8 + gid];
                    b[0] = scale_bf16x2(b[0], f0, f0);
                    b[1] = scale_bf16x2(b[1], f0, f0);
                    b[2] = scale_bf16x2(b[2], f1, f1);
                    b[3] = scale_bf16x2(b[3], f1, f1);
                }
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
                if (!is_u) {  // W staging [64][D] in the KR region
                    *reinterpret_cast<uint32_t *>(smem + SM::KR + swz_off<RB>(i, c)) =
                        pack_bf16x2(acc[n][2 * hr], acc[n][2 * hr + 1]);
                } else {      // U^T staging [D][64] in the QP region
                    *reinterpret_cast<uint16_t *>(smem + SM::QP + swz_off<128>(c, i)) = f32_to_bf16_bits(acc[n][2 * hr]);
                    *reinterpret_cast<uint16_t *>(smem + SM::QP + swz_off<128>(c + 1, i)) =
                        f32_to_bf16_bits(acc[n][2 * hr + 1]);
                }
            }
        }
    }
    __syncthreads();

    // ---- 6. W and U^T out to the record (Q~, K~, A_qk, gamma are already there) ----
    {
        const uint4 *sw = reinterpret_cast<const uint4 *>(smem + SM::KR);
        const uint4 *su = reinterpret_cast<const uint4 *>(smem + SM::QP);
        uint4 *gw = reinterpret_cast<uint4 *>(rec + R::W);
        uint4 *gu = reinterpret_cast<uint4 *>(rec + R::UT);
#pragma unroll
        for (int e = tid; e < R::TILE / 16; e += kThreads) gw[e] = sw[e];
#pragma unroll
        for (int e = tid; e < D * C * 2 / 16; e += kThreads) gu[e] = su[e];
    }
}

template <int D, typename IO>
cudaError_t launch_typed(const PrepParams &p, int64_t n_chunk_max, int32_t h, cudaStream_t st)
{
    auto kern = chunk_prep_kernel<D, IO>;
    constexpr int smem = PrepSmem<D>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(static_cast<unsigned>(n_chunk_max), static_cast<unsigned>(h)), kThreads, smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_prep(int d, int32_t io_dtype, const PrepParams &p, int64_t n_chunk_max, int32_t h,
                              cudaStream_t st)
{
    const bool bf = io_dtype == KDA_BF16;
    switch (d) {
    case 32: return bf ? launch_typed<32, __nv_bfloat16>(p, n_chunk_max, h, st) : launch_typed<32, float>(p, n_chunk_max, h, st);
    case 64: return bf ? launch_typed<64, __nv_bfloat16>(p, n_chunk_max, h, st) : launch_typed<64, float>(p, n_chunk_max, h, st);
    default: return bf ? launch_typed<128, __nv_bfloat16>(p, n_chunk_max, h, st) : launch_typed<128, float>(p, n_chunk_max, h, st);
    }
}

}  // namespace prefill
}  // namespace kda
