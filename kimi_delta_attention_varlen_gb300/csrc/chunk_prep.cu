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
// GPU mapping: one CTA (8 warps) per (chunk, head), heads fastest in the grid
// (the heads of a chunk run together: their input rows are whole [H][D] token
// rows and their records are adjacent), three CTAs per SM for bf16 inputs (two
// for fp32, whose row pass holds more registers).  All
// global loads of the chunk are issued up front: the q/k tiles by TMA tensor
// copies (bf16, head size >= 64; the maps' 128-byte swizzle is the tiles' own
// layout) or per-thread cp.async, v rows into L2 only (they move to shared
// memory after the Gram products, into the k R tile, the same way), and each
// warp's 8 consecutive g rows into registers, where the in-chunk cumulative
// sum runs (warp totals are exchanged once through shared memory).  The gated Gram products and W, U
// run on the tensor cores (bf16 operands, fp32 accumulate).  T' = (I + A_kk)^-1
// diag(beta) is formed blockwise: the four 16x16 diagonal inverses by fp32
// forward substitution, the six blocks below them by MMAs (T'_IJ = -T_II
// sum_K A_IK T'_KJ); then W = T' (K e^G) is a plain block product written in
// place over its right-hand side, and U^T = V^T T'^T is formed directly in the
// record's layout.  W and U^T leave through two bulk copies.
//
// Exponents: e^{G_i - G_j} = P_i F_IJ R_j with P_i = e^{G_i - G_mI},
// R_j = e^{G_mJ - G_j} (m = midpoint of the 16-row block) and F_IJ =
// e^{G_mI - G_mJ} <= 1 applied to the A fragments; P and R each span at most 8
// tokens of decay.  beta is folded into the columns of T' and e^G = P L_K
// (L_K = e^{G_mK}) into the fragments of the k P tile, so neither beta V nor
// beta k e^G needs a tile of its own.  The split is exact only while P and R
// stay in range: the row pass records the largest |G_i - G_mI| of the chunk,
// and a chunk where it exceeds 2^64 (a decay of more than 44 nats within
// 8 tokens of some channel) takes exact_gram instead, which forms every
// e^{G_i - G_j} (i >= j) from its own exponent difference, so any decay,
// however strong, underflows to zero where it should and nowhere else.
#include <cudaTypedefs.h>

#include <type_traits>

#include "prefill_common.cuh"

namespace kda {
namespace prefill {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kPrepWaitLimit = 1u << 22;  // bounded mbarrier polls (and about one second)

template <int D> struct PrepSmem {
    static constexpr int TILE = C * D * 2;                 // bf16 [64][D]
    // Matrix region: the six off-diagonal blocks of A_kk (bf16), the diagonal blocks of
    // T (bf16, as they are and column-scaled by beta), the six blocks of T' below them,
    // three 16x16 scratch blocks and the diagonal blocks of A_kk in fp32.  Before the
    // Gram products it holds the cumulative-sum exchange (warp totals and first rows,
    // fp32 [12][D]).
    static constexpr int AB = 0;                           // A_IK (K < I) bf16 [6][16][16]
    static constexpr int TD = AB + 6 * 512;                // T_II bf16 [4][16][16]
    static constexpr int TS = TD + 4 * 512;                // T_II diag(beta_I) bf16 [4][16][16]
    static constexpr int TO = TS + 4 * 512;                // T'_IJ (J < I) bf16 [6][16][16]
    static constexpr int SCR = TO + 6 * 512;               // per-warp 16x16 bf16 scratch [3]
    static constexpr int AD = SCR + 3 * 512;               // A_II fp32 [4][16][17]
    static constexpr int MEND = AD + 4 * 16 * 17 * 4;
    static constexpr int SUMS = 0;                         // fp32 [8][D] warp totals, [4][D] first rows
    static constexpr int MREG0 = MEND > 12 * D * 4 ? MEND : 12 * D * 4;
    // operand tiles on 1024-byte boundaries: whole 128-byte-swizzle atoms for the tensor copies
    static constexpr int MREG = (MREG0 + 1023) / 1024 * 1024;
    static constexpr int KP = MREG;      // k P: Gram A operand, W right-hand side -> W
    static constexpr int QP = KP + TILE; // q P: Gram A operand -> U^T staging [D][64]
    static constexpr int KR = QP + TILE; // k R: Gram B operand -> v (bf16), the U right-hand side -> U
    static constexpr int TAB = KR + TILE;                  // L[4][D] fp32, F[6][D] bf16
    static constexpr int BETA = TAB + 4 * D * 4 + 6 * D * 2;  // beta [64]
    static constexpr int BYTES = BETA + C * 4;
};

// Byte offset of element (r, c) (0..15) of 16x16 bf16 block `blk`: 32-byte rows, the two
// 16-byte halves swapped on every other group of four rows (conflict-free ldmatrix).
__device__ __forceinline__ uint32_t blk_off(int blk, int r, int c)
{
    return static_cast<uint32_t>(blk * 512 + r * 32 + ((((c >> 3) ^ (r >> 2)) & 1) << 4) + ((c & 7) << 1));
}

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

constexpr float kLog2e = 1.4426950408889634f;

// N consecutive fp32 values from shared memory (N = 1, 2, 4; aligned to N floats).
template <int N> __device__ __forceinline__ void load_f32(const float *p, float x[N])
{
    if constexpr (N == 4) {
        const float4 a = *reinterpret_cast<const float4 *>(p);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    } else if constexpr (N == 2) {
        const float2 a = *reinterpret_cast<const float2 *>(p);
        x[0] = a.x; x[1] = a.y;
    } else {
        x[0] = *p;
    }
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b)
{
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&a);
    const __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162 *>(&b);
    x = __hmul2(x, y);
    return *reinterpret_cast<uint32_t *>(&x);
}


// Slot of the factor F_IJ (J < I) in the F table.
__device__ __forceinline__ int fslot(int I, int J) { return I * (I - 1) / 2 + J; }

// N consecutive fp32 values from global memory (N = 1, 2, 4; aligned to N floats).
template <int N> __device__ __forceinline__ void ldg_f32(const float *p, float x[N])
{
    if constexpr (N == 4) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    } else if constexpr (N == 2) {
        const float2 a = __ldg(reinterpret_cast<const float2 *>(p));
        x[0] = a.x; x[1] = a.y;
    } else {
        x[0] = __ldg(p);
    }
}

// N consecutive fp32 values to shared or global memory (aligned to N floats).
template <int N> __device__ __forceinline__ void st_f32(float *p, const float x[N])
{
    if constexpr (N == 4) *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    else if constexpr (N == 2) *reinterpret_cast<float2 *>(p) = make_float2(x[0], x[1]);
    else *p = x[0];
}

// v[idx] for a warp-uniform runtime idx in 0..3, without local-memory indexing.
__device__ __forceinline__ float pick4(const float v0, const float v1, const float v2, const float v3, int idx)
{
    return idx == 0 ? v0 : idx == 1 ? v1 : idx == 2 ? v2 : v3;
}

// Largest |G_i - G_mI| (log2 units) for which the block split of the Gram is used:
// P, R <= 2^64, so a product P F R that underflows is below 2^-62 where it is lost.
constexpr float kSpanLimit = 64.f;

// Exact gated Gram for a chunk whose decay is too strong for the block split.
// Every e^{G_i - G_j} (i >= j) is the exponential of its own difference, so it
// underflows to zero exactly when the true factor is below fp32's range.  Writes
// what the split path writes: Q~, K~, A_qk (causal, zeros above) and gamma to the
// record, beta A_kk to the matrix region (blocks below the diagonal in bf16, the
// diagonal blocks in fp32), the W right-hand side k e^G into the k P tile with
// L_K = 1.  Scratch while it runs: G^T fp32 in the k P (channels < D/2) and k R
// tiles, q^T and k^T (bf16, unnormalised) in the q P tile and the matrix region
// (offset 0), row norms in the L table.  Rows past the chunk's length are zeros.
// Transposed tiles [channel][row] put row r of channel c at r ^ (c & 31).
template <int D, typename IO>
__device__ __forceinline__ void exact_gram(const IO *__restrict__ qg, const IO *__restrict__ kg,
                                        const float *__restrict__ gg, int32_t Hh, float scale, int32_t l2norm,
                                        char *smem, char *rec, int64_t t0, int len, int h)
{
    using SM = PrepSmem<D>;
    using R = Rec<D>;
    constexpr int CPL = D / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t H = Hh;
    float *rn = reinterpret_cast<float *>(smem + SM::TAB);  // [0, 64) q norms, [64, 128) k norms
    const float *sBeta = reinterpret_cast<const float *>(smem + SM::BETA);
    auto gt = [&](int c, int r) -> float * {  // G^T [c][r]
        char *base = c < D / 2 ? smem + SM::KP : smem + SM::KR;
        return reinterpret_cast<float *>(base) + (c % (D / 2)) * C + (r ^ (c & 31));
    };
    auto qt_at = [&](int c, int r) { return reinterpret_cast<uint16_t *>(smem + SM::QP) + c * C + (r ^ (c & 31)); };
    auto kt_at = [&](int c, int r) { return reinterpret_cast<uint16_t *>(smem + SM::AB) + c * C + (r ^ (c & 31)); };
    static_assert(SM::MREG >= SM::TILE, "k^T fits the matrix region");

    // (1) row norms: warp w owns rows 8w .. 8w + 7, lanes split the channels
    for (int j = 0; j < C / kWarps; ++j) {
        const int i = (C / kWarps) * warp + j;
        float qv[CPL], kv[CPL];
        if (i < len) {
            load_slice<IO, CPL>(qg + ((t0 + i) * H + h) * D + lane * CPL, qv);
            load_slice<IO, CPL>(kg + ((t0 + i) * H + h) * D + lane * CPL, kv);
        } else {
#pragma unroll
            for (int c = 0; c < CPL; ++c) qv[c] = kv[c] = 0.f;
        }
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            sq = fmaf(qv[c], qv[c], sq);
            sk = fmaf(kv[c], kv[c], sk);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
        }
        if (lane == 0) {
            rn[i] = l2norm ? rsqrtf(sq + 1e-6f) : 1.f;
            rn[C + i] = l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
        }
    }
    // (2) one thread per channel: the in-chunk cumulative sum G (log2 units), raw q and k
    //     as bf16 operands, and gamma = 2^{G_last}
    if (tid < D) {
        const int c = tid;
        float G = 0.f;
#pragma unroll 8
        for (int i = 0; i < C; ++i) {
            float gv = 0.f, qv = 0.f, kv = 0.f;
            if (i < len) {
                const int64_t o = ((t0 + i) * H + h) * D + c;
                gv = gg[o];
                qv = load_as_f32<IO>(qg + o);
                kv = load_as_f32<IO>(kg + o);
            }
            G = fmaf(gv, kLog2e, G);
            *gt(c, i) = G;
            *qt_at(c, i) = f32_to_bf16_bits(qv);
            *kt_at(c, i) = f32_to_bf16_bits(kv);
        }
        reinterpret_cast<float *>(rec + R::GAMMA)[c] = ex2_approx(G);
    }
    __syncthreads();

    // (3) thread t: row i = t / 4, columns j = (t % 4) + 4 m; sums over the channels of
    //     k_jc e^{G_ic - G_jc} times k_ic (A_kk) and q_ic (A_qk); -inf exponents above the diagonal
    const int i = tid >> 2, ph = tid & 3;
    float akk[C / 4], aqk[C / 4];
#pragma unroll
    for (int m = 0; m < C / 4; ++m) akk[m] = aqk[m] = 0.f;
#pragma unroll 1
    for (int c = 0; c < D; ++c) {
        const float Gi = *gt(c, i);
        const float qi = bf16_bits_to_f32(*qt_at(c, i)), ki = bf16_bits_to_f32(*kt_at(c, i));
#pragma unroll
        for (int m = 0; m < C / 4; ++m) {
            const int j = ph + 4 * m;
            const float d = j <= i ? Gi - *gt(c, j) : -INFINITY;
            const float t = bf16_bits_to_f32(*kt_at(c, j)) * ex2_approx(d);
            akk[m] = fmaf(ki, t, akk[m]);
            aqk[m] = fmaf(qi, t, aqk[m]);
        }
    }
    const float rqi = rn[i], rki = rn[C + i], bi = sBeta[i];
    float rkj[C / 4];
#pragma unroll
    for (int m = 0; m < C / 4; ++m) rkj[m] = rn[C + ph + 4 * m];

    // (4) one thread per channel: Q~ = scale q^ e^G and K~ = k^ e^{G_last - G} to the
    //     record; k^ e^G (the W right-hand side) kept in registers until G^T is free
    uint32_t kp[C / 2];
    if (tid < D) {
        const int c = tid;
        const float Gl = *gt(c, C - 1);
#pragma unroll
        for (int i2 = 0; i2 < C; i2 += 2) {
            float kpv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = i2 + e;
                float qv = 0.f, kv = 0.f;
                if (r < len) {
                    const int64_t o = ((t0 + r) * H + h) * D + c;
                    qv = load_as_f32<IO>(qg + o);
                    kv = load_as_f32<IO>(kg + o);
                }
                const float G = *gt(c, r);
                const float qh = qv * rn[r], kh = kv * rn[C + r];
                const float eg = ex2_approx(G);
                const uint32_t o2 = tile_off<D, C>(r, c);
                *reinterpret_cast<uint16_t *>(rec + R::qt_at(r, c)) = f32_to_bf16_bits(qh * eg * scale);
                *reinterpret_cast<uint16_t *>(rec + R::KT + o2) = f32_to_bf16_bits(kh * ex2_approx(Gl - G));
                kpv[e] = kh * eg;
            }
            kp[i2 / 2] = pack_bf16x2(kpv[0], kpv[1]);
        }
    }
    __syncthreads();  // every read of the scratch tiles is done

    // (5) results: k e^G into the k P tile, L = 1, beta A_kk to the matrix region, A_qk to the record
    if (tid < D) {
#pragma unroll
        for (int i2 = 0; i2 < C; i2 += 2) {
            *reinterpret_cast<uint16_t *>(smem + SM::KP + tile_off<D, C>(i2, tid)) =
                static_cast<uint16_t>(kp[i2 / 2] & 0xffffu);
            *reinterpret_cast<uint16_t *>(smem + SM::KP + tile_off<D, C>(i2 + 1, tid)) =
                static_cast<uint16_t>(kp[i2 / 2] >> 16);
        }
    }
    for (int e = tid; e < 4 * D; e += kThreads) rn[e] = 1.f;  // the norms were read above
    float *sAd = reinterpret_cast<float *>(smem + SM::AD);
    const int I = i >> 4;
#pragma unroll
    for (int m = 0; m < C / 4; ++m) {
        const int j = ph + 4 * m, J = j >> 4;
        const float ykk = j < i ? akk[m] * rki * rkj[m] * bi : 0.f;
        const float yqk = j <= i ? aqk[m] * rqi * rkj[m] * scale : 0.f;
        if (J < I)
            *reinterpret_cast<uint16_t *>(smem + SM::AB + blk_off(fslot(I, J), i - 16 * I, j - 16 * J)) =
                f32_to_bf16_bits(ykk);
        else if (J == I)
            sAd[I * 16 * 17 + (i - 16 * I) * 17 + (j - 16 * J)] = ykk;
        *reinterpret_cast<uint16_t *>(rec + R::AQK + swz_off<128>(i, j)) = f32_to_bf16_bits(yqk);
    }
}

// One (chunk, head): the record.  kExact = false: the block split, or, for a chunk whose
// decay is out of its range, nothing but an entry in the fix-up list (the CTA leaves before
// the Gram products); kExact = true: the exact Gram.  `ld_bar` (tensor-copy completion,
// phase 0 q and k, phase 1 v) is initialised by the kernel; each call completes two phases.
template <int D, typename IO, bool kExact>
__device__ __forceinline__ void prep_chunk(const PrepParams &p, const PrepMaps &maps, int64_t chunk, int h,
                                           char *smem, uint64_t &ld_bar, bool &gave_up)
{
    using SM = PrepSmem<D>;
    using R = Rec<D>;
    constexpr int ROWB = tile_row_bytes<D>();   // bytes per tile row
    constexpr int CPL = D / 32;                 // channels per lane in the row pass
    constexpr int ROWS = C / kWarps;            // consecutive rows per warp (8: half a 16-row block)
    constexpr int PRE = (sizeof(IO) == 2 || CPL < 4) ? ROWS : ROWS / 2;  // fp32 rows loaded per batch

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gid = lane >> 2, tig = lane & 3, mi = lane >> 3, ri = lane & 7;
    const int2 info = p.chunk_info[chunk];
    const int len = info.y;
    if (len <= 0) return;  // past the last chunk (uniform over the CTA)
    const int64_t t0 = info.x;
    const int64_t H = p.H;
    char *rec = p.records + (chunk * H + h) * static_cast<int64_t>(R::BYTES);

    float *sSum = reinterpret_cast<float *>(smem + SM::SUMS);
    float *sL = reinterpret_cast<float *>(smem + SM::TAB);
    uint16_t *sFb = reinterpret_cast<uint16_t *>(sL + 4 * D);  // F_IJ as bf16 [6][D]
    float *sBeta = reinterpret_cast<float *>(smem + SM::BETA);

    // ---- 1. issue every load of the chunk ----
    const IO *qg = static_cast<const IO *>(p.q);
    const IO *kg = static_cast<const IO *>(p.k);
    const IO *vg = static_cast<const IO *>(p.v);
    const int r0 = ROWS * warp;  // this warp's rows r0 .. r0 + ROWS - 1, all in block I
    const int I = warp >> 1;
    const int cb = lane * CPL;
    constexpr bool kStage = sizeof(IO) == 2;  // bf16 rows are staged into their swizzled tiles
    constexpr bool kTma = kStage && D >= 64;  // ... by tensor copies (128-byte swizzle = the tile layout)
    auto wait_loads = [&](uint32_t parity) {
        if (!gave_up && !mbar_wait(&ld_bar, parity, kPrepWaitLimit)) {
            gave_up = true;
            if (lane == 0) atomicExch(p.status, 3);
        }
    };
    Slice<IO, CPL> rq[kStage ? 1 : PRE], rk[kStage ? 1 : PRE];
    auto load_rows = [&](int j0) {
#pragma unroll
        for (int j = 0; j < PRE; ++j) {
            const int i = r0 + j0 + j;
            if (i < len) {
                const int64_t off = ((t0 + i) * H + h) * D + cb;
                rq[j].load(qg + off);
                rk[j].load(kg + off);
            } else {
                rq[j].zero();
                rk[j].zero();
            }
        }
    };
    if constexpr (kTma) {  // q -> QP, k -> KP: one tensor copy per 64-channel slab (rows past the
                           // sequence hold the next one's tokens or zeros; beta = 0 there cancels them)
        if (tid == 0) {
            mbar_arrive_expect_tx(&ld_bar, 2 * SM::TILE);
#pragma unroll
            for (int sl = 0; sl < D / 64; ++sl) {
                tma_load_3d(smem + SM::QP + sl * C * 128, &maps.q, 64 * sl, h, static_cast<int>(t0), &ld_bar);
                tma_load_3d(smem + SM::KP + sl * C * 128, &maps.k, 64 * sl, h, static_cast<int>(t0), &ld_bar);
            }
        }
    } else if constexpr (kStage) {  // q -> QP, k -> KP tiles, 16-byte chunks, zeros past the end
        constexpr int CH = D / 8;    // 16-byte chunks per row
#pragma unroll
        for (int e = tid; e < C * CH; e += kThreads) {
            const int i = e / CH, ch = e % CH;
            const int ii = i < len ? i : 0;
            const int64_t off = ((t0 + ii) * H + h) * D + 8 * ch;
            const uint32_t so = tile_off<D, C>(i, 8 * ch);
            const uint32_t nb = i < len ? 16u : 0u;
            cp_async16(smem_u32(smem + SM::QP + so), qg + off, nb);
            cp_async16(smem_u32(smem + SM::KP + so), kg + off, nb);
        }
    } else {
        load_rows(0);
    }
    float gr[ROWS][CPL];  // g of the warp's rows, then G (log2 units)
#pragma unroll
    for (int j = 0; j < ROWS; ++j) {
        if (r0 + j < len) {
            ldg_f32<CPL>(p.g + ((t0 + r0 + j) * H + h) * D + cb, gr[j]);
        } else {
#pragma unroll
            for (int c = 0; c < CPL; ++c) gr[j][c] = 0.f;
        }
    }
    if (tid < C) sBeta[tid] = tid < len ? p.beta[(t0 + tid) * H + h] : 0.f;
    if (tid < len) prefetch_l2(vg + ((t0 + tid) * H + h) * D, D * sizeof(IO));  // v is staged after the Gram

    // in-chunk cumulative sum of g per channel, in log2 units: inside the warp's
    // rows in registers, then across warps through their totals
#pragma unroll
    for (int j = 0; j < ROWS; ++j) {
        if constexpr (CPL % 2 == 0) {
#pragma unroll
            for (int c = 0; c < CPL; c += 2) {
                const float2 x = make_float2(gr[j][c], gr[j][c + 1]), l2 = make_float2(kLog2e, kLog2e);
                const float2 y = j == 0 ? mul2(x, l2) : fma2(x, l2, make_float2(gr[j - 1][c], gr[j - 1][c + 1]));
                gr[j][c] = y.x;
                gr[j][c + 1] = y.y;
            }
        } else {
#pragma unroll
            for (int c = 0; c < CPL; ++c) gr[j][c] = j == 0 ? gr[0][c] * kLog2e : fmaf(gr[j][c], kLog2e, gr[j - 1][c]);
        }
    }
    st_f32<CPL>(sSum + warp * D + cb, gr[ROWS - 1]);
    if (warp & 1) st_f32<CPL>(sSum + (kWarps + I) * D + cb, gr[0]);  // row 16 I + 8: the block midpoint
    // Range of the block split: |G_i - G_mI| (log2 units) of this warp's rows from its local
    // sums (an odd warp starts at its block's midpoint m; an even warp ends one row before it
    // and adds g at m).  A chunk where some channel exceeds kSpanLimit goes to the fix-up list,
    // whose kernel forms the whole record again with the exact Gram; this CTA carries on, and
    // what it writes is overwritten.  The list holds the item, chunk * H + h.
    bool wide = false;
    if constexpr (!kExact) {
        float gmid[CPL];
        if (warp & 1) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) gmid[c] = gr[0][c];
        } else {
            float g8[CPL] = {};
            if (r0 + ROWS < len) ldg_f32<CPL>(p.g + ((t0 + r0 + ROWS) * H + h) * D + cb, g8);
#pragma unroll
            for (int c = 0; c < CPL; ++c) gmid[c] = fmaf(g8[c], kLog2e, gr[ROWS - 1][c]);
        }
#pragma unroll
        for (int j = 0; j < ROWS; ++j)
#pragma unroll
            for (int c = 0; c < CPL; ++c) wide |= fabsf(gr[j][c] - gmid[c]) > kSpanLimit;
    }
    cp_async_wait_all();
    if (__syncthreads_or(wide) && tid == 0) p.fix_list[atomicAdd(p.fix_count, 1)] = static_cast<int32_t>(chunk * p.H + h);
    if constexpr (kTma) wait_loads(0);  // q and k are in their tiles
    float gm[4][CPL], glast[CPL], off[CPL];
    {
        float run[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) run[c] = off[c] = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            float t[CPL];
            load_f32<CPL>(sSum + w * D + cb, t);
            if (w == warp) {
#pragma unroll
                for (int c = 0; c < CPL; ++c) off[c] = run[c];
            }
            if (w & 1) {
                float f[CPL];
                load_f32<CPL>(sSum + (kWarps + (w >> 1)) * D + cb, f);
#pragma unroll
                for (int c = 0; c < CPL; ++c) gm[w >> 1][c] = run[c] + f[c];
            }
#pragma unroll
            for (int c = 0; c < CPL; ++c) run[c] += t[c];
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c) glast[c] = run[c];
    }
#pragma unroll
    for (int j = 0; j < ROWS; ++j) {
        if constexpr (CPL % 2 == 0) {
#pragma unroll
            for (int c = 0; c < CPL; c += 2) {
                const float2 x = add2(make_float2(gr[j][c], gr[j][c + 1]), make_float2(off[c], off[c + 1]));
                gr[j][c] = x.x;
                gr[j][c + 1] = x.y;
            }
        } else {
#pragma unroll
            for (int c = 0; c < CPL; ++c) gr[j][c] += off[c];
        }
    }

    // per-channel factors: F_IJ (warps 0-5, one (I, J) each), L_I = e^{G_mI}
    // (even warps), gamma = e^{G_last} (warp 7, to the record)
    float gmi[CPL], lI[CPL], ls[CPL], zz[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        gmi[c] = pick4(gm[0][c], gm[1][c], gm[2][c], gm[3][c], I);
        lI[c] = ex2_approx(gmi[c]);             // e^{G_mI}          <= 1
        ls[c] = lI[c] * p.scale;
        zz[c] = ex2_approx(glast[c] - gmi[c]);  // e^{G_last - G_mI}  <= 1
    }
    if (!(warp & 1)) st_f32<CPL>(sL + I * D + cb, lI);
    if (warp < 6) {
        const int fI = warp < 1 ? 1 : warp < 3 ? 2 : 3, fJ = warp - fI * (fI - 1) / 2;
        float f[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c)
            f[c] = ex2_approx(pick4(gm[0][c], gm[1][c], gm[2][c], gm[3][c], fI) -
                              pick4(gm[0][c], gm[1][c], gm[2][c], gm[3][c], fJ));
        store_bf16<CPL>(reinterpret_cast<char *>(sFb + warp * D), static_cast<uint32_t>(cb * 2), f);
    } else if (warp == 7) {
        float gam[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) gam[c] = ex2_approx(glast[c]);
        st_f32<CPL>(reinterpret_cast<float *>(rec + R::GAMMA) + cb, gam);
    }

    // ---- 2. row pass: normalise q, k; operand tiles in shared memory; Q~, K~ to the record ----
    // norms of the warp's 8 rows: 16 partial sums per lane reduced by a transposed butterfly
    // (lane L ends with the total of value L >> 1), one rsqrt per lane, then broadcast
    float nqs[ROWS], nks[ROWS];
    if constexpr (kStage) {
        float vsum[2 * ROWS];
#pragma unroll
        for (int j = 0; j < ROWS; ++j) {
            const uint32_t o = tile_off<D, C>(r0 + j, cb);
            float qv[CPL], kv[CPL];
            load_slice<__nv_bfloat16, CPL>(reinterpret_cast<const __nv_bfloat16 *>(smem + SM::QP + o), qv);
            load_slice<__nv_bfloat16, CPL>(reinterpret_cast<const __nv_bfloat16 *>(smem + SM::KP + o), kv);
            if constexpr (CPL % 2 == 0) {
                float2 sq = make_float2(0.f, 0.f), sk = make_float2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < CPL; c += 2) {
                    const float2 q2 = make_float2(qv[c], qv[c + 1]), k2 = make_float2(kv[c], kv[c + 1]);
                    sq = fma2(q2, q2, sq);
                    sk = fma2(k2, k2, sk);
                }
                vsum[2 * j] = sq.x + sq.y;
                vsum[2 * j + 1] = sk.x + sk.y;
            } else {
                float sq = 0.f, sk = 0.f;
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    sq += qv[c] * qv[c];
                    sk += kv[c] * kv[c];
                }
                vsum[2 * j] = sq;
                vsum[2 * j + 1] = sk;
            }
        }
#pragma unroll
        for (int mask = 16, half = ROWS; mask >= 2; mask >>= 1, half >>= 1) {
            const bool up = (lane & mask) != 0;
#pragma unroll
            for (int i = 0; i < half; ++i) {
                const float send = up ? vsum[i] : vsum[i + half];
                const float keep = up ? vsum[i + half] : vsum[i];
                vsum[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
            }
        }
        const float tot = vsum[0] + __shfl_xor_sync(0xffffffffu, vsum[0], 1);
        const float rn = p.l2norm ? rsqrtf(tot + 1e-6f) : 1.f;
#pragma unroll
        for (int j = 0; j < ROWS; ++j) {
            nqs[j] = __shfl_sync(0xffffffffu, rn, 4 * j);
            nks[j] = __shfl_sync(0xffffffffu, rn, 4 * j + 2);
        }
    }
#pragma unroll
    for (int j0 = 0; j0 < ROWS; j0 += PRE) {
        if (!kStage && j0 > 0) load_rows(j0);
#pragma unroll
        for (int j = 0; j < PRE; ++j) {
            const int i = r0 + j0 + j;
            const uint32_t o = tile_off<D, C>(i, cb);
            float qv[CPL], kv[CPL];
            if constexpr (kStage) {
                load_slice<__nv_bfloat16, CPL>(reinterpret_cast<const __nv_bfloat16 *>(smem + SM::QP + o), qv);
                load_slice<__nv_bfloat16, CPL>(reinterpret_cast<const __nv_bfloat16 *>(smem + SM::KP + o), kv);
            } else {
                rq[j].get(qv);
                rk[j].get(kv);
            }
            float nq, nk;
            if constexpr (kStage) {
                nq = nqs[j0 + j];
                nk = nks[j0 + j];
            } else {
                float sq = 0.f, sk = 0.f;
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    sq += qv[c] * qv[c];
                    sk += kv[c] * kv[c];
                }
#pragma unroll
                for (int o2 = 16; o2 > 0; o2 >>= 1) {
                    sq += __shfl_xor_sync(0xffffffffu, sq, o2);
                    sk += __shfl_xor_sync(0xffffffffu, sk, o2);
                }
                nq = p.l2norm ? rsqrtf(sq + 1e-6f) : 1.f;
                nk = p.l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
            }
            float kp[CPL], qp[CPL], kr[CPL], qt[CPL], kt[CPL];
            if constexpr (CPL % 2 == 0) {  // channel pairs through the packed fp32x2 instructions
#pragma unroll
                for (int c = 0; c < CPL; c += 2) {
                    const float d0 = gr[j0 + j][c] - gmi[c], d1 = gr[j0 + j][c + 1] - gmi[c + 1];
                    const float2 P = make_float2(ex2_approx(d0), ex2_approx(d1));     // e^{G_i - G_m}
                    const float2 Rr = make_float2(ex2_approx(-d0), ex2_approx(-d1));  // e^{G_m - G_i}
                    const float2 qh = mul2(make_float2(qv[c], qv[c + 1]), make_float2(nq, nq));
                    const float2 kh = mul2(make_float2(kv[c], kv[c + 1]), make_float2(nk, nk));
                    const float2 kp2 = mul2(kh, P), qp2 = mul2(qh, P), kr2 = mul2(kh, Rr);
                    const float2 qt2 = mul2(qp2, make_float2(ls[c], ls[c + 1]));
                    const float2 kt2 = mul2(kr2, make_float2(zz[c], zz[c + 1]));
                    kp[c] = kp2.x; kp[c + 1] = kp2.y;
                    qp[c] = qp2.x; qp[c + 1] = qp2.y;
                    kr[c] = kr2.x; kr[c + 1] = kr2.y;
                    qt[c] = qt2.x; qt[c + 1] = qt2.y;
                    kt[c] = kt2.x; kt[c + 1] = kt2.y;
                }
            } else {
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    const float gi = gr[j0 + j][c];
                    const float P = ex2_approx(gi - gmi[c]);   // e^{G_i - G_m}
                    const float Rr = ex2_approx(gmi[c] - gi);  // e^{G_m - G_i}
                    const float qh = qv[c] * nq, kh = kv[c] * nk;
                    kp[c] = kh * P;
                    qp[c] = qh * P;
                    kr[c] = kh * Rr;
                    qt[c] = qp[c] * ls[c];
                    kt[c] = kr[c] * zz[c];
                }
            }
            store_bf16<CPL>(smem + SM::KP, o, kp);  // each lane rewrites exactly the bytes it read
            store_bf16<CPL>(smem + SM::QP, o, qp);
            store_bf16<CPL>(smem + SM::KR, o, kr);
            store_bf16<CPL>(rec, R::qt_at(i, cb), qt);
            store_bf16<CPL>(rec + R::KT, o, kt);
        }
    }
    __syncthreads();
    if constexpr (kExact) {
        exact_gram<D, IO>(qg, kg, p.g, p.H, p.scale, p.l2norm, smem, rec, t0, len, h);
    } else {
        // A_qk blocks above the diagonal are zero (the record is used as a full 64 x 64 operand)
        for (int e = tid; e < 6 * 16 * 2; e += kThreads) {
            const int b = e >> 5, r = (e >> 1) & 15, ch = e & 1;
            const int I = b < 3 ? 0 : b < 5 ? 1 : 2;        // upper blocks (I, J), J > I
            const int J = b < 3 ? b + 1 : b < 5 ? b - 1 : 3;
            *reinterpret_cast<uint4 *>(rec + R::AQK + swz_off<128>(16 * I + r, 16 * J + 8 * ch)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        // ---- 3. gated Gram products, 20 (matrix, I, J) block pairs over 8 warps ----
        // A_kk (x beta_i, strictly lower) -> bf16 tile for the substitution products, and its
        // diagonal blocks in fp32 for their inverses; A_qk (x scale, causal) -> the record.
        float *sAd = reinterpret_cast<float *>(smem + SM::AD);  // [4][16][17] fp32
        {
            // Pairs by slot: u = 0 an off-diagonal pair (warp w: the w-th of 12), u = 1 a diagonal
            // pair (the w-th of 8), u = 2 (warps 0-3) the off-diagonal pair 8 + w.  Off-diagonal
            // pairs scale by F_IJ; diagonal ones need no factor.  The first six of each kind are A_kk.
            constexpr int MAXP = 3;
            const int npairs = warp < 4 ? 3 : 2;
            int pI[MAXP], pJ[MAXP];
            bool pqk[MAXP];
#pragma unroll
            for (int u = 0; u < MAXP; ++u) {
                if (u == 1) {  // diagonal: index w in 0..7
                    pqk[u] = warp >= 4;
                    pI[u] = pJ[u] = warp & 3;
                } else {       // off-diagonal: index w or 8 + w in 0..11
                    const int o = u == 0 ? warp : 8 + warp;
                    const int sl = o % 6;  // F slot (I, J), J < I
                    pqk[u] = o >= 6;
                    pI[u] = sl < 1 ? 1 : sl < 3 ? 2 : 3;
                    pJ[u] = sl - pI[u] * (pI[u] - 1) / 2;
                }
            }
            float acc[MAXP][2][4] = {};
            // One k-step of pair u; off-diagonal pairs: a <- a * F_IJ on the fragment's four
            // channels (bf16x2 products).
            auto step = [&](int u, int ks, auto scaled) {
                const int I = pI[u], J = pJ[u];
                uint32_t a[4], b[4];
                ldmatrix_x4(a, smem_u32(smem + (pqk[u] ? SM::QP : SM::KP) +
                                        tile_off<D, C>(16 * I + ri + 8 * (mi & 1), 16 * ks + 8 * (mi >> 1))));
                if constexpr (decltype(scaled)::value) {
                    const uint16_t *f = sFb + fslot(I, J) * D + 16 * ks + 2 * tig;
                    const uint32_t f01 = *reinterpret_cast<const uint32_t *>(f);
                    const uint32_t f23 = *reinterpret_cast<const uint32_t *>(f + 8);
                    a[0] = mul_bf16x2(a[0], f01);
                    a[1] = mul_bf16x2(a[1], f01);
                    a[2] = mul_bf16x2(a[2], f23);
                    a[3] = mul_bf16x2(a[3], f23);
                }
                ldmatrix_x4(b, smem_u32(smem + SM::KR +
                                        tile_off<D, C>(16 * J + ri + 8 * (mi >> 1), 16 * ks + 8 * (mi & 1))));
                mma_bf16(acc[u][0], a, b[0], b[1]);
                mma_bf16(acc[u][1], a, b[2], b[3]);
            };
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {  // every warp: an off-diagonal and a diagonal pair
                step(0, ks, std::true_type{});
                step(1, ks, std::false_type{});
            }
            if (npairs > 2) {  // warps 0-3: one more off-diagonal pair
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) step(2, ks, std::true_type{});
            }
            // Epilogue of pair u (one branch per pair on its kind, none per element).
            auto epilogue = [&](int u) {
                const int I = pI[u], J = pJ[u];
                if (!pqk[u]) {  // beta_i A_kk, strictly lower -> bf16 tile (+ fp32 copy of a diagonal block)
                    float *d = I == J ? sAd + I * 16 * 17 : nullptr;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            const int i = 16 * I + gid + 8 * hr, j = 16 * J + 8 * nt + 2 * tig;
                            const float bi = sBeta[i];
                            const float y0 = j < i ? acc[u][nt][2 * hr] * bi : 0.f;
                            const float y1 = j + 1 < i ? acc[u][nt][2 * hr + 1] * bi : 0.f;
                            if (I != J)
                                *reinterpret_cast<uint32_t *>(smem + SM::AB + blk_off(fslot(I, J), i - 16 * I, j - 16 * J)) =
                                    pack_bf16x2(y0, y1);
                            if (d) {  // rows of 17 floats: scalar stores (odd rows are not 8-byte aligned)
                                d[(i - 16 * I) * 17 + (j - 16 * J)] = y0;
                                d[(i - 16 * I) * 17 + (j - 16 * J) + 1] = y1;
                            }
                        }
                    }
                } else {  // scale A_qk, causal -> the record
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            const int i = 16 * I + gid + 8 * hr, j = 16 * J + 8 * nt + 2 * tig;
                            const float y0 = j <= i ? acc[u][nt][2 * hr] * p.scale : 0.f;
                            const float y1 = j + 1 <= i ? acc[u][nt][2 * hr + 1] * p.scale : 0.f;
                            *reinterpret_cast<uint32_t *>(rec + R::AQK + swz_off<128>(i, j)) = pack_bf16x2(y0, y1);
                        }
                    }
                }
            };
            epilogue(0);
            epilogue(1);
            if (npairs > 2) epilogue(2);
        }
    }  // block split
    __syncthreads();

    // v -> the k R tile (free after the Gram products), bf16, zeros past the end; its
    // latency overlaps the diagonal inverses (the rows were prefetched into L2)
    if constexpr (kTma) {
        if (tid == 0) {
            fence_proxy_async_smem();  // the Gram's reads of k R precede the tensor copies into it
            mbar_arrive_expect_tx(&ld_bar, SM::TILE);
#pragma unroll
            for (int sl = 0; sl < D / 64; ++sl)
                tma_load_3d(smem + SM::KR + sl * C * 128, &maps.v, 64 * sl, h, static_cast<int>(t0), &ld_bar);
        }
    } else if constexpr (kStage) {
        constexpr int CH = D / 8;
#pragma unroll
        for (int e = tid; e < C * CH; e += kThreads) {
            const int i = e / CH, ch = e % CH;
            const int ii = i < len ? i : 0;
            cp_async16(smem_u32(smem + SM::KR + tile_off<D, C>(i, 8 * ch)), vg + ((t0 + ii) * H + h) * D + 8 * ch,
                       i < len ? 16u : 0u);
        }
    } else {
#pragma unroll
        for (int e = tid; e < C * (D / 4); e += kThreads) {
            const int i = e / (D / 4), c4 = 4 * (e % (D / 4));
            float x[4] = {0.f, 0.f, 0.f, 0.f};
            if (i < len) load_slice<IO, 4>(vg + ((t0 + i) * H + h) * D + c4, x);
            store_bf16<4>(smem + SM::KR, tile_off<D, C>(i, c4), x);
        }
    }
    // ---- 4. inverses of the diagonal blocks, T_II = (I + A_II)^-1, fp32 forward substitution;
    //         stored as they are (TD) and with their columns scaled by beta (TS) ----
    if (warp < 4 && lane < 16) {  // one column per lane
        const int I = warp, j = lane;
        const float *A = reinterpret_cast<const float *>(smem + SM::AD) + I * 16 * 17;
        // Right-looking: once tcol[k] is final it is subtracted from every later row, so
        // row i still accumulates its terms in the order k = 0, 1, .., i - 1 but the
        // dependent chain is one step per row instead of one per term.
        float tcol[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) tcol[i] = i == j ? 1.f : 0.f;
#pragma unroll
        for (int kk = 0; kk < 15; ++kk)
#pragma unroll
            for (int i = kk + 1; i < 16; ++i) tcol[i] -= A[i * 17 + kk] * tcol[kk];
        const float bj = sBeta[16 * I + j];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            *reinterpret_cast<uint16_t *>(smem + SM::TD + blk_off(I, i, j)) = f32_to_bf16_bits(tcol[i]);
            *reinterpret_cast<uint16_t *>(smem + SM::TS + blk_off(I, i, j)) = f32_to_bf16_bits(tcol[i] * bj);
        }
    }
    __syncthreads();

    // ---- 5. the off-diagonal blocks of T' = (I + A_kk)^-1 diag(beta):
    //         T'_IJ = -T_II sum_{J<=K<I} A_IK T'_KJ.  Warp 0 forms (1,0), (2,0), (3,0), warp 1
    //         (2,1), (3,1), warp 2 (3,2): each block needs only the diagonal blocks and the
    //         warp's own earlier results. ----
    if (warp < 3) {
        char *scr = smem + SM::SCR + warp * 512;
        auto tblock = [&](int I, int J) {
            float x[2][4] = {};
            for (int K = J; K < I; ++K) {
                uint32_t a[4], b[4];
                ldmatrix_x4(a, smem_u32(smem + SM::AB + blk_off(fslot(I, K), ri + 8 * (mi & 1), 8 * (mi >> 1))));
                const int tb = K == J ? SM::TS + J * 512 : SM::TO + fslot(K, J) * 512;
                ldmatrix_x4_trans(b, smem_u32(smem + tb + blk_off(0, ri + 8 * (mi & 1), 8 * (mi >> 1))));
                mma_bf16(x[0], a, b[0], b[1]);
                mma_bf16(x[1], a, b[2], b[3]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
                    *reinterpret_cast<uint32_t *>(scr + blk_off(0, gid + 8 * hr, 8 * nt + 2 * tig)) =
                        pack_bf16x2(x[nt][2 * hr], x[nt][2 * hr + 1]);
            __syncwarp();
            float y[2][4] = {};
            uint32_t a[4], b[4];
            ldmatrix_x4(a, smem_u32(smem + SM::TD + blk_off(I, ri + 8 * (mi & 1), 8 * (mi >> 1))));
            ldmatrix_x4_trans(b, smem_u32(scr + blk_off(0, ri + 8 * (mi & 1), 8 * (mi >> 1))));
            mma_bf16(y[0], a, b[0], b[1]);
            mma_bf16(y[1], a, b[2], b[3]);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
                    *reinterpret_cast<uint32_t *>(smem + SM::TO + blk_off(fslot(I, J), gid + 8 * hr, 8 * nt + 2 * tig)) =
                        pack_bf16x2(-y[nt][2 * hr], -y[nt][2 * hr + 1]);
            __syncwarp();  // the block is read by this warp's next block; scr is rewritten
        };
        if (warp == 0) {
            tblock(1, 0);
            tblock(2, 0);
            tblock(3, 0);
        } else if (warp == 1) {
            tblock(2, 1);
            tblock(3, 1);
        } else {
            tblock(3, 2);
        }
    }
    cp_async_wait_all();  // v has landed (each thread its own copies; the barrier publishes them)
    __syncthreads();
    if constexpr (kTma) wait_loads(1);  // ... or its tensor copies have completed

    // ---- 6. W = T' (K e^G) and U = T' V, block row I from blocks K <= I: warps 0-3 W,
    //         warps 4-7 U, each warp D / NW columns.  The right-hand sides are read into
    //         registers once (k P tile with e^G = P L_K applied to the fragments, or v);
    //         W_I overwrites its rows of the k P tile in place, U^T goes to the q P tile
    //         in the record's layout. ----
    {
        constexpr int NW = D / 16 < 4 ? D / 16 : 4;  // warps per matrix with work
        constexpr int COLS = D / NW, NP = COLS / 16;
        const int q4 = warp & 3;
        const int c0 = q4 * COLS;
        auto product_w = [&]() {
            char *ytile = smem + SM::KP;  // right-hand sides in, W rows out
            uint32_t b[4][NP][4];
#pragma unroll
            for (int K = 0; K < 4; ++K)
#pragma unroll
                for (int np = 0; np < NP; ++np) {
                    ldmatrix_x4_trans(b[K][np], smem_u32(ytile + tile_off<D, C>(16 * K + ri + 8 * (mi & 1),
                                                                              c0 + 16 * np + 8 * (mi >> 1))));
                    // row k of block K times L_K = e^{G_mK}, column gid of each n8 tile
                    const float l0 = sL[K * D + c0 + 16 * np + gid], l1 = sL[K * D + c0 + 16 * np + 8 + gid];
                    const uint32_t f0 = pack_bf16x2(l0, l0), f1 = pack_bf16x2(l1, l1);
                    b[K][np][0] = mul_bf16x2(b[K][np][0], f0);
                    b[K][np][1] = mul_bf16x2(b[K][np][1], f0);
                    b[K][np][2] = mul_bf16x2(b[K][np][2], f1);
                    b[K][np][3] = mul_bf16x2(b[K][np][3], f1);
                }
            __syncwarp();  // every lane holds its fragments before Y overwrites the tile
#pragma unroll
            for (int I = 0; I < 4; ++I) {
                float acc[2 * NP][4] = {};
#pragma unroll
                for (int K = 0; K <= I; ++K) {
                    uint32_t a[4];
                    const int tb = K == I ? SM::TS + I * 512 : SM::TO + fslot(I, K) * 512;
                    ldmatrix_x4(a, smem_u32(smem + tb + blk_off(0, ri + 8 * (mi & 1), 8 * (mi >> 1))));
#pragma unroll
                    for (int np = 0; np < NP; ++np) {
                        mma_bf16(acc[2 * np], a, b[K][np][0], b[K][np][1]);
                        mma_bf16(acc[2 * np + 1], a, b[K][np][2], b[K][np][3]);
                    }
                }
#pragma unroll
                for (int n = 0; n < 2 * NP; ++n) {
                    const uint32_t co = tile_off<D, C>(gid, c0 + 8 * n + 2 * tig) - gid * ROWB;
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int i = 16 * I + gid + 8 * hr;
                        const float y0 = acc[n][2 * hr], y1 = acc[n][2 * hr + 1];
                        *reinterpret_cast<uint32_t *>(ytile + static_cast<uint32_t>(i) * ROWB + co) = pack_bf16x2(y0, y1);
                    }
                }
            }
        };
        // U^T = V^T T'^T formed directly (A: V_K^T by transposed loads of the v tile, B: T'_IK^T
        // by plain loads of the T' blocks): its accumulators are U^T rows, stored as bf16 pairs in
        // the record's layout; the U rows themselves are never needed.
        auto product_ut = [&]() {
            const char *vtile = smem + SM::KR;
            char *utile = smem + SM::QP;  // U^T [D][64] bf16, 128-byte swizzled rows
            uint32_t a[4][NP][4];
#pragma unroll
            for (int K = 0; K < 4; ++K)
#pragma unroll
                for (int np = 0; np < NP; ++np)
                    ldmatrix_x4_trans(a[K][np], smem_u32(vtile + tile_off<D, C>(16 * K + ri + 8 * (mi >> 1),
                                                                               c0 + 16 * np + 8 * (mi & 1))));
#pragma unroll
            for (int I = 0; I < 4; ++I) {
                float acc[NP][2][4] = {};
#pragma unroll
                for (int K = 0; K <= I; ++K) {
                    uint32_t bt[4];
                    const int tb = K == I ? SM::TS + I * 512 : SM::TO + fslot(I, K) * 512;
                    ldmatrix_x4(bt, smem_u32(smem + tb + blk_off(0, ri + 8 * (mi >> 1), 8 * (mi & 1))));
#pragma unroll
                    for (int np = 0; np < NP; ++np) {
                        mma_bf16(acc[np][0], a[K][np], bt[0], bt[1]);
                        mma_bf16(acc[np][1], a[K][np], bt[2], bt[3]);
                    }
                }
#pragma unroll
                for (int np = 0; np < NP; ++np)
#pragma unroll
                    for (int hn = 0; hn < 2; ++hn)
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            const int c = c0 + 16 * np + gid + 8 * hr;  // value row of U^T
                            const int t = 16 * I + 8 * hn + 2 * tig;    // token column pair
                            *reinterpret_cast<uint32_t *>(utile + swz_off<128>(c, t)) =
                                pack_bf16x2(acc[np][hn][2 * hr], acc[np][hn][2 * hr + 1]);
                        }
            }
        };
        if (q4 < NW) {
            if (warp >= 4) product_ut();
            else product_w();
        }
    }
    fence_proxy_async_smem();  // the W and U^T tiles are read by the bulk copies below
    __syncthreads();

    // ---- 6. W and U^T out to the record (Q~, K~, A_qk and gamma are already there) ----
    if (tid == 0) {
        constexpr int kSlabs = D >= 128 ? D / 64 : 1;  // W's 64-column slabs: rows 0..63 of [W; Q~]
#pragma unroll
        for (int s = 0; s < kSlabs; ++s)
            bulk_s2g(rec + R::w_at(0, 64 * s), smem + SM::KP + s * (R::TILE / kSlabs), R::TILE / kSlabs);
        bulk_s2g(rec + R::UT, smem + SM::QP, D * C * 2);
        bulk_commit();
        bulk_wait_all_read();  // shared memory stays valid until the copies have read it
    }
}

template <int D, typename IO> __device__ __forceinline__ void init_load_barrier(uint64_t &ld_bar)
{
    if constexpr (sizeof(IO) == 2 && D >= 64) {
        if (threadIdx.x == 0) {
            mbar_init(&ld_bar, 1);
            fence_mbar_init();
        }
    }
}

// One CTA per (chunk, head), heads fastest in the grid: the heads of one chunk run together.
template <int D, typename IO>
__global__ void __launch_bounds__(kThreads, sizeof(IO) == 2 ? 3 : 2)  // bf16: 3 CTAs per SM (≈69 KB smem each)
chunk_prep_kernel(PrepParams p, const __grid_constant__ PrepMaps maps)
{
    extern __shared__ __align__(1024) char smem[];
    __shared__ __align__(8) uint64_t ld_bar;
    bool gave_up = false;
    init_load_barrier<D, IO>(ld_bar);
    prep_chunk<D, IO, false>(p, maps, p.chunk_base + blockIdx.x / p.H, static_cast<int>(blockIdx.x % p.H), smem, ld_bar,
                             gave_up);
}

// The (chunk, head) items the block split left in the fix-up list, with the exact Gram;
// persistent CTAs stride over the list (most calls find it empty and return at once).
template <int D, typename IO>
__global__ void __launch_bounds__(kThreads, 1)
chunk_prep_exact_kernel(PrepParams p, const __grid_constant__ PrepMaps maps)
{
    extern __shared__ __align__(1024) char smem[];
    __shared__ __align__(8) uint64_t ld_bar;
    const int32_t n = *p.fix_count;
    if (static_cast<int32_t>(blockIdx.x) >= n) return;
    bool gave_up = false;
    init_load_barrier<D, IO>(ld_bar);
    for (int32_t i = blockIdx.x; i < n; i += gridDim.x) {
        const int32_t item = p.fix_list[i];
        prep_chunk<D, IO, true>(p, maps, item / p.H, item % p.H, smem, ld_bar, gave_up);
        __syncthreads();  // shared memory and the barrier are reused by the next item
    }
}

template <int D, typename IO>
cudaError_t launch_typed(const PrepParams &p, int64_t n_chunk_max, int32_t h, cudaStream_t st)
{
    if (p.total_tokens < 1) return cudaSuccess;  // no chunk has rows: every CTA would exit at once
    if (n_chunk_max * h > 0x7fffffffLL) return cudaErrorInvalidConfiguration;  // one-dimensional grid
    auto kern = chunk_prep_kernel<D, IO>;
    constexpr int smem = PrepSmem<D>::BYTES;
    PrepMaps maps{};
    if constexpr (sizeof(IO) == 2 && D >= 64) {
        if (!encode_rows(&maps.q, p.q, p.total_tokens, h, D) || !encode_rows(&maps.k, p.k, p.total_tokens, h, D) ||
            !encode_rows(&maps.v, p.v, p.total_tokens, h, D))
            return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(n_chunk_max * h), kThreads, smem, st>>>(p, maps);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    auto fix = chunk_prep_exact_kernel<D, IO>;
    if ((e = cudaFuncSetAttribute(fix, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
    const int64_t items = n_chunk_max * h, grid = items < 2 * sm_count() ? items : 2 * sm_count();
    fix<<<static_cast<unsigned>(grid), kThreads, smem, st>>>(p, maps);
    return cudaGetLastError();
}

}  // namespace

// cuTensorMapEncodeTiled from the driver, resolved once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// Map of a bf16 [T][H][D] input: dims (D, H, T), boxes of 64 channels x 1 head x 64
// tokens, 128-byte swizzle (the tiles' layout), zeros outside the tensor.
bool encode_rows(CUtensorMap *m, const void *base, int64_t T, int32_t H, int D)
{
    const PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
    if (fn == nullptr || T < 1) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
    const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(C)};
    const cuuint32_t elem[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_rows_f32(CUtensorMap *m, const float *base, int64_t T, int32_t H, int D)
{
    const PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
    if (fn == nullptr || T < 1) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4, static_cast<cuuint64_t>(H) * D * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(D), 1, static_cast<cuuint32_t>(C)};
    const cuuint32_t elem[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_chunk_prep(int d, int32_t io_dtype, const PrepParams &p, int64_t n_chunk_max, int32_t h,
                              cudaStream_t st)
{
    const bool bf = io_dtype == KDA_BF16;
    switch (d) {
    case 32:
        return bf ? launch_typed<32, __nv_bfloat16>(p, n_chunk_max, h, st) : launch_typed<32, float>(p, n_chunk_max, h, st);
    case 64:
        return bf ? launch_typed<64, __nv_bfloat16>(p, n_chunk_max, h, st) : launch_typed<64, float>(p, n_chunk_max, h, st);
    default:
        return bf ? launch_typed<128, __nv_bfloat16>(p, n_chunk_max, h, st)
                  : launch_typed<128, float>(p, n_chunk_max, h, st);
    }
}

}  // namespace prefill
}  // namespace kda
