// Fused chunked prefill for head size 128 with bf16 inputs and outputs: one
// persistent CTA per SM takes (sequence, head) items, longest sequences first,
// and runs the chunk preparation of chunk i + 1 in eight warps while eight
// other warps run the inter-chunk state pass of chunk i.  The per-chunk
// quantities never leave the SM: they pass from one half of the CTA to the
// other through a two-stage ring in shared memory (and, for U^T, in tensor
// memory).
//
// The method is the chunkwise form of the gated delta rule, S_t = (I - beta_t
// k_t k_t^T) Diag(e^{g_t}) S_{t-1} + beta_t k_t v_t^T, o_t = scale S_t^T q_t
// ("KDA's challenges for AI infra", section 1.1), chunk by chunk in the order
// of the "Support Kimi-K3 on NPU" report's extend listing: l2norm, in-chunk
// gate cumsum, gated K K^T / Q K^T, (I + A)^-1, W and U, the state pass and
// the outputs.  Here the per-channel exponentials are taken through one
// reference per chunk and channel, G_r = (max_i G_i + min_i G_i) / 2 (log2
// units), so every factor lies within 2^60 of 1 when the chunk's span of G is
// at most 120:
//   Qp = scale q^ 2^{G - G_r},  Kp = k^ 2^{G - G_r},  Kr = k^ 2^{G_r - G},
//   A_qk = Qp Kr^T (causal),  A_kk = Kp Kr^T (strictly lower) x beta_i,
//   T' = (I + A_kk)^-1 diag(beta),  W' = T' Kp,  U = T' V.
// With the state kept as S^ = S 2^{-(G_last - G_r)} of the chunk that produced
// it, the state pass needs no Q~, K~ or W tiles of its own:
//   S_r = S^ m  (m = 2^{G_last - G_r} of the previous chunk x 2^{G_r})
//   X = W' S_r,  V_new = U - X,  O = Qp S_r + A_qk V_new,  S^ <- S_r + Kr^T V_new
// because W S = T' Kp diag(2^{G_r}) S, scale q^ 2^G S = Qp diag(2^{G_r}) S and
// S_new 2^{-(G_last - G_r)} = diag(2^{G_r}) S + Kr^T V_new.  A chunk whose span is
// wider takes the exact path: every e^{G_i - G_j} of its gated Gram is the
// exponential of its own difference, and it supplies the plain operands
// (Qp = Q~, Kp = k^ e^G, Kr = K~) with m_op = 2^{G_last - G_r} of the previous
// chunk, m_st = that x 2^{G_last}, and 2^{-(G_last - G_r)} = 1.
//
// Warps 0-7 (the pass) own the state: S^ (fp32) in tensor memory, the bf16
// operand S_r in shared memory; one thread issues their tcgen05 MMAs.  Warps
// 8-15 (the preparation) own the gated Gram (tcgen05, M = 128 = [Qp; Kp],
// N = 64), the blockwise triangular solve (fp32 diagonal blocks, mma.sync for
// the blocks below them) and the W'^T = Kp^T T'^T and U^T = V^T T'^T products
// (tcgen05, MN-major A).  q, k and v arrive by TMA tensor copies straight into
// their tiles; the next chunk's rows are prefetched into L2.  Every mbarrier
// wait is bounded: on expiry the status word gets 5, the group stops and the
// CTA frees its tensor memory.  The preparation's serial chain is the kernel's
// critical path, so registers move to it: the pass's warpgroups drop to 88 per
// thread and the preparation's rise to 168 (setmaxnreg); of the splits from
// 72 / 184 to 112 / 144 this one runs the varlen batch fastest.
#include <cudaTypedefs.h>

#include "prefill_common.cuh"
#include "tcgen05.cuh"

namespace kda {
namespace prefill {
namespace {

constexpr int kD = 128;
constexpr int kThreads = 512;
constexpr int kGroup = 256;  // warps 0-7: the state pass; warps 8-15: the chunk preparation
constexpr int kPassRegs = 88, kPrepRegs = 168;  // registers per thread of each half after the split
static_assert(kGroup * kPassRegs + kGroup * kPrepRegs == kThreads * 128 && kPassRegs % 8 == 0 && kPrepRegs % 8 == 0,
              "the split redistributes exactly the registers the CTA is launched with");
constexpr uint32_t kWait = 1u << 22;
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kSpanMax = 120.f;  // widest in-chunk span of G (log2 units) for the scaled path
constexpr float kGrowMax = 60.f;   // largest G (log2 units) for the scaled path

// Shared memory, from a 1 KiB-aligned base.
struct FS {
    // Stage s at s * STAGE: the chunk's operands for the state pass.
    static constexpr int QK = 0;        // Qp slab 0 | Kp slab 0 | Qp slab 1 | Kp slab 1 (8 KiB each); the
                                        // Gram's A = [Qp; Kp]; later W'^T [128][64] in the two Kp slabs
    static constexpr int KR = 32768;    // Kr [64][128] (two 64-channel slabs)
    static constexpr int AQK = 49152;   // A_qk [64][64]
    static constexpr int VEC = 57344;   // m_op[128], m_st[128], f[128] fp32
    static constexpr int META = VEC + 1536;  // int32[16]
    static constexpr int STAGE = 59392;
    static constexpr int V = 2 * STAGE;          // v [64][128] (TMA target)
    static constexpr int TP = V + 16384;         // T' [64][64]
    static constexpr int SOP = TP + 8192;        // S_r^T [128][128] bf16; V_new^T [128][64] reuses slab 0
    static constexpr int OST = SOP + 32768;      // output staging [64][128] bf16
    static constexpr int SCR = OST + 16384;      // preparation scratch (16 KiB)
    static constexpr int TAB = SCR + 16384;      // beta[64], fprev[128], norms[128], item word
    static constexpr int BYTES = TAB + 2048;
    // inside SCR: the cumsum exchange, then the triangular solve's blocks
    static constexpr int TOT = SCR, LMAX = SCR + 4096, LMIN = SCR + 8192;  // fp32 [8][128] each
    static constexpr int AB = SCR;                // A_IK (K < I) bf16 [6][16][16]
    static constexpr int TD = SCR + 3072;         // T_II bf16 [4][16][16]
    static constexpr int BLK = SCR + 5120;        // per-warp 16x16 bf16 scratch [3]
    static constexpr int AD = SCR + 6656;         // A_II fp32 [4][16][17]
    static_assert(AD + 4 * 16 * 17 * 4 <= SCR + 16384, "solve blocks fit");
    static constexpr int BETA = TAB, FPREV = TAB + 256, NORM = TAB + 768, ITEM = TAB + 1280;
};

// Tensor memory columns.
constexpr uint32_t kColS = 0, kColX = 128, kColY = 192, kColG = 320, kColU = 384, kTmemCols = 512;

// Stage metadata (int32 words).
enum { M_KIND = 0, M_B, M_H, M_C, M_NCH, M_T0, M_LEN };
enum { K_CHUNK = 1, K_EMPTY = 2, K_END = 3 };

struct FusedParams {
    const __nv_bfloat16 *q, *k, *v;
    const float *g, *beta;
    const int32_t *cu, *seq_order;
    int32_t *status;        // word 0: status (5: a bounded wait of this kernel expired)
    int32_t *item_counter;  // next (sequence, head) item; zeroed by the chunk table kernel
    int64_t n_items;        // num_seqs * H
    int32_t H;
    float scale;
    int32_t l2norm;
    StateEnds se;
    __nv_bfloat16 *out;
};

struct FusedMaps {
    CUtensorMap q, k, v, g;  // g: for L2 prefetches only
};

__device__ __forceinline__ void group_sync(int id) { asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(kGroup) : "memory"); }

__device__ __forceinline__ bool group_or(int id, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(id), "r"(kGroup)
        : "memory");
    return r != 0;
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A and B, fp32 D,
// each operand K-major or MN-major.
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool a_mn, bool b_mn)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ uint4 pack8f(const float *x)
{
    return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                      pack_bf16x2(x[6], x[7]));
}

// Byte offset of (row, col) of a [rows][128] bf16 tile in 64-column slabs of rows x 128 bytes.
__device__ __forceinline__ uint32_t slab_off(int rows, int row, int col)
{
    return static_cast<uint32_t>((col >> 6) * rows * 128) + swz_off<128>(row, col & 63);
}
// Element (row i, channel c) of Qp / Kp in a stage's interleaved [Qp0 | Kp0 | Qp1 | Kp1].
__device__ __forceinline__ uint32_t qp_off(int i, int c) { return (c >> 6) * 16384 + swz_off<128>(i, c & 63); }
__device__ __forceinline__ uint32_t kp_off(int i, int c) { return 8192 + (c >> 6) * 16384 + swz_off<128>(i, c & 63); }
// Element (channel c, token t) of W'^T [128][64] (MN-major B rows) in the two Kp slabs.
__device__ __forceinline__ uint32_t wt_off(int c, int t) { return 8192 + (c >> 6) * 16384 + swz_off<128>(c & 63, t); }

// Byte offset of element (r, c) (0..15) of 16x16 bf16 block `blk` (the solve's ldmatrix layout).
__device__ __forceinline__ uint32_t blk_off(int blk, int r, int c)
{
    return static_cast<uint32_t>(blk * 512 + r * 32 + ((((c >> 3) ^ (r >> 2)) & 1) << 4) + ((c & 7) << 1));
}
__device__ __forceinline__ int fslot(int I, int J) { return I * (I - 1) / 2 + J; }

// Waits for the barrier's phase `parity`, the thread suspended between polls (up to about
// 1 us each, woken when the phase completes) so that a waiting thread takes no issue slots
// from the working warps; gives up after about one second of the global timer.
__device__ __forceinline__ bool mbar_wait_suspend(uint64_t *bar, uint32_t parity)
{
    const uint32_t a = smem_u32(bar);
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n"
            " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(a), "r"(parity), "r"(1000u)
            : "memory");
        if (done) return true;
        const uint64_t t = global_ns();
        if (t0 == 0) t0 = t;
        else if (t - t0 > 1000000000ull || i >= kWait) return false;
    }
}

struct Waiter {
    int32_t *status;
    bool gave_up = false;
    __device__ __forceinline__ bool wait(uint64_t *bar, uint32_t parity)
    {
        if (gave_up) return false;
        if (!mbar_wait_suspend(bar, parity)) {
            gave_up = true;
            atomicExch(status, 5);
        }
        return !gave_up;
    }
};

struct Bars {
    uint64_t full[2], empty[2], ld, pmma, smma;
};

// ------------------------------------------------------------ preparation ---

// G (fp32 [64][128], log2 units) of the exact path: rows 0-31 over the Kr tile, rows 32-63
// over the scratch.
__device__ __forceinline__ float *exact_g_row(char *sm, char *st, int i)
{
    return i < 32 ? reinterpret_cast<float *>(st + FS::KR) + i * kD
                  : reinterpret_cast<float *>(sm + FS::SCR) + (i - 32) * kD;
}

// Exact gated Gram of one chunk (a span too wide for the scaled operands): every
// e^{G_i - G_j} (i >= j) from its own exponent difference.  Leaves A_qk in the stage,
// beta A_kk in the solve blocks, and the plain operands Q~ (scale q^ e^G), k^ e^G and
// K~ (k^ e^{G_last - G}) in the Qp, Kp and Kr tiles.  G is in its rows (exact_g_row),
// written by the caller; the first barrier here publishes it.
__device__ __noinline__ void prep_exact(char *sm, char *st, int ptid, float scale, int32_t l2norm, int r0, int cb)
{
    const int lane = ptid & 31;
    float *norm = reinterpret_cast<float *>(sm + FS::NORM);  // [0, 64) q, [64, 128) k
    const float *beta = reinterpret_cast<const float *>(sm + FS::BETA);
    auto gq = [&](int i) { return exact_g_row(sm, st, i); };
    auto ld_bf = [&](const char *base, uint32_t off) {
        return bf16_bits_to_f32(*reinterpret_cast<const uint16_t *>(base + off));
    };
    // norms of the raw q, k rows (in place in the stage)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int i = r0 + j;
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float qv = ld_bf(st, qp_off(i, cb + c)), kv = ld_bf(st, kp_off(i, cb + c));
            sq = fmaf(qv, qv, sq);
            sk = fmaf(kv, kv, sk);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
        }
        if (lane == 0) {
            norm[i] = l2norm ? rsqrtf(sq + 1e-6f) : 1.f;
            norm[64 + i] = l2norm ? rsqrtf(sk + 1e-6f) : 1.f;
        }
    }
    group_sync(1);
    // thread: row i = ptid / 4, columns j = ptid % 4 + 4 m
    const int i = ptid >> 2, ph = ptid & 3;
    float akk[16], aqk[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) akk[m] = aqk[m] = 0.f;
#pragma unroll 1
    for (int c = 0; c < kD; ++c) {
        const float Gi = gq(i)[c];
        const float qi = ld_bf(st, qp_off(i, c)), ki = ld_bf(st, kp_off(i, c));
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int j = ph + 4 * m;
            const float d = j <= i ? Gi - gq(j)[c] : -INFINITY;
            const float t = ld_bf(st, kp_off(j, c)) * ex2_approx(d);
            akk[m] = fmaf(ki, t, akk[m]);
            aqk[m] = fmaf(qi, t, aqk[m]);
        }
    }
    const float rqi = norm[i], rki = norm[64 + i], bi = beta[i];
    float rkj[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) rkj[m] = norm[64 + ph + 4 * m];
    // the plain operands of this thread's rows, kept packed until the scratch is free
    uint32_t pq[8][2], pk[8][2], pr[8][2];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int r = r0 + j;
        float vq[4], vk[4], vr[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float Gv = gq(r)[cb + c], Gl = gq(C - 1)[cb + c];
            const float e = ex2_approx(Gv);
            const float qh = ld_bf(st, qp_off(r, cb + c)) * norm[r];
            const float kh = ld_bf(st, kp_off(r, cb + c)) * norm[64 + r];
            vq[c] = qh * e * scale;
            vk[c] = kh * e;
            vr[c] = kh * ex2_approx(Gl - Gv);
        }
        pq[j][0] = pack_bf16x2(vq[0], vq[1]);
        pq[j][1] = pack_bf16x2(vq[2], vq[3]);
        pk[j][0] = pack_bf16x2(vk[0], vk[1]);
        pk[j][1] = pack_bf16x2(vk[2], vk[3]);
        pr[j][0] = pack_bf16x2(vr[0], vr[1]);
        pr[j][1] = pack_bf16x2(vr[2], vr[3]);
    }
    group_sync(1);  // every read of G, the raw q and k is done
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int r = r0 + j;
        *reinterpret_cast<uint2 *>(st + qp_off(r, cb)) = make_uint2(pq[j][0], pq[j][1]);
        *reinterpret_cast<uint2 *>(st + kp_off(r, cb)) = make_uint2(pk[j][0], pk[j][1]);
        *reinterpret_cast<uint2 *>(st + FS::KR + slab_off(64, r, cb)) = make_uint2(pr[j][0], pr[j][1]);
    }
    float *ad = reinterpret_cast<float *>(sm + FS::AD);
    const int I = i >> 4;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int j = ph + 4 * m, J = j >> 4;
        const float ykk = j < i ? akk[m] * rki * rkj[m] * bi : 0.f;
        const float yqk = j <= i ? aqk[m] * rqi * rkj[m] * scale : 0.f;
        if (J < I)
            *reinterpret_cast<uint16_t *>(sm + FS::AB + blk_off(fslot(I, J), i - 16 * I, j - 16 * J)) =
                f32_to_bf16_bits(ykk);
        else if (J == I)
            ad[I * 16 * 17 + (i - 16 * I) * 17 + (j - 16 * J)] = ykk;
        *reinterpret_cast<uint16_t *>(st + FS::AQK + swz_off<128>(i, j)) = f32_to_bf16_bits(yqk);
    }
}

// T' = (I + A_kk)^-1 diag(beta) into the [64][64] tile TP: the four 16 x 16 diagonal
// inverses by fp32 forward substitution (right-looking, one column per lane), then the
// blocks below them, T'_IJ = -T_II sum_{J <= K < I} A_IK T'_KJ, by mma.sync
// (warp 0: (1,0), (2,0), (3,0); warp 1: (2,1), (3,1); warp 2: (3,2)).
__device__ __forceinline__ void prep_solve(char *sm, int ptid)
{
    const int lane = ptid & 31, pw = ptid >> 5;
    const int gid = lane >> 2, tig = lane & 3, mi = lane >> 3, ri = lane & 7;
    const float *beta = reinterpret_cast<const float *>(sm + FS::BETA);
    char *tp = sm + FS::TP;
    if (pw < 4 && lane < 16) {
        const int I = pw, j = lane;
        const float *A = reinterpret_cast<const float *>(sm + FS::AD) + I * 16 * 17;
        float tcol[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) tcol[i] = i == j ? 1.f : 0.f;
#pragma unroll
        for (int kk = 0; kk < 15; ++kk)
#pragma unroll
            for (int i = kk + 1; i < 16; ++i) tcol[i] -= A[i * 17 + kk] * tcol[kk];
        const float bj = beta[16 * I + j];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            *reinterpret_cast<uint16_t *>(sm + FS::TD + blk_off(I, i, j)) = f32_to_bf16_bits(tcol[i]);
            *reinterpret_cast<uint16_t *>(tp + swz_off<128>(16 * I + i, 16 * I + j)) = f32_to_bf16_bits(tcol[i] * bj);
        }
    }
    group_sync(1);
    if (pw < 3) {
        char *scr = sm + FS::BLK + pw * 512;
        auto tblock = [&](int I, int J) {
            float x[2][4] = {};
            for (int K = J; K < I; ++K) {
                uint32_t a[4], b[4];
                ldmatrix_x4(a, smem_u32(sm + FS::AB + blk_off(fslot(I, K), ri + 8 * (mi & 1), 8 * (mi >> 1))));
                ldmatrix_x4_trans(b, smem_u32(tp + swz_off<128>(16 * K + ri + 8 * (mi & 1), 16 * J + 8 * (mi >> 1))));
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
            ldmatrix_x4(a, smem_u32(sm + FS::TD + blk_off(I, ri + 8 * (mi & 1), 8 * (mi >> 1))));
            ldmatrix_x4_trans(b, smem_u32(scr + blk_off(0, ri + 8 * (mi & 1), 8 * (mi >> 1))));
            mma_bf16(y[0], a, b[0], b[1]);
            mma_bf16(y[1], a, b[2], b[3]);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
                    *reinterpret_cast<uint32_t *>(tp + swz_off<128>(16 * I + gid + 8 * hr, 16 * J + 8 * nt + 2 * tig)) =
                        pack_bf16x2(-y[nt][2 * hr], -y[nt][2 * hr + 1]);
            __syncwarp();  // the block is read by this warp's next block; scr is rewritten
        };
        if (pw == 0) {
            tblock(1, 0);
            tblock(2, 0);
            tblock(3, 0);
        } else if (pw == 1) {
            tblock(2, 1);
            tblock(3, 1);
        } else {
            tblock(3, 2);
        }
    }
}

__device__ void prep_loop(const FusedParams &p, const FusedMaps &maps, char *sm, Bars &bar, uint32_t tmem,
                          Waiter &w)
{
    const int tid = threadIdx.x, ptid = tid - kGroup, lane = tid & 31, pw = ptid >> 5;
    const int quad = (tid >> 5) & 3, part = pw >> 2;  // TMEM lane quadrant of this warp; column half
    const int r0 = 8 * pw, cb = 4 * lane;            // row pass: rows r0 .. r0 + 7, channels cb .. cb + 3
    const int64_t H = p.H;
    const bool leader = ptid == 0;
    float *beta_s = reinterpret_cast<float *>(sm + FS::BETA);
    float *fprev = reinterpret_cast<float *>(sm + FS::FPREV);
    int32_t *item_word = reinterpret_cast<int32_t *>(sm + FS::ITEM);
    uint32_t ld_phase = 0, pmma_phase = 0;

    int64_t b = 0, tok_begin = 0, tok_end = 0;
    int h = 0, n_chunks = 0, c = 0;
    for (uint32_t n = 0;; ++n) {
        const int s = static_cast<int>(n & 1);
        char *st = sm + s * FS::STAGE;
        int32_t *meta = reinterpret_cast<int32_t *>(st + FS::META);
        int kind = K_CHUNK;
        if (c >= n_chunks) {  // the next item (or the end)
            if (leader) *item_word = atomicAdd(p.item_counter, 1);
            group_sync(1);
            const int64_t k = *item_word;
            group_sync(1);  // the word is rewritten at the next fetch
            if (k >= p.n_items) {
                kind = K_END;
            } else {
                b = p.seq_order[k / H];
                h = static_cast<int>(k % H);
                tok_begin = p.cu[b];
                tok_end = p.cu[b + 1];
                n_chunks = tok_end > tok_begin ? static_cast<int>((tok_end - tok_begin + C - 1) / C) : 0;
                c = 0;
                if (ptid < kD) fprev[ptid] = 1.f;
                if (n_chunks == 0) kind = K_EMPTY;
            }
        }
        // this chunk's gates and beta, loaded before waiting for the stage
        const int64_t t0 = tok_begin + static_cast<int64_t>(c) * C;
        const int len = kind == K_CHUNK ? static_cast<int>(tok_end - t0 < C ? tok_end - t0 : C) : 0;
        float G[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (r0 + j < len) {
                const float4 x = __ldg(reinterpret_cast<const float4 *>(p.g + ((t0 + r0 + j) * H + h) * kD + cb));
                G[j][0] = x.x; G[j][1] = x.y; G[j][2] = x.z; G[j][3] = x.w;
            } else {
                G[j][0] = G[j][1] = G[j][2] = G[j][3] = 0.f;
            }
        }
        const float beta_v = ptid < len ? p.beta[(t0 + ptid) * H + h] : 0.f;
        if (leader) w.wait(&bar.empty[s], ((n >> 1) & 1) ^ 1);  // the barrier below orders the rest
        if (group_or(1, w.gave_up)) return;
        if (kind != K_CHUNK) {
            if (leader) {
                meta[M_KIND] = kind;
                meta[M_B] = static_cast<int32_t>(b);
                meta[M_H] = h;
                mbar_arrive(&bar.full[s]);
            }
            if (kind == K_END) return;
            continue;
        }
        if (leader) {
            meta[M_KIND] = K_CHUNK;
            meta[M_B] = static_cast<int32_t>(b);
            meta[M_H] = h;
            meta[M_C] = c;
            meta[M_NCH] = n_chunks;
            meta[M_T0] = static_cast<int32_t>(t0);
            meta[M_LEN] = len;
        }
        // the six tensor copies (q, k, v x two 64-channel slabs) and the next chunk's L2
        // prefetches, one per warp lane 0, so that no thread issues them all in turn
        if (lane == 0) {
            const int sl = pw & 1, x = 64 * sl, z = static_cast<int>(t0);
            if (pw < 6) {
                char *dst = pw < 2 ? st + FS::QK + sl * 16384 : pw < 4 ? st + FS::QK + 8192 + sl * 16384
                                                                       : sm + FS::V + sl * 8192;
                const CUtensorMap *map = pw < 2 ? &maps.q : pw < 4 ? &maps.k : &maps.v;
                mbar_arrive_expect_tx(&bar.ld, 8192);  // six arrivals complete a phase, with their bytes
                tma_load_3d(dst, map, x, h, z, &bar.ld);
                if (c + 1 < n_chunks) tma_prefetch_3d(map, x, h, z + C);  // the next chunk into L2
            } else if (pw == 6 && c + 1 < n_chunks) {
                tma_prefetch_3d(&maps.g, 0, h, z + C);
            }
        }

        if (ptid < C) beta_s[ptid] = beta_v;
        // ---- gates: in-chunk cumulative sum (log2 units), the reference and the span ----
        float lmax[4], lmin[4];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const float2 x = make_float2(G[j][e], G[j][e + 1]), l2 = make_float2(kLog2eF, kLog2eF);
                const float2 y = j == 0 ? mul2(x, l2) : fma2(x, l2, make_float2(G[j - 1][e], G[j - 1][e + 1]));
                G[j][e] = y.x;
                G[j][e + 1] = y.y;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                lmax[e] = j == 0 ? G[0][e] : fmaxf(lmax[e], G[j][e]);
                lmin[e] = j == 0 ? G[0][e] : fminf(lmin[e], G[j][e]);
            }
        }
        *reinterpret_cast<float4 *>(sm + FS::TOT + (pw * kD + cb) * 4) = make_float4(G[7][0], G[7][1], G[7][2], G[7][3]);
        *reinterpret_cast<float4 *>(sm + FS::LMAX + (pw * kD + cb) * 4) = make_float4(lmax[0], lmax[1], lmax[2], lmax[3]);
        *reinterpret_cast<float4 *>(sm + FS::LMIN + (pw * kD + cb) * 4) = make_float4(lmin[0], lmin[1], lmin[2], lmin[3]);
        group_sync(1);
        float off[4], gmax[4], gmin[4], glast[4];
        {
            float run[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ww = 0; ww < 8; ++ww) {
                const float4 t = *reinterpret_cast<const float4 *>(sm + FS::TOT + (ww * kD + cb) * 4);
                const float4 mx = *reinterpret_cast<const float4 *>(sm + FS::LMAX + (ww * kD + cb) * 4);
                const float4 mn = *reinterpret_cast<const float4 *>(sm + FS::LMIN + (ww * kD + cb) * 4);
                const float tv[4] = {t.x, t.y, t.z, t.w}, xv[4] = {mx.x, mx.y, mx.z, mx.w}, nv[4] = {mn.x, mn.y, mn.z, mn.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (ww == pw) off[e] = run[e];
                    gmax[e] = ww == 0 ? run[e] + xv[e] : fmaxf(gmax[e], run[e] + xv[e]);
                    gmin[e] = ww == 0 ? run[e] + nv[e] : fminf(gmin[e], run[e] + nv[e]);
                    run[e] += tv[e];
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) glast[e] = run[e];
        }
        bool wide_c = false;
        float gref[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            gref[e] = 0.5f * (gmax[e] + gmin[e]);
            wide_c |= !(gmax[e] - gmin[e] <= kSpanMax) || !(gmax[e] <= kGrowMax);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) G[j][e] += off[e];
        if (leader) w.wait(&bar.ld, ld_phase);  // q, k (in place in the stage) and v have landed
        ld_phase ^= 1u;
        // (the barrier also publishes the landed tiles and ends every read of the exchange)
        const bool exact = group_or(1, wide_c);

        float *vec = reinterpret_cast<float *>(st + FS::VEC);
        if (!exact) {
            // ---- row pass: norms, then Qp, Kp in place and Kr ----
            float vsum[16];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint2 qa = *reinterpret_cast<const uint2 *>(st + qp_off(r0 + j, cb));
                const uint2 ka = *reinterpret_cast<const uint2 *>(st + kp_off(r0 + j, cb));
                const float qv[4] = {bf16_lo(qa.x), bf16_hi(qa.x), bf16_lo(qa.y), bf16_hi(qa.y)};
                const float kv[4] = {bf16_lo(ka.x), bf16_hi(ka.x), bf16_lo(ka.y), bf16_hi(ka.y)};
                float2 sq = mul2(make_float2(qv[0], qv[1]), make_float2(qv[0], qv[1]));
                float2 sk = mul2(make_float2(kv[0], kv[1]), make_float2(kv[0], kv[1]));
                sq = fma2(make_float2(qv[2], qv[3]), make_float2(qv[2], qv[3]), sq);
                sk = fma2(make_float2(kv[2], kv[3]), make_float2(kv[2], kv[3]), sk);
                vsum[2 * j] = sq.x + sq.y;
                vsum[2 * j + 1] = sk.x + sk.y;
            }
            // transposed butterfly: lane L ends with the total of value L >> 1
#pragma unroll
            for (int mask = 16, half = 8; mask >= 2; mask >>= 1, half >>= 1) {
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
            for (int j = 0; j < 8; ++j) {
                const float nq = __shfl_sync(0xffffffffu, rn, 4 * j) * p.scale;
                const float nk = __shfl_sync(0xffffffffu, rn, 4 * j + 2);
                const int i = r0 + j;
                const uint2 qa = *reinterpret_cast<const uint2 *>(st + qp_off(i, cb));
                const uint2 ka = *reinterpret_cast<const uint2 *>(st + kp_off(i, cb));
                const float qv[4] = {bf16_lo(qa.x), bf16_hi(qa.x), bf16_lo(qa.y), bf16_hi(qa.y)};
                const float kv[4] = {bf16_lo(ka.x), bf16_hi(ka.x), bf16_lo(ka.y), bf16_hi(ka.y)};
                float oq[4], ok[4], orr[4];
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const float d0 = G[j][e] - gref[e], d1 = G[j][e + 1] - gref[e + 1];
                    const float2 P = make_float2(ex2_approx(d0), ex2_approx(d1));
                    const float2 R = make_float2(ex2_approx(-d0), ex2_approx(-d1));
                    const float2 qh = mul2(make_float2(qv[e], qv[e + 1]), make_float2(nq, nq));
                    const float2 kh = mul2(make_float2(kv[e], kv[e + 1]), make_float2(nk, nk));
                    const float2 a = mul2(qh, P), bb = mul2(kh, P), rr = mul2(kh, R);
                    oq[e] = a.x; oq[e + 1] = a.y;
                    ok[e] = bb.x; ok[e + 1] = bb.y;
                    orr[e] = rr.x; orr[e + 1] = rr.y;
                }
                *reinterpret_cast<uint2 *>(st + qp_off(i, cb)) = make_uint2(pack_bf16x2(oq[0], oq[1]), pack_bf16x2(oq[2], oq[3]));
                *reinterpret_cast<uint2 *>(st + kp_off(i, cb)) = make_uint2(pack_bf16x2(ok[0], ok[1]), pack_bf16x2(ok[2], ok[3]));
                *reinterpret_cast<uint2 *>(st + FS::KR + slab_off(64, i, cb)) =
                    make_uint2(pack_bf16x2(orr[0], orr[1]), pack_bf16x2(orr[2], orr[3]));
            }
            if (pw == 0) {  // per-channel factors of the pass: m = f_prev 2^{G_r}, f = 2^{G_last - G_r}
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float m = fprev[cb + e] * ex2_approx(gref[e]);
                    const float f = ex2_approx(glast[e] - gref[e]);
                    vec[cb + e] = m;
                    vec[kD + cb + e] = m;
                    vec[2 * kD + cb + e] = f;
                    fprev[cb + e] = f;
                }
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            group_sync(1);
            tc::fence_after_sync();
            // ---- gated Gram on the tensor cores: [Qp; Kp] Kr^T, M = 128, N = 64, K = 128 ----
            if (leader) {
                const uint32_t a0 = smem_u32(st + FS::QK), b0 = smem_u32(st + FS::KR);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t a = tc::sdesc_sw128(a0 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                    const uint64_t bd = tc::sdesc_sw128(b0 + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
                    tc::mma_bf16(tmem + kColG, a, bd, idesc(128, 64, false, false), ks > 0 ? 1u : 0u);
                }
                tc::commit(&bar.pmma);
                w.wait(&bar.pmma, pmma_phase);
            }
            pmma_phase ^= 1u;
            group_sync(1);
            tc::fence_after_sync();
            // epilogue: lanes 0-63 A_qk (causal) -> the stage; lanes 64-127 beta A_kk -> solve blocks
            {
                uint32_t r[32];
                tc::ld32(tmem + (static_cast<uint32_t>(32 * quad) << 16) + kColG + 32 * part, r);
                tc::wait_ld();
                const int row = 32 * quad + lane, j0 = 32 * part;
                if (quad < 2) {
                    const int i = row;
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) y[e] = j0 + 8 * q8 + e <= i ? __uint_as_float(r[8 * q8 + e]) : 0.f;
                        *reinterpret_cast<uint4 *>(st + FS::AQK + swz_off<128>(i, j0 + 8 * q8)) = pack8f(y);
                    }
                } else {
                    const int i = row - 64, I = i >> 4;
                    const float bi = beta_s[i];
                    float *ad = reinterpret_cast<float *>(sm + FS::AD);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const int j = j0 + e, J = j >> 4;
                        const float y0 = j < i ? __uint_as_float(r[e]) * bi : 0.f;
                        const float y1 = j + 1 < i ? __uint_as_float(r[e + 1]) * bi : 0.f;
                        if (J < I) {
                            *reinterpret_cast<uint32_t *>(sm + FS::AB + blk_off(fslot(I, J), i - 16 * I, j - 16 * J)) =
                                pack_bf16x2(y0, y1);
                        } else if (J == I) {
                            ad[I * 16 * 17 + (i - 16 * I) * 17 + (j - 16 * J)] = y0;
                            ad[I * 16 * 17 + (i - 16 * I) * 17 + (j - 16 * J) + 1] = y1;
                        }
                    }
                }
            }
        } else {
            // ---- exact path: G rows to the scratch, the exact Gram and the plain operands ----
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<float4 *>(exact_g_row(sm, st, r0 + j) + cb) =
                    make_float4(G[j][0], G[j][1], G[j][2], G[j][3]);
            prep_exact(sm, st, ptid, p.scale, p.l2norm, r0, cb);
            if (pw == 0) {  // plain state: m_op = f_prev, m_st = f_prev 2^{G_last}, f = 1
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float fp = fprev[cb + e];
                    vec[cb + e] = fp;
                    vec[kD + cb + e] = fp * ex2_approx(glast[e]);
                    vec[2 * kD + cb + e] = 1.f;
                    fprev[cb + e] = 1.f;
                }
            }
        }
        group_sync(1);
        prep_solve(sm, ptid);
        fence_proxy_async_smem();
        tc::fence_before_sync();
        group_sync(1);
        tc::fence_after_sync();
        // ---- W'^T = Kp^T T'^T -> Gram columns, U^T = V^T T'^T -> U buffer s (M = 128, N = 64, K = 64) ----
        if (leader) {
            const uint32_t kp0 = smem_u32(st + FS::QK + 8192), v0 = smem_u32(sm + FS::V), t0s = smem_u32(sm + FS::TP);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t bd = tc::sdesc_sw128(t0s + ks * 32, 16, 1024);
                tc::mma_bf16(tmem + kColG, tc::sdesc_sw128(kp0 + ks * 2048, 16384, 1024), bd,
                             idesc(128, 64, true, false), ks > 0 ? 1u : 0u);
                tc::mma_bf16(tmem + kColU + 64 * s, tc::sdesc_sw128(v0 + ks * 2048, 8192, 1024), bd,
                             idesc(128, 64, true, false), ks > 0 ? 1u : 0u);
            }
            tc::commit(&bar.pmma);
            w.wait(&bar.pmma, pmma_phase);
        }
        pmma_phase ^= 1u;
        group_sync(1);
        tc::fence_after_sync();
        // W'^T (lane = channel) -> the Kp slabs, as the MN-major B operand of X^T = S_r^T W'^T
        {
            uint32_t r[32];
            tc::ld32(tmem + (static_cast<uint32_t>(32 * quad) << 16) + kColG + 32 * part, r);
            tc::wait_ld();
            const int ch = 32 * quad + lane;
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = __uint_as_float(r[8 * q8 + e]);
                *reinterpret_cast<uint4 *>(st + wt_off(ch, 32 * part + 8 * q8)) = pack8f(y);
            }
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        group_sync(1);
        if (leader) mbar_arrive(&bar.full[s]);
        ++c;
    }
}

// ---------------------------------------------------------------- pass ---

__device__ void pass_loop(const FusedParams &p, char *sm, Bars &bar, uint32_t tmem, Waiter &w)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = warp & 3, part = warp >> 2;
    const int v = 32 * quad + lane;  // value row = TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * quad) << 16);
    const int64_t H = p.H;
    const int64_t per_seq = H * kD * kD;
    const bool leader = tid == 0;
    __nv_bfloat16 *os = reinterpret_cast<__nv_bfloat16 *>(sm + FS::OST);
    uint32_t smma_phase = 0, ybuf = 0;
    // the previous chunk, whose outputs are still in tensor memory
    bool prev = false;
    int64_t prev_t0 = 0;
    int prev_len = 0, prev_h = 0;
    uint32_t prev_y = 0;

    auto stage_outputs = [&]() {
        uint32_t y[32];
        tc::ld32(tl + prev_y + 32 * part, y);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) os[(32 * part + e) * kD + v] = __float2bfloat16_rn(__uint_as_float(y[e]));
    };
    auto store_outputs = [&]() {
        const uint4 *src = reinterpret_cast<const uint4 *>(os);
#pragma unroll
        for (int e = tid; e < C * (kD * 2 / 16); e += kGroup) {
            const int t = e >> 4, q16 = e & 15;
            if (t < prev_len) reinterpret_cast<uint4 *>(p.out + ((prev_t0 + t) * H + prev_h) * kD)[q16] = src[e];
        }
    };
    // S (this thread's row v, columns c0 .. c0 + 31) = S^ f -> a state buffer with its dtype's cast
    auto put_state = [&](void *dst, int32_t dtype, int64_t base, int hh, const float *f) {
#pragma unroll 1
        for (int j = 0; j < 2; ++j) {
            const int c0 = 64 * part + 32 * j;
            uint32_t r[32];
            tc::ld32(tl + kColS + c0, r);
            tc::wait_ld();
            const int64_t row = base + (static_cast<int64_t>(hh) * kD + v) * kD + c0;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const float4 fv = *reinterpret_cast<const float4 *>(f + c0 + e);
                store_state4(dst, dtype, row + e,
                             make_float4(__uint_as_float(r[e]) * fv.x, __uint_as_float(r[e + 1]) * fv.y,
                                         __uint_as_float(r[e + 2]) * fv.z, __uint_as_float(r[e + 3]) * fv.w));
            }
        }
    };

    for (uint32_t n = 0;; ++n) {
        const int s = static_cast<int>(n & 1);
        char *st = sm + s * FS::STAGE;
        const int32_t *meta = reinterpret_cast<const int32_t *>(st + FS::META);
        if (leader) w.wait(&bar.full[s], (n >> 1) & 1);  // the barrier below publishes the stage
        if (group_or(2, w.gave_up)) break;  // together, if any wait of this group expired
        const int kind = meta[M_KIND];
        if (kind == K_END) break;
        const int64_t b = meta[M_B];
        const int h = meta[M_H];
        if (kind == K_EMPTY) {  // no tokens: the final state is the initial one
            const int64_t ib = init_base(p.se, b, per_seq), ob = out_base(p.se, b);
            const int64_t row = (static_cast<int64_t>(h) * kD + v) * kD + 64 * part;
#pragma unroll 4
            for (int e = 0; e < 64; e += 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (ib >= 0) x = load_state4(p.se.init, p.se.init_dtype, ib + row + e);
                if (p.se.final_state != nullptr) store_state4(p.se.final_state, KDA_F32, b * per_seq + row + e, x);
                if (ob >= 0) store_state4(p.se.out_cache, p.se.out_dtype, ob + row + e, x);
            }
            group_sync(2);
            if (leader) mbar_arrive(&bar.empty[s]);
            continue;
        }
        const int c = meta[M_C], n_chunks = meta[M_NCH], len = meta[M_LEN];
        const int64_t t0 = meta[M_T0];
        const float *vec = reinterpret_cast<const float *>(st + FS::VEC);
        const uint32_t ycol = kColY + 64 * ybuf;  // alternates per chunk: the previous chunk's is still read
        ybuf ^= 1u;

        if (c == 0) {  // initial state -> S^ (a new item's scale is 1)
            const int64_t ib = init_base(p.se, b, per_seq);
            const int64_t row = (static_cast<int64_t>(h) * kD + v) * kD;
#pragma unroll 1
            for (int j = 0; j < 2; ++j) {
                const int c0 = 64 * part + 32 * j;
                uint32_t r[32];
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (ib >= 0) x = load_state4(p.se.init, p.se.init_dtype, ib + row + c0 + e);
                    r[e] = __float_as_uint(x.x);
                    r[e + 1] = __float_as_uint(x.y);
                    r[e + 2] = __float_as_uint(x.z);
                    r[e + 3] = __float_as_uint(x.w);
                }
                tc::st32(tl + kColS + c0, r);
            }
            tc::wait_st();
        }
        // (A) S_r = S^ m_op -> bf16 operand; S^ <- S^ m_st (m_st = m_op unless the chunk took the exact path)
        {
            uint32_t r[2][32];
            tc::ld32(tl + kColS + 64 * part, r[0]);
            tc::ld32(tl + kColS + 64 * part + 32, r[1]);
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int c0 = 64 * part + 32 * j;
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {
                    float a[8];
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const int cc = c0 + 8 * q8 + e;
                        const float2 mo = *reinterpret_cast<const float2 *>(vec + cc);
                        const float2 ms = *reinterpret_cast<const float2 *>(vec + kD + cc);
                        const float2 x = make_float2(__uint_as_float(r[j][8 * q8 + e]), __uint_as_float(r[j][8 * q8 + e + 1]));
                        const float2 yo = mul2(x, mo), ys = mul2(x, ms);
                        a[e] = yo.x;
                        a[e + 1] = yo.y;
                        r[j][8 * q8 + e] = __float_as_uint(ys.x);
                        r[j][8 * q8 + e + 1] = __float_as_uint(ys.y);
                    }
                    *reinterpret_cast<uint4 *>(sm + FS::SOP + slab_off(128, v, c0 + 8 * q8)) = pack8f(a);
                }
                tc::st32(tl + kColS + c0, r[j]);
            }
            tc::wait_st();
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        group_sync(2);
        tc::fence_after_sync();
        // (B) X^T = S_r^T W'^T (B MN-major), Y^T = S_r^T Qp^T (B K-major): M = 128, N = 64, K = 128
        if (leader) {
            const uint32_t sa = smem_u32(sm + FS::SOP), qk = smem_u32(st + FS::QK);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t a = tc::sdesc_sw128(sa + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                tc::mma_bf16(tmem + kColX, a, tc::sdesc_sw128(qk + 8192 + (ks >> 2) * 16384 + (ks & 3) * 2048, 8192, 1024),
                             idesc(128, 64, false, true), ks > 0 ? 1u : 0u);
                tc::mma_bf16(tmem + ycol, a, tc::sdesc_sw128(qk + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                             idesc(128, 64, false, false), ks > 0 ? 1u : 0u);
            }
            tc::commit(&bar.smma);
        }
        if (prev) stage_outputs();  // the previous chunk's outputs, while these MMAs run
        if (leader) w.wait(&bar.smma, smma_phase);
        smma_phase ^= 1u;
        group_sync(2);
        tc::fence_after_sync();
        // (C) V_new^T = U^T - X^T (this thread's 32 token columns) -> bf16 operand in slab 0
        {
            uint32_t x[32], u[32];
            tc::ld32(tl + kColX + 32 * part, x);
            tc::ld32(tl + kColU + 64 * s + 32 * part, u);
            tc::wait_ld();
            float d[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) d[e] = __uint_as_float(u[e]) - __uint_as_float(x[e]);
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8)
                *reinterpret_cast<uint4 *>(sm + FS::SOP + swz_off<128>(v, 32 * part + 8 * q8)) = pack8f(d + 8 * q8);
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        group_sync(2);
        tc::fence_after_sync();
        // (D) Y^T += V_new^T A_qk^T (N = 64), S^T += V_new^T Kr (N = 128, B MN-major), K = 64
        if (leader) {
            const uint32_t sa = smem_u32(sm + FS::SOP), aq = smem_u32(st + FS::AQK), kr = smem_u32(st + FS::KR);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t a = tc::sdesc_sw128(sa + ks * 32, 16, 1024);
                tc::mma_bf16(tmem + ycol, a, tc::sdesc_sw128(aq + ks * 32, 16, 1024), idesc(128, 64, false, false), 1u);
                tc::mma_bf16(tmem + kColS, a, tc::sdesc_sw128(kr + ks * 2048, 8192, 1024), idesc(128, 128, false, true), 1u);
            }
            tc::commit(&bar.smma);
        }
        if (prev) store_outputs();  // staged before the barrier above
        if (leader) w.wait(&bar.smma, smma_phase);
        smma_phase ^= 1u;
        group_sync(2);
        tc::fence_after_sync();
        // the state after this chunk is S^ f: checkpoint, and the final state after the last chunk
        {
            const float *f = vec + 2 * kD;
            const int64_t tlen = p.cu[b + 1] - p.cu[b];
            const int64_t ck = ckpt_slot(p.se, b, c, tlen);
            if (ck >= 0) put_state(p.se.ckpt, p.se.ckpt_dtype, ck * per_seq, h, f);
            if (c == n_chunks - 1) {
                if (p.se.final_state != nullptr) put_state(p.se.final_state, KDA_F32, b * per_seq, h, f);
                const int64_t ob = out_base(p.se, b);
                if (ob >= 0) put_state(p.se.out_cache, p.se.out_dtype, ob, h, f);
            }
        }
        tc::fence_before_sync();
        group_sync(2);  // every read of stage s (operands, factors) is over
        if (leader) mbar_arrive(&bar.empty[s]);
        prev = true;
        prev_t0 = t0;
        prev_len = len;
        prev_h = h;
        prev_y = ycol;
    }
    if (!group_or(2, w.gave_up) && prev) {
        stage_outputs();
        group_sync(2);
        store_outputs();
    }
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_fused_kernel(const __grid_constant__ FusedParams p, const __grid_constant__ FusedMaps maps)
{
    extern __shared__ char smem_raw[];
    // 1 KiB-aligned base, by indexing the shared array (which keeps the address space known)
    char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ __align__(8) Bars bar;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5;
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar.full[s], 1);
            mbar_init(&bar.empty[s], 1);
        }
        mbar_init(&bar.ld, 6);  // one per tensor copy of a chunk
        mbar_init(&bar.pmma, 1);
        mbar_init(&bar.smma, 1);
        fence_mbar_init();
    }
    // T' blocks above the diagonal stay zero
    for (int e = tid; e < 6 * 16 * 2; e += kThreads) {
        const int bk = e >> 5, r = (e >> 1) & 15, ch = e & 1;
        const int I = bk < 3 ? 0 : bk < 5 ? 1 : 2;
        const int J = bk < 3 ? bk + 1 : bk < 5 ? bk - 1 : 3;
        *reinterpret_cast<uint4 *>(sm + FS::TP + swz_off<128>(16 * I + r, 16 * J + 8 * ch)) = make_uint4(0u, 0u, 0u, 0u);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base;
    Waiter w{p.status};
    // Registers move from the pass to the preparation: launched at 128 per thread (512 threads,
    // the whole 65,536-register file), warpgroups 0-1 drop to 88 and warpgroups 2-3 rise to 168,
    // 8 x 32 x 88 + 8 x 32 x 168 = 65,536, so the increase is always satisfiable.
    if (warp < 8) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kPassRegs) : "memory");
        pass_loop(p, sm, bar, tmem, w);
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kPrepRegs) : "memory");
        prep_loop(p, maps, sm, bar, tmem, w);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_prefill_fused(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                 const int32_t *cu, const int32_t *seq_order, int32_t *status, int32_t *item_counter,
                                 int64_t num_seqs, int64_t total_tokens, int32_t h, float scale, int32_t l2norm,
                                 const StateEnds &se, void *out, cudaStream_t st)
{
    FusedMaps maps{};
    if (total_tokens > 0 && (!encode_rows(&maps.q, q, total_tokens, h, kD) || !encode_rows(&maps.k, k, total_tokens, h, kD) ||
                             !encode_rows(&maps.v, v, total_tokens, h, kD) ||
                             !encode_rows_f32(&maps.g, g, total_tokens, h, kD)))
        return cudaErrorInvalidValue;
    FusedParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.g = g;
    p.beta = beta;
    p.cu = cu;
    p.seq_order = seq_order;
    p.status = status;
    p.item_counter = item_counter;
    p.n_items = num_seqs * h;
    p.H = h;
    p.scale = scale;
    p.l2norm = l2norm;
    p.se = se;
    p.out = static_cast<__nv_bfloat16 *>(out);
    constexpr int smem = FS::BYTES + 1024;  // + slack to align the base to 1 KiB
    // The register split (setmaxnreg) needs the kernel launched with exactly 128 registers per
    // thread: with fewer, the preparation's increase could never be satisfied.
    static const int regs = [] {
        cudaFuncAttributes fa{};
        return cudaFuncGetAttributes(&fa, prefill_fused_kernel) == cudaSuccess ? fa.numRegs : -1;
    }();
    if (regs * kThreads != kGroup * (kPassRegs + kPrepRegs)) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(prefill_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = p.n_items < sm_count() ? p.n_items : sm_count();
    prefill_fused_kernel<<<static_cast<unsigned>(grid), kThreads, smem, st>>>(p, maps);
    return cudaGetLastError();
}

}  // namespace prefill
}  // namespace kda
