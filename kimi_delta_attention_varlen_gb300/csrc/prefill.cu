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
//                           ceil(len/64)), a per-chunk table (first token,
//                           length), checkpoint offsets and a longest-first
//                           sequence order.
//   2. chunk_prep_kernel    one CTA per (chunk, head), fully parallel: every
//                           quantity above that does not depend on S, written
//                           to the workspace as one record per (chunk, head)
//                           (chunk_prep.cu).
//   3. the state pass, which walks each sequence's chunks in order:
//      state_pass_tc_kernel one CTA per (sequence, head), S in tensor memory
//                           (state_pass_tc.cu; head size 128, bf16 output,
//                           enough pairs to fill the GPU), or
//      state_pass_split_kernel  two CTAs per (sequence, head), 64 value
//                           columns each, S in tensor memory with the key as
//                           the lane (state_pass_split.cu; head size 128, bf16
//                           output, few pairs), or
//      state_pass_kernel    one CTA per (sequence, head, value slice), S in
//                           registers (fp32 accumulators), double-buffering
//                           the records into shared memory with bulk copies
//                           (head sizes 32 and 64, fp32 outputs); for few
//                           pairs at head size 128 with fp32 outputs its
//                           warp-pair form (state_pass_pair_kernel) splits
//                           each value group's key channels over two warps.
//   One long sequence at head size 128 (bf16) runs 2. and 3. in segments of
//   256 chunks, the pass of a segment overlapping the next one's preparation
//   on a second stream.
// All products run on the tensor cores (bf16 operands, fp32 accumulation).
//
// Exponent ranges.  Factors e^{G_i - G_j} are split through a reference row:
// off-diagonal 16x16 blocks use the block midpoints, e^{G_i - G_j} =
// P_i F_IJ R_j with P_i = e^{G_i - G_mI}, F_IJ = e^{G_mI - G_mJ} <= 1 and
// R_j = e^{G_mJ - G_j}; each of P and R spans at most 8 tokens of decay, so
// the products stay in fp32/bf16 range while that decay is above -80.  All
// inter-chunk factors (e^G, e^{G_last - G}, e^{G_last}) are <= 1 for g <= 0.
#include <atomic>
#include <mutex>

#include "prefill_common.cuh"

namespace kda {

int64_t sm_count()
{
    static std::atomic<int32_t> count[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    int32_t n = count[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

namespace {

using prefill::C;
using prefill::Rec;
using prefill::tile_off;
using prefill::PassParams;
using prefill::init_base;
using prefill::out_base;
using prefill::ckpt_slot;
using prefill::load_state2;
using prefill::store_state2;
constexpr uint32_t kWaitLimit = 1u << 22;  // bounded mbarrier polls
constexpr int64_t kSegChunks = 256;         // chunks per segment of the segmented prefill

// The segmented prefill's second stream (the highest priority, non-blocking) and its events, one
// set per device, created on first use and kept for the process; calls that use them hold the mutex
// while they enqueue.
struct SegStreams {
    cudaStream_t aux = nullptr;
    cudaEvent_t fork = nullptr, seg = nullptr, join = nullptr;
};
std::mutex g_seg_mu;
SegStreams g_seg[64];

cudaError_t seg_streams(SegStreams **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    SegStreams &r = g_seg[dev];
    if (r.aux == nullptr) {
        int least = 0, greatest = 0;
        if ((e = cudaDeviceGetStreamPriorityRange(&least, &greatest)) != cudaSuccess) return e;
        SegStreams n;
        if ((e = cudaStreamCreateWithPriority(&n.aux, cudaStreamNonBlocking, greatest)) != cudaSuccess) return e;
        for (cudaEvent_t *ev : {&n.fork, &n.seg, &n.join})
            if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
        r = n;
    }
    *out = &r;
    return cudaSuccess;
}

// ---------------------------------------------------------- chunk table ---

// Exclusive prefix sum of count(len_b) over the sequences into off[0 .. B]
// (off[B] = total), by one block of 1024 threads.  Returns the total.
template <typename F>
__device__ int32_t block_prefix(const int32_t *__restrict__ cu, int64_t B, int32_t *__restrict__ off, F count,
                                int32_t *warp_tot, int32_t *carry)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) *carry = 0;
    __syncthreads();
    for (int64_t base = 0; base < B; base += 1024) {
        const int64_t b = base + tid;
        const int32_t n = b < B ? count(cu[b + 1] - cu[b]) : 0;
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
        const int32_t before = *carry + (warp > 0 ? warp_tot[warp - 1] : 0) + x - n;
        if (b < B) off[b] = before;
        __syncthreads();
        if (tid == 1023) *carry = before + n;
        __syncthreads();
    }
    const int32_t total = *carry;
    if (tid == 0) off[B] = total;
    __syncthreads();
    return total;
}

constexpr int64_t kTableStaged = 4096;  // batches up to this many sequences are ranked by length

__global__ void __launch_bounds__(1024)
chunk_table_kernel(const int32_t *__restrict__ cu, int64_t B, int64_t n_chunk_max, int32_t *__restrict__ chunk_off,
                   int32_t *__restrict__ seq_order, int2 *__restrict__ chunk_info, int32_t ckpt_every,
                   int32_t *__restrict__ ckpt_off, int32_t *__restrict__ status)
{
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry;
    __shared__ int32_t s_cu[kTableStaged + 1], s_off[kTableStaged + 1];
    const int tid = threadIdx.x;
    if (tid == 0) {
        status[0] = 0;
        status[1] = 0;  // the fix-up list of the chunk preparation is empty
        status[2] = 0;  // the fused kernel's next (sequence, head) item
    }
    const int32_t total = block_prefix(
        cu, B, chunk_off, [](int32_t len) { return len > 0 ? (len + C - 1) / C : 0; }, warp_tot, &carry);
    // cu_seqlens[B] > total_tokens (a broken caller precondition) would give more chunks than
    // the workspace holds records for: record it and clamp the offsets, so that no state pass
    // reads a record beyond the workspace.
    if (total > n_chunk_max) {  // uniform: every thread read the same total
        if (tid == 0) *status = 4;
        for (int64_t b = tid; b <= B; b += 1024)
            if (chunk_off[b] > n_chunk_max) chunk_off[b] = static_cast<int32_t>(n_chunk_max);
        __syncthreads();
    }
    if (ckpt_every > 0)  // checkpoints of sequence b: after every ckpt_every tokens, up to its length
        block_prefix(
            cu, B, ckpt_off, [ckpt_every](int32_t len) { return len > 0 ? len / ckpt_every : 0; }, warp_tot, &carry);
    // Small batches: cu_seqlens and the chunk offsets staged in shared memory for the
    // searches below (one parallel read instead of dependent global loads).
    const bool staged = B <= kTableStaged;
    if (staged) {
        for (int64_t b = tid; b <= B; b += 1024) {
            s_cu[b] = cu[b];
            s_off[b] = chunk_off[b];
        }
        __syncthreads();
    }
    auto cu_at = [&](int64_t b) { return staged ? s_cu[b] : cu[b]; };
    auto off_at = [&](int64_t b) { return staged ? s_off[b] : chunk_off[b]; };
    // Per chunk: its first token and length ({0, 0} past the last chunk), so a
    // chunk's CTA finds its rows with one load.
    for (int64_t c = tid; c < n_chunk_max; c += 1024) {
        int2 info = make_int2(0, 0);
        if (c < total) {
            int64_t lo = 0, hi = B - 1;  // the b with chunk_off[b] <= c < chunk_off[b + 1]
            while (lo < hi) {
                const int64_t mid = (lo + hi + 1) / 2;
                if (off_at(mid) <= c) lo = mid;
                else hi = mid - 1;
            }
            const int32_t t0 = cu_at(lo) + static_cast<int32_t>(c - off_at(lo)) * C;
            const int32_t left = cu_at(lo + 1) - t0;
            info = make_int2(t0, left < C ? left : C);
        }
        chunk_info[c] = info;
    }
    // Longest sequences first, so their serial chunk chains start early.
    if (staged) {
        for (int64_t b = tid; b < B; b += 1024) {
            const int32_t lb = s_cu[b + 1] - s_cu[b];
            int32_t rank = 0;
            for (int64_t o = 0; o < B; ++o) {
                const int32_t lo = s_cu[o + 1] - s_cu[o];
                rank += (lo > lb) || (lo == lb && o < b);
            }
            seq_order[rank] = static_cast<int32_t>(b);
        }
    } else {
        for (int64_t b = tid; b < B; b += 1024) seq_order[b] = static_cast<int32_t>(b);
    }
}

// ----------------------------------------------------------- state pass ---


template <int D, typename IO, int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
state_pass_kernel(PassParams p)
{
    using R = Rec<D>;
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
    const int64_t per_seq = H * D * D;
    // element offset of (v = vg0 + gid + 8 hr, k = 8 n + 2 tig) within a state
    auto elem = [&](int n, int hr) {
        return (static_cast<int64_t>(h) * D + vg0 + gid + 8 * hr) * D + 8 * n + 2 * tig;
    };
    auto put_state = [&](void *dst, int32_t dtype, int64_t base) {
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr)
                store_state2(dst, dtype, base + elem(n, hr), make_float2(s[n][2 * hr], s[n][2 * hr + 1]));
    };
    {
        const int64_t base = init_base(p.se, b, per_seq);
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                float2 x = make_float2(0.f, 0.f);
                if (base >= 0) x = load_state2(p.se.init, p.se.init_dtype, base + elem(n, hr));
                s[n][2 * hr] = x.x;
                s[n][2 * hr + 1] = x.y;
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
                const int r = 16 * np + ri + 8 * (mi >> 1), c = 16 * ks + 8 * (mi & 1);
                uint32_t bw[4], bq[4];
                ldmatrix_x4(bw, smem_u32(sb + R::w_at(r, c)));
                ldmatrix_x4(bq, smem_u32(sb + R::qt_at(r, c)));
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
                const uint32_t u1 =
                    *reinterpret_cast<const uint32_t *>(ut + swz_off<128>(vl0 + gid + 8, 8 * n + 2 * tig));
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
                    ldmatrix_x4(ba, smem_u32(sb + R::AQK +
                                             swz_off<128>(16 * tp + ri + 8 * (mi >> 1), 16 * ks + 8 * (mi & 1))));
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
                    ldmatrix_x4_trans(bk, smem_u32(sb + R::KT + tile_off<D, C>(16 * ks + ri + 8 * (mi & 1),
                                                                                 16 * np + 8 * (mi >> 1))));
                    mma_bf16(s[2 * np], va[ks], bk[0], bk[1]);
                    mma_bf16(s[2 * np + 1], va[ks], bk[2], bk[3]);
                }
            }
        }
        __syncthreads();  // every warp is done with this stage
        if (tid == 0 && i + 2 < n_chunks) issue(i + 2, st);
        const int64_t ck = ckpt_slot(p.se, b, i, tok_end - tok_begin);  // S is the state after chunk i
        if (ck >= 0) put_state(p.se.ckpt, p.se.ckpt_dtype, ck * per_seq);
    }

    if (p.se.final_state != nullptr) put_state(p.se.final_state, KDA_F32, b * per_seq);
    const int64_t ob = out_base(p.se, b);
    if (ob >= 0) put_state(p.se.out_cache, p.se.out_dtype, ob);
}

// Warp-pair variant of the state pass for few (sequence, head) pairs: each 16-row value group
// of S^T is held by two warps, one per half of the key channels.  Per chunk the two halves
// are swapped as bf16 fragments through shared memory; warp A (role 0) forms X^T = S^T W^T and
// V_new^T = U^T - X^T, warp B (role 1) forms Y^T = S^T Q~^T and O^T = Y^T + V_new^T A_qk^T, and
// each updates its own half, S^T <- S^T Diag(gamma) + V_new^T K~.  A chunk then costs a warp
// 96 (A) or 116 (B) tensor-core instructions instead of 212, which is what bounds the chunk
// when every warp has a scheduler to itself.
template <int D, typename IO, int PAIRS>
__global__ void __launch_bounds__(PAIRS * 64)
state_pass_pair_kernel(PassParams p)
{
    using R = Rec<D>;
    constexpr int VT = 16 * PAIRS;          // value columns per CTA
    constexpr int NSPLIT = D / VT;
    constexpr int HEAD = R::UT;             // W, Q~, K~, A_qk, gamma
    constexpr int UT_BYTES = VT * C * 2;    // this CTA's rows of U^T
    constexpr int STAGE = HEAD + UT_BYTES;
    constexpr int KH = D / 2;               // key channels per warp
    constexpr int KSH = KH / 16;            // k-steps per half
    constexpr int XS = KSH * 512;           // half of S^T as bf16 A fragments [KSH][32 lanes][16 B]
    constexpr int XV = 4 * 512;             // V_new^T as bf16 A fragments [4][32 lanes][16 B]
    constexpr int XG = 2 * XS + XV;         // exchange bytes per group
    static_assert(NSPLIT * VT == D && KSH >= 1, "value split");
    extern __shared__ __align__(1024) char smem[];
    __shared__ __align__(8) uint64_t bars[2];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gid = lane >> 2, tig = lane & 3, mi = lane >> 3, ri = lane & 7;
    const int grp = warp >> 1, role = warp & 1;  // role = the key half this warp owns
    const int64_t H = p.H;
    const int64_t item = blockIdx.x;
    const int vs = static_cast<int>(item % NSPLIT);
    const int h = static_cast<int>((item / NSPLIT) % H);
    const int64_t b = p.seq_order[item / (NSPLIT * H)];
    const int32_t c_begin = p.chunk_off[b], n_chunks = p.chunk_off[b + 1] - c_begin;
    const int64_t tok_begin = p.cu[b], tok_end = p.cu[b + 1];
    const int vl0 = 16 * grp;               // first value column of this group within the CTA
    const int vg0 = vs * VT + vl0;          // ... within the head
    const int kb = role * KH;               // first key channel of this warp's half
    char *xg = smem + 2 * STAGE + grp * XG;  // this group's exchange area
    IO *sO = reinterpret_cast<IO *>(smem + 2 * STAGE + PAIRS * XG) + grp * (C * 16);
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;\n" ::"r"(1 + grp) : "memory"); };

    // S^T accumulator fragments of this warp's half:
    // s[n][e] = S^T(v = vg0 + gid + 8 (e >> 1), k = kb + 8 n + 2 tig + (e & 1))
    float s[KH / 8][4];
    const int64_t per_seq = H * D * D;
    auto elem = [&](int n, int hr) {
        return (static_cast<int64_t>(h) * D + vg0 + gid + 8 * hr) * D + kb + 8 * n + 2 * tig;
    };
    auto put_state = [&](void *dst, int32_t dtype, int64_t base) {
#pragma unroll
        for (int n = 0; n < KH / 8; ++n)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr)
                store_state2(dst, dtype, base + elem(n, hr), make_float2(s[n][2 * hr], s[n][2 * hr + 1]));
    };
    {
        const int64_t base = init_base(p.se, b, per_seq);
#pragma unroll
        for (int n = 0; n < KH / 8; ++n) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                float2 x = make_float2(0.f, 0.f);
                if (base >= 0) x = load_state2(p.se.init, p.se.init_dtype, base + elem(n, hr));
                s[n][2 * hr] = x.x;
                s[n][2 * hr + 1] = x.y;
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

        // (1) S^T as bf16 A fragments (M = 16 value rows, K = key channels): this warp's half
        //     packed and published, the partner's half read back
        uint32_t slo[KSH][4], shi[KSH][4];  // key steps of the first and second half
        {
            uint32_t own[KSH][4];
#pragma unroll
            for (int ks = 0; ks < KSH; ++ks) {
                own[ks][0] = pack_bf16x2(s[2 * ks][0], s[2 * ks][1]);
                own[ks][1] = pack_bf16x2(s[2 * ks][2], s[2 * ks][3]);
                own[ks][2] = pack_bf16x2(s[2 * ks + 1][0], s[2 * ks + 1][1]);
                own[ks][3] = pack_bf16x2(s[2 * ks + 1][2], s[2 * ks + 1][3]);
                *reinterpret_cast<uint4 *>(xg + role * XS + (ks * 32 + lane) * 16) =
                    make_uint4(own[ks][0], own[ks][1], own[ks][2], own[ks][3]);
            }
            pair_sync();
#pragma unroll
            for (int ks = 0; ks < KSH; ++ks) {
                const uint4 o = *reinterpret_cast<const uint4 *>(xg + (role ^ 1) * XS + (ks * 32 + lane) * 16);
                if (role == 0) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) slo[ks][e] = own[ks][e];
                    shi[ks][0] = o.x; shi[ks][1] = o.y; shi[ks][2] = o.z; shi[ks][3] = o.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) shi[ks][e] = own[ks][e];
                    slo[ks][0] = o.x; slo[ks][1] = o.y; slo[ks][2] = o.z; slo[ks][3] = o.w;
                }
            }
        }
        // (2) role 0: X^T = S^T W^T; role 1: Y^T = S^T Q~^T   (N = 64 chunk rows)
        float x[8][4] = {};
        {
#pragma unroll
            for (int np = 0; np < 4; ++np) {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int r = 16 * np + ri + 8 * (mi >> 1), c = 16 * ks + 8 * (mi & 1);
                    uint32_t bw[4];
                    ldmatrix_x4(bw, smem_u32(sb + (role ? R::qt_at(r, c) : R::w_at(r, c))));
                    const uint32_t *a = ks < KSH ? slo[ks % KSH] : shi[ks % KSH];
                    mma_bf16(x[2 * np], a, bw[0], bw[1]);
                    mma_bf16(x[2 * np + 1], a, bw[2], bw[3]);
                }
            }
        }
        // (3) role 0: V_new^T = U^T - X^T as bf16 A fragments (K = chunk rows), published;
        //     role 1 reads them
        uint32_t va[4][4];
        if (role == 0) {
            const char *ut = sb + HEAD;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const uint32_t u0 = *reinterpret_cast<const uint32_t *>(ut + swz_off<128>(vl0 + gid, 8 * n + 2 * tig));
                const uint32_t u1 =
                    *reinterpret_cast<const uint32_t *>(ut + swz_off<128>(vl0 + gid + 8, 8 * n + 2 * tig));
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
                *reinterpret_cast<uint4 *>(xg + 2 * XS + (ks * 32 + lane) * 16) =
                    make_uint4(va[ks][0], va[ks][1], va[ks][2], va[ks][3]);
            }
        }
        pair_sync();
        if (role == 1) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint4 o = *reinterpret_cast<const uint4 *>(xg + 2 * XS + (ks * 32 + lane) * 16);
                va[ks][0] = o.x; va[ks][1] = o.y; va[ks][2] = o.z; va[ks][3] = o.w;
            }
            // (4) O^T = Y^T + V_new^T A_qk^T   (A_qk causal: chunk row t needs s <= t)
#pragma unroll
            for (int tp = 0; tp < 4; ++tp) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    if (ks <= tp) {
                        uint32_t ba[4];
                        ldmatrix_x4(ba, smem_u32(sb + R::AQK +
                                                 swz_off<128>(16 * tp + ri + 8 * (mi >> 1), 16 * ks + 8 * (mi & 1))));
                        mma_bf16(x[2 * tp], va[ks], ba[0], ba[1]);
                        mma_bf16(x[2 * tp + 1], va[ks], ba[2], ba[3]);
                    }
                }
            }
            // output rows through the group's staging tile [64][16]
#pragma unroll
            for (int n = 0; n < 8; ++n) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = 8 * n + 2 * tig + (e & 1);
                    const int vl = gid + 8 * (e >> 1);
                    sO[t * 16 + vl] = from_f32<IO>(x[n][e]);
                }
            }
            __syncwarp();
            constexpr int PARTS = 16 * static_cast<int>(sizeof(IO)) / 16;  // uint4 per staged row
            const uint4 *src = reinterpret_cast<const uint4 *>(sO);
            for (int e = lane; e < C * PARTS; e += 32) {
                const int t = e / PARTS, part = e % PARTS;
                if (t < len) {
                    IO *dst = out + ((t0 + t) * H + h) * D + vg0;
                    reinterpret_cast<uint4 *>(dst)[part] = src[e];
                }
            }
            __syncwarp();
        }
        // (5) this warp's half: S^T <- S^T Diag(gamma) + V_new^T K~
        {
            const float *gam = reinterpret_cast<const float *>(sb + R::GAMMA) + kb;
#pragma unroll
            for (int n = 0; n < KH / 8; ++n) {
                const float2 gm = *reinterpret_cast<const float2 *>(gam + 8 * n + 2 * tig);
                s[n][0] *= gm.x;
                s[n][1] *= gm.y;
                s[n][2] *= gm.x;
                s[n][3] *= gm.y;
            }
#pragma unroll
            for (int np = 0; np < KH / 16; ++np) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t bk[4];
                    ldmatrix_x4_trans(bk, smem_u32(sb + R::KT + tile_off<D, C>(16 * ks + ri + 8 * (mi & 1),
                                                                                 kb + 16 * np + 8 * (mi >> 1))));
                    mma_bf16(s[2 * np], va[ks], bk[0], bk[1]);
                    mma_bf16(s[2 * np + 1], va[ks], bk[2], bk[3]);
                }
            }
        }
        __syncthreads();  // every warp is done with this stage (and with the exchange area)
        if (tid == 0 && i + 2 < n_chunks) issue(i + 2, st);
        const int64_t ck = ckpt_slot(p.se, b, i, tok_end - tok_begin);  // S is the state after chunk i
        if (ck >= 0) put_state(p.se.ckpt, p.se.ckpt_dtype, ck * per_seq);
    }

    if (p.se.final_state != nullptr) put_state(p.se.final_state, KDA_F32, b * per_seq);
    const int64_t ob = out_base(p.se, b);
    if (ob >= 0) put_state(p.se.out_cache, p.se.out_dtype, ob);
}

// Multiprocessors of the current device (queried once per device; no synchronisation).

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

template <int D, typename IO, int PAIRS>
cudaError_t launch_pair(const PassParams &pp, int64_t items, cudaStream_t st)
{
    constexpr int VT = 16 * PAIRS;
    constexpr int STAGE = Rec<D>::UT + VT * C * 2;
    constexpr int XG = 2 * (D / 32) * 512 + 4 * 512;
    const int smem = 2 * STAGE + PAIRS * XG + PAIRS * C * 16 * static_cast<int>(sizeof(IO));
    auto kern = state_pass_pair_kernel<D, IO, PAIRS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(items * (D / VT)), PAIRS * 64, smem, st>>>(pp);
    return cudaGetLastError();
}


template <int D, typename IO>
cudaError_t launch_typed(const PrefillArgs &a, const PrefillLayout &L, cudaStream_t st)
{
    char *ws = static_cast<char *>(a.workspace);
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    int32_t *chunk_off = reinterpret_cast<int32_t *>(ws + L.off_chunk_off);
    int32_t *seq_order = reinterpret_cast<int32_t *>(ws + L.off_seq_order);
    int2 *chunk_info = reinterpret_cast<int2 *>(ws + L.off_chunk_info);
    int32_t *ckpt_off = reinterpret_cast<int32_t *>(ws + L.off_ckpt_off);
    char *records = ws + L.off_records;
    const int32_t ckpt_every = a.se.ckpt != nullptr ? a.se.ckpt_every : 0;

    auto mark = [&](int i) -> cudaError_t {
        return a.events && a.events[i] ? cudaEventRecord(static_cast<cudaEvent_t>(a.events[i]), st) : cudaSuccess;
    };
    cudaError_t e = mark(0);
    if (e != cudaSuccess) return e;
    chunk_table_kernel<<<1, 1024, 0, st>>>(a.cu_seqlens, a.num_seqs, L.n_chunk_max, chunk_off, seq_order, chunk_info,
                                           ckpt_every, ckpt_off, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if ((e = mark(1)) != cudaSuccess) return e;

    // Head size 128, bf16, and a workspace without room for the records: the fused kernel
    // (chunk preparation and state pass in one persistent CTA per SM, no records in memory).
    if constexpr (D == 128 && sizeof(IO) == 2) {
        if (a.ws_bytes < L.total) {
            StateEnds se = a.se;
            se.ckpt_every = ckpt_every;
            se.ckpt_off = ckpt_off;
            e = prefill::launch_prefill_fused(a.q, a.k, a.v, a.g, a.beta, a.cu_seqlens, seq_order, status, status + 2,
                                              a.num_seqs, a.total_tokens, a.h, a.scale, a.l2norm, se, a.out, st);
            if (e != cudaSuccess) return e;
            if ((e = mark(2)) != cudaSuccess) return e;
            return mark(3);
        }
    }

    prefill::PrepParams pp{a.q, a.k, a.v, a.g, a.beta, chunk_info, a.h, a.scale, a.l2norm, records, status,
                           a.total_tokens, status + 1, reinterpret_cast<int32_t *>(ws + L.off_fix_list), 0};
    StateEnds se = a.se;
    se.ckpt_every = ckpt_every;
    se.ckpt_off = ckpt_off;
    PassParams sp{a.cu_seqlens, chunk_off, seq_order, status, records, a.h, se, a.out};
    const int64_t items = a.num_seqs * a.h;

    // One long sequence with few heads (head size 128, bf16): its chunks in segments of kSegChunks.
    // The value-split state pass of segment s runs on a second stream of the highest priority while
    // segment s + 1 is prepared on the SMs it leaves free; the pass alone would leave most SMs idle
    // for its serial chain.  Events order everything after the caller's stream and back onto it.
    if constexpr (D == 128 && sizeof(IO) == 2) {
        if (L.off_seg_state != 0 && items * prefill::state_pass_split_slices() <= sm_count() &&
            L.n_chunk_max >= 2 * kSegChunks) {
            std::lock_guard<std::mutex> lock(g_seg_mu);
            SegStreams *ss = nullptr;
            if ((e = seg_streams(&ss)) != cudaSuccess) return e;
            sp.seg_state = reinterpret_cast<float *>(ws + L.off_seg_state);
            if ((e = cudaEventRecord(ss->fork, st)) != cudaSuccess) return e;
            if ((e = cudaStreamWaitEvent(ss->aux, ss->fork, 0)) != cudaSuccess) return e;
            for (int64_t lo = 0; lo < L.n_chunk_max; lo += kSegChunks) {
                const int64_t hi = lo + kSegChunks < L.n_chunk_max ? lo + kSegChunks : L.n_chunk_max;
                pp.chunk_base = lo;
                if ((e = prefill::launch_chunk_prep(D, a.io_dtype, pp, hi - lo, a.h, st)) != cudaSuccess) return e;
                if ((e = cudaMemsetAsync(status + 1, 0, sizeof(int32_t), st)) != cudaSuccess) return e;  // fix-up list
                if ((e = cudaEventRecord(ss->seg, st)) != cudaSuccess) return e;
                if ((e = cudaStreamWaitEvent(ss->aux, ss->seg, 0)) != cudaSuccess) return e;
                sp.seg_lo = static_cast<int32_t>(lo);
                sp.seg_hi = hi < L.n_chunk_max ? static_cast<int32_t>(hi) : 0x7fffffff;
                if ((e = prefill::launch_state_pass_split(sp, items, ss->aux)) != cudaSuccess) return e;
            }
            if ((e = mark(2)) != cudaSuccess) return e;  // every segment prepared
            if ((e = cudaEventRecord(ss->join, ss->aux)) != cudaSuccess) return e;
            if ((e = cudaStreamWaitEvent(st, ss->join, 0)) != cudaSuccess) return e;
            return mark(3);
        }
    }

    if (L.n_chunk_max > 0) {
        e = prefill::launch_chunk_prep(D, a.io_dtype, pp, L.n_chunk_max, a.h, st);
        if (e != cudaSuccess) return e;
    }

    if ((e = mark(2)) != cudaSuccess) return e;
    // Enough CTAs to cover the SMs: split the value columns when there are few
    // (sequence, head) pairs.  Columns of S evolve independently.
    int warps = D / 16;
    while (warps > 1 && items * (D / (16 * warps)) < 120) warps /= 2;
    if constexpr (D == 128 && sizeof(IO) == 2) {  // the tensor-memory state passes
        // value columns split over CTAs while the split fits one wave, else one CTA per (sequence, head)
        e = items * prefill::state_pass_split_slices() <= sm_count() ? prefill::launch_state_pass_split(sp, items, st)
                                                                    : prefill::launch_state_pass_tc(sp, items, st);
        if (e != cudaSuccess) return e;
        return mark(3);
    } else if constexpr (D == 128) {  // fp32: at most two 16-column groups per CTA: two warps per group
        if (warps == 8) e = launch_pass<D, IO, 8>(sp, items, st);
        else if (warps == 4) e = launch_pass<D, IO, 4>(sp, items, st);
        else if (warps == 2) e = launch_pair<D, IO, 2>(sp, items, st);
        else e = launch_pair<D, IO, 1>(sp, items, st);
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
    const int rb = prefill::rec_bytes_for(d);
    if (rb == 0 || total_tokens < 0 || num_seqs < 1 || h < 1) return false;
    auto up = [](size_t x, size_t a) { return (x + a - 1) / a * a; };
    PrefillLayout L{};
    L.n_chunk_max = (total_tokens + (C - 1) * num_seqs) / C;  // >= sum of ceil(len / C)
    L.rec_bytes = static_cast<size_t>(rb);
    L.off_chunk_off = 256;
    L.off_seq_order = up(L.off_chunk_off + 4 * static_cast<size_t>(num_seqs + 1), 256);
    L.off_chunk_info = up(L.off_seq_order + 4 * static_cast<size_t>(num_seqs), 256);
    L.off_ckpt_off = up(L.off_chunk_info + 8 * static_cast<size_t>(L.n_chunk_max), 256);
    L.off_fix_list = up(L.off_ckpt_off + 4 * static_cast<size_t>(num_seqs + 1), 256);
    L.compact = L.off_fix_list;
    L.off_records = up(L.off_fix_list + 4 * static_cast<size_t>(L.n_chunk_max) * static_cast<size_t>(h), 1024);
    L.total = L.off_records + static_cast<size_t>(L.n_chunk_max) * static_cast<size_t>(h) * L.rec_bytes;
    if (num_seqs == 1 && d == 128) {  // the segmented prefill of one sequence keeps its state here between segments
        L.off_seg_state = up(L.total, 256);
        L.total = L.off_seg_state + static_cast<size_t>(h) * d * d * 4;
    }
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
