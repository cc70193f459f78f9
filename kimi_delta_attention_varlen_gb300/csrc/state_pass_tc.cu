// Inter-chunk state pass on the 5th-generation tensor cores (tcgen05, TMEM),
// for head size 128 with bf16 output: one CTA of 512 threads per (sequence,
// head), walking the sequence's chunks in order.
//
// Per chunk, with S the K x V state and the chunk's record (W, Q~, K~, A_qk,
// gamma, U^T) in shared memory:
//   X^T = S^T W^T,  Y^T = S^T Q~^T                    (M = 128 value rows, N = 64)
//   V_new^T = U^T - X^T                               (threads, one value row each)
//   O^T = Y^T + V_new^T A_qk^T,  S^T <- S^T diag(gamma) + V_new^T K~   (N = 64, 128)
// which is the chunkwise form of S_t = (I - beta k k^T) Diag(e^g) S + beta k v^T,
// o_t = scale S^T q of the "KDA's challenges for AI infra" page (section 1.1),
// in the order of the "Support Kimi-K3 on NPU" report's extend listing.
//
// Layout: S^T (fp32, 128 lanes x 128 columns), X^T (64 columns) and two
// Y^T/O^T buffers (64 columns each) live in tensor memory.  Value row v is TMEM
// lane v; four warps share each 32-lane quadrant and split its columns.  The
// A operands of the MMAs, S^T and V_new^T in bf16, are written by the threads
// into tensor memory too (two values per column), so the tensor cores read only
// the B operands from shared memory: W, Q~, A_qk (K-major) and K~ (MN-major),
// straight from the bulk-copied record in the 128-byte-swizzle layout.  One
// thread issues the MMAs;
// mbarriers signal their completion.  Records are double-buffered: the copy of
// chunk i + 1 starts in chunk i once chunk i - 1's MMAs are done, and each copy
// prefetches the record kTcAhead chunks further on into L2.  The outputs of chunk
// i - 1 move from tensor memory to a staging tile while the first MMA group of
// chunk i runs and from there to global memory while the second group runs, so
// neither half waits on a barrier of its own.  Every wait is bounded; an
// expired wait sets the workspace status word and the CTA stops waiting (and
// still frees its TMEM).
#include "prefill_common.cuh"
#include "tcgen05.cuh"

namespace kda {
namespace prefill {
namespace {

constexpr int kTcCompute = 512;                // sixteen warps
constexpr int kTcThreads = kTcCompute;
constexpr int kTcParts = kTcCompute / 128;   // warps sharing one 32-lane TMEM quadrant
constexpr int kTcSCols = 128 / kTcParts;     // S^T columns per thread
constexpr int kTcYCols = 64 / kTcParts;      // X^T / Y^T columns per thread
constexpr uint32_t kTcWaitLimit = 1u << 22;
constexpr int kTcAhead = 2;                     // records prefetched into L2 beyond the two stages
constexpr int kTcD = 128;
using RT = Rec<kTcD>;
constexpr int kStage = (RT::BYTES + 1023) / 1024 * 1024;  // one record, padded to 1 KiB
constexpr int kOS = 2 * kStage;          // output staging bf16 [64 tokens][128 values]
constexpr int kTcSmem = kOS + 16384 + 1024;  // + slack to align the base to 1 KiB
// Tensor memory: S^T fp32 (128 columns), two [X^T | Y^T] buffers (128 columns each: X^T, then
// Y^T / O^T), and the MMAs' A operands in bf16, two values per 32-bit column: S^T (64 columns)
// and V_new^T (32).
constexpr uint32_t kColS = 0, kColXY = 128, kColA = 384, kColV = 448, kTmemCols = 512;

__device__ __forceinline__ void compute_sync()  // the compute warps (named barrier 1)
{
    asm volatile("bar.sync 1, %0;\n" ::"n"(kTcCompute) : "memory");
}

// 2n fp32 values (as bits) -> n bf16 pairs
template <int N> __device__ __forceinline__ void pack_pairs(const uint32_t *r, uint32_t (&p)[N])
{
#pragma unroll
    for (int e = 0; e < N; ++e) p[e] = pack_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
}

// N (32 or 16) consecutive TMEM columns of this thread's lane
template <int N> __device__ __forceinline__ void ld_cols(uint32_t t, uint32_t (&r)[N])
{
    if constexpr (N == 32) tc::ld32(t, r);
    else tc::ld16(t, r);
}

__global__ void __launch_bounds__(kTcThreads, 1)
state_pass_tc_kernel(PassParams p)
{
    extern __shared__ char smem_raw[];
    char *smem = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // two record stages; X|Y done, S done, O done per stage
    __shared__ __align__(8) uint64_t bars[6];
    __shared__ uint32_t tmem_base;
    uint64_t *const bar_xy = &bars[2], *const bar_s = &bars[3], *const bar_o = &bars[4];

    const int tid = threadIdx.x, warp = tid >> 5;
    const int quad = warp & 3, part = (warp >> 2) & 3;  // TMEM lane quadrant; which part of the columns
    const int v = 32 * quad + (tid & 31);          // value row = TMEM lane
    const int64_t H = p.H;
    const int64_t item = blockIdx.x;
    const int h = static_cast<int>(item % H);
    const int64_t b = p.seq_order[item / H];
    const int32_t c_begin = p.chunk_off[b], n_chunks = p.chunk_off[b + 1] - c_begin;
    const int64_t tok_begin = p.cu[b], tok_end = p.cu[b + 1];

    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        for (int j = 0; j < 6; ++j) mbar_init(&bars[j], 1);
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base;

    // record of chunk i -> stage i & 1 (thread 0); records kTcAhead chunks further on -> L2
    auto issue = [&](int32_t i) {
        if (i < n_chunks) {
            const char *rec = p.records + (static_cast<int64_t>(c_begin + i) * H + h) * RT::BYTES;
            mbar_arrive_expect_tx(&bars[i & 1], RT::BYTES);
            bulk_g2s(smem + (i & 1) * kStage, rec, RT::BYTES, &bars[i & 1]);
        }
        if (i + kTcAhead < n_chunks)
            prefetch_l2(p.records + (static_cast<int64_t>(c_begin + i + kTcAhead) * H + h) * RT::BYTES, RT::BYTES);
    };
    if (tid == 0) {
        issue(0);
        issue(1);
    }
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * quad) << 16);  // this warp's lanes

    const int64_t row_v = (static_cast<int64_t>(h) * kTcD + v) * kTcD;  // element offset of [v][0] within a state
    // 32 consecutive fp32 values of S^T row v (columns c0 ...) -> a state buffer, with its dtype's cast
    auto put_row = [&](void *dst, int32_t dtype, int64_t base, int c0, const uint32_t r[32]) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
            store_state4(dst, dtype, base + row_v + c0 + e,
                         make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                                     __uint_as_float(r[e + 3])));
    };

    // initial state: this thread's columns of S^T row v (= cache row [v][k])
    {
        const int64_t base = init_base(p.se, b, H * kTcD * kTcD);
#pragma unroll
        for (int j = 0; j < kTcSCols / 32; ++j) {
            const int c0 = kTcSCols * part + 32 * j;
            uint32_t r[32];
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (base >= 0) x = load_state4(p.se.init, p.se.init_dtype, base + row_v + c0 + e);
                r[e] = __float_as_uint(x.x);
                r[e + 1] = __float_as_uint(x.y);
                r[e + 2] = __float_as_uint(x.z);
                r[e + 3] = __float_as_uint(x.w);
            }
            tc::st32(tl + kColS + c0, r);
        }
        tc::wait_st();
    }

    constexpr uint32_t kIdN64 = tc::idesc_bf16(128, 64, false);
    constexpr uint32_t kIdN128 = tc::idesc_bf16(128, 128, false);
    constexpr uint32_t kIdN128Mn = tc::idesc_bf16(128, 128, true);
    uint32_t phase_xy = 0, phase_s = 0;
    bool gave_up = false;
    auto wait_bar = [&](uint64_t *bar, uint32_t parity) {
        if (!gave_up && !mbar_wait(bar, parity, kTcWaitLimit)) {
            gave_up = true;
            if ((tid & 31) == 0) atomicExch(p.status, 2);
        }
    };
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);

    // Outputs of chunk c (O^T in the Y half of buffer c & 1): TMEM -> staging [t][v] once the O
    // MMAs have completed (stage_outputs), then, after a barrier of the compute warps, whole
    // output rows from the staging to global memory (store_outputs).
    __nv_bfloat16 *os = reinterpret_cast<__nv_bfloat16 *>(smem + kOS);
    auto stage_outputs = [&](int32_t c) {
        wait_bar(&bar_o[c & 1], (c >> 1) & 1);
        tc::fence_after_sync();
        uint32_t y[kTcYCols];
        ld_cols(tl + kColXY + 128 * (c & 1) + 64 + kTcYCols * part, y);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < kTcYCols; ++e)
            os[(kTcYCols * part + e) * kTcD + v] = __float2bfloat16_rn(__uint_as_float(y[e]));
    };
    auto store_outputs = [&](int32_t c) {
        const int64_t t0 = tok_begin + static_cast<int64_t>(c) * C;
        const int len = static_cast<int>(tok_end - t0 < C ? tok_end - t0 : C);
        const uint4 *src = reinterpret_cast<const uint4 *>(os);
#pragma unroll
        for (int e = tid; e < C * (kTcD * 2 / 16); e += kTcCompute) {
            const int t = e >> 4, part = e & 15;
            if (t < len) reinterpret_cast<uint4 *>(out + ((t0 + t) * H + h) * kTcD)[part] = src[e];
        }
    };

    for (int32_t i = 0; i < n_chunks; ++i) {
        const int st = i & 1;
        wait_bar(&bars[st], (i >> 1) & 1);
        const char *sb = smem + st * kStage;
        const float4 *gam4 = reinterpret_cast<const float4 *>(sb + RT::GAMMA);
        const uint32_t xy = kColXY + 128 * static_cast<uint32_t>(st);

        // S is now the state after chunk i - 1: a checkpoint when that chunk ends on one.
        if (p.se.ckpt != nullptr && i > 0) {
            const int64_t ck = ckpt_slot(p.se, b, i - 1, tok_end - tok_begin);
            if (ck >= 0) {
#pragma unroll 1
                for (int j = 0; j < kTcSCols / 32; ++j) {
                    const int c0 = kTcSCols * part + 32 * j;
                    uint32_t r[32];
                    tc::ld32(tl + kColS + c0, r);
                    tc::wait_ld();
                    put_row(p.se.ckpt, p.se.ckpt_dtype, ck * H * kTcD * kTcD, c0, r);
                }
            }
        }
        // (A) S^T row v, this warp's 64 columns -> bf16 operand (undecayed); decay the TMEM copy by gamma
#pragma unroll
        for (int j = 0; j < kTcSCols / 32; ++j) {
            const int c0 = kTcSCols * part + 32 * j;
            uint32_t r[32];
            tc::ld32(tl + kColS + c0, r);
            tc::wait_ld();
            {
                uint32_t a[16];
                pack_pairs(r, a);
                tc::st16(tl + kColA + c0 / 2, a);
            }
#pragma unroll
            for (int e = 0; e < 32; e += 4) {  // channel pairs through the packed fp32x2 multiply
                const float4 gv = gam4[(c0 + e) >> 2];
                const float2 a = mul2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])),
                                      make_float2(gv.x, gv.y));
                const float2 b2 = mul2(make_float2(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3])),
                                       make_float2(gv.z, gv.w));
                r[e] = __float_as_uint(a.x);
                r[e + 1] = __float_as_uint(a.y);
                r[e + 2] = __float_as_uint(b2.x);
                r[e + 3] = __float_as_uint(b2.y);
            }
            tc::st32(tl + kColS + c0, r);
        }
        tc::wait_st();
        tc::fence_before_sync();
        compute_sync();
        tc::fence_after_sync();

        // (B) [X^T | Y^T] = S^T [W; Q~]^T: M = 128, N = 128 (W rows, then Q~ rows), K = 128 in 8 steps
        if (tid == 0) {
            const uint32_t wq = smem_u32(sb + RT::WQ);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_bf16_ts(tmem + xy, tmem + kColA + 8 * ks,
                                tc::sdesc_sw128(wq + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024), kIdN128,
                                ks > 0 ? 1u : 0u);
            tc::commit(bar_xy);
        }
        __syncwarp();
        if (i > 0) {
            stage_outputs(i - 1);  // the previous chunk's outputs into the staging, while these MMAs run
            // every read of chunk i - 1's stage is over (its O products have completed): chunk i + 1
            if (tid == 0) issue(i + 1);
        }
        wait_bar(bar_xy, phase_xy);
        phase_xy ^= 1u;
        tc::fence_after_sync();

        // (C) V_new^T row v, this thread's 16 token columns = U^T - X^T -> bf16 operand in tensor memory
        {
            uint32_t x[kTcYCols];
            ld_cols(tl + xy + kTcYCols * part, x);
            tc::wait_ld();
            const char *ut = sb + RT::UT;
            uint32_t w[kTcYCols / 2];
#pragma unroll
            for (int q = 0; q < kTcYCols / 8; ++q) {
                const uint4 u = *reinterpret_cast<const uint4 *>(ut + swz_off<128>(v, kTcYCols * part + 8 * q));
                const uint32_t *xx = x + 8 * q;
                w[4 * q] = pack_bf16x2(bf16_lo(u.x) - __uint_as_float(xx[0]), bf16_hi(u.x) - __uint_as_float(xx[1]));
                w[4 * q + 1] = pack_bf16x2(bf16_lo(u.y) - __uint_as_float(xx[2]), bf16_hi(u.y) - __uint_as_float(xx[3]));
                w[4 * q + 2] = pack_bf16x2(bf16_lo(u.z) - __uint_as_float(xx[4]), bf16_hi(u.z) - __uint_as_float(xx[5]));
                w[4 * q + 3] = pack_bf16x2(bf16_lo(u.w) - __uint_as_float(xx[6]), bf16_hi(u.w) - __uint_as_float(xx[7]));
            }
            tc::st8(tl + kColV + (kTcYCols * part) / 2, w);
            tc::wait_st();
        }
        tc::fence_before_sync();
        compute_sync();
        tc::fence_after_sync();

        // (D) S^T += V_new^T K~ (N = 128, K~ MN-major; committed alone: the next chunk waits for it),
        // then O^T = Y^T + V_new^T A_qk^T (N = 64); K = 64.  This stage is refilled in the next chunk
        // once the O MMAs have completed (gamma in A and U^T in C were read before the barrier above).
        if (tid == 0) {
            const uint32_t aq = smem_u32(sb + RT::AQK), kt = smem_u32(sb + RT::KT);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_bf16_ts(tmem + kColS, tmem + kColV + 8 * ks, tc::sdesc_sw128(kt + ks * 2048, 8192, 1024),
                                kIdN128Mn, 1u);
            tc::commit(bar_s);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_bf16_ts(tmem + xy + 64, tmem + kColV + 8 * ks, tc::sdesc_sw128(aq + ks * 32, 16, 1024),
                                kIdN64, 1u);
            tc::commit(&bar_o[st]);
        }
        __syncwarp();
        if (i > 0) store_outputs(i - 1);  // staged before the barrier above; stored while these MMAs run
        wait_bar(bar_s, phase_s);
        phase_s ^= 1u;
        tc::fence_after_sync();
    }
    if (gave_up && tid == 0)  // copies still in flight land before the CTA exits
        for (int32_t i = n_chunks > 2 ? n_chunks - 2 : 0; i < n_chunks; ++i) mbar_wait(&bars[i & 1], (i >> 1) & 1, kTcWaitLimit);
    if (n_chunks > 0) {
        compute_sync();  // the staging's last rows (chunk n - 2) have been stored
        stage_outputs(n_chunks - 1);
        compute_sync();
        store_outputs(n_chunks - 1);
    }

    // final state -> packed fp32, the cache row out_idx[b], and the last checkpoint if it ends there
    {
        const int64_t per_seq = H * kTcD * kTcD;
        const int64_t ob = out_base(p.se, b);
        const int64_t ck = n_chunks > 0 ? ckpt_slot(p.se, b, n_chunks - 1, tok_end - tok_begin) : -1;
        if (p.se.final_state != nullptr || ob >= 0 || ck >= 0) {
#pragma unroll
            for (int j = 0; j < kTcSCols / 32; ++j) {
                const int c0 = kTcSCols * part + 32 * j;
                uint32_t r[32];
                tc::ld32(tl + kColS + c0, r);
                tc::wait_ld();
                if (p.se.final_state != nullptr) put_row(p.se.final_state, KDA_F32, b * per_seq, c0, r);
                if (ob >= 0) put_row(p.se.out_cache, p.se.out_dtype, ob, c0, r);
                if (ck >= 0) put_row(p.se.ckpt, p.se.ckpt_dtype, ck * per_seq, c0, r);
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_state_pass_tc(const PassParams &p, int64_t items, cudaStream_t st)
{
    cudaError_t e = cudaFuncSetAttribute(state_pass_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (e != cudaSuccess) return e;
    state_pass_tc_kernel<<<static_cast<unsigned>(items), kTcThreads, kTcSmem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace prefill
}  // namespace kda
