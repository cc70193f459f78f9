// Inter-chunk state pass on the tensor cores for few (sequence, head) pairs:
// head size 128, bf16 output, the value columns of each state split over two
// CTAs (64 columns each), so a batch of one long sequence still spreads over
// twice as many SMs as it has heads.  Columns of S evolve independently: the
// recurrence S_t = (I - beta k k^T) Diag(e^g) S + beta k v^T of the "KDA's
// challenges for AI infra" page (section 1.1) multiplies S from the left only,
// and its chunkwise form in the "Support Kimi-K3 on NPU" report's extend
// listing keeps that property:
//   [-V_new; Y] = [-I; 0] U + [W; Q~] S     (M = 128: 64 rows of each, N = 64 columns, K = 64 + 128)
//   S <- diag(gamma) S + K~^T V_new,  O = Y + A_qk V_new    (K = 64 tokens)
//
// Layout.  S (fp32, 128 key lanes x 64 columns) lives in tensor memory with the
// key as the lane, so the decay diag(gamma) is one scalar per thread; three
// [-V_new; Y] buffers (-V_new in lanes 0..63, Y / O in lanes 64..127) and the
// constant A operand [-I; 0] (bf16, 128 lanes x 64) sit beside it.  U enters
// through that identity product (its B operand is this CTA's half of the
// record's U^T, K-major), so the threads only negate and round -V_new.  The B
// operands S and V_new in bf16 are written by the threads into shared memory
// as 64-column MN-major tiles in the 128-byte-swizzle layout; the other A
// operands come straight from the bulk-copied record: [W; Q~] and A_qk
// K-major, K~ MN-major (as K~^T).  The O product takes M = 128 rows of which
// A_qk is the second half, so that it lands on Y's lanes: its first 64 rows are
// the 8 KB of the record before A_qk, and they add into -V_new's lanes after
// those have been read.
//
// Threads: eight compute warps (warp w serves TMEM lanes 32 (w % 4) ... and
// columns 32 (w / 4) ... of the slice), an MMA warp and a copy warp.  The
// compute warps signal the MMA warp through named barriers (operands written)
// and never issue or wait on an MMA issue themselves; mbarriers signal
// [-V_new; Y] (to the V_new step), S (to the next chunk) and O (to the output
// rows and the copy warp).  Records are triple-buffered, and each CTA copies
// only its half of U^T (prefetching later records into L2 as well made the
// pass 3 % slower).  The warps of lanes 0..63 form V_new while those of lanes
// 64..127 move the previous chunk's output rows out of tensor memory.  A launch
// may cover one segment of every sequence's chunks (the segmented prefill of one
// long sequence): a segment after the first starts from the fp32 state the
// previous one left in the workspace, one before the last ends in it.  Every
// wait is bounded; an expired wait sets the workspace status word and the CTA
// stops waiting, waits (bounded) for its own copies in flight, and still frees
// its TMEM.
#include "prefill_common.cuh"
#include "tcgen05.cuh"

namespace kda {
namespace prefill {
namespace {

constexpr int kSpD = 128;
constexpr int kSpNV = 64;                          // value columns per CTA
constexpr int kSpSlices = kSpD / kSpNV;
constexpr int kSpCompute = 256;                    // eight compute warps
constexpr int kSpMmaWarp = kSpCompute / 32;        // then the MMA warp ...
constexpr int kSpCopyWarp = kSpMmaWarp + 1;        // ... and the copy warp
constexpr int kSpThreads = kSpCompute + 64;
constexpr uint32_t kSpWaitLimit = 1u << 22;
using RS = Rec<kSpD>;
constexpr int kSpStages = 3;
constexpr int kSpMain = RS::UT;                    // [W; Q~], K~, A_qk, gamma
constexpr int kSpUt = kSpNV * C * 2;               // this CTA's rows of U^T
constexpr int kSpUtOff = (kSpMain + 1023) / 1024 * 1024;  // U^T rows at a swizzle-atom boundary
constexpr int kSpStage = kSpUtOff + kSpUt;
constexpr int kSpSop = kSpStages * kSpStage;       // S bf16 [128 keys][64 columns], MN-major
constexpr int kSpVop = kSpSop + kSpD * 128;        // V_new bf16 [64 tokens][64 columns], MN-major
constexpr int kSpSmem = kSpVop + C * 128 + 1024;   // + slack to align the base to 1 KiB
static_assert(kSpSmem + 256 <= 227 * 1024, "shared memory");
// Tensor memory: S (64 columns), three [-V_new; Y] buffers (64 columns each), [-I; 0] (32 columns)
constexpr uint32_t kSpColS = 0, kSpColXY = 64, kSpColI = 256, kSpTmemCols = 512;
constexpr int kSpBufs = 3;
// The O product's A operand starts 64 rows (8 KB) before A_qk, inside the record.
static_assert(RS::AQK >= C * 128 && kSpMain % 16 == 0 && kSpStage % 1024 == 0, "record layout");
// named barriers: the compute warps arrive, the MMA warp waits
constexpr int kBarOperandsS = 2, kBarOperandsV = 3, kBarCount = kSpCompute + 32;

__host__ __device__ constexpr uint32_t sp_idesc(bool a_mn, bool b_mn)  // M = 128, N = 64, bf16 -> fp32
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(kSpNV >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
}

__device__ __forceinline__ void named_arrive(int id)
{
    asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "n"(kBarCount) : "memory");
}
__device__ __forceinline__ void named_sync(int id)
{
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "n"(kBarCount) : "memory");
}

__device__ __forceinline__ float load_state1(const void *base, int32_t dtype, int64_t e)
{
    if (dtype == KDA_F32) return static_cast<const float *>(base)[e];
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t *>(base)[e]) << 16);
}

__device__ __forceinline__ void store_state1(void *base, int32_t dtype, int64_t e, float x)
{
    if (dtype == KDA_F32) static_cast<float *>(base)[e] = x;
    else static_cast<__nv_bfloat16 *>(base)[e] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ uint4 pack8_bits(const uint32_t *r)
{
    return make_uint4(pack_bf16x2(__uint_as_float(r[0]), __uint_as_float(r[1])),
                      pack_bf16x2(__uint_as_float(r[2]), __uint_as_float(r[3])),
                      pack_bf16x2(__uint_as_float(r[4]), __uint_as_float(r[5])),
                      pack_bf16x2(__uint_as_float(r[6]), __uint_as_float(r[7])));
}

__global__ void __launch_bounds__(kSpThreads, 1)
state_pass_split_kernel(PassParams p)
{
    extern __shared__ char smem_raw[];
    char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    // record stages; [X; Y] done; S done; O done per stage
    __shared__ __align__(8) uint64_t bars[2 * kSpStages + 2];
    __shared__ uint32_t tmem_base;
    uint64_t *const bar_x = &bars[kSpStages], *const bar_s = &bars[kSpStages + 1], *const bar_o = &bars[kSpStages + 2];

    const int tid = threadIdx.x, warp = tid >> 5;
    const int quad = warp & 3, part = (warp >> 2) & 1;
    const int lane = 32 * quad + (tid & 31);        // key (S), token (X) or 64 + token (Y) of this thread
    const int64_t H = p.H;
    const int64_t item = blockIdx.x / kSpSlices;
    const int slice = static_cast<int>(blockIdx.x % kSpSlices);
    const int v0 = kSpNV * slice + 32 * part;       // this thread's 32 columns
    const int h = static_cast<int>(item % H);
    const int64_t b = p.seq_order[item / H];
    // this launch's chunks of the sequence: the segment [seg_lo, seg_hi) of its n_all chunks
    const int32_t n_all = p.chunk_off[b + 1] - p.chunk_off[b];
    const int32_t c_lo = p.seg_lo > 0 ? p.seg_lo : 0, c_hi = p.seg_hi < n_all ? p.seg_hi : n_all;
    const int32_t n_chunks = c_hi > c_lo ? c_hi - c_lo : 0;
    if (n_chunks == 0 && (n_all > 0 || c_lo > 0)) return;  // nothing of this sequence here (uniform over the CTA)
    const bool first = c_lo == 0, last = c_hi >= n_all;     // the segment starts / ends the sequence
    const int32_t c_begin = p.chunk_off[b] + c_lo;          // record index of the segment's first chunk
    const int64_t tok_seq = p.cu[b], tok_end = p.cu[b + 1];
    const int64_t tok_begin = tok_seq + static_cast<int64_t>(c_lo) * C;  // first token of the segment

    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, kSpTmemCols);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        for (int j = 0; j < 2 * kSpStages + 2; ++j) mbar_init(&bars[j], 1);
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base;
    if (warp < kSpMmaWarp) {  // [-I; 0]: lane t < 64 holds -1 at K = t (column t / 2, the high half for odd t)
        uint32_t id[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            id[j] = (lane < C && (lane >> 1) == 16 * part + j) ? ((lane & 1) ? 0xBF800000u : 0x0000BF80u) : 0u;
        tc::st16(tmem + (static_cast<uint32_t>(32 * quad) << 16) + kSpColI + 16 * part, id);
        tc::wait_st();
    }
    tc::fence_before_sync();
    __syncthreads();  // the MMA warp reads [-I; 0] from here on
    tc::fence_after_sync();
    constexpr uint32_t kIdKB = sp_idesc(false, true);   // A K-major ([W; Q~], A_qk), B MN-major
    constexpr uint32_t kIdMB = sp_idesc(true, true);    // A MN-major (K~^T), B MN-major
    const uint32_t sop_a = smem_u32(smem + kSpSop), vop_a = smem_u32(smem + kSpVop);

    if (warp == kSpCopyWarp) {  // ---- records: chunk i -> stage i % 3, refilled once chunk i's O products complete
        if ((tid & 31) == 0) {
            auto issue = [&](int32_t i) {
                const char *rec = p.records + (static_cast<int64_t>(c_begin + i) * H + h) * RS::BYTES;
                char *dst = smem + (i % kSpStages) * kSpStage;
                uint64_t *bar = &bars[i % kSpStages];
                mbar_arrive_expect_tx(bar, kSpMain + kSpUt);
                bulk_g2s(dst, rec, kSpMain, bar);
                bulk_g2s(dst + kSpUtOff, rec + RS::UT + slice * kSpUt, kSpUt, bar);
            };
            int32_t last = -1;
            for (int32_t i = 0; i < n_chunks && i < kSpStages; ++i) issue(last = i);
            for (int32_t i = 0; i + kSpStages < n_chunks; ++i) {
                if (!mbar_wait(&bar_o[i % kSpStages], (i / kSpStages) & 1, kSpWaitLimit)) {
                    atomicExch(p.status, 2);
                    break;
                }
                issue(last = i + kSpStages);
            }
            // every copy this CTA issued has landed before it exits
            for (int32_t i = last; i >= 0 && i > last - kSpStages; --i)
                if (!mbar_wait(&bars[i % kSpStages], (i / kSpStages) & 1, kSpWaitLimit)) atomicExch(p.status, 2);
        }
        __syncwarp();
        __syncthreads();
        return;
    }
    if (warp == kSpMmaWarp) {  // ---- MMAs, issued by one thread once the compute warps' operands are written
        constexpr uint32_t kIdKK = sp_idesc(false, false);  // A K-major ([-I; 0] in TMEM), B K-major (U^T)
        bool failed = false;
        // [-V_new; Y] of chunk c starts as [-I; 0] U (c's record landed), before its S is known
        auto issue_u = [&](int32_t c) {
            if (!failed && !mbar_wait(&bars[c % kSpStages], (c / kSpStages) & 1, kSpWaitLimit)) {
                failed = true;
                atomicExch(p.status, 2);
            }
            const uint32_t ut = smem_u32(smem + (c % kSpStages) * kSpStage + kSpUtOff);
            const uint32_t xy = kSpColXY + 64 * static_cast<uint32_t>(c % kSpBufs);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_bf16_ts(tmem + xy, tmem + kSpColI + 8 * ks, tc::sdesc_sw128(ut + ks * 32, 16, 1024), kIdKK,
                                ks > 0 ? 1u : 0u);
        };
        if ((tid & 31) == 0 && n_chunks > 0) issue_u(0);
        __syncwarp();
        bool u_next = false;  // chunk i + 1's U product issued
        for (int32_t i = 0; i < n_chunks; ++i) {
            const char *sb = smem + (i % kSpStages) * kSpStage;
            const uint32_t xy = kSpColXY + 64 * static_cast<uint32_t>(i % kSpBufs);
            named_sync(kBarOperandsS);
            tc::fence_after_sync();
            if ((tid & 31) == 0) {  // += [W; Q~] S, K = 128 keys; the commit also covers the previous O products
                const uint32_t wq = smem_u32(sb + RS::WQ);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_bf16(tmem + xy, tc::sdesc_sw128(wq + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                 tc::sdesc_sw128(sop_a + ks * 2048, 8192, 1024), kIdKB, 1u);
                tc::commit(bar_x);
                // chunk i + 1's U product fills the tensor cores while the threads form V_new, if its
                // record has landed (else it follows the O products)
                const int32_t c = i + 1;
                u_next = c < n_chunks && mbar_test(&bars[c % kSpStages], (c / kSpStages) & 1);
                if (u_next) issue_u(c);
            }
            __syncwarp();
            named_sync(kBarOperandsV);
            tc::fence_after_sync();
            if ((tid & 31) == 0) {
                // S += K~^T V_new (committed alone: the next chunk waits for it), then O = Y + A_qk V_new
                // (A from 8 KB before A_qk: A_qk is rows 64..127, on Y's lanes); K = 64.  The next chunk's
                // U product goes to the buffer of chunk i - 2, whose outputs were stored during chunk i - 1.
                const uint32_t aq = smem_u32(sb + RS::AQK), kt = smem_u32(sb + RS::KT);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + kSpColS, tc::sdesc_sw128(kt + ks * 2048, 8192, 1024),
                                 tc::sdesc_sw128(vop_a + ks * 2048, 8192, 1024), kIdMB, 1u);
                tc::commit(bar_s);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + xy, tc::sdesc_sw128(aq - C * 128 + ks * 32, 16, 1024),
                                 tc::sdesc_sw128(vop_a + ks * 2048, 8192, 1024), kIdKB, 1u);
                tc::commit(&bar_o[i % kSpStages]);
                if (i + 1 < n_chunks && !u_next) issue_u(i + 1);
            }
            __syncwarp();
        }
        __syncthreads();
        return;
    }

    // ---- compute warps ----
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * quad) << 16);  // this warp's lanes
    // element offset of state row [h][v][k] for this thread's key k = lane and column v
    auto srow = [&](int v) { return (static_cast<int64_t>(h) * kSpD + v) * kSpD + lane; };

    // initial state: S[k][v0 ... v0 + 31] for key k = lane (after the first segment: the previous one's end)
    {
        const void *src = first ? p.se.init : p.seg_state;
        const int32_t dtype = first ? p.se.init_dtype : KDA_F32;
        const int64_t base = first ? init_base(p.se, b, H * kSpD * kSpD) : b * H * kSpD * kSpD;
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
            r[j] = __float_as_uint(base >= 0 ? load_state1(src, dtype, base + srow(v0 + j)) : 0.f);
        tc::st32(tl + kSpColS + 32 * part, r);
        tc::wait_st();
    }
    auto put_state = [&](void *dst, int32_t dtype, int64_t base, const uint32_t r[32]) {
#pragma unroll
        for (int j = 0; j < 32; ++j) store_state1(dst, dtype, base + srow(v0 + j), __uint_as_float(r[j]));
    };

    uint32_t phase_x = 0, phase_s = 0;
    bool gave_up = false;
    auto wait_bar = [&](uint64_t *bar, uint32_t parity) {
        if (!gave_up && !mbar_wait(bar, parity, kSpWaitLimit)) {
            gave_up = true;
            if ((tid & 31) == 0) atomicExch(p.status, 2);
        }
    };
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
    char *const sop = smem + kSpSop, *const vop = smem + kSpVop;

    // O rows of chunk c (buffer c % 3, lanes 64..127) -> out[t][h][v0 ... v0 + 31]; warps of quadrants 2, 3
    auto store_outputs = [&](int32_t c) {
        wait_bar(&bar_o[c % kSpStages], (c / kSpStages) & 1);
        tc::fence_after_sync();
        uint32_t y[32];
        tc::ld32(tl + kSpColXY + 64 * (c % kSpBufs) + 32 * part, y);
        tc::wait_ld();
        const int64_t t = tok_begin + static_cast<int64_t>(c) * C + (lane - C);
        if (t < tok_end) {
            uint4 *dst = reinterpret_cast<uint4 *>(out + (t * H + h) * kSpD + v0);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = pack8_bits(y + 8 * q);
        }
    };

    for (int32_t i = 0; i < n_chunks; ++i) {
        wait_bar(&bars[i % kSpStages], (i / kSpStages) & 1);
        const char *sb = smem + (i % kSpStages) * kSpStage;
        const uint32_t xy = kSpColXY + 64 * static_cast<uint32_t>(i % kSpBufs);

        // S is the state after chunk i - 1: a checkpoint when that chunk ends on one.
        if (p.se.ckpt != nullptr && i > 0) {
            const int64_t ck = ckpt_slot(p.se, b, c_lo + i - 1, tok_end - tok_seq);
            if (ck >= 0) {
                uint32_t r[32];
                tc::ld32(tl + kSpColS + 32 * part, r);
                tc::wait_ld();
                put_state(p.se.ckpt, p.se.ckpt_dtype, ck * H * kSpD * kSpD, r);
            }
        }
        // (A) S row k (this thread's 32 columns) -> bf16 operand (undecayed); decay the TMEM copy by gamma_k
        {
            uint32_t r[32];
            tc::ld32(tl + kSpColS + 32 * part, r);
            tc::wait_ld();
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4 *>(sop + swz_off<128>(lane, 32 * part + 8 * q)) = pack8_bits(r + 8 * q);
            const float gk = reinterpret_cast<const float *>(sb + RS::GAMMA)[lane];
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * gk);
            tc::st32(tl + kSpColS + 32 * part, r);
        }
        tc::wait_st();
        fence_proxy_async_smem();  // generic-proxy operand writes -> visible to the tensor cores
        tc::fence_before_sync();
        named_arrive(kBarOperandsS);

        if (quad >= 2) {
            if (i > 0) store_outputs(i - 1);  // the previous chunk's outputs, while the MMAs run
        } else {
            // (C) V_new row t (token lanes 0..63), this thread's 32 columns -> bf16 operand, once this
            // chunk's [-V_new; Y] and the previous chunk's O products (readers of the operand) are done
            wait_bar(bar_x, phase_x);
            tc::fence_after_sync();
            uint32_t x[32];
            tc::ld32(tl + xy + 32 * part, x);
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] ^= 0x80000000u;  // -(-V_new)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4 *>(vop + swz_off<128>(lane, 32 * part + 8 * q)) = pack8_bits(x + 8 * q);
            fence_proxy_async_smem();
        }
        phase_x ^= 1u;
        tc::fence_before_sync();
        named_arrive(kBarOperandsV);
        wait_bar(bar_s, phase_s);
        phase_s ^= 1u;
        tc::fence_after_sync();
    }
    if (n_chunks > 0 && quad >= 2) store_outputs(n_chunks - 1);

    // final state -> packed fp32 and the cache row out_idx[b] (or, before the sequence's last
    // segment, the segment state), and the checkpoint of the segment's last chunk if it ends on one
    {
        const int64_t per_seq = H * kSpD * kSpD;
        const int64_t ob = last ? out_base(p.se, b) : -1;
        const int64_t ck = n_chunks > 0 ? ckpt_slot(p.se, b, c_hi - 1, tok_end - tok_seq) : -1;
        float *fin = last ? p.se.final_state : p.seg_state;
        if (fin != nullptr || ob >= 0 || ck >= 0) {
            uint32_t r[32];
            tc::ld32(tl + kSpColS + 32 * part, r);
            tc::wait_ld();
            if (fin != nullptr) put_state(fin, KDA_F32, b * per_seq, r);
            if (ob >= 0) put_state(p.se.out_cache, p.se.out_dtype, ob, r);
            if (ck >= 0) put_state(p.se.ckpt, p.se.ckpt_dtype, ck * per_seq, r);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kSpTmemCols);
}

}  // namespace

int state_pass_split_slices() { return kSpSlices; }

cudaError_t launch_state_pass_split(const PassParams &p, int64_t items, cudaStream_t st)
{
    cudaError_t e =
        cudaFuncSetAttribute(state_pass_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSpSmem);
    if (e != cudaSuccess) return e;
    state_pass_split_kernel<<<static_cast<unsigned>(items * kSpSlices), kSpThreads, kSpSmem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace prefill
}  // namespace kda
