// Short causal convolution ahead of the recurrence: q, k and v each pass a
// depthwise causal convolution of width W with a convolution state per
// request (the infra page, sections 6.5 and 8.2.3: causal_conv1d_fn in
// prefill, causal_conv1d_update in decode).  Per channel c:
//   y_t = act(bias_c + sum_{i<W} w[c][i] x_{t-(W-1)+i}),  act = identity | SiLU,
// inputs before a sequence start taken from its state (the last W-1 inputs,
// oldest first; zeros when absent).  fp32 arithmetic; inputs and outputs bf16
// or fp32; states in fp32 or bf16 (stored values are inputs, so a bf16 state
// of bf16 inputs is exact).
//
// Both kernels are HBM-bound streams: each thread owns 8 consecutive channels
// (16-byte bf16 vectors) and a tile of consecutive tokens, keeping its window
// of W - 1 earlier inputs in registers; warps read and write whole 512-byte
// spans of a token row.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kConvThreads = 128;
constexpr int kVec = 8;  // channels per thread
static_assert(kConvThreads * kVec == kConvChannelsPerBlock, "channel block of the host-side grid checks");

template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
    uint4 u;
    __device__ __forceinline__ void load(const void *p) { u = *reinterpret_cast<const uint4 *>(p); }
    __device__ __forceinline__ void get(float x[8]) const
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = bf16_lo(w[i]);
            x[2 * i + 1] = bf16_hi(w[i]);
        }
    }
};
template <> struct Vec8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const void *p)
    {
        a = reinterpret_cast<const float4 *>(p)[0];
        b = reinterpret_cast<const float4 *>(p)[1];
    }
    __device__ __forceinline__ void get(float x[8]) const
    {
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
};

// 8 values of a state / io buffer (fp32 or bf16 by `dtype`) at element offset e.
__device__ __forceinline__ void load8(const void *base, int32_t dtype, int64_t e, float x[8])
{
    if (dtype == KDA_F32) {
        const float4 a = *reinterpret_cast<const float4 *>(static_cast<const float *>(base) + e);
        const float4 b = *(reinterpret_cast<const float4 *>(static_cast<const float *>(base) + e) + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
        const uint4 u = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + e);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = bf16_lo(w[i]);
            x[2 * i + 1] = bf16_hi(w[i]);
        }
    }
}
__device__ __forceinline__ void store8(void *base, int32_t dtype, int64_t e, const float x[8])
{
    if (dtype == KDA_F32) {
        float4 *p = reinterpret_cast<float4 *>(static_cast<float *>(base) + e);
        p[0] = make_float4(x[0], x[1], x[2], x[3]);
        p[1] = make_float4(x[4], x[5], x[6], x[7]);
    } else {
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(base) + e) =
            make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                       pack_bf16x2(x[6], x[7]));
    }
}

// SiLU with the fast exponential and division (a few ulps; for y << 0 the
// denominator overflows and the result is the limit 0).
__device__ __forceinline__ float activate(float y, int32_t act)
{
    return act == 1 ? __fdividef(y, 1.f + __expf(-y)) : y;
}

__device__ __forceinline__ float tanh_approx(float x)
{
    float y;
    asm("tanh.approx.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// SiLU for bf16 outputs: y * sigmoid(y) with sigmoid(y) = (1 + tanh(y / 2)) / 2
// from one hardware tanh (relative error about 2^-11 on the sigmoid, below half a
// bf16 step of the output, which is rounded to 2^-9 anyway).
__device__ __forceinline__ float activate_bf16(float y, int32_t act)
{
    if (act != 1) return y;
    const float h = 0.5f * y;
    return fmaf(h, tanh_approx(h), h);
}

struct ConvArgs {
    const void *x;
    int32_t io_dtype;
    const int32_t *cu;
    int64_t B, T, C;
    const float *weight, *bias;
    int32_t act;
    const void *init;
    void *final_state;
    int32_t state_dtype;
    void *y;
};

// Taps and bias of channels c0 .. c0 + 7: w[j][i] = weight[c0 + j][i].
template <int W> __device__ __forceinline__ void load_taps(const ConvArgs &a, int64_t c0, float w[8][W], float b[8])
{
    const float4 *wp = reinterpret_cast<const float4 *>(a.weight + c0 * W);  // 8 W floats, 16-byte aligned
    float t[8 * W];
#pragma unroll
    for (int q = 0; q < 2 * W; ++q) {
        const float4 v = wp[q];
        t[4 * q] = v.x; t[4 * q + 1] = v.y; t[4 * q + 2] = v.z; t[4 * q + 3] = v.w;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int i = 0; i < W; ++i) w[j][i] = t[j * W + i];
#pragma unroll
    for (int j = 0; j < 8; ++j) b[j] = 0.f;
    if (a.bias != nullptr) {
        const float4 b0 = reinterpret_cast<const float4 *>(a.bias + c0)[0];
        const float4 b1 = reinterpret_cast<const float4 *>(a.bias + c0)[1];
        b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w; b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
    }
}

// Tokens [t0, t0 + TT) x channels [c0, c0 + 8) per thread.
template <int W, typename IO, int TT>
__global__ void __launch_bounds__(kConvThreads, 3)
conv_varlen_kernel(ConvArgs a)
{
    // channel blocks fastest: the blocks of one token tile run together (whole rows of x and y)
    const int64_t ncb = (a.C + kConvThreads * kVec - 1) / (kConvThreads * kVec);
    const int64_t c0 = ((static_cast<int64_t>(blockIdx.x) % ncb) * kConvThreads + threadIdx.x) * kVec;
    const int64_t t0 = (static_cast<int64_t>(blockIdx.x) / ncb) * TT;
    if (c0 >= a.C || t0 >= a.T) return;
    const int64_t C = a.C;
    const IO *x = static_cast<const IO *>(a.x);
    // this tile's rows and the W - 1 rows before it, all loads in flight at once
    // (the earlier rows are used unless the tile starts a sequence)
    Vec8<IO> xr[TT], xp[W - 1];
#pragma unroll
    for (int j = 0; j < TT; ++j)
        if (t0 + j < a.T) xr[j].load(x + (t0 + j) * C + c0);
#pragma unroll
    for (int i = 0; i < W - 1; ++i)
        if (t0 - (W - 1) + i >= 0) xp[i].load(x + (t0 - (W - 1) + i) * C + c0);
    float w[8][W], bias[8];
    load_taps<W>(a, c0, w, bias);
    // the sequence holding t0: the last b with cu[b] <= t0
    int64_t lo = 0, hi = a.B - 1;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) / 2;
        if (a.cu[mid] <= t0) lo = mid;
        else hi = mid - 1;
    }
    int64_t b = lo;
    int64_t start = a.cu[b], end = a.cu[b + 1];
    // window of the W - 1 inputs before t0 (oldest first)
    float win[W - 1][8];
#pragma unroll
    for (int i = 0; i < W - 1; ++i) {
        const int64_t tau = t0 - (W - 1) + i;
        if (tau >= start) {
            xp[i].get(win[i]);
        } else if (a.init != nullptr) {  // state row (W - 1) - (start - tau) of sequence b
            load8(a.init, a.state_dtype, (b * (W - 1) + (W - 1) - (start - tau)) * C + c0, win[i]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) win[i][j] = 0.f;
        }
    }
    IO *y = static_cast<IO *>(a.y);
    if (t0 + TT <= end) {  // the whole tile inside one sequence (the common case): no branches
        IO *yp = y + t0 * C + c0;
#pragma unroll
        for (int jt = 0; jt < TT; ++jt) {
            float xt[8], out[8];
            xr[jt].get(xt);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float acc = bias[j];
#pragma unroll
                for (int i = 0; i < W - 1; ++i) acc = fmaf(w[j][i], win[(jt + i) % (W - 1)][j], acc);
                acc = fmaf(w[j][W - 1], xt[j], acc);
                out[j] = sizeof(IO) == 2 ? activate_bf16(acc, a.act) : activate(acc, a.act);
            }
            store8(yp, a.io_dtype, 0, out);
            yp += C;
#pragma unroll
            for (int j = 0; j < 8; ++j) win[jt % (W - 1)][j] = xt[j];  // ring: the oldest entry is replaced
        }
        if (t0 + TT == end && a.final_state != nullptr) {  // the tile ends the sequence: its final state
#pragma unroll
            for (int i = 0; i < W - 1; ++i)
                store8(a.final_state, a.state_dtype, (b * (W - 1) + i) * C + c0, win[(TT + i) % (W - 1)]);
        }
        return;
    }
#pragma unroll
    for (int jt = 0; jt < TT; ++jt) {
        const int64_t t = t0 + jt;
        if (t >= a.T) break;
        if (t == end) {  // a new sequence starts here (skipping empty ones): its state
            do {
                ++b;
                start = a.cu[b];
                end = a.cu[b + 1];
            } while (end == t && b + 1 < a.B);
#pragma unroll
            for (int i = 0; i < W - 1; ++i) {
                if (a.init != nullptr) {
                    load8(a.init, a.state_dtype, (b * (W - 1) + i) * C + c0, win[i]);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) win[i][j] = 0.f;
                }
            }
        }
        float xt[8], out[8];
        xr[jt].get(xt);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float acc = bias[j];
#pragma unroll
            for (int i = 0; i < W - 1; ++i) acc = fmaf(w[j][i], win[i][j], acc);
            acc = fmaf(w[j][W - 1], xt[j], acc);
            out[j] = sizeof(IO) == 2 ? activate_bf16(acc, a.act) : activate(acc, a.act);
        }
        store8(y, a.io_dtype, t * C + c0, out);
#pragma unroll
        for (int i = 0; i + 1 < W - 1; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) win[i][j] = win[i + 1][j];
#pragma unroll
        for (int j = 0; j < 8; ++j) win[W - 2][j] = xt[j];
        if (t == end - 1 && a.final_state != nullptr) {  // the sequence's last token: its final state
#pragma unroll
            for (int i = 0; i < W - 1; ++i) store8(a.final_state, a.state_dtype, (b * (W - 1) + i) * C + c0, win[i]);
        }
    }
}

// Final states of empty sequences: their initial states (or zeros).
template <int W>
__global__ void __launch_bounds__(kConvThreads)
conv_empty_kernel(ConvArgs a)
{
    const int64_t c0 = (static_cast<int64_t>(blockIdx.y) * kConvThreads + threadIdx.x) * kVec;
    const int64_t b = blockIdx.x;
    if (c0 >= a.C || a.cu[b + 1] != a.cu[b]) return;
#pragma unroll
    for (int i = 0; i < W - 1; ++i) {
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const int64_t e = (b * (W - 1) + i) * a.C + c0;
        if (a.init != nullptr) load8(a.init, a.state_dtype, e, v);
        store8(a.final_state, a.state_dtype, e, v);
    }
}

struct UpdateArgs {
    const void *x;
    int32_t io_dtype;
    int64_t R, C;
    const float *weight, *bias;
    int32_t act;
    CacheDesc cache;
    const void *idx;
    int32_t idx_type;
    void *y;
};

// One token per request, on its conv-state cache row in place.
template <int W>
__global__ void __launch_bounds__(kConvThreads)
conv_update_kernel(UpdateArgs u)
{
    const int64_t c0 = (static_cast<int64_t>(blockIdx.y) * kConvThreads + threadIdx.x) * kVec;
    const int64_t r = blockIdx.x;
    if (c0 >= u.C) return;
    const int64_t row = u.idx_type == KDA_I64 ? static_cast<const int64_t *>(u.idx)[r]
                                              : static_cast<const int32_t *>(u.idx)[r];
    const bool valid = row >= 0 && row < u.cache.n_rows;
    ConvArgs a{};
    a.weight = u.weight;
    a.bias = u.bias;
    float w[8][W], bias[8];
    load_taps<W>(a, c0, w, bias);
    float win[W][8];
#pragma unroll
    for (int i = 0; i < W - 1; ++i) {
        if (valid) {
            load8(u.cache.data, u.cache.dtype, row * u.cache.row_stride + i * u.C + c0, win[i]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) win[i][j] = 0.f;
        }
    }
    load8(u.x, u.io_dtype, r * u.C + c0, win[W - 1]);
    float out[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float acc = bias[j];
#pragma unroll
        for (int i = 0; i < W; ++i) acc = fmaf(w[j][i], win[i][j], acc);
        out[j] = activate(acc, u.act);
    }
    store8(u.y, u.io_dtype, r * u.C + c0, out);
    if (valid) {
#pragma unroll
        for (int i = 0; i < W - 1; ++i)
            store8(u.cache.data, u.cache.dtype, row * u.cache.row_stride + i * u.C + c0, win[i + 1]);
    }
}

template <int W> cudaError_t varlen_w(const ConvArgs &a, cudaStream_t st)
{
    const unsigned gy = static_cast<unsigned>((a.C + kConvThreads * kVec - 1) / (kConvThreads * kVec));
    if (a.T > 0) {
        if ((a.T + 15) / 8 * static_cast<int64_t>(gy) > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        if (a.io_dtype == KDA_BF16) {
            constexpr int TT = 16;
            conv_varlen_kernel<W, __nv_bfloat16, TT>
                <<<static_cast<unsigned>((a.T + TT - 1) / TT * gy), kConvThreads, 0, st>>>(a);
        } else {
            constexpr int TT = 8;
            conv_varlen_kernel<W, float, TT>
                <<<static_cast<unsigned>((a.T + TT - 1) / TT * gy), kConvThreads, 0, st>>>(a);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (a.final_state != nullptr) {
        conv_empty_kernel<W><<<dim3(static_cast<unsigned>(a.B), gy), kConvThreads, 0, st>>>(a);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

template <int W> cudaError_t update_w(const UpdateArgs &u, cudaStream_t st)
{
    const unsigned gy = static_cast<unsigned>((u.C + kConvThreads * kVec - 1) / (kConvThreads * kVec));
    conv_update_kernel<W><<<dim3(static_cast<unsigned>(u.R), gy), kConvThreads, 0, st>>>(u);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv1d_varlen(const Conv1dArgs &p, cudaStream_t st)
{
    ConvArgs a{p.x, p.io_dtype, p.cu_seqlens, p.num_seqs, p.total_tokens, p.channels, p.weight, p.bias,
               p.activation, p.init_state, p.final_state, p.state_dtype, p.y};
    switch (p.width) {
    case 2: return varlen_w<2>(a, st);
    case 3: return varlen_w<3>(a, st);
    default: return varlen_w<4>(a, st);
    }
}

cudaError_t launch_conv1d_update(const Conv1dUpdateArgs &p, cudaStream_t st)
{
    UpdateArgs u{p.x, p.io_dtype, p.batch, p.channels, p.weight, p.bias, p.activation, p.cache, p.idx, p.idx_type,
                 p.y};
    switch (p.width) {
    case 2: return update_w<2>(u, st);
    case 3: return update_w<3>(u, st);
    default: return update_w<4>(u, st);
    }
}

}  // namespace kda
