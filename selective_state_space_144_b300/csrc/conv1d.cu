// conv1d.cu -- the causal depthwise conv1d (+ SiLU) that feeds the scan, for
// sm_103a: the prefill over a whole sequence and the one-token decode update.
//
// Operation ("Deep dive into Mamba: architecture and implementation of
// selective state-space models", section 3.2: Conv1d with kernel d_conv,
// padding d_conv - 1 and one group per channel, with bias; section 5.2 and
// the MambaBlock of "State space models and Mamba": the first L outputs are
// kept, then SiLU):
//     out[b,t,d] = silu(bias[d] + sum_k w[d,k] * x[b, t - (d_conv-1) + k, d])
// where inputs before t = 0 come from a conv state (the d_conv-1 inputs that
// preceded the sequence, oldest first) or are zero.
//
// Both kernels move each input and output once and are bound by HBM.  The
// prefill kernel gives a thread V consecutive channels (8 bytes of input per
// time step: 4 bf16 or 2 fp32 channels; V = 1 when the channel count or the
// pointers do not allow it) and a tile of kTileT time steps, whose input
// rows (plus a halo of d_conv-1 rows) it loads into registers all at once
// before computing; a warp's loads of one time row are 32 consecutive 8-byte
// words.
#include "msc_device.cuh"
#include "msc_internal.h"

namespace msc {

constexpr int kConvThreads = 128;
constexpr int kTileT = 16;

template <typename T, int V> struct Vec;
template <> struct Vec<float, 1> { using type = float; };
template <> struct Vec<float, 2> { using type = float2; };
template <> struct Vec<__nv_bfloat16, 1> { using type = __nv_bfloat16; };
template <> struct Vec<__nv_bfloat16, 4> { using type = uint2; };

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

// Raw 8-byte word of V channels (V = 8 / sizeof(T)) <-> V floats.
template <typename T>
__device__ __forceinline__ void unpack_word(uint2 q, float* v) {
    if constexpr (sizeof(T) == 4) {
        v[0] = __uint_as_float(q.x);
        v[1] = __uint_as_float(q.y);
    } else {
        v[0] = __uint_as_float(q.x << 16);
        v[1] = __uint_as_float(q.x & 0xffff0000u);
        v[2] = __uint_as_float(q.y << 16);
        v[3] = __uint_as_float(q.y & 0xffff0000u);
    }
}

template <typename T>
__device__ __forceinline__ uint2 pack_word(const float* v) {
    uint2 q;
    if constexpr (sizeof(T) == 4) {
        q.x = __float_as_uint(v[0]);
        q.y = __float_as_uint(v[1]);
    } else {
        const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
        const __nv_bfloat162 c = __floats2bfloat162_rn(v[2], v[3]);
        q.x = *reinterpret_cast<const uint32_t*>(&a);
        q.y = *reinterpret_cast<const uint32_t*>(&c);
    }
    return q;
}

// Prefill.  Grid (channel groups of kConvThreads * V, time tiles of kTileT,
// batch).  KC = d_conv, H = KC - 1.  A thread first loads the H + kTileT
// input rows of its channels that its tile needs (the H halo rows from the
// previous tile or the conv state) -- all loads in flight together, the
// kernel being bound by memory latency and bandwidth -- then computes and
// stores kTileT outputs.  The CTA whose tile holds the last step writes the
// conv state (the last H inputs); with L == 0 one tile of no steps does that.
template <typename T, int V, int KC>
__global__ void __launch_bounds__(kConvThreads)
causal_conv1d_kernel(const T* __restrict__ x, const float* __restrict__ w,
                     const float* __restrict__ bias, const T* __restrict__ state_in,
                     T* __restrict__ out, T* __restrict__ state_out, int64_t L,
                     int64_t d_inner, int silu_on) {
    constexpr int H = KC - 1;
    constexpr int R = H + kTileT;  // rows held: halo, then the tile
    using W = typename Vec<T, V>::type;
    const int64_t d0 = ((int64_t)blockIdx.x * kConvThreads + threadIdx.x) * V;
    if (d0 >= d_inner) return;
    const int64_t b = blockIdx.z;
    const int64_t t0 = (int64_t)blockIdx.y * kTileT;
    const int nt = (int)min((int64_t)kTileT, L - t0 > 0 ? L - t0 : 0);  // steps here

    W raw[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t s = t0 - H + r;
        if (s >= 0 && r < H + nt) raw[r] = *reinterpret_cast<const W*>(x + (b * L + s) * d_inner + d0);
    }
    float wv[V][KC], bv[V];
#pragma unroll
    for (int c = 0; c < V; ++c) {
#pragma unroll
        for (int k = 0; k < KC; ++k) wv[c][k] = __ldg(w + (d0 + c) * KC + k);
        bv[c] = bias ? __ldg(bias + d0 + c) : 0.0f;
    }
    auto row = [&](int r, float (&v)[V]) {  // input row t0 - H + r as floats
        const int64_t s = t0 - H + r;
        if (s >= 0) {
            if constexpr (V == 1) {
                v[0] = to_f32(raw[r]);  // a register value: no memory load
            } else {
                unpack_word<T>(*reinterpret_cast<const uint2*>(&raw[r]), v);
            }
        } else {
#pragma unroll
            for (int c = 0; c < V; ++c)
                v[c] = state_in ? Elem<T>::load(state_in + ((b * d_inner + d0 + c) * H + H + s))
                                : 0.0f;
        }
    };
    float win[H + 1][V];  // rows j .. j + H of the current output step
#pragma unroll
    for (int j = 0; j < H; ++j) row(j, win[j]);
    T* op = out + (b * L + t0) * d_inner + d0;
#pragma unroll
    for (int t = 0; t < kTileT; ++t) {
        if (t < nt) {
            row(H + t, win[H]);
            float y[V];
#pragma unroll
            for (int c = 0; c < V; ++c) {
                float acc = bv[c];
#pragma unroll
                for (int k = 0; k <= H; ++k) acc = fmaf(wv[c][k], win[k][c], acc);
                y[c] = silu_on ? silu(acc) : acc;
            }
            if constexpr (V == 1) {
                Elem<T>::store(op + (int64_t)t * d_inner, y[0]);
            } else {
                *reinterpret_cast<uint2*>(op + (int64_t)t * d_inner) = pack_word<T>(y);
            }
#pragma unroll
            for (int j = 0; j < H; ++j)
#pragma unroll
                for (int c = 0; c < V; ++c) win[j][c] = win[j + 1][c];
        }
    }
    if (state_out && t0 + kTileT >= L) {
#pragma unroll
        for (int c = 0; c < V; ++c)
#pragma unroll
            for (int j = 0; j < H; ++j)
                Elem<T>::store(state_out + (b * d_inner + d0 + c) * H + j, win[j][c]);
    }
}

// Decode: one thread per (batch, channel); its state row is H inputs.  (A
// thread per 8-byte group of channels, reading the state rows as words,
// measured slower on the 256 x 5120 decode shape.)
template <typename T, int KC>
__global__ void __launch_bounds__(256)
conv1d_update_kernel(T* __restrict__ state, const T* __restrict__ x,
                     const float* __restrict__ w, const float* __restrict__ bias,
                     T* __restrict__ out, int64_t n, int64_t d_inner, int silu_on) {
    constexpr int H = KC - 1;
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;  // flat (b, d)
    if (i >= n) return;
    const int64_t d = i % d_inner;
    float st[H > 0 ? H : 1];
#pragma unroll
    for (int k = 0; k < H; ++k) st[k] = to_f32(state[i * H + k]);  // rewritten below
    const float cur = Elem<T>::load(x + i);
    float acc = bias ? __ldg(bias + d) : 0.0f;
#pragma unroll
    for (int k = 0; k < H; ++k) acc = fmaf(__ldg(w + d * KC + k), st[k], acc);
    acc = fmaf(__ldg(w + d * KC + H), cur, acc);
    Elem<T>::store(out + i, silu_on ? silu(acc) : acc);
#pragma unroll
    for (int k = 0; k + 1 < H; ++k) Elem<T>::store(state + i * H + k, st[k + 1]);
    if (H > 0) Elem<T>::store(state + i * H + (H > 0 ? H - 1 : 0), cur);
}

template <typename T, int V, int KC>
static cudaError_t launch_conv_v(const ConvArgs& a, cudaStream_t s) {
    const int64_t groups = (a.d_inner + (int64_t)kConvThreads * V - 1) / ((int64_t)kConvThreads * V);
    const int64_t tiles = a.L > 0 ? (a.L + kTileT - 1) / kTileT : 1;
    const dim3 grid((unsigned)groups, (unsigned)tiles, (unsigned)a.batch);
    causal_conv1d_kernel<T, V, KC><<<grid, kConvThreads, 0, s>>>(
        static_cast<const T*>(a.x), a.w, a.bias, static_cast<const T*>(a.state_in),
        static_cast<T*>(a.out), static_cast<T*>(a.state_out), a.L, a.d_inner, a.silu);
    return cudaGetLastError();
}

template <typename T, int KC>
static cudaError_t launch_conv_k(const ConvArgs& a, cudaStream_t s) {
    constexpr int VW = 8 / (int)sizeof(T);  // channels per 8-byte vector
    if (a.vec) return launch_conv_v<T, VW, KC>(a, s);
    return launch_conv_v<T, 1, KC>(a, s);
}

template <typename T, int KC>
static cudaError_t launch_update_k(const ConvArgs& a, cudaStream_t s) {
    const int64_t n = a.batch * a.d_inner;
    conv1d_update_kernel<T, KC><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(
        static_cast<T*>(a.state_out), static_cast<const T*>(a.x), a.w, a.bias,
        static_cast<T*>(a.out), n, a.d_inner, a.silu);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t dispatch(const ConvArgs& a, bool update, cudaStream_t s) {
#define MSC_CONV_CASE(K)                                                        \
    case K:                                                                     \
        return update ? launch_update_k<T, K>(a, s) : launch_conv_k<T, K>(a, s);
    switch (a.d_conv) {
        MSC_CONV_CASE(1)
        MSC_CONV_CASE(2)
        MSC_CONV_CASE(3)
        MSC_CONV_CASE(4)
        MSC_CONV_CASE(5)
        MSC_CONV_CASE(6)
        MSC_CONV_CASE(7)
        MSC_CONV_CASE(8)
        default:
            return cudaErrorInvalidValue;
    }
#undef MSC_CONV_CASE
}

cudaError_t launch_causal_conv1d(const ConvArgs& a, msc_dtype dtype, cudaStream_t s) {
    return dtype == MSC_BF16 ? dispatch<__nv_bfloat16>(a, false, s) : dispatch<float>(a, false, s);
}

cudaError_t launch_conv1d_update(const ConvArgs& a, msc_dtype dtype, cudaStream_t s) {
    return dtype == MSC_BF16 ? dispatch<__nv_bfloat16>(a, true, s) : dispatch<float>(a, true, s);
}

}  // namespace msc
