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
#include <type_traits>

#include "msc_device.cuh"
#include "msc_internal.h"

namespace msc {

constexpr int kConvThreads = 64;  // 2 warps: finer CTAs than 128 threads measured 2-3 % faster
constexpr int kTileT = 32;

template <typename T, int V> struct Vec;
template <> struct Vec<float, 1> { using type = float; };
template <> struct Vec<float, 2> { using type = float2; };
template <> struct Vec<__nv_bfloat16, 1> { using type = __nv_bfloat16; };
template <> struct Vec<__nv_bfloat16, 4> { using type = uint2; };

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

// Input word of a thread (V channels) as channel pairs.
template <typename T, int V>
__device__ __forceinline__ void word_pairs(const typename Vec<T, V>::type& q,
                                           u64 (&p)[(V + 1) / 2]) {
    if constexpr (V == 1) {
        const float v = to_f32(q);
        p[0] = pk2(v, v);
    } else if constexpr (sizeof(T) == 4) {
        p[0] = *reinterpret_cast<const u64*>(&q);
    } else {
        p[0] = pk2(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xffff0000u));
        p[1] = pk2(__uint_as_float(q.y << 16), __uint_as_float(q.y & 0xffff0000u));
    }
}

// Prefill.  Grid (channel groups of kConvThreads * V, time tiles of kTileT,
// batch).  KC = d_conv, H = KC - 1.  A thread first loads the H + kTileT
// input rows of its channels that its tile needs (the H halo rows from the
// previous tile) -- all loads in flight together -- then computes kTileT
// outputs on channel pairs (fma.rn.f32x2) and stores them.  Interior tiles
// (halo inside the sequence, tile full) run without any per-step test; the
// first tile takes its halo from the conv state (or zeros) and the last may
// be partial.  The CTA whose tile holds the last step writes the conv state
// (the last H inputs); with L == 0 one tile of no steps does that.
template <typename T, int V, int KC>
__global__ void __launch_bounds__(kConvThreads)
causal_conv1d_kernel(const T* __restrict__ x, const float* __restrict__ w,
                     const float* __restrict__ bias, const T* __restrict__ state_in,
                     T* __restrict__ out, T* __restrict__ state_out, int64_t L,
                     int64_t d_inner, int silu_on) {
    constexpr int H = KC - 1;
    constexpr int R = H + kTileT;  // rows held: halo, then the tile
    constexpr int P = (V + 1) / 2; // channel pairs (V = 1: one, upper half unused)
    using W = typename Vec<T, V>::type;
    const int64_t d0 = ((int64_t)blockIdx.x * kConvThreads + threadIdx.x) * V;
    if (d0 >= d_inner) return;
    const int64_t b = blockIdx.z;
    const int64_t t0 = (int64_t)blockIdx.y * kTileT;
    const int nt = (int)min((int64_t)kTileT, L - t0 > 0 ? L - t0 : 0);  // steps here

    u64 w2[P][KC], b2[P];
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int64_t c0 = d0 + 2 * p, c1 = V == 1 ? c0 : c0 + 1;
#pragma unroll
        for (int k = 0; k < KC; ++k) w2[p][k] = pk2(__ldg(w + c0 * KC + k), __ldg(w + c1 * KC + k));
        b2[p] = bias ? pk2(__ldg(bias + c0), __ldg(bias + c1)) : pk2(0.0f, 0.0f);
    }
    const T* xb = x + (b * L + t0 - H) * d_inner + d0;  // row r of the tile: xb + r * d_inner
    T* op = out + (b * L + t0) * d_inner + d0;
    u64 win[H + 1][P];  // rows t .. t + H of output step t

    auto tile = [&](auto edge_tag) {
        constexpr bool EDGE = decltype(edge_tag)::value;
        W raw[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (!EDGE || (t0 - H + r >= 0 && r < H + nt))
                raw[r] = *reinterpret_cast<const W*>(xb + (int64_t)r * d_inner);
        }
#pragma unroll
        for (int j = 0; j < H; ++j) {
            if (!EDGE || t0 - H + j >= 0) {
                word_pairs<T, V>(raw[j], win[j]);
            } else {  // before the sequence: conv state, oldest first, or zero
                const int64_t s = t0 - H + j;
                float v[2 * P];
#pragma unroll
                for (int c = 0; c < 2 * P; ++c)
                    v[c] = (state_in && c < V)
                        ? Elem<T>::load(state_in + ((b * d_inner + d0 + c) * H + H + s))
                        : 0.0f;
#pragma unroll
                for (int p = 0; p < P; ++p) win[j][p] = pk2(v[2 * p], v[2 * p + 1]);
            }
        }
#pragma unroll
        for (int t = 0; t < kTileT; ++t) {
            if (EDGE && t >= nt) break;
            word_pairs<T, V>(raw[H + t], win[H]);
            u64 y[P];
#pragma unroll
            for (int p = 0; p < P; ++p) {
                u64 acc = b2[p];
#pragma unroll
                for (int k = 0; k <= H; ++k) acc = fma2(w2[p][k], win[k][p], acc);
                y[p] = silu_on ? silu2(acc) : acc;
            }
            T* o = op + (int64_t)t * d_inner;
            if constexpr (V == 1) {
                Elem<T>::store(o, lo2(y[0]));
            } else if constexpr (sizeof(T) == 4) {
                *reinterpret_cast<u64*>(o) = y[0];
            } else {
                const __nv_bfloat162 a2 = __floats2bfloat162_rn(lo2(y[0]), hi2(y[0]));
                const __nv_bfloat162 c2 = __floats2bfloat162_rn(lo2(y[1]), hi2(y[1]));
                uint2 q;
                q.x = *reinterpret_cast<const uint32_t*>(&a2);
                q.y = *reinterpret_cast<const uint32_t*>(&c2);
                *reinterpret_cast<uint2*>(o) = q;
            }
#pragma unroll
            for (int j = 0; j < H; ++j)
#pragma unroll
                for (int p = 0; p < P; ++p) win[j][p] = win[j + 1][p];
        }
    };
    if (t0 >= H && t0 + kTileT <= L)
        tile(std::integral_constant<bool, false>{});
    else
        tile(std::integral_constant<bool, true>{});

    if (state_out && t0 + kTileT >= L) {
#pragma unroll
        for (int j = 0; j < H; ++j)
#pragma unroll
            for (int p = 0; p < P; ++p) {
                Elem<T>::store(state_out + (b * d_inner + d0 + 2 * p) * H + j, lo2(win[j][p]));
                if (2 * p + 1 < V)
                    Elem<T>::store(state_out + (b * d_inner + d0 + 2 * p + 1) * H + j,
                                   hi2(win[j][p]));
            }
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
    Elem<T>::store(out + i, silu_on ? silu_rcp(acc) : acc);  // same rounding as the prefill
#pragma unroll
    for (int k = 0; k + 1 < H; ++k) Elem<T>::store(state + i * H + k, st[k + 1]);
    if (H > 0) Elem<T>::store(state + i * H + (H > 0 ? H - 1 : 0), cur);
}

// Decode, batch rows per thread: a thread owns channel d of kUpdRows
// consecutive batch rows, so its weights and bias are loaded once and the
// rows' state and input loads (independent of one another) are all in
// flight together.  The same operations per (row, channel) as above.
constexpr int kUpdRows = 8;
template <typename T, int KC>
__global__ void __launch_bounds__(256)
conv1d_update_rows_kernel(T* __restrict__ state, const T* __restrict__ x,
                          const float* __restrict__ w, const float* __restrict__ bias,
                          T* __restrict__ out, int64_t batch, int64_t d_inner, int silu_on) {
    constexpr int H = KC - 1;
    const int64_t d = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (d >= d_inner) return;
    const int64_t b0 = (int64_t)blockIdx.y * kUpdRows;
    float wk[KC];
#pragma unroll
    for (int k = 0; k < KC; ++k) wk[k] = __ldg(w + d * KC + k);
    const float bs = bias ? __ldg(bias + d) : 0.0f;
    float st[kUpdRows][H > 0 ? H : 1], cur[kUpdRows];
#pragma unroll
    for (int r = 0; r < kUpdRows; ++r) {
        const int64_t i = (b0 + r < batch ? b0 + r : batch - 1) * d_inner + d;
#pragma unroll
        for (int k = 0; k < H; ++k) st[r][k] = to_f32(state[i * H + k]);
        cur[r] = Elem<T>::load(x + i);
    }
#pragma unroll
    for (int r = 0; r < kUpdRows; ++r) {
        if (b0 + r >= batch) break;
        const int64_t i = (b0 + r) * d_inner + d;
        float acc = bs;
#pragma unroll
        for (int k = 0; k < H; ++k) acc = fmaf(wk[k], st[r][k], acc);
        acc = fmaf(wk[H], cur[r], acc);
        Elem<T>::store(out + i, silu_on ? silu_rcp(acc) : acc);  // same rounding as the prefill
#pragma unroll
        for (int k = 0; k + 1 < H; ++k) Elem<T>::store(state + i * H + k, st[r][k + 1]);
        if (H > 0) Elem<T>::store(state + i * H + (H > 0 ? H - 1 : 0), cur[r]);
    }
}

template <typename T, int V, int KC>
static cudaError_t launch_conv_v(const ConvArgs& a, cudaStream_t s) {
    const int64_t groups = (a.d_inner + (int64_t)kConvThreads * V - 1) / ((int64_t)kConvThreads * V);
    const int64_t tiles = a.L > 0 ? (a.L + kTileT - 1) / kTileT : 1;
    const dim3 grid((unsigned)groups, (unsigned)tiles, (unsigned)a.batch);
    const ProfileMark m = profile_begin(s, MSC_PROF_CONV);
    causal_conv1d_kernel<T, V, KC><<<grid, kConvThreads, 0, s>>>(
        static_cast<const T*>(a.x), a.w, a.bias, static_cast<const T*>(a.state_in),
        static_cast<T*>(a.out), static_cast<T*>(a.state_out), a.L, a.d_inner, a.silu);
    profile_end(m, s);
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
    const ProfileMark m = profile_begin(s, MSC_PROF_CONV_UPDATE);
    const int64_t rgroups = (a.batch + kUpdRows - 1) / kUpdRows;
    if (a.batch >= kUpdRows && rgroups <= 65535) {
        const dim3 grid((unsigned)((a.d_inner + 255) / 256), (unsigned)rgroups);
        conv1d_update_rows_kernel<T, KC><<<grid, 256, 0, s>>>(
            static_cast<T*>(a.state_out), static_cast<const T*>(a.x), a.w, a.bias,
            static_cast<T*>(a.out), a.batch, a.d_inner, a.silu);
    } else {
        conv1d_update_kernel<T, KC><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(
            static_cast<T*>(a.state_out), static_cast<const T*>(a.x), a.w, a.bias,
            static_cast<T*>(a.out), n, a.d_inner, a.silu);
    }
    profile_end(m, s);
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
