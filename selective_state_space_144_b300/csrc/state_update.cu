// state_update.cu -- single-token selective state update (decode) for sm_103a.
//
// One step of the scan's recurrence with the state read from and written
// back to HBM in place (the "Mamba decoding" example of "State space models
// and Mamba": constant memory per generated token):
//     delta = softplus(dt + dt_bias);  h = exp(delta*A) * h + delta*B*u
//     out = (C . h + D*u) * silu(z)
// (delta*B is replaced by the zero-order-hold input matrix when asked).
// The step is bound by streaming the fp32 state (8 bytes per state element
// per step).  state_update_row_kernel (N = 8, 16, 32, aligned arrays) keeps
// a whole channel per thread; state_update_kernel is the general form, a
// thread per 4 consecutive states with a shuffle reduction over the lanes of
// a channel.
#include "msc_device.cuh"
#include "msc_internal.h"

namespace msc {

template <typename T, int G, bool VEC>
__global__ void __launch_bounds__(kUpdateThreads)
state_update_kernel(UpdateArgs a) {
    const int64_t gid = (int64_t)blockIdx.x * kUpdateThreads + threadIdx.x;
    const int g = (int)(gid % G);
    const int64_t nch = a.batch * a.d_inner;
    const int64_t ch_raw = gid / G;
    const bool valid = ch_raw < nch;
    const int64_t ch = valid ? ch_raw : nch - 1;  // idle lanes read in bounds
    const int64_t b = ch / a.d_inner;
    const int64_t d = ch - b * a.d_inner;
    const int N = (int)a.N;
    const int n0 = g * 4;

    float* srow = a.state + ch * N;
    float h[4];
    if (VEC) {
        if (n0 < N) {
            const float4 q = *reinterpret_cast<const float4*>(srow + n0);
            h[0] = q.x; h[1] = q.y; h[2] = q.z; h[3] = q.w;
        } else {
            h[0] = h[1] = h[2] = h[3] = 0.0f;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) h[j] = (n0 + j < N) ? srow[n0 + j] : 0.0f;
    }
    float A2[4], iA[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float Av = (n0 + j < N) ? __ldg(a.A + d * N + n0 + j) : 0.0f;
        A2[j] = Av * kLog2e;
        iA[j] = a.zoh ? 1.0f / Av : 0.0f;
    }

    const float bias = a.dt_bias ? __ldg(a.dt_bias + d) : 0.0f;
    const float x = Elem<T>::load(static_cast<const T*>(a.dt) + ch) + bias;
    const float uu = Elem<T>::load(static_cast<const T*>(a.u) + ch);
    const float delta = softplus(x);
    const float du = delta * uu;
    float Bv[4], Cv[4], Bq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    load_row4<T, VEC>(static_cast<const T*>(a.B) + b * N, n0, N, Bv);
    load_row4<T, VEC>(static_cast<const T*>(a.C) + b * N, n0, N, Cv);
    float tra = 0.0f, trc = 0.0f, uq = 0.0f;  // exponential trapezoid
    if (a.trap) {
        const float lt = Elem<T>::load(static_cast<const T*>(a.lam) + ch);
        tra = (1.0f - lt) * delta;
        trc = (lt * delta) * uu;
        if (a.u_prev && a.B_prev) {
            uq = Elem<T>::load(static_cast<const T*>(a.u_prev) + ch);
            load_row4<T, false>(static_cast<const T*>(a.B_prev) + b * N, n0, N, Bq);
        }
    }
    float y = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float x2 = delta * A2[j];
        const float dA = ex2(x2);
        const float inj = a.trap  ? fmaf(tra, uq * Bq[j], trc * Bv[j])
                          : a.zoh ? zoh_gain(x2, dA, delta, iA[j]) * uu * Bv[j]
                                  : du * Bv[j];
        h[j] = fmaf(dA, h[j], inj);
        y = fmaf(Cv[j], h[j], y);
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
    if (!valid) return;
    if (VEC) {
        if (n0 < N)
            *reinterpret_cast<float4*>(srow + n0) = make_float4(h[0], h[1], h[2], h[3]);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (n0 + j < N) srow[n0 + j] = h[j];
    }
    if (g == 0) {
        y = fmaf(a.D ? __ldg(a.D + d) : 0.0f, uu, y);
        if (a.z) y *= silu(Elem<T>::load(static_cast<const T*>(a.z) + ch));
        Elem<T>::store(static_cast<T*>(a.out) + ch, y);
    }
}

// Channel-per-thread decode step for N in {8, 16, 32}: a thread keeps all N
// states of its channel, so softplus and the gate are evaluated once per
// channel; B and C of the batch row are staged once per CTA in shared memory
// as fp32.  Grid (d_inner / 128, batch): no index division.  The state moves
// as N/4 16-byte loads and stores per thread (the warp's 32 x N*4 bytes are
// contiguous, so every fetched sector is used).  The kernel is bound by the
// latency of those loads, so every global load of the thread -- state, A,
// u, dt, z, bias, D -- is issued before the barrier that publishes B and C.
template <typename T, int N>
__global__ void __launch_bounds__(128)
state_update_row_kernel(UpdateArgs a) {
    __shared__ float sB[N], sC[N], sBq[N];
    const int b = blockIdx.y;
    const int64_t d_raw = (int64_t)blockIdx.x * 128 + threadIdx.x;
    const bool valid = d_raw < a.d_inner;
    const int64_t d = valid ? d_raw : a.d_inner - 1;  // idle threads read in bounds
    const int64_t ch = (int64_t)b * a.d_inner + d;
    float4* srow = reinterpret_cast<float4*>(a.state + ch * N);
    const float4* arow = reinterpret_cast<const float4*>(a.A + d * N);
    float h[N], Av[N];
#pragma unroll
    for (int q = 0; q < N / 4; ++q) {
        const float4 v = __ldcs(srow + q);  // streamed: read once, written once
        h[4 * q] = v.x; h[4 * q + 1] = v.y; h[4 * q + 2] = v.z; h[4 * q + 3] = v.w;
        const float4 w = __ldg(arow + q);
        Av[4 * q] = w.x; Av[4 * q + 1] = w.y; Av[4 * q + 2] = w.z; Av[4 * q + 3] = w.w;
    }
    const float bias = a.dt_bias ? __ldg(a.dt_bias + d) : 0.0f;
    const float Dd = a.D ? __ldg(a.D + d) : 0.0f;
    const float x = Elem<T>::load(static_cast<const T*>(a.dt) + ch) + bias;
    const float uu = Elem<T>::load(static_cast<const T*>(a.u) + ch);
    const float zz = a.z ? Elem<T>::load(static_cast<const T*>(a.z) + ch) : 0.0f;
    const bool prev = a.trap && a.u_prev && a.B_prev;
    const float lt = a.trap ? Elem<T>::load(static_cast<const T*>(a.lam) + ch) : 0.0f;
    const float uq = prev ? Elem<T>::load(static_cast<const T*>(a.u_prev) + ch) : 0.0f;
    if (threadIdx.x < N) {
        sB[threadIdx.x] = Elem<T>::load(static_cast<const T*>(a.B) + (int64_t)b * N + threadIdx.x);
        sC[threadIdx.x] = Elem<T>::load(static_cast<const T*>(a.C) + (int64_t)b * N + threadIdx.x);
        sBq[threadIdx.x] =
            prev ? Elem<T>::load(static_cast<const T*>(a.B_prev) + (int64_t)b * N + threadIdx.x)
                 : 0.0f;
    }
    const float delta = softplus(x);
    const float du = delta * uu;
    __syncthreads();
    float y = 0.0f;
    if (a.trap) {  // exponential trapezoid
        const float tra = (1.0f - lt) * delta, trc = (lt * delta) * uu;
#pragma unroll
        for (int n = 0; n < N; ++n) {
            const float dA = ex2(delta * (Av[n] * kLog2e));
            h[n] = fmaf(dA, h[n], fmaf(tra, uq * sBq[n], trc * sB[n]));
            y = fmaf(sC[n], h[n], y);
        }
    } else if (a.zoh) {
#pragma unroll
        for (int n = 0; n < N; ++n) {
            const float x2 = delta * (Av[n] * kLog2e);
            const float dA = ex2(x2);
            h[n] = fmaf(dA, h[n], zoh_gain(x2, dA, delta, 1.0f / Av[n]) * uu * sB[n]);
            y = fmaf(sC[n], h[n], y);
        }
    } else {
#pragma unroll
        for (int n = 0; n < N; ++n) {
            const float dA = ex2(delta * (Av[n] * kLog2e));  // same rounding as the scan
            h[n] = fmaf(dA, h[n], du * sB[n]);
            y = fmaf(sC[n], h[n], y);
        }
    }
    if (!valid) return;
#pragma unroll
    for (int q = 0; q < N / 4; ++q)
        __stcs(srow + q, make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]));
    y = fmaf(Dd, uu, y);
    if (a.z) y *= silu(zz);
    Elem<T>::store(static_cast<T*>(a.out) + ch, y);
}

template <typename T, bool VEC>
static cudaError_t launch_update_v(const UpdateArgs& a, cudaStream_t s) {
    if (VEC && a.batch <= 65535 && (a.N == 8 || a.N == 16 || a.N == 32) &&
        reinterpret_cast<uintptr_t>(a.A) % 16 == 0) {
        const dim3 grid((unsigned)((a.d_inner + 127) / 128), (unsigned)a.batch);
        switch (a.N) {
            case 8: state_update_row_kernel<T, 8><<<grid, 128, 0, s>>>(a); break;
            case 16: state_update_row_kernel<T, 16><<<grid, 128, 0, s>>>(a); break;
            default: state_update_row_kernel<T, 32><<<grid, 128, 0, s>>>(a); break;
        }
        return cudaGetLastError();
    }
    const int G = lanes_per_channel(a.N);
    const int64_t threads = a.batch * a.d_inner * G;
    const unsigned nb = (unsigned)((threads + kUpdateThreads - 1) / kUpdateThreads);
    switch (G) {
        case 1: state_update_kernel<T, 1, VEC><<<nb, kUpdateThreads, 0, s>>>(a); break;
        case 2: state_update_kernel<T, 2, VEC><<<nb, kUpdateThreads, 0, s>>>(a); break;
        case 4: state_update_kernel<T, 4, VEC><<<nb, kUpdateThreads, 0, s>>>(a); break;
        case 8: state_update_kernel<T, 8, VEC><<<nb, kUpdateThreads, 0, s>>>(a); break;
        default: state_update_kernel<T, 16, VEC><<<nb, kUpdateThreads, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_state_update(const UpdateArgs& a, msc_dtype dtype, cudaStream_t s) {
    if (dtype == MSC_BF16)
        return a.vec ? launch_update_v<__nv_bfloat16, true>(a, s)
                     : launch_update_v<__nv_bfloat16, false>(a, s);
    return a.vec ? launch_update_v<float, true>(a, s) : launch_update_v<float, false>(a, s);
}

}  // namespace msc
