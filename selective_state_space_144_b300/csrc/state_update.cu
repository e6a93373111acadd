// state_update.cu -- single-token selective state update (decode) for sm_103a.
//
// One step of the scan's recurrence with the state read from and written
// back to HBM in place (the "Mamba decoding" example of "State space models
// and Mamba": constant memory per generated token):
//     delta = softplus(dt + dt_bias);  h = exp(delta*A) * h + delta*B*u
//     out = (C . h + D*u) * silu(z)
// (delta*B is replaced by the zero-order-hold input matrix when asked).
// The step is bound by streaming the fp32 state (8 bytes per state element
// per step).  state_update_stream_kernel (N = 16, Euler, aligned arrays)
// streams it through shared memory with bulk copies; state_update_row_kernel
// (N = 8, 16, 32, aligned arrays) keeps a whole channel per thread;
// state_update_kernel is the general form, a thread per 4 consecutive states
// with a shuffle reduction over the lanes of a channel.
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
    const float tq = tra * uq;  // the previous token's u weighted by (1-lambda)*delta
    float y = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float x2 = delta * A2[j];
        const float dA = ex2(x2);
        const float inj = a.trap  ? fmaf(trc, Bv[j], tq * Bq[j])
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
        const float tq = tra * uq;
#pragma unroll
        for (int n = 0; n < N; ++n) {
            const float dA = ex2(delta * (Av[n] * kLog2e));
            h[n] = fmaf(dA, h[n], fmaf(trc, sB[n], tq * sBq[n]));
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

// Set (bit 0) by a decode kernel whose bounded wait for a copy gave up.
__device__ unsigned int g_update_error;

// Decode step with the state streamed by the copy engine (N = 16, 32, 64).  A CTA owns one tile of CH = 2048 / N channels (8 KB of state) of
// every R-th batch row (rows r, r+R, ...) and walks those tiles through a
// ring of SS shared-memory stages: one thread issues 1-D bulk copies of each
// tile's state rows, u, dt, z (CH elements each) and the row's B, C into a
// stage, completing the stage's mbarrier, AHEAD tiles ahead; the CTA updates
// the states in place in shared memory and the same thread copies the
// tile's state back with a bulk store.  So the HBM stream is kept in flight
// by the copy engine rather than by the threads' registers, and A, dt_bias
// and D of the CTA's channels are read once per CTA.  Work split inside a
// tile: TPC = N / 4 threads per channel, thread t owning the float4 of
// states (t % TPC) of channels t / TPC + k * (128 / TPC), k = 0..3, so every
// shared access of a warp is 512 contiguous bytes; the TPC partial C.h of a
// channel are summed with log2(TPC) shuffles.
constexpr int kStreamThreads = 128;

// SS stages; the tile AHEAD steps ahead is loaded while one is updated and
// the store of an earlier one (SS - AHEAD stages) may still read its stage.
// TRAP: the exponential trapezoid's lambda and previous-token u (kX each)
// and B row follow the C row.
// A tile is CH = 2048 / N channels (8 KB of state); a channel's N states
// are N/4 threads' float4s.
template <typename T, int N_, int SS, bool TRAP = false>
struct StreamLayout {
    static constexpr int N = N_;
    static constexpr int CH = 2048 / N;                                 // channels per tile
    static constexpr int TPC = N / 4;                                   // threads per channel
    static constexpr int kState = CH * N * 4;                           // 8192
    static constexpr int kX = CH * (int)sizeof(T);                      // u / dt / z
    static constexpr int kBC = N * (int)sizeof(T);                      // B / C row
    static constexpr int kBCa = ((kBC + 15) / 16) * 16;
    static constexpr int kU = kState, kDt = kU + kX, kZ = kDt + kX;
    static constexpr int kB = kZ + kX, kC = kB + kBCa;
    static constexpr int kLam = kC + kBCa, kUp = kLam + kX, kBp = kUp + kX;
    static constexpr int kEnd = TRAP ? kBp + kBC : kC + kBC;
    static constexpr int kStage = ((kEnd + 127) / 128) * 128;
    static constexpr int kBar = SS * kStage;
    static constexpr int kTotal = kBar + SS * 8;
};

template <typename T, int N_, int SS, int AHEAD, int DISC>
__global__ void __launch_bounds__(kStreamThreads)
state_update_stream_kernel(UpdateArgs a, int nJ, int R, uint32_t wait_limit) {
    static_assert(AHEAD >= 1 && AHEAD <= SS - 2, "a stage for the update and one for a store");
    constexpr int kStreamStages = SS;
    constexpr int kStreamAhead = AHEAD;
    constexpr bool ZOH = DISC == 1, TRAP = DISC == 2;
    using Lay = StreamLayout<T, N_, SS, TRAP>;
    constexpr int N = Lay::N;
    constexpr int CH = Lay::CH, TPC = Lay::TPC;
    constexpr int CPP = kStreamThreads / TPC;  // channels per pass of the CTA's threads
    static_assert(CH == 4 * CPP, "four passes cover a tile");
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x;
    const int q = tid % TPC;
    const int j = blockIdx.x % nJ;
    const int r = blockIdx.x / nJ;
    const int64_t c0 = (int64_t)j * CH;
    const int nch = (int)min((int64_t)CH, a.d_inner - c0);
    const int nt = r < a.batch ? (int)((a.batch - 1 - r) / R + 1) : 0;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + Lay::kBar;
    const uint32_t xbytes = (uint32_t)(nch * sizeof(T));
    // trapezoid: the previous token's u and B, when both are given
    const bool prev = TRAP && a.u_prev && a.B_prev;
    const uint32_t tx = (uint32_t)(nch * N * 4) + (a.z ? 3u : 2u) * xbytes + 2u * Lay::kBC +
                        (TRAP ? xbytes : 0u) + (prev ? xbytes + (uint32_t)Lay::kBC : 0u);

    if (tid == 0) {
        for (int s2 = 0; s2 < kStreamStages; ++s2) mbar_init(bar0 + 8 * s2, 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int t) {  // thread 0: tile t (batch row r + t*R) into stage t % S
        const int st = t % kStreamStages;
        const uint32_t dst = sbase + st * Lay::kStage;
        const uint32_t bar = bar0 + 8 * st;
        const int64_t b = r + (int64_t)t * R;
        const int64_t ch = b * a.d_inner + c0;
        fence_proxy_async_smem();  // earlier generic accesses of the stage come first
        mbar_expect_tx(bar, tx);
        bulk_load(dst, a.state + ch * N, (uint32_t)(nch * N * 4), bar);
        bulk_load(dst + Lay::kU, static_cast<const T*>(a.u) + ch, xbytes, bar);
        bulk_load(dst + Lay::kDt, static_cast<const T*>(a.dt) + ch, xbytes, bar);
        if (a.z) bulk_load(dst + Lay::kZ, static_cast<const T*>(a.z) + ch, xbytes, bar);
        bulk_load(dst + Lay::kB, static_cast<const T*>(a.B) + b * N, Lay::kBC, bar);
        bulk_load(dst + Lay::kC, static_cast<const T*>(a.C) + b * N, Lay::kBC, bar);
        if constexpr (TRAP) {
            bulk_load(dst + Lay::kLam, static_cast<const T*>(a.lam) + ch, xbytes, bar);
            if (prev) {
                bulk_load(dst + Lay::kUp, static_cast<const T*>(a.u_prev) + ch, xbytes, bar);
                bulk_load(dst + Lay::kBp, static_cast<const T*>(a.B_prev) + b * N, Lay::kBC,
                          bar);
            }
        }
    };
    int issued = 0;
    if (tid == 0) {
        issued = a.starve ? 0 : min(kStreamAhead, nt);
        for (int t = 0; t < issued; ++t) issue(t);
    }

    // per-channel constants of the CTA's channels, once
    float A2[4][4], bias[4], Dd[4];
    [[maybe_unused]] float iA[ZOH ? 4 : 1][4];  // zero-order hold: 1/A
    bool valid[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int cl = it * CPP + tid / TPC;
        valid[it] = cl < nch;
        const int64_t d = c0 + (valid[it] ? cl : 0);
        const float4 av = __ldg(reinterpret_cast<const float4*>(a.A + d * N) + q);
        A2[it][0] = av.x * kLog2e; A2[it][1] = av.y * kLog2e;
        A2[it][2] = av.z * kLog2e; A2[it][3] = av.w * kLog2e;
        if constexpr (ZOH) {
            iA[it][0] = 1.0f / av.x; iA[it][1] = 1.0f / av.y;
            iA[it][2] = 1.0f / av.z; iA[it][3] = 1.0f / av.w;
        }
        bias[it] = a.dt_bias ? __ldg(a.dt_bias + d) : 0.0f;
        Dd[it] = a.D ? __ldg(a.D + d) : 0.0f;
    }

    bool ok = true;
    int t = 0;
    for (; t < nt; ++t) {
        const int st = t % kStreamStages;
        // refill: tile t + Ahead goes into the stage tile t + Ahead - S used;
        // its state store (committed two iterations ago) must have read it
        if (tid == 0 && t + kStreamAhead < nt && !a.starve) {
            bulk_wait_read<SS - AHEAD - 1>();
            issue(t + kStreamAhead);
            issued = t + kStreamAhead + 1;
        }
        ok = __syncthreads_and(mbar_wait(bar0 + 8 * st, (t / kStreamStages) & 1, wait_limit));
        if (!ok) break;
        unsigned char* sp = smem + st * Lay::kStage;
        const T* su = reinterpret_cast<const T*>(sp + Lay::kU);
        const T* sdt = reinterpret_cast<const T*>(sp + Lay::kDt);
        const T* sz = reinterpret_cast<const T*>(sp + Lay::kZ);
        float Bv[4], Cv[4];
        [[maybe_unused]] float Bq[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // trapezoid: B_prev
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            Bv[k] = lds_scalar<T>(reinterpret_cast<const T*>(sp + Lay::kB) + 4 * q + k);
            Cv[k] = lds_scalar<T>(reinterpret_cast<const T*>(sp + Lay::kC) + 4 * q + k);
            if constexpr (TRAP) {
                if (prev) Bq[k] = lds_scalar<T>(reinterpret_cast<const T*>(sp + Lay::kBp) + 4 * q + k);
            }
        }
        const int64_t b = r + (int64_t)t * R;
        T* outp = static_cast<T*>(a.out) + b * a.d_inner + c0;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int cl = it * CPP + tid / TPC;
            float4* hp = reinterpret_cast<float4*>(sp) + it * kStreamThreads + tid;
            float4 h = *hp;
            const float uu = lds_scalar<T>(su + cl);
            const float delta = softplus(lds_scalar<T>(sdt + cl) + bias[it]);
            const float du = delta * uu;
            float hv[4] = {h.x, h.y, h.z, h.w};
            float y = 0.0f;
            // the input term as the scan forms it (same operations, same order;
            // the trapezoid's as in the scan's steps after an octet's first)
            [[maybe_unused]] float tra = 0.0f, trc = 0.0f, uq = 0.0f;
            if constexpr (TRAP) {
                const float lt = lds_scalar<T>(reinterpret_cast<const T*>(sp + Lay::kLam) + cl);
                tra = (1.0f - lt) * delta;
                trc = (lt * delta) * uu;
                uq = prev ? lds_scalar<T>(reinterpret_cast<const T*>(sp + Lay::kUp) + cl) : 0.0f;
            }
            [[maybe_unused]] const float tq = tra * uq;  // weighted previous u
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float x2 = delta * A2[it][k];
                const float dA = ex2(x2);  // same rounding as the scan
                float inj;
                if constexpr (ZOH)
                    inj = zoh_gain(x2, dA, delta, iA[it][k]) * uu * Bv[k];
                else if constexpr (TRAP)
                    inj = fmaf(trc, Bv[k], tq * Bq[k]);
                else
                    inj = du * Bv[k];
                hv[k] = fmaf(dA, hv[k], inj);
                y = fmaf(Cv[k], hv[k], y);
            }
            *hp = make_float4(hv[0], hv[1], hv[2], hv[3]);
#pragma unroll
            for (int o = 1; o < TPC; o <<= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
            if (q == 0 && valid[it]) {
                y = fmaf(Dd[it], uu, y);
                if (a.z) y *= silu(lds_scalar<T>(sz + cl));
                Elem<T>::store(outp + cl, y);
            }
        }
        fence_proxy_async_smem();  // this thread's states, visible to the bulk store
        __syncthreads();           // ... and every thread's
        if (tid == 0) {
            bulk_store(a.state + (b * a.d_inner + c0) * N, sbase + st * Lay::kStage,
                       (uint32_t)(nch * N * 4));
            bulk_commit();
        }
    }
    if (!ok) {
        // a copy never completed: flag it and give the loads still in flight
        // a bounded chance to land before the shared memory is released
        if (tid == 0) {
            atomicOr(&g_update_error, 1u);
            for (int w = t; w < issued; ++w)
                mbar_wait(bar0 + 8 * (w % kStreamStages), (w / kStreamStages) & 1, wait_limit);
        }
    }
    if (tid == 0) bulk_wait_all();  // the stores have read shared memory and landed
}

bool stream_update_supported(const UpdateArgs& a, size_t es) {
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    // d_state 8 measured no faster than the thread-per-channel kernel (22.7
    // against 21.8 us on 256 x 5120): its state is small next to the inputs
    return (a.N == 16 || a.N == 32 || a.N == 64) &&
           (a.d_inner * (int64_t)es) % 16 == 0 && al16(a.state) && al16(a.A) &&
           al16(a.u) && al16(a.dt) && al16(a.B) && al16(a.C) && (!a.z || al16(a.z)) &&
           (!a.trap || (al16(a.lam) && (!a.u_prev || al16(a.u_prev)) &&
                        (!a.B_prev || al16(a.B_prev))));
}

template <typename T, int N, int SS, int AHEAD, int DISC>
static cudaError_t launch_stream_s(const UpdateArgs& a, int ctas_per_sm, cudaStream_t s) {
    using Lay = StreamLayout<T, N, SS, DISC == 2>;
    const int nJ = (int)((a.d_inner + Lay::CH - 1) / Lay::CH);
    const int64_t target = (int64_t)a.sms * ctas_per_sm;
    int64_t R = target / nJ;
    R = R < 1 ? 1 : (R > a.batch ? a.batch : R);
    const int64_t grid = (int64_t)nJ * R;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    auto kern = state_update_stream_kernel<T, N, SS, AHEAD, DISC>;
    if (Lay::kTotal > 48 * 1024)
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kTotal);
    kern<<<(unsigned)grid, kStreamThreads, Lay::kTotal, s>>>(a, nJ, (int)R, a.wait_limit);
    return cudaGetLastError();
}

// Three stages, one tile loading ahead, eight CTAs per SM (27 KB of shared
// memory each): measured on the 256 x 5120 x 16 step, 28.6 us with a cold
// L2 against 45.1 us for six stages four ahead at three CTAs per SM -- many
// small CTAs keep more tiles in flight than a few deep rings.
template <typename T, int N>
static cudaError_t launch_stream_n(const UpdateArgs& a, cudaStream_t s) {
    if (a.trap) return launch_stream_s<T, N, 3, 1, 2>(a, 8, s);
    // zero-order hold: more arithmetic per tile, so a deeper ring (4 stages,
    // 2 ahead, 6 CTAs per SM) measured 36.5-37.0 against 37.8-38.3 us; for the
    // trapezoid (larger stages) it measured 51 against 40 us
    if (a.zoh) return launch_stream_s<T, N, 4, 2, 1>(a, 6, s);
    return launch_stream_s<T, N, 3, 1, 0>(a, 8, s);
}

template <typename T>
static cudaError_t launch_stream(const UpdateArgs& a, cudaStream_t s) {
    switch (a.N) {
        case 16: return launch_stream_n<T, 16>(a, s);
        case 32: return launch_stream_n<T, 32>(a, s);
        default: return launch_stream_n<T, 64>(a, s);
    }
}

template <typename T, bool VEC>
static cudaError_t launch_update_v(const UpdateArgs& a, cudaStream_t s) {
    if (a.stream_ok && stream_update_supported(a, sizeof(T)))
        return launch_stream<T>(a, s);
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

cudaError_t update_error_word(unsigned int* value, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_update_error, sizeof(unsigned int));
    if (e == cudaSuccess && clear && *value) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_update_error, &zero, sizeof(unsigned int));
    }
    return e;
}

cudaError_t launch_state_update(const UpdateArgs& a, msc_dtype dtype, cudaStream_t s) {
    if (dtype == MSC_BF16)
        return a.vec ? launch_update_v<__nv_bfloat16, true>(a, s)
                     : launch_update_v<__nv_bfloat16, false>(a, s);
    return a.vec ? launch_update_v<float, true>(a, s) : launch_update_v<float, false>(a, s);
}

}  // namespace msc
