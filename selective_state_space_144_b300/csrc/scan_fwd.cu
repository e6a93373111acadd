// scan_fwd.cu -- the fused selective-scan forward kernels for sm_103a.
//
// Operation ("Deep dive into Mamba: architecture and implementation of
// selective state-space models", sections 4.4 and 5.2; gate and step-size
// bias from the MambaBlock of "State space models and Mamba"):
//     delta = softplus(dt + dt_bias);  h = exp(delta*A) * h + delta*B*u
//     y = C . h + D*u;  out = y * silu(z)
// (optionally with the zero-order-hold input matrix in place of delta*B, and
// an initial state h0 in place of zero) fused in one pass per time chunk: nothing of size (batch, L, d_inner, N)
// ever exists in memory; the state lives in registers.
//
// Work split.  A thread owns one channel d and 4 consecutive states of it;
// G = ceil(N/4) (rounded to a power of two) neighbouring lanes of a warp
// share a channel and add their partial C.h with butterfly shuffles.  When
// batch * d_inner channels do not fill the GPU, time is cut into K chunks
// (the segmented scan of the presentation article, section 3.2, and the
// chunk + recompute scheme of "Deep dive into Mamba", section 7.3):
//   pass 1 (chunks 0..K-2): run each chunk from a zero state, keep its end
//          state b_k and its transfer coefficient a_k = prod of the decays;
//   prefix:  fold (a_j, b_j) in order into the state entering every chunk
//          -- the associative combine (a1, b1) then (a2, b2) ->
//          (a2*a1, a2*b1 + b2) -- one thread per (batch, channel, state);
//   pass 2 (all chunks): rerun each chunk from its entering state and emit
//          outputs.
// The exponential uses the MUFU ex2 unit with log2(e) folded into A once.
#include "msc_device.cuh"
#include "msc_internal.h"

namespace msc {

template <typename T, int G, bool VEC, bool OUTPUT>
__global__ void __launch_bounds__(kScanThreads)
scan_chunk_kernel(ScanArgs a, int kgrid) {
    constexpr int CPB = kScanThreads / G;  // channels per block
    const int g = threadIdx.x % G;
    const int cl = threadIdx.x / G;
    int64_t bid = blockIdx.x;
    const int tile = (int)(bid % a.ntile);
    bid /= a.ntile;
    const int k = (int)(bid % kgrid);
    const int64_t b = bid / kgrid;
    const int64_t d_raw = (int64_t)tile * CPB + cl;
    const bool dvalid = d_raw < a.d_inner;
    const int64_t d = dvalid ? d_raw : a.d_inner - 1;  // idle lanes read in bounds
    const int N = (int)a.N;
    const int n0 = g * 4;

    const int64_t t0 = (int64_t)k * a.chunk;
    const int64_t t1 = min(t0 + a.chunk, a.L);

    float A2[4], iA[4], h[4], P[4];
    const float* h0 = (OUTPUT && k == 0) ? a.h0 : nullptr;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int n = n0 + j;
        const float Av = (n < N) ? __ldg(a.A + d * N + n) : 0.0f;
        A2[j] = Av * kLog2e;
        iA[j] = a.zoh ? 1.0f / Av : 0.0f;
        h[j] = (h0 && n < N) ? h0[(b * a.d_inner + d) * N + n] : 0.0f;
        P[j] = 1.0f;
    }
    if (OUTPUT && k > 0) {
        // state entering chunk k (carry_prefix_kernel, from the summaries)
        const int64_t w = ((b * (a.K - 1) + k - 1) * a.d_inner + d) * N;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (n0 + j < N) h[j] = a.ws_b[w + n0 + j];
    }

    const float bias = a.dt_bias ? __ldg(a.dt_bias + d) : 0.0f;
    const float Dd = a.D ? __ldg(a.D + d) : 0.0f;
    const int64_t base = b * a.L * a.d_inner + d;  // element (b, 0, d)
    const T* up = static_cast<const T*>(a.u) + base;
    const T* dtp = static_cast<const T*>(a.dt) + base;
    const T* zp = a.z ? static_cast<const T*>(a.z) + base : nullptr;
    T* op = static_cast<T*>(a.out) + base;
    const T* Bp = static_cast<const T*>(a.B) + b * a.L * N;
    const T* Cp = static_cast<const T*>(a.C) + b * a.L * N;
    const T* lamp = a.trap ? static_cast<const T*>(a.lam) + base : nullptr;

    // exponential trapezoid: B*u of the step before the current one, seeded
    // from the step before the chunk (or the caller's u_prev / B_prev)
    float bx[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (a.trap && (t0 > 0 || (a.u_prev && a.B_prev))) {
        float Bq[4];
        float uq;
        if (t0 > 0) {
            uq = Elem<T>::load(up + (t0 - 1) * a.d_inner);
            load_row4<T, false>(Bp + (t0 - 1) * N, n0, N, Bq);
        } else {
            uq = Elem<T>::load(static_cast<const T*>(a.u_prev) + b * a.d_inner + d);
            load_row4<T, false>(static_cast<const T*>(a.B_prev) + b * N, n0, N, Bq);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) bx[j] = uq * Bq[j];
    }

#pragma unroll 2
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t off = t * a.d_inner;
        const float x = Elem<T>::load(dtp + off) + bias;
        const float uu = Elem<T>::load(up + off);
        const float delta = softplus(x);
        const float du = delta * uu;
        float Bv[4];
        load_row4<T, VEC>(Bp + t * N, n0, N, Bv);
        // input term of state j: delta*B*u, the zero-order hold's gain*u*B,
        // or the trapezoid's (1-lambda)*delta*(B*u)_{t-1} + (lambda*delta*u)*B
        float tra = 0.0f, trc = 0.0f;
        if (a.trap) {
            const float lt = Elem<T>::load(lamp + off);
            tra = (1.0f - lt) * delta;
            trc = (lt * delta) * uu;
        }
        auto inject = [&](int j, float x2, float dA) {
            if (a.trap) {
                const float v = fmaf(tra, bx[j], trc * Bv[j]);
                bx[j] = uu * Bv[j];
                return v;
            }
            return a.zoh ? zoh_gain(x2, dA, delta, iA[j]) * uu * Bv[j] : du * Bv[j];
        };
        if (OUTPUT) {
            float Cv[4];
            load_row4<T, VEC>(Cp + t * N, n0, N, Cv);
            float y = 0.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float x2 = delta * A2[j];
                const float dA = ex2(x2);
                h[j] = fmaf(dA, h[j], inject(j, x2, dA));
                y = fmaf(Cv[j], h[j], y);
            }
#pragma unroll
            for (int o = G / 2; o > 0; o >>= 1)
                y += __shfl_xor_sync(0xffffffffu, y, o);
            if (g == 0 && dvalid) {
                y = fmaf(Dd, uu, y);
                if (zp) y *= silu(Elem<T>::load(zp + off));
                Elem<T>::store(op + off, y);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float x2 = delta * A2[j];
                const float dA = ex2(x2);
                h[j] = fmaf(dA, h[j], inject(j, x2, dA));
                P[j] *= dA;
            }
        }
    }
    if (!dvalid) return;
    if (OUTPUT) {
        if (k == a.K - 1 && a.last_state) {
            float* ls = a.last_state + (b * a.d_inner + d) * N;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (n0 + j < N) ls[n0 + j] = h[j];
        }
    } else {
        const int64_t w = ((b * (a.K - 1) + k) * a.d_inner + d) * N;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (n0 + j < N) {
                a.ws_a[w + n0 + j] = P[j];
                a.ws_b[w + n0 + j] = h[j];
            }
        }
    }
}

// Entering states of the time chunks from their summaries: one thread per
// (batch, channel, state) folds (a_k, b_k), k = 0..K-2, in order with the
// combine (a1, b1) then (a2, b2) -> (a2*a1, a2*b1 + b2) applied to a state
// (presentation article, section 3.2), starting from h0 (or zero), and
// overwrites b_k with the state entering chunk k+1.  The output kernels then
// read one state per chunk instead of folding all earlier summaries.
__global__ void __launch_bounds__(256)
carry_prefix_kernel(const float* __restrict__ ws_a, float* ws_b, const float* __restrict__ h0,
                    int64_t batch, int K, int64_t dn) {
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;  // (b, d, n) flat
    if (i >= batch * dn) return;
    const int64_t b = i / dn, e = i - b * dn;
    float h = h0 ? h0[i] : 0.0f;
    const int64_t base = b * (int64_t)(K - 1) * dn + e;
#pragma unroll 8
    for (int k = 0; k < K - 1; ++k) {
        const int64_t w = base + (int64_t)k * dn;
        h = fmaf(ws_a[w], h, ws_b[w]);
        ws_b[w] = h;
    }
}

cudaError_t launch_carry_prefix(const ScanArgs& a, cudaStream_t s) {
    const int64_t dn = a.d_inner * a.N;
    const int64_t n = a.batch * dn;
    carry_prefix_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a.ws_a, a.ws_b, a.h0,
                                                                   a.batch, a.K, dn);
    return cudaGetLastError();
}

int lanes_per_channel(int64_t N) {
    return N <= 4 ? 1 : N <= 8 ? 2 : N <= 16 ? 4 : N <= 32 ? 8 : 16;
}

ScanPlan make_scan_plan(int64_t batch, int64_t L, int64_t d_inner, int64_t N,
                        int sm_count, int64_t force_chunks, int64_t min_chunk) {
    ScanPlan p{};
    p.G = lanes_per_channel(N);
    const int64_t cpb = kScanThreads / p.G;
    p.ntile = (int)((d_inner + cpb - 1) / cpb);
    const int64_t blocks1 = batch * p.ntile;
    int64_t K = 1;
    if (L > 0) {
        if (force_chunks > 0) {
            K = force_chunks;
        } else {
            const int64_t target = (int64_t)sm_count * 8;  // 32 warps per SM
            K = blocks1 > 0 ? (target + blocks1 - 1) / blocks1 : 1;
            const int64_t maxK = L / (min_chunk > 0 ? min_chunk : 1);
            K = K < maxK ? K : maxK;
        }
        K = K < 1 ? 1 : K;
        K = K > L ? L : K;
        p.chunk = (L + K - 1) / K;
        K = (L + p.chunk - 1) / p.chunk;
    } else {
        p.chunk = 1;
    }
    p.K = (int)K;
    p.tma = 0;
    p.ws_carry = K > 1 ? 2 * (size_t)batch * (size_t)(K - 1) * (size_t)d_inner *
                             (size_t)N * sizeof(float)
                       : 0;
    p.ws_bc = 0;
    p.ws_bytes = p.ws_carry;
    return p;
}

static size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

ScanPlan make_tma_plan(int64_t batch, int64_t L, int64_t d_inner, int64_t N, int sm_count,
                       int64_t force_chunks, int64_t min_chunk, bool need_bc, int64_t force_lanes) {
    ScanPlan p{};
    p.tma = 1;
    const int64_t target = (int64_t)sm_count * 8;  // 2 warps per SM sub-partition
    // 2 lanes per channel (8 states each for N = 16) need half the shared-
    // memory traffic and shuffles per update of 4 lanes; take them when the
    // channels alone still fill the GPU, and always for N <= 32 when forced
    int G = 4;
    if (force_lanes == 2 && N <= 32 && d_inner % 16 == 0) {
        G = 2;
    } else if (force_lanes == 0 && N <= 32 && d_inner % 16 == 0 &&
               batch * (d_inner / 16) >= target) {
        G = 2;
    }
    p.G = G;
    const int64_t cpw = 32 / G;
    p.ntile = (int)(d_inner / cpw);
    const int64_t TT = tma_scan_tile(N);
    const int64_t warps1 = batch * p.ntile;  // one warp per CTA
    int64_t K = 1;
    if (L > 0) {
        if (force_chunks > 0) {
            K = force_chunks;
        } else {
            // Once time must be cut, cut it finer than the minimum that fills
            // the GPU: the summary pass of a chunk whose decays stay near 1
            // walks all of it, so shorter chunks shorten the slowest warps'
            // walks, and several waves of CTAs even out the rest.
            constexpr int64_t kChunkWaves = 7;
            K = warps1 >= target ? 1 : (kChunkWaves * target + warps1 - 1) / warps1;
            const int64_t maxK = L / (min_chunk > 0 ? min_chunk : 1);
            K = K < maxK ? K : maxK;
        }
        K = K < 1 ? 1 : K;
        int64_t chunk = (L + K - 1) / K;
        chunk = (chunk + TT - 1) / TT * TT;  // chunk boundaries on tile boundaries
        p.chunk = chunk;
        K = (L + chunk - 1) / chunk;
    } else {
        p.chunk = TT;
    }
    p.K = (int)K;
    p.ws_carry = K > 1 ? round256(2 * (size_t)batch * (size_t)(K - 1) * (size_t)d_inner *
                                  (size_t)N * sizeof(float))
                       : 0;
    p.ws_bc = need_bc ? 2 * round256((size_t)batch * (size_t)L * (size_t)N * sizeof(float)) : 0;
    p.ws_bytes = p.ws_carry + p.ws_bc;
    return p;
}

template <typename T, int G, bool VEC>
static cudaError_t launch_scan_g(const ScanArgs& a, const ScanPlan& p,
                                 cudaStream_t s) {
    if (p.K > 1) {
        const int64_t nb = a.batch * (int64_t)(p.K - 1) * p.ntile;
        scan_chunk_kernel<T, G, VEC, false>
            <<<(unsigned)nb, kScanThreads, 0, s>>>(a, p.K - 1);
        const cudaError_t e = launch_carry_prefix(a, s);
        if (e != cudaSuccess) return e;
    }
    const int64_t nb = a.batch * (int64_t)p.K * p.ntile;
    const ProfileMark m = profile_begin(s, MSC_PROF_SCAN);
    scan_chunk_kernel<T, G, VEC, true><<<(unsigned)nb, kScanThreads, 0, s>>>(a, p.K);
    profile_end(m, s);
    profile_count(p.K > 1 ? 3 : 1);
    return cudaGetLastError();
}

template <typename T, bool VEC>
static cudaError_t launch_scan_v(const ScanArgs& a, const ScanPlan& p,
                                 cudaStream_t s) {
    switch (p.G) {
        case 1: return launch_scan_g<T, 1, VEC>(a, p, s);
        case 2: return launch_scan_g<T, 2, VEC>(a, p, s);
        case 4: return launch_scan_g<T, 4, VEC>(a, p, s);
        case 8: return launch_scan_g<T, 8, VEC>(a, p, s);
        default: return launch_scan_g<T, 16, VEC>(a, p, s);
    }
}

cudaError_t launch_scan(const ScanArgs& a, const ScanPlan& p, msc_dtype dtype,
                        cudaStream_t s) {
    if (dtype == MSC_BF16) {
        return a.vec ? launch_scan_v<__nv_bfloat16, true>(a, p, s)
                     : launch_scan_v<__nv_bfloat16, false>(a, p, s);
    }
    return a.vec ? launch_scan_v<float, true>(a, p, s)
                 : launch_scan_v<float, false>(a, p, s);
}

}  // namespace msc
