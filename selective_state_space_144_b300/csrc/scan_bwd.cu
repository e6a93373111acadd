// scan_bwd.cu -- backward pass of the selective scan (Euler form) for sm_103a.
//
// Gradients of a loss of (out, last_state) with respect to u, dt, A, B, C,
// D, z, dt_bias and h0, given dout and dlast_state.  The pages' design
// recomputes the states instead of storing them ("Deep dive into Mamba",
// section 7.3: chunk + recompute; the Mamba series article, section 3); here:
//   1. the checkpoints: the state entering every segment of kSeg steps
//      (batch x (segments - 1) x d_inner x N fp32, segment 0 starting from
//      h0) -- from the forward's TMA chunk summaries and carry prefix with
//      chunks of kSeg steps where the shape allows, else from
//      scan_bwd_ckpt_kernel, which runs the recurrence once keeping them;
//   2. scan_bwd_kernel walks the segments from last to first: it recomputes
//      the segment's states from its checkpoint into shared memory, then
//      runs the adjoint recurrence backwards,
//          dy_t = dout_t silu(z_t),  dh_t = C_t dy_t + exp(delta_{t+1} A) dh_{t+1},
//      forming per step du, ddt (through softplus' = sigmoid) and dz (through
//      silu'), and accumulating dA, dD, ddt_bias in registers and dB, dC (sums
//      over channels) in per-segment shared-memory accumulators (warp sums
//      added there atomically, no barrier per step), flushed with one global
//      atomic add per (batch, step, state) and CTA.
// Thread layout as the element-load forward kernels: G lanes per channel,
// 4 states per lane, 128 threads per CTA, grid (channel tiles, batch).
#include "msc_device.cuh"
#include "msc_internal.h"

namespace msc {

constexpr int kBwdThreads = 128;
constexpr int kSeg = 32;  // steps per recomputed segment (states kept in shared memory)

__device__ __forceinline__ float sigmoid_f(float x) {
    return __fdividef(1.0f, 1.0f + ex2(-x * kLog2e));
}

template <typename T, int G, bool VEC>
__global__ void __launch_bounds__(kBwdThreads)
scan_bwd_ckpt_kernel(BwdArgs a) {
    constexpr int CPB = kBwdThreads / G;
    const int g = threadIdx.x % G;
    const int64_t d_raw = (int64_t)blockIdx.x * CPB + threadIdx.x / G;
    const int64_t b = blockIdx.y;
    const bool dvalid = d_raw < a.d_inner;
    const int64_t d = dvalid ? d_raw : a.d_inner - 1;
    const int N = (int)a.N, n0 = g * 4;
    float A2[4], h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int n = n0 + j;
        A2[j] = (n < N) ? __ldg(a.A + d * N + n) * kLog2e : 0.0f;
        h[j] = (a.h0 && n < N) ? a.h0[(b * a.d_inner + d) * N + n] : 0.0f;
    }
    const float bias = a.dt_bias ? __ldg(a.dt_bias + d) : 0.0f;
    const int64_t base = b * a.L * a.d_inner + d;
    const T* up = static_cast<const T*>(a.u) + base;
    const T* dtp = static_cast<const T*>(a.dt) + base;
    const T* Bp = static_cast<const T*>(a.B) + b * a.L * N;
    // segment sg + 1 enters with the state after step (sg + 1) * kSeg - 1,
    // kept at index sg (the layout of the forward's chunk carries)
    for (int64_t sg = 0; sg < a.nseg - 1; ++sg) {
#pragma unroll 8
        for (int t = 0; t < kSeg; ++t) {
            const int64_t off = (sg * kSeg + t) * a.d_inner;
            const float delta = softplus(Elem<T>::load(dtp + off) + bias);
            const float du = delta * Elem<T>::load(up + off);
            float Bv[4];
            load_row4<T, VEC>(Bp + (sg * kSeg + t) * N, n0, N, Bv);
#pragma unroll
            for (int j = 0; j < 4; ++j) h[j] = fmaf(ex2(delta * A2[j]), h[j], du * Bv[j]);
        }
        if (dvalid) {
            float* c = a.ckpt + ((b * (a.nseg - 1) + sg) * a.d_inner + d) * N;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (n0 + j < N) c[n0 + j] = h[j];
        }
    }
}

template <typename T, int G, bool VEC>
__global__ void __launch_bounds__(kBwdThreads)
scan_bwd_kernel(BwdArgs a) {
    constexpr int CPB = kBwdThreads / G;
    extern __shared__ float4 hbuf[];  // [kSeg][kBwdThreads] states after each step, then
                                      // float acc[2][kSeg][N]: the segment's dB, dC sums
    float* const acc = reinterpret_cast<float*>(hbuf + kSeg * kBwdThreads);
    const int g = threadIdx.x % G;
    const int lane = threadIdx.x & 31;
    const int64_t d_raw = (int64_t)blockIdx.x * CPB + threadIdx.x / G;
    const int64_t b = blockIdx.y;
    const bool dvalid = d_raw < a.d_inner;
    const int64_t d = dvalid ? d_raw : a.d_inner - 1;
    const int N = (int)a.N, n0 = g * 4;

    float A2[4], An[4], dh[4], dAacc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int n = n0 + j;
        An[j] = (n < N) ? __ldg(a.A + d * N + n) : 0.0f;
        A2[j] = An[j] * kLog2e;
        dh[j] = (dvalid && a.dlast && n < N) ? a.dlast[(b * a.d_inner + d) * N + n] : 0.0f;
        dAacc[j] = 0.0f;
    }
    const float bias = a.dt_bias ? __ldg(a.dt_bias + d) : 0.0f;
    const float Dd = a.D ? __ldg(a.D + d) : 0.0f;
    float dDacc = 0.0f, dbacc = 0.0f;
    const int64_t base = b * a.L * a.d_inner + d;
    const T* up = static_cast<const T*>(a.u) + base;
    const T* dtp = static_cast<const T*>(a.dt) + base;
    const T* zp = a.z ? static_cast<const T*>(a.z) + base : nullptr;
    const T* gp = static_cast<const T*>(a.dout) + base;
    const T* Bp = static_cast<const T*>(a.B) + b * a.L * N;
    const T* Cp = static_cast<const T*>(a.C) + b * a.L * N;
    const int64_t obase = b * a.L * N;

    for (int64_t sgi = a.nseg - 1; sgi >= 0; --sgi) {
        const int64_t t0 = sgi * kSeg;
        const int64_t t1 = min(t0 + kSeg, a.L);
        for (int i = threadIdx.x; i < 2 * kSeg * N; i += kBwdThreads) acc[i] = 0.0f;
        __syncthreads();
        // (1) recompute the segment's states from its checkpoint
        float hs0[4], h[4];
        const float* ck = sgi > 0 ? a.ckpt + ((b * (a.nseg - 1) + sgi - 1) * a.d_inner + d) * N
                                  : (a.h0 ? a.h0 + (b * a.d_inner + d) * N : nullptr);
#pragma unroll
        for (int j = 0; j < 4; ++j) hs0[j] = h[j] = (ck && n0 + j < N) ? ck[n0 + j] : 0.0f;
        const int nk = (int)(t1 - t0);
        const int64_t ds = a.d_inner;
        {
            const T* pdt = dtp + t0 * ds;
            const T* pu = up + t0 * ds;
            const T* pB = Bp + t0 * N;
#pragma unroll 8
            for (int k = 0; k < nk; ++k, pdt += ds, pu += ds, pB += N) {
                const float delta = softplus(Elem<T>::load(pdt) + bias);
                const float du = delta * Elem<T>::load(pu);
                float Bv[4];
                load_row4<T, VEC>(pB, n0, N, Bv);
#pragma unroll
                for (int j = 0; j < 4; ++j) h[j] = fmaf(ex2(delta * A2[j]), h[j], du * Bv[j]);
                hbuf[k * kBwdThreads + threadIdx.x] = make_float4(h[0], h[1], h[2], h[3]);
            }
        }
        // (2) the adjoint, last step of the segment first; each step's global
        // inputs are loaded one step ahead (before the previous step's
        // reduction barrier) so that their latency overlaps it
        struct In {
            float dt, u, z, go, B[4], C[4];
        };
        // running pointers at the step being loaded (k - 1 while k is computed)
        int64_t off_ld = (t1 - 1) * ds;
        const T* pB = Bp + (t1 - 1) * N;
        const T* pC = Cp + (t1 - 1) * N;
        auto load_in = [&](In& v) {
            v.dt = Elem<T>::load(dtp + off_ld);
            v.u = Elem<T>::load(up + off_ld);
            v.z = zp ? Elem<T>::load(zp + off_ld) : 0.0f;
            v.go = dvalid ? Elem<T>::load(gp + off_ld) : 0.0f;
            load_row4<T, VEC>(pB, n0, N, v.B);
            load_row4<T, VEC>(pC, n0, N, v.C);
        };
        In nxt;
        load_in(nxt);
        int64_t off = off_ld;
        for (int k = nk - 1; k >= 0; --k, off -= ds) {
            const In cur = nxt;
            if (k > 0) {
                off_ld -= ds;
                pB -= N;
                pC -= N;
                load_in(nxt);
            }
            const float x = cur.dt + bias;
            const float delta = softplus(x);
            const float uu = cur.u;
            const float go = cur.go;
            const float* Bv = cur.B;
            const float* Cv = cur.C;
            const float4 hv = hbuf[k * kBwdThreads + threadIdx.x];
            const float ht[4] = {hv.x, hv.y, hv.z, hv.w};
            float hp[4];
            if (k > 0) {
                const float4 pv = hbuf[(k - 1) * kBwdThreads + threadIdx.x];
                hp[0] = pv.x; hp[1] = pv.y; hp[2] = pv.z; hp[3] = pv.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) hp[j] = hs0[j];
            }
            // y_t (before the gate), needed for dz
            float y = 0.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j) y = fmaf(Cv[j], ht[j], y);
#pragma unroll
            for (int o = G / 2; o > 0; o >>= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
            y = fmaf(Dd, uu, y);
            float dy = go, dz = 0.0f;
            if (zp) {
                const float zz = cur.z;
                const float s = sigmoid_f(zz);
                dy = go * zz * s;
                dz = go * y * s * fmaf(zz, 1.0f - s, 1.0f);
            }
            float ddel = 0.0f, dus = 0.0f, dBp[4], dCp[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float ea = ex2(delta * A2[j]);
                dh[j] = fmaf(Cv[j], dy, dh[j]);
                dCp[j] = dy * ht[j];
                const float da = dh[j] * hp[j];
                dAacc[j] = fmaf(da * ea, delta, dAacc[j]);
                ddel = fmaf(da * ea, An[j], ddel);
                ddel = fmaf(dh[j] * Bv[j], uu, ddel);
                dBp[j] = dh[j] * delta * uu;
                dus = fmaf(dh[j] * delta, Bv[j], dus);
                dh[j] *= ea;
            }
#pragma unroll
            for (int o = G / 2; o > 0; o >>= 1) {
                ddel += __shfl_xor_sync(0xffffffffu, ddel, o);
                dus += __shfl_xor_sync(0xffffffffu, dus, o);
            }
            if (g == 0 && dvalid) {
                const float ddt = ddel * sigmoid_f(x);
                Elem<T>::store(static_cast<T*>(a.du) + base + off, fmaf(dy, Dd, dus));
                Elem<T>::store(static_cast<T*>(a.ddt) + base + off, ddt);
                if (a.dz) Elem<T>::store(static_cast<T*>(a.dz) + base + off, dz);
                dDacc = fmaf(dy, uu, dDacc);
                dbacc += ddt;
            }
            // dB_t, dC_t: sum over the CTA's channels (lanes G apart hold the
            // same states of neighbouring channels), then one add per state
#pragma unroll
            for (int o = G; o < 32; o <<= 1) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    dBp[j] += __shfl_xor_sync(0xffffffffu, dBp[j], o);
                    dCp[j] += __shfl_xor_sync(0xffffffffu, dCp[j], o);
                }
            }
            if (lane < G) {  // the warp's sums into the segment accumulators
                float* ab = acc + k * N;
                float* ac = acc + (kSeg + k) * N;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (n0 + j < N) {
                        atomicAdd(ab + n0 + j, dBp[j]);
                        atomicAdd(ac + n0 + j, dCp[j]);
                    }
                }
            }
        }
        // (3) the segment's dB, dC: one global add per (step, state) and CTA
        __syncthreads();
        for (int i = threadIdx.x; i < 2 * kSeg * N; i += kBwdThreads) {
            const int which = i / (kSeg * N), r = i % (kSeg * N);
            const int64_t t = t0 + r / N;
            if (t < t1) atomicAdd((which ? a.dC : a.dB) + obase + t * N + r % N, acc[i]);
        }
        __syncthreads();
    }
    if (!dvalid) return;
    if (a.dh0) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (n0 + j < N) a.dh0[(b * a.d_inner + d) * N + n0 + j] = dh[j];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (n0 + j < N) atomicAdd(a.dA + d * N + n0 + j, dAacc[j]);
    if (g == 0) {
        if (a.dD) atomicAdd(a.dD + d, dDacc);
        if (a.ddt_bias) atomicAdd(a.ddt_bias + d, dbacc);
    }
}

size_t scan_bwd_ckpt_bytes(int64_t batch, int64_t L, int64_t d_inner, int64_t N) {
    const int64_t nseg = (L + kSeg - 1) / kSeg;
    return (size_t)batch * (size_t)(nseg > 1 ? nseg - 1 : 1) * (size_t)d_inner * (size_t)N *
           sizeof(float);
}

template <typename T, int G, bool VEC>
static cudaError_t launch_bwd_g(BwdArgs a, cudaStream_t s) {
    constexpr int CPB = kBwdThreads / G;
    const dim3 grid((unsigned)((a.d_inner + CPB - 1) / CPB), (unsigned)a.batch);
    if (a.nseg > 1) {
        scan_bwd_ckpt_kernel<T, G, VEC><<<grid, kBwdThreads, 0, s>>>(a);
        profile_count(1);
    }
    const size_t smem = (size_t)kSeg * kBwdThreads * sizeof(float4) +
                        2 * (size_t)kSeg * (size_t)a.N * sizeof(float);
    auto kern = scan_bwd_kernel<T, G, VEC>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const ProfileMark m = profile_begin(s, MSC_PROF_SCAN_BWD);
    kern<<<grid, kBwdThreads, smem, s>>>(a);
    profile_end(m, s);
    profile_count(1);
    return cudaGetLastError();
}

template <typename T, bool VEC>
static cudaError_t launch_bwd_v(const BwdArgs& a, cudaStream_t s) {
    switch (lanes_per_channel(a.N)) {
        case 1: return launch_bwd_g<T, 1, VEC>(a, s);
        case 2: return launch_bwd_g<T, 2, VEC>(a, s);
        case 4: return launch_bwd_g<T, 4, VEC>(a, s);
        case 8: return launch_bwd_g<T, 8, VEC>(a, s);
        default: return launch_bwd_g<T, 16, VEC>(a, s);
    }
}

cudaError_t launch_scan_bwd(const BwdArgs& a, msc_dtype dtype, cudaStream_t s) {
    if (dtype == MSC_BF16)
        return a.vec ? launch_bwd_v<__nv_bfloat16, true>(a, s)
                     : launch_bwd_v<__nv_bfloat16, false>(a, s);
    return a.vec ? launch_bwd_v<float, true>(a, s) : launch_bwd_v<float, false>(a, s);
}

}  // namespace msc
