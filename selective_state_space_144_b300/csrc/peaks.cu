// peaks.cu -- roofline denominators measured on the running GPU: MUFU ex2
// throughput, FP32 FFMA and packed FFMA2 throughput, the rate of the scan's
// per-update arithmetic alone, and a streaming copy.
// Each entry point launches its kernel once on `stream` and returns the
// device time in milliseconds, bracketed by CUDA events on that stream.
// The operation counts the caller divides by are stated per function.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 8 independent chains x <- 2^-x per thread and iteration: 8 ex2 each.
__global__ void k_ex2(float* sink, int64_t iters) {
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = 0.25f + 0.05f * i + 1e-7f * threadIdx.x;
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = ex2_ftz(-x[i]);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += x[i];
    if (s == 1234.5f) sink[0] = s;
}

// 8 independent FFMA chains per thread and iteration.
__global__ void k_ffma(float* sink, int64_t iters, float a, float b) {
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = 0.5f + 0.01f * i + 1e-7f * threadIdx.x;
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = fmaf(x[i], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += x[i];
    if (s == 1234.5f) sink[0] = s;
}

// 8 independent packed fma.rn.f32x2 chains per thread and iteration
// (16 fp32 FMAs).
__global__ void k_ffma2(float* sink, int64_t iters, float a, float b) {
    unsigned long long x[8], av, bv;
    asm("mov.b64 %0, {%1, %1};" : "=l"(av) : "f"(a));
    asm("mov.b64 %0, {%1, %1};" : "=l"(bv) : "f"(b));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float lo = 0.5f + 0.01f * i + 1e-7f * threadIdx.x, hi = lo + 0.003f;
        asm("mov.b64 %0, {%1, %2};" : "=l"(x[i]) : "f"(lo), "f"(hi));
    }
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x[i]) : "l"(av), "l"(bv));
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float lo, hi;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x[i]));
        s += lo + hi;
    }
    if (s == 1234.5f) sink[0] = s;
}

// The scan's per-update arithmetic with no memory traffic at all, as the
// scan kernels issue it: a lane holds 4 states as two fp32 pairs and per
// step forms dA = 2^(delta*A2) on MUFU (mul.f32x2 + 2 ex2), the input term
// (delta*u)*B (mul.f32x2), h = dA*h + input (fma.f32x2) and the partial
// C.h (fma.f32x2), then adds the pair's halves.  Its rate is the ceiling
// the scan's update core can reach on this GPU: per update one MUFU
// operation and four FMA-pipe operations (two packed instructions of two
// lanes each), issued through the same sub-partition.
__device__ __forceinline__ unsigned long long pk2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float lo2(unsigned long long v) {
    return __uint_as_float(static_cast<unsigned>(v & 0xffffffffull));
}
__device__ __forceinline__ float hi2(unsigned long long v) {
    return __uint_as_float(static_cast<unsigned>(v >> 32));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float ex2_f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void k_scan_core(float* sink, int64_t iters) {
    unsigned long long A2[2], h[2], B[2], C[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        A2[i] = pk2(-1.4426950f * (2 * i + 1), -1.4426950f * (2 * i + 2));
        h[i] = pk2(0.f, 0.f);
        B[i] = pk2(0.1f * i - 0.7f, 0.2f - 0.1f * i);
        C[i] = pk2(0.3f - 0.02f * i, 0.1f * i);
    }
    float dl = 0.01f + 1e-6f * threadIdx.x, du = 0.5f, acc = 0.f;
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float vdl = dl + 1e-7f * j, vdu = du - 1e-7f * j;
            const unsigned long long dl2 = pk2(vdl, vdl), du2 = pk2(vdu, vdu);
            unsigned long long y2 = pk2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const unsigned long long x2 = mul2(dl2, A2[i]);
                const unsigned long long dA = pk2(ex2_f(lo2(x2)), ex2_f(hi2(x2)));
                h[i] = fma2(dA, h[i], mul2(du2, B[i]));
                y2 = fma2(C[i], h[i], y2);
            }
            acc += lo2(y2) + hi2(y2);
        }
        dl = fmaf(dl, 0.999f, 1e-5f);
        du = fmaf(du, 0.999f, 1e-4f);
    }
    if (acc == 1234.5f) sink[0] = acc;
}

// MUFU and the FMA pipe together: per iteration and thread 8 independent
// ex2 and K2 packed fma.rn.f32x2 per pair of ex2 (K2 = 0 gives the ex2 rate
// with its operand arithmetic alone, K2 = 4 the scan core's ratio), so the
// caller can see how far the two pipes overlap.
// NE = false drops the ex2 (and their operand FMAs): the FMA work alone.
// SCALAR: 2*K2 scalar fma.rn.f32 instead of K2 packed ones (the same FLOPs).
template <int K2, bool NE = true, bool SCALAR = false>
__global__ void k_mufu_fma(float* sink, int64_t iters) {
    float e[8], g[16];
    unsigned long long f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        e[i] = -0.1f * (i + 1) - 1e-7f * threadIdx.x;
        f[i] = pk2(0.5f + 0.01f * i, 0.3f);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) g[i] = 0.5f + 0.01f * i;
    const unsigned long long a = pk2(0.9999f, 0.9998f), b = pk2(1e-4f, 2e-4f);
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            if constexpr (NE) {
                e[i] = ex2_f(-e[i] * 0.5f - 0.01f);
                e[i + 1] = ex2_f(-e[i + 1] * 0.5f - 0.01f);
            }
            if constexpr (SCALAR) {
#pragma unroll
                for (int k = 0; k < 2 * K2; ++k) {
                    float& x = g[(2 * i + k) & 15];
                    asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(x) : "f"(0.9999f), "f"(1e-4f));
                }
            } else {
#pragma unroll
                for (int k = 0; k < K2; ++k) f[(i + k) & 7] = fma2(f[(i + k) & 7], a, b);
            }
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += e[i] + lo2(f[i]) + hi2(f[i]);
#pragma unroll
    for (int i = 0; i < 16; ++i) s += g[i];
    if (s == 1234.5f) sink[0] = s;
}

__global__ void k_copy(float4* __restrict__ dst, const float4* __restrict__ src, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = src[i];
}

template <typename F>
int timed(cudaStream_t s, float* ms, F launch) {
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) return 1;
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return 1;
    }
    cudaEventRecord(e0, s);
    launch();
    cudaEventRecord(e1, s);
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) err = cudaEventSynchronize(e1);
    if (err == cudaSuccess) err = cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return err == cudaSuccess ? 0 : 1;
}

}  // namespace

extern "C" {

// ex2 operations = blocks * threads * iters * 8.
int msc_peak_ex2(float* sink, int blocks, int threads, int64_t iters, cudaStream_t s,
                 float* ms) {
    return timed(s, ms, [&] { k_ex2<<<blocks, threads, 0, s>>>(sink, iters); });
}

// fp32 FMAs = blocks * threads * iters * 8.
int msc_peak_ffma(float* sink, int blocks, int threads, int64_t iters, cudaStream_t s,
                  float* ms) {
    return timed(s, ms,
                 [&] { k_ffma<<<blocks, threads, 0, s>>>(sink, iters, 0.9999f, 1e-4f); });
}

// fp32 FMAs = blocks * threads * iters * 16 (8 packed instructions).
int msc_peak_ffma2(float* sink, int blocks, int threads, int64_t iters, cudaStream_t s,
                   float* ms) {
    return timed(s, ms,
                 [&] { k_ffma2<<<blocks, threads, 0, s>>>(sink, iters, 0.9999f, 1e-4f); });
}

// state updates = blocks * threads * iters * 32 (8 steps x 4 states).
int msc_peak_scan_core(float* sink, int blocks, int threads, int64_t iters, cudaStream_t s,
                       float* ms) {
    return timed(s, ms, [&] { k_scan_core<<<blocks, threads, 0, s>>>(sink, iters); });
}

// ex2 operations = blocks * threads * iters * 8, with k2 (0, 2 or 4) packed
// FMAs per pair of them.
int msc_peak_mufu_fma(float* sink, int blocks, int threads, int64_t iters, int k2,
                      cudaStream_t s, float* ms) {
    if (k2 == 4) return timed(s, ms, [&] { k_mufu_fma<4><<<blocks, threads, 0, s>>>(sink, iters); });
    if (k2 == 2) return timed(s, ms, [&] { k_mufu_fma<2><<<blocks, threads, 0, s>>>(sink, iters); });
    return timed(s, ms, [&] { k_mufu_fma<0><<<blocks, threads, 0, s>>>(sink, iters); });
}

// The same loop in five mixes (per pair of ex2, with their two operand
// FMAs): 0 ex2 alone, 1 + 2 packed FMAs, 2 + 4 packed FMAs, 3 + 8 scalar
// FMAs, 4 the 4 packed FMAs without the ex2.  Iterations of 4 such groups per
// thread; time in ms.
int msc_peak_mix(float* sink, int blocks, int threads, int64_t iters, int mix,
                 cudaStream_t s, float* ms) {
    switch (mix) {
        case 0: return timed(s, ms, [&] { k_mufu_fma<0><<<blocks, threads, 0, s>>>(sink, iters); });
        case 1: return timed(s, ms, [&] { k_mufu_fma<2><<<blocks, threads, 0, s>>>(sink, iters); });
        case 2: return timed(s, ms, [&] { k_mufu_fma<4><<<blocks, threads, 0, s>>>(sink, iters); });
        case 3:
            return timed(s, ms, [&] {
                k_mufu_fma<4, true, true><<<blocks, threads, 0, s>>>(sink, iters);
            });
        case 4:
            return timed(s, ms, [&] {
                k_mufu_fma<4, false><<<blocks, threads, 0, s>>>(sink, iters);
            });
        default: return 1;
    }
}

// bytes moved = 2 * n16 * 16 (read + write); n16 = number of 16-byte words.
int msc_peak_copy(void* dst, const void* src, int64_t n16, int blocks, cudaStream_t s,
                  float* ms) {
    return timed(s, ms, [&] {
        k_copy<<<blocks, 256, 0, s>>>(static_cast<float4*>(dst),
                                      static_cast<const float4*>(src), n16);
    });
}

}  // extern "C"
