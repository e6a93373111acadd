// peaks.cu -- roofline denominators measured on the running GPU: MUFU ex2
// throughput, FP32 FFMA and packed FFMA2 throughput, and a streaming copy.
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

// The scan's per-update arithmetic without memory traffic: per iteration and
// thread 16 state updates (1 ex2, 2 FMUL, 2 FFMA each).
__global__ void k_update_core(float* sink, int64_t iters) {
    float A2[16], h[16], Bv[16], Cv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        A2[j] = -1.4426950f * (j + 1);
        h[j] = 0.f;
        Bv[j] = 0.1f * j - 0.7f;
        Cv[j] = 0.3f - 0.02f * j;
    }
    float delta = 0.01f + 1e-6f * threadIdx.x, du = 0.5f, acc = 0.f;
    for (int64_t it = 0; it < iters; ++it) {
        float y = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float dA = ex2_ftz(delta * A2[j]);
            h[j] = fmaf(dA, h[j], du * Bv[j]);
            y = fmaf(Cv[j], h[j], y);
        }
        acc += y;
        delta = fmaf(delta, 0.999f, 1e-5f);
        du = fmaf(du, 0.999f, 1e-4f);
    }
    if (acc == 1234.5f) sink[0] = acc;
}

// Shared-memory load throughput by access pattern: each iteration every
// lane issues 8 independent volatile loads of W bytes (W = 4, 8 or 16) from
// 8 precomputed addresses (so the loop is 8 loads + 8 adds).  The element
// a lane reads within each 512-byte block is set by `pattern`:
//   0 all lanes the same       1 lane & 3       2 lane >> 2      3 lane
//   4 lane >> 4                5 lane >> 3      6 lane & 7
template <int W>
__global__ void k_lds(float* sink, int64_t iters, int pattern) {
    __shared__ __align__(16) float sm[4096];
    for (int i = threadIdx.x; i < 4096; i += blockDim.x) sm[i] = 0.001f * i;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    int sel;
    switch (pattern) {
        case 0: sel = 0; break;
        case 1: sel = lane & 3; break;
        case 2: sel = lane >> 2; break;
        case 3: sel = lane; break;
        case 4: sel = lane >> 4; break;
        case 5: sel = lane >> 3; break;
        default: sel = lane & 7; break;
    }
    constexpr int E = W / 4;  // floats per load
    unsigned addr[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
        addr[r] = static_cast<unsigned>(__cvta_generic_to_shared(sm + r * 128 * E / 4 * 4 + sel * E));
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            if (E == 4) {
                float x, y, z, w;
                asm volatile("ld.volatile.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(x), "=f"(y), "=f"(z), "=f"(w) : "r"(addr[r]));
                acc[r] += x;
            } else if (E == 2) {
                float x, y;
                asm volatile("ld.volatile.shared.v2.f32 {%0, %1}, [%2];"
                             : "=f"(x), "=f"(y) : "r"(addr[r]));
                acc[r] += x;
            } else {
                float x;
                asm volatile("ld.volatile.shared.f32 %0, [%1];" : "=f"(x) : "r"(addr[r]));
                acc[r] += x;
            }
        }
    }
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r) s += acc[r];
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

// state updates = blocks * threads * iters * 16.
int msc_peak_update_core(float* sink, int blocks, int threads, int64_t iters,
                         cudaStream_t s, float* ms) {
    return timed(s, ms, [&] { k_update_core<<<blocks, threads, 0, s>>>(sink, iters); });
}

// shared loads (warp instructions) = blocks * (threads / 32) * iters * 8.
int msc_peak_lds(float* sink, int blocks, int threads, int64_t iters, int width_bytes,
                 int pattern, cudaStream_t s, float* ms) {
    if (width_bytes == 16)
        return timed(s, ms,
                     [&] { k_lds<16><<<blocks, threads, 0, s>>>(sink, iters, pattern); });
    if (width_bytes == 8)
        return timed(s, ms,
                     [&] { k_lds<8><<<blocks, threads, 0, s>>>(sink, iters, pattern); });
    return timed(s, ms, [&] { k_lds<4><<<blocks, threads, 0, s>>>(sink, iters, pattern); });
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
