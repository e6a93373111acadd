// msc_device.cuh -- fp32 device arithmetic shared by the scan and decode
// kernels: the step-size nonlinearity (softplus), the gate (silu), the
// exponential, and typed loads/stores for fp32 and bf16 storage.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "msc_ptx.cuh"

namespace msc {

constexpr float kLog2e = 1.4426950408889634f;

// 2^x on the MUFU pipe (PTX ex2.approx, flush-to-zero: results below the
// fp32 normal range become 0, which is the limit the decay tends to).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log(1 + e) for e in [0, 1] as e * P(2e - 1); P interpolates log1p(e)/e at
// the 9 Chebyshev nodes of [0, 1] (coefficients from gen_log1p_poly.py).
// Max relative error about 1.9e-7 in fp32, i.e. accurate where 1 + e
// rounding would lose the low bits of small e.
__device__ __forceinline__ float log1p_unit(float e) {
    const float s = fmaf(2.0f, e, -1.0f);
    float p = 2.0023837e-05f;
    p = fmaf(p, s, -6.695044e-05f);
    p = fmaf(p, s, 0.00018186837f);
    p = fmaf(p, s, -0.0006321981f);
    p = fmaf(p, s, 0.0022891003f);
    p = fmaf(p, s, -0.008463899f);
    p = fmaf(p, s, 0.033152375f);
    p = fmaf(p, s, -0.14426334f);
    p = fmaf(p, s, 0.8109302f);
    return __fmul_rn(e, p);
}

// softplus(x) = log(1 + e^x) = max(x, 0) + log(1 + e^-|x|).  The step size
// of the selective scan (the Delta of the pages' selection mechanism).  The
// last multiply and add are separately rounded (not fused), so that every
// kernel -- scalar here, on pairs in the TMA scan -- gets the same delta bit
// for bit, and a backward pass recomputing states from checkpoints that a
// forward kernel wrote walks the very same states.
__device__ __forceinline__ float softplus(float x) {
    const float e = ex2(-fabsf(x) * kLog2e);
    return __fadd_rn(fmaxf(x, 0.0f), log1p_unit(e));
}

// silu(z) = z * sigmoid(z) = z / (1 + e^-z).  For z -> -inf the divisor
// overflows to inf and the fast divide returns 0, the limit of silu.
__device__ __forceinline__ float silu(float z) {
    return __fdividef(z, 1.0f + ex2(-z * kLog2e));
}

// Zero-order-hold input gain of one state ("State space models and Mamba",
// discretisation; "Deep dive into Mamba", section 12): with A diagonal,
// Bbar_n = (exp(delta*A_n) - 1) / A_n * B_n = delta * phi1(delta*A_n) * B_n,
// phi1(x) = (e^x - 1) / x.  Inputs: x2 = delta*A_n*log2(e) (the exponent
// already formed for dA), dA = 2^x2, delta, and iA = 1/A_n.
//   |delta*A_n| < 1/4: delta * phi1 from its Taylor series to degree 4 in
//     x2 (coefficients (ln 2)^k / (k+1)!); truncation < 1.5e-6 relative
//     (the remainder x^5/6! + ... against phi1 >= 0.88), fp32 Horner
//     < 1e-7;
//   otherwise: dA * iA - iA in one FMA, where |dA - 1| > 0.22 keeps the
//     relative error of the 2-ulp exponential below 1.1e-6.
// The two branches thus meet at about the same error.  A_n = 0 takes the
// first branch and gives delta exactly.
constexpr float kZohSwitch = 0.36067376f;  // 1/4 in units of log2(e)
constexpr float kZohC1 = 0.34657359f;      // (ln 2)^k / (k+1)!, k = 1..4
constexpr float kZohC2 = 0.080075502f;
constexpr float kZohC3 = 0.013876027f;
constexpr float kZohC4 = 0.0019236258f;

__device__ __forceinline__ float zoh_gain(float x2, float dA, float delta, float iA) {
    float p = kZohC4;
    p = fmaf(p, x2, kZohC3);
    p = fmaf(p, x2, kZohC2);
    p = fmaf(p, x2, kZohC1);
    p = fmaf(p, x2, 1.0f);
    const float small = delta * p;
    const float large = fmaf(dA, iA, -iA);
    return fabsf(x2) < kZohSwitch ? small : large;
}

// 1/x on the MUFU pipe (PTX rcp.approx, flush-to-zero).
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// silu with the reciprocal written out, z * (1 / (1 + e^-z)): the scalar
// twin of silu2 (same operations per value), for kernels whose results must
// match a paired evaluation bit for bit.
__device__ __forceinline__ float silu_rcp(float z) {
    return z * rcp_approx(ex2(-z * kLog2e) + 1.0f);
}

// silu of both halves of a pair: z / (1 + e^-z).
__device__ __forceinline__ u64 silu2(u64 z2) {
    const float z0 = lo2(z2), z1 = hi2(z2);
    const u64 d = add2(pk2(ex2(-z0 * kLog2e), ex2(-z1 * kLog2e)), pk2(1.0f, 1.0f));
    return mul2(z2, pk2(rcp_approx(lo2(d)), rcp_approx(hi2(d))));
}

// ---- typed element access -------------------------------------------------
template <typename T> struct Elem;

template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float* p) { return __ldg(p); }
    static __device__ __forceinline__ void store(float* p, float v) { *p = v; }
    // store under a predicate, without a branch
    // (no memory clobber: for outputs the storing kernel does not read back)
    static __device__ __forceinline__ void store_if(bool pred, float* p, float v) {
        asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
                     "@q st.global.f32 [%0], %1;\n\t}" ::"l"(p), "f"(v), "r"((int)pred));
    }
    // 4 consecutive elements, p 16-byte aligned
    static __device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
        const float4 q = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    }
};

template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float bits_to_float(uint32_t b16) {
        return __uint_as_float(b16 << 16);
    }
    static __device__ __forceinline__ float load(const __nv_bfloat16* p) {
        const unsigned short b = __ldg(reinterpret_cast<const unsigned short*>(p));
        return bits_to_float(b);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, float v) {
        *p = __float2bfloat16_rn(v);
    }
    static __device__ __forceinline__ void store_if(bool pred, __nv_bfloat16* p, float v) {
        const unsigned short b = __bfloat16_as_ushort(__float2bfloat16_rn(v));
        asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
                     "@q st.global.b16 [%0], %1;\n\t}" ::"l"(p), "h"(b), "r"((int)pred));
    }
    // 4 consecutive elements, p 8-byte aligned
    static __device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
        const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
        v[0] = __uint_as_float(q.x << 16);
        v[1] = __uint_as_float(q.x & 0xffff0000u);
        v[2] = __uint_as_float(q.y << 16);
        v[3] = __uint_as_float(q.y & 0xffff0000u);
    }
};

// A shared-memory element as fp32 (bf16: its bits are the high half).
template <typename T> __device__ __forceinline__ float lds_scalar(const T* p);
template <> __device__ __forceinline__ float lds_scalar<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float lds_scalar<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(p))
                           << 16);
}

// Load elements [n0, n0 + 4) of a row of `n` elements into v, zero past n.
template <typename T, bool VEC>
__device__ __forceinline__ void load_row4(const T* row, int n0, int n, float (&v)[4]) {
    if (VEC) {  // n % 4 == 0 and the row 4-element aligned
        if (n0 < n) {
            Elem<T>::load4(row + n0, v);
        } else {
            v[0] = v[1] = v[2] = v[3] = 0.0f;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            v[j] = (n0 + j < n) ? Elem<T>::load(row + n0 + j) : 0.0f;
    }
}

}  // namespace msc
