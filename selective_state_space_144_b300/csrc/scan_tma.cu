// scan_tma.cu -- the selective-scan forward for B300: TMA-staged tiles,
// fp32 state in registers, packed fp32x2 arithmetic.
//
// Operation ("Deep dive into Mamba: architecture and implementation of
// selective state-space models", sections 4.4 and 5.2; gate and step-size
// bias from the MambaBlock of "State space models and Mamba"):
//     delta = softplus(dt + dt_bias);  h = exp(delta*A) * h + delta*B*u
//     y = C . h + D*u;  out = y * silu(z)
// optionally with the zero-order-hold input matrix (exp(delta*A) - 1)/A * B
// in place of delta*B ("State space models and Mamba", discretisation) and
// an initial state h0 in place of zero (split prefill);
// all fused: the discretised A and B, and the states, never leave the chip
// (the kernel fusion and SRAM residency of the presentation article,
// section 3.3 -- restated here for TMA and registers).
//
// Work split.  One CTA is one warp and owns CPW = 32/G consecutive channels
// of one batch row for one time chunk.  Lane l works on channel l % CPW and
// on the NS = N/G consecutive states g*NS ... of it, g = l / CPW, held in
// registers as fp32 pairs.  Lanes that hold the same states are contiguous,
// so the per-step reads of B and C from shared memory are broadcasts that
// the shared-memory crossbar serves at full width.  Per tile of TT steps
// one lane issues five 3-D TMA loads into a ring of S stages -- u, dt, z as
// [TT x CPW] boxes and B, C (fp32) as [TT x N] boxes -- completing an
// mbarrier per stage; every lane waits on it (bounded).
//
// Time advances in octets of 8 steps.  Per octet each lane
//   * computes delta = softplus(dt + dt_bias) and delta*u for the 8/G steps
//     s = g, g+G, ... of the NEXT octet of its channel (in fp32 pairs) and
//     posts them to shared memory: the per-(step, channel) work is done
//     once, one octet ahead so that its latency overlaps the state updates;
//   * runs the 8 steps of the current octet on its states: dA = 2^(delta*A2)
//     on MUFU (A2 = A*log2 e), h = dA*h + (delta*u)*B, y += C*h, with
//     fma/mul.rn.f32x2 on state pairs; the 8 partial C.h stay in registers;
//   * reduce-scatters the partial C.h over the G lanes of its channel with
//     butterfly shuffles, ending with the full sums of steps g, g+G, ...,
//     adds D*u, applies the gate and stores those outputs.
// Steps past the end of the chunk get delta = 0, i.e. dA = 1 and no input:
// the state passes through unchanged and nothing is stored.
//
// Time chunks (K > 1) follow the segmented scan of the presentation
// article, section 3.2: the summary kernel runs chunks 0..K-2 from a zero
// state and records (prod dA, end state); carry_prefix_kernel folds them in
// order with the combine (a1, b1) then (a2, b2) -> (a2*a1, a2*b1 + b2) into
// the state entering every chunk; the output kernel starts from it.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <type_traits>

#include "msc_device.cuh"
#include "msc_internal.h"
#include "msc_ptx.cuh"

namespace msc {

// Set (bit 0) by a kernel whose bounded wait for a TMA copy gave up.
__device__ unsigned int g_scan_error;

constexpr int kOct = 8;  // steps per iteration
// Row stride (in float2) of a channel's (delta, delta*u) row in shared
// memory: the steps of a group padded by 2 (8 -> 10, 16 -> 18) so that the
// prologue's 8-byte stores from 8 channels and the core's 16-byte loads
// (2 steps) hit distinct banks.
constexpr int kDUStride = kOct + 2;

// Shared memory of one CTA: S stages of [u | dt | z | (lambda) | B | C]
// tiles, the (delta, delta*u) buffers (trapezoid: two sets), the barriers.
template <typename T, int G, int NS, int TT, int S, bool TRAP = false, int OCT = kOct>
struct TmaLayout {
    static constexpr int DUS = OCT + 2;                 // sDU row stride (float2)
    static constexpr int CPW = 32 / G;                  // channels per warp
    static constexpr int N = G * NS;
    static constexpr int NX = TRAP ? 4 : 3;             // [TT x CPW] tiles per stage
    static constexpr int kX = TT * CPW * (int)sizeof(T); // one of u / dt / z / lambda
    static constexpr int kBC = TT * N * 4;              // one of B / C (fp32) per stage
    static constexpr int kLam = 3 * kX;                 // lambda tile (trapezoid)
    static constexpr int kBoff = NX * kX;               // B tile
    static constexpr int kCoff = kBoff + kBC;           // C tile
    static constexpr int kStage = NX * kX + 2 * kBC;
    static constexpr int kDU = S * kStage;              // float2 [2][CPW][DUS]
    static constexpr int kDUsz = 2 * CPW * DUS * 8;
    static constexpr int kBar = kDU + (TRAP ? 2 : 1) * kDUsz;
    static constexpr int kTotal = kBar + S * 8;
    static_assert(kX % 128 == 0 && kBC % 128 == 0, "TMA destinations must stay 128B aligned");
    static_assert(TT % OCT == 0, "tiles hold whole groups of steps");
};

template <typename T> __device__ __forceinline__ float lds_elem(const T* p);
template <> __device__ __forceinline__ float lds_elem<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float lds_elem<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(p))
                           << 16);
}

// softplus of both halves of a pair: max(x, 0) + log1p(e), e = e^-|x|,
// log1p(e) = e * P(2e - 1) (the polynomial of log1p_unit, evaluated on pairs).
__device__ __forceinline__ u64 softplus2(u64 x2) {
    const float x0 = lo2(x2), x1 = hi2(x2);
    const u64 e = pk2(ex2(-fabsf(x0) * kLog2e), ex2(-fabsf(x1) * kLog2e));
    const u64 s = fma2(e, pk2(2.0f, 2.0f), pk2(-1.0f, -1.0f));
    u64 p = pk2(2.0023837e-05f, 2.0023837e-05f);
    p = fma2(p, s, pk2(-6.695044e-05f, -6.695044e-05f));
    p = fma2(p, s, pk2(0.00018186837f, 0.00018186837f));
    p = fma2(p, s, pk2(-0.0006321981f, -0.0006321981f));
    p = fma2(p, s, pk2(0.0022891003f, 0.0022891003f));
    p = fma2(p, s, pk2(-0.008463899f, -0.008463899f));
    p = fma2(p, s, pk2(0.033152375f, 0.033152375f));
    p = fma2(p, s, pk2(-0.14426334f, -0.14426334f));
    p = fma2(p, s, pk2(0.8109302f, 0.8109302f));
    return add2(pk2(fmaxf(x0, 0.0f), fmaxf(x1, 0.0f)), mul2(e, p));
}

// Zero-order-hold input gain of a state pair: zoh_gain (msc_device.cuh) on
// both halves, same operations in the same order (niA2 = -iA2).
__device__ __forceinline__ u64 zoh_gain2(u64 x2, u64 dA, u64 dl2, u64 iA2, u64 niA2) {
    u64 p = pk2(kZohC4, kZohC4);
    p = fma2(p, x2, pk2(kZohC3, kZohC3));
    p = fma2(p, x2, pk2(kZohC2, kZohC2));
    p = fma2(p, x2, pk2(kZohC1, kZohC1));
    p = fma2(p, x2, pk2(1.0f, 1.0f));
    const u64 small = mul2(dl2, p);
    const u64 large = fma2(dA, iA2, niA2);
    return pk2(fabsf(lo2(x2)) < kZohSwitch ? lo2(small) : lo2(large),
               fabsf(hi2(x2)) < kZohSwitch ? hi2(small) : hi2(large));
}

// Input term of a state pair: (delta*u)*B, or with zero-order hold
// (gain*u)*B, where `du2` carries delta*u, respectively u (see octet_prologue).
template <bool ZOH>
__device__ __forceinline__ u64 injection2(u64 x2, u64 dA, u64 dl2, u64 du2, u64 iA2, u64 niA2,
                                          u64 B2) {
    if constexpr (ZOH)
        return mul2(mul2(zoh_gain2(x2, dA, dl2, iA2, niA2), du2), B2);
    else
        return mul2(du2, B2);
}

// Reduce-scatter of the V per-step partial sums over the G lanes of a
// channel (lanes ch, ch + CPW, ...): afterwards out[m] holds the full sum of
// step g + G*m, m < V/G.
template <int G, int V = kOct>
__device__ __forceinline__ void reduce_scatter(const float (&y)[V], int lane,
                                               float (&out)[V / G]) {
    constexpr int CPW = 32 / G;
    if constexpr (G == 2) {
        const bool b0 = (lane / CPW) & 1;
#pragma unroll
        for (int m = 0; m < V / 2; ++m) {  // pair (2m, 2m+1): keep step 2m + b0
            const float send = b0 ? y[2 * m] : y[2 * m + 1];
            const float keep = b0 ? y[2 * m + 1] : y[2 * m];
            out[m] = keep + __shfl_xor_sync(0xffffffffu, send, CPW);
        }
    } else {
        static_assert(G == 4, "2 or 4 lanes per channel");
        const int g = lane / CPW;
        const bool b1 = (g >> 1) & 1, b0 = g & 1;
        float k[V / 2];
#pragma unroll
        for (int m = 0; m < V / 2; ++m) {  // steps (p, p+2), p = 4q + {0,1}: keep p + 2*b1
            const int p = (m & 1) + 4 * (m >> 1);
            const float send = b1 ? y[p] : y[p + 2];
            const float keep = b1 ? y[p + 2] : y[p];
            k[m] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * CPW);
        }
#pragma unroll
        for (int m = 0; m < V / 4; ++m) {  // (k[2m], k[2m+1]) = steps (4m+2b1, +1): keep +b0
            const float send = b0 ? k[2 * m] : k[2 * m + 1];
            const float keep = b0 ? k[2 * m + 1] : k[2 * m];
            out[m] = keep + __shfl_xor_sync(0xffffffffu, send, CPW);
        }
    }
}

// Per-(step, channel) prologue of one octet: delta = softplus(dt + dt_bias)
// and delta*u (ZOH: u, the gain being per state; trapezoid: lambda*delta*u,
// with ((1-lambda)*delta, u) in `dst2`) for steps g + G*m (m < 8/G) of the
// octet whose first row is `row0` of the tile at `stage`; written to `dst`
// (the lane's channel row of one sDU buffer, indexed by step) for the core.  The u of those steps is returned as pairs for the D*u
// term.  MASK: steps at or past `nsteps` get delta = 0 and no input (the
// state passes through).
template <typename T, int G, int TT, bool MASK, int DISC, bool GATE = false, int OCT = kOct>
__device__ __forceinline__ void octet_prologue(const unsigned char* stage, int row0, int lane_x,
                                               float2* dst, float2* dst2, u64 bias2,
                                               int s0_first, int nsteps,
                                               u64 (&uu)[OCT / G / 2],
                                               u64* gz = nullptr, bool has_z = false) {
    constexpr int CPW = 32 / G;
    constexpr int PPL = OCT / G / 2;
    const T* sx = reinterpret_cast<const T*>(stage) + row0 * CPW + lane_x;
#pragma unroll
    for (int p = 0; p < PPL; ++p) {
        const int r0 = G * (2 * p) * CPW, r1 = r0 + G * CPW;
        uu[p] = pk2(lds_elem<T>(sx + r0), lds_elem<T>(sx + r1));
        if constexpr (GATE) {  // silu(z) of the same steps, for the output epilogue
            if (has_z)
                gz[p] = silu2(pk2(lds_elem<T>(sx + 2 * TT * CPW + r0),
                                  lds_elem<T>(sx + 2 * TT * CPW + r1)));
        }
        const u64 x =
            add2(pk2(lds_elem<T>(sx + TT * CPW + r0), lds_elem<T>(sx + TT * CPW + r1)), bias2);
        const u64 dl = softplus2(x);
        u64 du, tra = 0;
        if constexpr (DISC == 2) {  // trapezoid: (lambda*delta)*u here, (1-lambda)*delta in dst2
            const u64 lt =
                pk2(lds_elem<T>(sx + 3 * TT * CPW + r0), lds_elem<T>(sx + 3 * TT * CPW + r1));
            du = mul2(mul2(lt, dl), uu[p]);
            tra = mul2(fma2(lt, pk2(-1.0f, -1.0f), pk2(1.0f, 1.0f)), dl);
        } else if constexpr (DISC == 1) {
            du = uu[p];
        } else {
            du = mul2(dl, uu[p]);
        }
        if (MASK) {
            const int s0 = s0_first + G * (2 * p);
            const bool v0 = s0 < nsteps, v1 = s0 + G < nsteps;
            dst[(2 * p) * G] = make_float2(v0 ? lo2(dl) : 0.0f, v0 ? lo2(du) : 0.0f);
            dst[(2 * p + 1) * G] = make_float2(v1 ? hi2(dl) : 0.0f, v1 ? hi2(du) : 0.0f);
            if constexpr (DISC == 2) {
                dst2[(2 * p) * G] = make_float2(v0 ? lo2(tra) : 0.0f, v0 ? lo2(uu[p]) : 0.0f);
                dst2[(2 * p + 1) * G] = make_float2(v1 ? hi2(tra) : 0.0f, v1 ? hi2(uu[p]) : 0.0f);
            }
        } else {
            dst[(2 * p) * G] = make_float2(lo2(dl), lo2(du));
            dst[(2 * p + 1) * G] = make_float2(hi2(dl), hi2(du));
            if constexpr (DISC == 2) {
                dst2[(2 * p) * G] = make_float2(lo2(tra), lo2(uu[p]));
                dst2[(2 * p + 1) * G] = make_float2(hi2(tra), hi2(uu[p]));
            }
        }
    }
}

// Exponential trapezoid: B*u of the step before a chunk for the lane's NS
// states -- step tc0 - 1 of the caller's u and B, or, for the first chunk,
// the caller's u_prev / B_prev (zero when absent).
template <typename T, int NS>
__device__ __forceinline__ void trap_seed(const ScanArgs& a, int b, int64_t d, int n0,
                                          int64_t tc0, u64 (&bx)[NS / 2]) {
    const T* ur;
    const T* Br;
    if (tc0 > 0) {
        ur = static_cast<const T*>(a.u) + ((int64_t)b * a.L + tc0 - 1) * a.d_inner + d;
        Br = static_cast<const T*>(a.B) + ((int64_t)b * a.L + tc0 - 1) * a.N + n0;
    } else if (a.u_prev && a.B_prev) {
        ur = static_cast<const T*>(a.u_prev) + (int64_t)b * a.d_inner + d;
        Br = static_cast<const T*>(a.B_prev) + (int64_t)b * a.N + n0;
    } else {
        return;
    }
    const float uq = Elem<T>::load(ur);
#pragma unroll
    for (int i = 0; i < NS / 2; ++i)
        bx[i] = pk2(uq * Elem<T>::load(Br + 2 * i), uq * Elem<T>::load(Br + 2 * i + 1));
}

template <typename T, int G, int NS, int TT, int S, int DISC, int OCT, bool CK = false>
__global__ void __launch_bounds__(32)
scan_tma_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dt,
                const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B,
                const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_lam,
                const ScanArgs a, const int kgrid) {
    constexpr bool ZOH = DISC == 1, TRAP = DISC == 2;
    using Lay = TmaLayout<T, G, NS, TT, S, TRAP, OCT>;
    constexpr int kDUStride = Lay::DUS;
    constexpr int kD2 = Lay::kDUsz / 8;  // second (delta) buffer, trapezoid only
    constexpr int CPW = Lay::CPW;
    constexpr int N = Lay::N;
    constexpr int NP = NS / 2;         // state pairs per lane
    constexpr int OPT = TT / OCT;     // octets per tile
    constexpr int SPL = OCT / G;      // steps per lane in the prologue / epilogue
    constexpr int PPL = SPL / 2;       // ... as fp32 pairs
    extern __shared__ __align__(128) unsigned char smem[];

    const int lane = threadIdx.x;
    const int ch = lane % CPW;
    const int g = lane / CPW;
    const int n0 = g * NS;
    int64_t bid = blockIdx.x;
    const int tile = (int)(bid % a.ntile);
    bid /= a.ntile;
    const int k = (int)(bid % kgrid);
    const int b = (int)(bid / kgrid);
    const int d0 = tile * CPW;
    const int64_t d = d0 + ch;
    const int64_t tc0 = (int64_t)k * a.chunk;
    const int nsteps = (int)min(a.chunk, a.L - tc0);
    const int ntiles = (nsteps + TT - 1) / TT;
    const bool has_z = a.z != nullptr;
    const uint32_t tx_bytes =
        (uint32_t)((2 + (has_z ? 1 : 0) + (TRAP ? 1 : 0)) * Lay::kX + 2 * Lay::kBC);

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + Lay::kBar;
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_u);
        prefetch_tensormap(&tm_dt);
        prefetch_tensormap(&tm_B);
        prefetch_tensormap(&tm_C);
        if (has_z) prefetch_tensormap(&tm_z);
        if (TRAP) prefetch_tensormap(&tm_lam);
    }
    __syncwarp();

    // u, dt, z, lambda are read once (evicted first); B and C, read by every
    // channel tile of the batch row, keep the default policy
    const uint64_t once = lane == 0 ? l2_evict_first_policy() : 0;
    auto issue = [&](int i) {  // lane 0: tile i of this chunk into stage i % S
        const uint32_t st = sbase + (i % S) * Lay::kStage;
        const uint32_t bar = bar0 + 8 * (i % S);
        const int32_t tt = (int32_t)(tc0 + (int64_t)i * TT);
        mbar_expect_tx(bar, tx_bytes);
        tma_load_3d_hint(st, &tm_u, bar, d0, tt, b, once);
        tma_load_3d_hint(st + Lay::kX, &tm_dt, bar, d0, tt, b, once);
        if (has_z) tma_load_3d_hint(st + 2 * Lay::kX, &tm_z, bar, d0, tt, b, once);
        if (TRAP) tma_load_3d_hint(st + Lay::kLam, &tm_lam, bar, d0, tt, b, once);
        tma_load_3d(st + Lay::kBoff, &tm_B, bar, 0, tt, b);
        tma_load_3d(st + Lay::kCoff, &tm_C, bar, 0, tt, b);
    };
    int issued = a.starve ? 0 : min(S, ntiles);
    if (lane == 0)
        for (int i = 0; i < issued; ++i) issue(i);

    // per-channel constants and the starting state
    const float bias = a.dt_bias ? __ldg(a.dt_bias + d) : 0.0f;
    const float Dd = a.D ? __ldg(a.D + d) : 0.0f;
    u64 A2[NP], iA2[NP], niA2[NP], hp[NP];
    const float* h0 = (a.h0 && k == 0) ? a.h0 + ((int64_t)b * a.d_inner + d) * N + n0 : nullptr;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        const float* Ar = a.A + d * N + n0 + 2 * i;
        const float a0 = __ldg(Ar), a1 = __ldg(Ar + 1);
        A2[i] = pk2(a0 * kLog2e, a1 * kLog2e);
        iA2[i] = ZOH ? pk2(1.0f / a0, 1.0f / a1) : pk2(0.0f, 0.0f);
        niA2[i] = ZOH ? pk2(-lo2(iA2[i]), -hi2(iA2[i])) : pk2(0.0f, 0.0f);
        hp[i] = h0 ? pk2(h0[2 * i], h0[2 * i + 1]) : pk2(0.0f, 0.0f);
    }
    if (k > 0) {  // state entering chunk k (carry_prefix_kernel)
        const int64_t w = ((int64_t)(b * (a.K - 1) + k - 1) * a.d_inner + d) * N + n0;
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const float2 v = *reinterpret_cast<const float2*>(a.ws_b + w + 2 * i);
            hp[i] = pk2(v.x, v.y);
        }
    }
    // trapezoid: B*u of the step before the chunk (or the caller's u_prev, B_prev)
    u64 bxp[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) bxp[i] = pk2(0.0f, 0.0f);
    if (TRAP) trap_seed<T, NS>(a, b, d, n0, tc0, bxp);

    float2* const sDU = reinterpret_cast<float2*>(smem + Lay::kDU);
    const u64 bias2 = pk2(bias, bias);
    const int lane_x = g * CPW + ch;  // element (row g, channel ch) of a [row][CPW] tile


    bool ok = ntiles == 0 || __all_sync(0xffffffffu, mbar_wait(bar0, 0, a.wait_limit));
    int waited = (ntiles > 0 && ok) ? 1 : 0;  // tiles [0, waited) are known complete
    // Per octet parity: the prologue's u and silu(z) of the lane's output
    // steps, and the core's per-step partial sums C.h.  The output epilogue
    // of an octet runs one octet later, beside the next octet's core, so
    // that its shuffle and store chains overlap independent work.
    u64 uz[2][PPL], gz[2][PPL];
    float yv[2][OCT];
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int p = 0; p < PPL; ++p) uz[q][p] = gz[q][p] = pk2(0.0f, 0.0f);
    if (ok && ntiles > 0)
        octet_prologue<T, G, TT, true, DISC, true, OCT>(smem, 0, lane_x, sDU + ch * kDUStride + g,
                                                   sDU + ch * kDUStride + g + kD2, bias2, g,
                                                   nsteps, uz[0], gz[0], has_z);
    __syncwarp();

    const u64 D2 = pk2(Dd, Dd);
    const int64_t dinner = a.d_inner;
    const int64_t gstride = (int64_t)G * dinner;  // output rows G apart
    T* out_p = static_cast<T*>(a.out) + ((int64_t)b * a.L + tc0 + g) * dinner + d;
    int st_idx = 0;                               // stage of tile i

    // Outputs of steps g + G*m of channel ch of the octet of parity Q whose
    // first row is chunk step sb, at op: reduce-scatter the partial sums,
    // add D*u, apply the gate, store.  MASKED: only steps before nsteps.
    auto epilogue = [&](auto q_tag, auto masked_tag, int sb, T* op) {
        constexpr int Q = decltype(q_tag)::value;
        constexpr bool MASKED = decltype(masked_tag)::value;
        float ys[SPL];
        reduce_scatter<G, OCT>(yv[Q], lane, ys);
#pragma unroll
        for (int p = 0; p < PPL; ++p) {
            u64 y2 = fma2(D2, uz[Q][p], pk2(ys[2 * p], ys[2 * p + 1]));
            if (has_z) y2 = mul2(y2, gz[Q][p]);
            T* o = op + (2 * p) * gstride;
            if (!MASKED) {
                Elem<T>::store(o, lo2(y2));
                Elem<T>::store(o + gstride, hi2(y2));
            } else {
                const int s0 = sb + g + G * (2 * p);
                if (s0 < nsteps) Elem<T>::store(o, lo2(y2));
                if (s0 + G < nsteps) Elem<T>::store(o + gstride, hi2(y2));
            }
        }
    };
    using P0 = std::integral_constant<int, 0>;
    using P1 = std::integral_constant<int, 1>;
    using Unmasked = std::integral_constant<bool, false>;
    using Masked = std::integral_constant<bool, true>;

    // One tile: OPT octets, unrolled so that every shared-memory offset and
    // every parity index is a constant.  FULL: the tile lies inside the
    // chunk, no step is masked.  OPT is even, so the octet of parity 1 that
    // ends a tile is the one pending when the next tile starts.
    static_assert(OPT % 2 == 0, "parity ring needs an even number of octets per tile");
    auto tile_body = [&](int i, auto full_tag) {
        constexpr bool FULL = decltype(full_tag)::value;
        const unsigned char* st = smem + st_idx * Lay::kStage;
        const int nxt_idx = st_idx + 1 == S ? 0 : st_idx + 1;
        const float* sB0 = reinterpret_cast<const float*>(st + Lay::kBoff) + n0;
        const float* sC0 = reinterpret_cast<const float*>(st + Lay::kCoff) + n0;
        bool flushed = false;
#pragma unroll
        for (int oo = 0; oo < OPT; ++oo) {
            const int sb = i * TT + OCT * oo;  // chunk step of the octet's first row
            if (!FULL && sb >= nsteps) {        // past the end of a partial tile:
                if (oo > 0) {                   // emit the pending octet, oo - 1
                    if ((oo - 1) & 1)
                        epilogue(P1{}, Masked{}, sb - OCT, out_p - OCT * dinner);
                    else
                        epilogue(P0{}, Masked{}, sb - OCT, out_p - OCT * dinner);
                }
                flushed = true;
                break;
            }
            // checkpoint for the backward pass: the state entering this
            // octet when it starts an interval of 2^ckpt_shift steps
            if (CK && ((tc0 + sb) & ((1 << a.ckpt_shift) - 1)) == 0) {
                float* cp = a.ckpt_out +
                            (((int64_t)b * a.ckpt_rows + ((tc0 + sb) >> a.ckpt_shift)) * a.d_inner +
                             d) * N + n0;
                // streaming stores: read again only by the backward pass
                if constexpr (NP == 1) {
                    __stcs(reinterpret_cast<float2*>(cp), make_float2(lo2(hp[0]), hi2(hp[0])));
                } else {
#pragma unroll
                    for (int i2 = 0; i2 < NP; i2 += 2)
                        __stcs(reinterpret_cast<float4*>(cp) + i2 / 2,
                               make_float4(lo2(hp[i2]), hi2(hp[i2]), lo2(hp[i2 + 1]),
                                           hi2(hp[i2 + 1])));
                }
            }
            // (1) the state updates of this octet
            const float4* sd =
                reinterpret_cast<const float4*>(sDU + ((oo & 1) * CPW + ch) * kDUStride);
            [[maybe_unused]] const float4* sd2 = sd + kD2 / 2;  // trapezoid: ((1-lambda)*delta, u)
            const float* sB = sB0 + OCT * oo * N;
            const float* sC = sC0 + OCT * oo * N;
#pragma unroll
            for (int j = 0; j < OCT; ++j) {
                const float4 v2 = sd[j >> 1];  // steps j & ~1 and (j & ~1) + 1
                const float vdl = (j & 1) ? v2.z : v2.x, vdu = (j & 1) ? v2.w : v2.y;
                const u64 dl2 = pk2(vdl, vdl), du2 = pk2(vdu, vdu);
                [[maybe_unused]] u64 tr2 = 0, ux2 = 0, qn2 = 0;
                if constexpr (TRAP) {
                    const float4 w2 = sd2[j >> 1];
                    const float vtr = (j & 1) ? w2.z : w2.x, vux = (j & 1) ? w2.w : w2.y;
                    tr2 = pk2(vtr, vtr);
                    ux2 = pk2(vux, vux);
                    if (j + 1 < OCT) {  // the next step's (1-lambda)*delta times this u
                        const float4 wn = sd2[(j + 1) >> 1];
                        const float qn = ((j + 1) & 1 ? wn.z : wn.x) * vux;
                        qn2 = pk2(qn, qn);
                    }
                }
                u64 Bp[NP], Cp[NP];
                if constexpr (NP == 1) {  // 2 states: one 8-byte read each
                    Bp[0] = *reinterpret_cast<const u64*>(sB + j * N);
                    Cp[0] = *reinterpret_cast<const u64*>(sC + j * N);
                } else {                  // 16-byte reads, two pairs each
#pragma unroll
                    for (int i2 = 0; i2 < NP; i2 += 2) {
                        const ulonglong2 bq =
                            *reinterpret_cast<const ulonglong2*>(sB + j * N + 2 * i2);
                        Bp[i2] = bq.x;
                        Bp[i2 + 1] = bq.y;
                        const ulonglong2 cq =
                            *reinterpret_cast<const ulonglong2*>(sC + j * N + 2 * i2);
                        Cp[i2] = cq.x;
                        Cp[i2 + 1] = cq.y;
                    }
                }
                u64 y2 = pk2(0.0f, 0.0f);
#pragma unroll
                for (int i2 = 0; i2 < NP; ++i2) {
                    const u64 x2 = mul2(dl2, A2[i2]);
                    const u64 dA = pk2(ex2(lo2(x2)), ex2(hi2(x2)));
                    u64 inj;
                    if constexpr (TRAP) {
                        // bxp: the previous step's u*B, already weighted by this
                        // step's (1-lambda)*delta except across octets, where
                        // the next octet's weights are not posted yet
                        if (j == 0)
                            inj = fma2(tr2, bxp[i2], mul2(du2, Bp[i2]));
                        else
                            inj = fma2(du2, Bp[i2], bxp[i2]);
                        bxp[i2] = j + 1 < OCT ? mul2(qn2, Bp[i2]) : mul2(ux2, Bp[i2]);
                    } else {
                        inj = injection2<ZOH>(x2, dA, dl2, du2, iA2[i2], niA2[i2], Bp[i2]);
                    }
                    hp[i2] = fma2(dA, hp[i2], inj);
                    y2 = fma2(Cp[i2], hp[i2], y2);
                }
                yv[oo & 1][j] = lo2(y2) + hi2(y2);
            }
            // (2) outputs of the previous octet (the last of the previous
            //     tile for oo = 0, a full tile: unmasked)
            if (oo > 0) {
                if ((oo - 1) & 1)
                    epilogue(P1{}, std::integral_constant<bool, !FULL>{}, sb - OCT,
                             out_p - OCT * dinner);
                else
                    epilogue(P0{}, std::integral_constant<bool, !FULL>{}, sb - OCT,
                             out_p - OCT * dinner);
            } else if (i > 0) {
                epilogue(P1{}, Unmasked{}, sb - OCT, out_p - OCT * dinner);
            }
            // (3) the next octet's step sizes, u and gate (next tile: wait
            //     for it first)
            float2* const dnx = sDU + (((oo + 1) & 1) * CPW + ch) * kDUStride + g;
            u64(&un)[PPL] = uz[(oo + 1) & 1];
            u64* gn = gz[(oo + 1) & 1];
            if (oo + 1 < OPT) {
                octet_prologue<T, G, TT, !FULL, DISC, true, OCT>(st, OCT * (oo + 1), lane_x, dnx,
                                                            dnx + kD2, bias2, sb + OCT + g,
                                                            nsteps, un, gn, has_z);
            } else if (i + 1 < ntiles) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * nxt_idx,
                                                       ((i + 1) / S) & 1, a.wait_limit));
                if (!ok) return;
                waited = i + 2;
                const unsigned char* stn = smem + nxt_idx * Lay::kStage;
                if ((i + 2) * TT <= nsteps)
                    octet_prologue<T, G, TT, false, DISC, true, OCT>(stn, 0, lane_x, dnx, dnx + kD2,
                                                                bias2, sb + OCT + g, nsteps,
                                                                un, gn, has_z);
                else
                    octet_prologue<T, G, TT, true, DISC, true, OCT>(stn, 0, lane_x, dnx, dnx + kD2,
                                                               bias2, sb + OCT + g, nsteps,
                                                               un, gn, has_z);
            }
            out_p += OCT * dinner;
            __syncwarp();
        }
        // the chunk's last octet of a full tile is still pending
        if (FULL && i + 1 == ntiles && !flushed)
            epilogue(P1{}, Unmasked{}, i * TT + TT - OCT, out_p - OCT * dinner);
        if (!FULL && !flushed)  // a partial tile whose octets were all run
            epilogue(P1{}, Masked{}, i * TT + TT - OCT, out_p - OCT * dinner);
        // (4) the tile is consumed: refill its stage
        if (i + S < ntiles) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(i + S);
            }
            issued = i + S + 1;
        }
        st_idx = nxt_idx;
    };

    for (int i = 0; ok && i < ntiles; ++i) {
        if ((i + 1) * TT <= nsteps)
            tile_body(i, std::integral_constant<bool, true>{});
        else
            tile_body(i, std::integral_constant<bool, false>{});
    }

    if (!ok) {
        // a copy never completed: flag it, give the copies still in flight a
        // bounded chance to land in this CTA's shared memory, then leave
        if (lane == 0) atomicOr(&g_scan_error, 1u);
        for (int i = waited; i < issued; ++i) mbar_wait(bar0 + 8 * (i % S), (i / S) & 1, a.wait_limit);
        return;
    }

    if (k == a.K - 1 && a.last_state) {
        float* ls = a.last_state + ((int64_t)b * a.d_inner + d) * N + n0;
#pragma unroll
        for (int i = 0; i < NP; ++i)
            *reinterpret_cast<float2*>(ls + 2 * i) = make_float2(lo2(hp[i]), hi2(hp[i]));
    }
}

// Chunk summary for the time-chunked scan (chunks 0..K-2, all full): the
// transfer coefficient a = prod of dA over the chunk and the chunk's end
// state from zero, b = sum_t (prod_{l>t} dA_l) dB_t u_t.  The chunk is walked
// backwards from its last step (Presentation article, section 3.2: segment
// summaries merged by the associative combine) with
//     b += P * dBu_t,   P = prod_{l>t} dA_l = 2^(A log2(e) * R),
//     R = sum_{l>t} delta_l   (one scalar per channel, grown by delta_t)
// -- the product of the later decays is an exponential of the sum of their
// step sizes, so it costs one exponent multiply and one ex2 per state and
// step, like a decay, and no running product.  The zero-order hold needs
// each step's own decay for its input gain and keeps P *= dA_t instead.
// The walk stops once every state of every lane of the warp has
// P < 2^-40: the remaining terms are below fp32 resolution of b and of the
// carry a*h (with A <= 0 the decays are <= 1, so P only falls; for A > 0 or
// NaN the walk covers the whole chunk).  Same lane layout, TMA ring and
// prologue as scan_tma_kernel; only u, dt and B are loaded.
constexpr float kSummaryCut = 9.094947e-13f;  // 2^-40
constexpr float kSummaryCutLog2 = -40.0f;

template <typename T, int G, int NS, int TT, int S, int DISC>
__global__ void __launch_bounds__(32)
scan_summary_kernel(const __grid_constant__ CUtensorMap tm_u,
                    const __grid_constant__ CUtensorMap tm_dt,
                    const __grid_constant__ CUtensorMap tm_B,
                    const __grid_constant__ CUtensorMap tm_lam, const ScanArgs a, const int kgrid) {
    constexpr bool ZOH = DISC == 1, TRAP = DISC == 2;
    using Lay = TmaLayout<T, G, NS, TT, S, TRAP>;
    constexpr int kD2 = Lay::kDUsz / 8;
    constexpr int CPW = Lay::CPW;
    constexpr int N = Lay::N;
    constexpr int NP = NS / 2;
    constexpr int OPT = TT / kOct;
    constexpr int PPL = kOct / G / 2;
    extern __shared__ __align__(128) unsigned char smem[];

    const int lane = threadIdx.x;
    const int ch = lane % CPW;
    const int g = lane / CPW;
    const int n0 = g * NS;
    int64_t bid = blockIdx.x;
    const int tile = (int)(bid % a.ntile);
    bid /= a.ntile;
    const int k = (int)(bid % kgrid);
    const int b = (int)(bid / kgrid);
    const int d0 = tile * CPW;
    const int64_t d = d0 + ch;
    const int64_t tc0 = (int64_t)k * a.chunk;
    const int ntiles = (int)(a.chunk / TT);  // summarised chunks are whole tiles
    const uint32_t tx_bytes = (uint32_t)((TRAP ? 3 : 2) * Lay::kX + Lay::kBC);

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + Lay::kBar;
    if (lane == 0) {
        for (int s2 = 0; s2 < S; ++s2) mbar_init(bar0 + 8 * s2, 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_u);
        prefetch_tensormap(&tm_dt);
        prefetch_tensormap(&tm_B);
        if (TRAP) prefetch_tensormap(&tm_lam);
    }
    __syncwarp();
    // r-th tile in walking order = tile ntiles-1-r of the chunk, stage r % S
    auto issue = [&](int r) {
        const uint32_t st = sbase + (r % S) * Lay::kStage;
        const uint32_t bar = bar0 + 8 * (r % S);
        const int32_t tt = (int32_t)(tc0 + (int64_t)(ntiles - 1 - r) * TT);
        mbar_expect_tx(bar, tx_bytes);
        tma_load_3d(st, &tm_u, bar, d0, tt, b);
        tma_load_3d(st + Lay::kX, &tm_dt, bar, d0, tt, b);
        if (TRAP) tma_load_3d(st + Lay::kLam, &tm_lam, bar, d0, tt, b);
        tma_load_3d(st + Lay::kBoff, &tm_B, bar, 0, tt, b);
    };
    int issued = a.starve ? 0 : min(S, ntiles);
    if (lane == 0)
        for (int r = 0; r < issued; ++r) issue(r);

    const float bias = a.dt_bias ? __ldg(a.dt_bias + d) : 0.0f;
    const u64 bias2 = pk2(bias, bias);
    u64 A2[NP], iA2[NP], niA2[NP], Pp[NP], bp[NP];
    u64 pend[NP];  // trapezoid: P * (1-lambda)*delta of the step after, awaiting B*u
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        const float* Ar = a.A + d * N + n0 + 2 * i;
        const float a0 = __ldg(Ar), a1 = __ldg(Ar + 1);
        A2[i] = pk2(a0 * kLog2e, a1 * kLog2e);
        iA2[i] = ZOH ? pk2(1.0f / a0, 1.0f / a1) : pk2(0.0f, 0.0f);
        niA2[i] = ZOH ? pk2(-lo2(iA2[i]), -hi2(iA2[i])) : pk2(0.0f, 0.0f);
        Pp[i] = pk2(1.0f, 1.0f);
        pend[i] = pk2(0.0f, 0.0f);
        bp[i] = pk2(0.0f, 0.0f);
    }
    float R = 0.0f;  // Euler, trapezoid: sum of delta over the steps walked
    float2* const sDU = reinterpret_cast<float2*>(smem + Lay::kDU);
    const int lane_x = g * CPW + ch;
    u64 uu[PPL];

    bool ok = ntiles == 0 || __all_sync(0xffffffffu, mbar_wait(bar0, 0, a.wait_limit));
    int waited = (ntiles > 0 && ok) ? 1 : 0;
    if (ok && ntiles > 0)
        octet_prologue<T, G, TT, false, DISC>(smem, kOct * (OPT - 1), lane_x,
                                              sDU + ch * kDUStride + g,
                                              sDU + ch * kDUStride + g + kD2, bias2, 0, 0, uu);
    __syncwarp();

    bool done = false;
    int c = 0;  // octets processed: sDU buffer c & 1
    for (int r = 0; ok && !done && r < ntiles; ++r) {
        const unsigned char* st = smem + (r % S) * Lay::kStage;
        const float* sB0 = reinterpret_cast<const float*>(st + Lay::kBoff) + n0;
#pragma unroll
        for (int oo = OPT - 1; oo >= 0; --oo, ++c) {
            // (1) the octet's steps, last to first
            const float4* sd =
                reinterpret_cast<const float4*>(sDU + ((c & 1) * CPW + ch) * kDUStride);
            [[maybe_unused]] const float4* sd2 = sd + kD2 / 2;
            const float* sB = sB0 + kOct * oo * N;
#pragma unroll
            for (int j = kOct - 1; j >= 0; --j) {
                const float4 v2 = sd[j >> 1];
                const float vdl = (j & 1) ? v2.z : v2.x, vdu = (j & 1) ? v2.w : v2.y;
                const u64 dl2 = pk2(vdl, vdl), du2 = pk2(vdu, vdu);
                [[maybe_unused]] u64 tr2 = 0, ux2 = 0;
                if constexpr (TRAP) {
                    const float4 w2 = sd2[j >> 1];
                    const float vtr = (j & 1) ? w2.z : w2.x, vux = (j & 1) ? w2.w : w2.y;
                    tr2 = pk2(vtr, vtr);
                    ux2 = pk2(vux, vux);
                }
                u64 Bp[NP];
                if constexpr (NP == 1) {
                    Bp[0] = *reinterpret_cast<const u64*>(sB + j * N);
                } else {
#pragma unroll
                    for (int i2 = 0; i2 < NP; i2 += 2) {
                        const ulonglong2 bq =
                            *reinterpret_cast<const ulonglong2*>(sB + j * N + 2 * i2);
                        Bp[i2] = bq.x;
                        Bp[i2 + 1] = bq.y;
                    }
                }
                [[maybe_unused]] const u64 R2 = pk2(R, R);
#pragma unroll
                for (int i2 = 0; i2 < NP; ++i2) {
                    if constexpr (ZOH) {
                        const u64 x2 = mul2(dl2, A2[i2]);
                        const u64 dA = pk2(ex2(lo2(x2)), ex2(hi2(x2)));
                        bp[i2] = fma2(Pp[i2],
                                      injection2<true>(x2, dA, dl2, du2, iA2[i2], niA2[i2], Bp[i2]),
                                      bp[i2]);
                        Pp[i2] = mul2(Pp[i2], dA);
                    } else {
                        const u64 x2 = mul2(R2, A2[i2]);
                        const u64 P = pk2(ex2(lo2(x2)), ex2(hi2(x2)));
                        if constexpr (TRAP) {
                            // this step's B*u meets the later step's deferred
                            // weight, and this step's own (lambda*delta*u)*B its
                            // weight P
                            bp[i2] = fma2(pend[i2], mul2(ux2, Bp[i2]), bp[i2]);
                            bp[i2] = fma2(P, mul2(du2, Bp[i2]), bp[i2]);
                            pend[i2] = mul2(P, tr2);
                        } else {
                            bp[i2] = fma2(P, mul2(du2, Bp[i2]), bp[i2]);
                        }
                    }
                }
                if constexpr (!ZOH) R += lo2(dl2);
            }
            // (2) the previous octet's step sizes (previous tile: wait first)
            float2* const dnx = sDU + (((c + 1) & 1) * CPW + ch) * kDUStride + g;
            if (oo > 0) {
                octet_prologue<T, G, TT, false, DISC>(st, kOct * (oo - 1), lane_x, dnx, dnx + kD2, bias2, 0, 0, uu);
            } else if (r + 1 < ntiles) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * ((r + 1) % S),
                                                       ((r + 1) / S) & 1, a.wait_limit));
                if (!ok) break;
                waited = r + 2;
                octet_prologue<T, G, TT, false, DISC>(smem + ((r + 1) % S) * Lay::kStage,
                                                kOct * (OPT - 1), lane_x, dnx, dnx + kD2, bias2, 0, 0, uu);
            }
            __syncwarp();
            // (3) stop once every later-decay product is below fp32 resolution
            //     (Euler, trapezoid: compared through its base-2 exponent)
            float pmax = -INFINITY;
#pragma unroll
            for (int i2 = 0; i2 < NP; ++i2) {
                const u64 v2 = ZOH ? Pp[i2] : mul2(pk2(R, R), A2[i2]);
                pmax = fmaxf(pmax, fmaxf(lo2(v2), hi2(v2)));
            }
            if (__all_sync(0xffffffffu, pmax < (ZOH ? kSummaryCut : kSummaryCutLog2))) {
                done = true;
                break;
            }
        }
        if (!ok || done) break;
        // (4) the tile is consumed: refill its stage with a tile further back
        if (r + S < ntiles) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(r + S);
            }
            issued = r + S + 1;
        }
    }
    // copies still in flight (early stop or a failed wait) land before exit
    for (int r = waited; r < issued; ++r) mbar_wait(bar0 + 8 * (r % S), (r / S) & 1, a.wait_limit);
    if (!ok) {
        if (lane == 0) atomicOr(&g_scan_error, 1u);
        return;
    }
    if (TRAP && !done) {  // the first step's (1-lambda)*delta term: B*u before the chunk
        u64 bxq[NP];
#pragma unroll
        for (int i = 0; i < NP; ++i) bxq[i] = pk2(0.0f, 0.0f);
        trap_seed<T, NS>(a, b, d, n0, tc0, bxq);
#pragma unroll
        for (int i = 0; i < NP; ++i) bp[i] = fma2(pend[i], bxq[i], bp[i]);
    }
    if constexpr (!ZOH) {  // the product of every walked step's decay
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const u64 x2 = mul2(pk2(R, R), A2[i]);
            Pp[i] = pk2(ex2(lo2(x2)), ex2(hi2(x2)));
        }
    }
    const int64_t w = ((int64_t)(b * (a.K - 1) + k) * a.d_inner + d) * N + n0;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        *reinterpret_cast<float2*>(a.ws_a + w + 2 * i) = make_float2(lo2(Pp[i]), hi2(Pp[i]));
        *reinterpret_cast<float2*>(a.ws_b + w + 2 * i) = make_float2(lo2(bp[i]), hi2(bp[i]));
    }
}

// Backward of the Euler scan on TMA tiles, checkpoints included.  One warp
// per CTA on CPW = 8 channels of one batch row, lane (ch, g) = (l % 8, l / 8)
// holding states g*NS .. g*NS+NS-1 of channel ch as fp32 pairs (the
// forward's lane layout).  The sequence is cut into tiles of TT steps, and
// the CTA makes one pass of 2*nt - 1 rounds over them through a TMA ring of
// S stages:
//   * forward rounds, tiles 0 .. nt-2 (u, dt, B loaded): the recurrence from
//     h0 (or zero), the state entering each next tile stored to the
//     checkpoint rows (batch, tile, d_inner, N) in global memory (they stay
//     in L2) -- skipped when a.ext_ckpt says the forward scan wrote those
//     rows already, the pass then starting at the last tile;
//   * reverse rounds, tiles nt-1 .. 0 (u, dt, z, dout, B, C loaded):
//       1. a tile prologue: every lane computes the per-(step, channel)
//          scalars for TT/4 of the tile's (step, channel) pairs -- delta,
//          delta*u, dy = dout*silu(z), u, softplus'(x) = sigmoid(x) and the
//          gate's slope for dz -- once, into a table in shared memory;
//       2. the tile's states recomputed from its entering state (the
//          forward's registers for the last tile, a checkpoint otherwise)
//          into a per-lane buffer, [TT][32 lanes][NS];
//       3. the adjoint from the tile's last step to its first, per state:
//            dh += C dy;  dC = dy h_t;  dae = dh h_{t-1} a   (a = e^{delta A})
//            dA += dae delta;  ddelta += dae A;  S += dh B;  dB = dh delta u;
//            dh *= a
//          then ddelta += u S and du = dy D + delta S over the channel's
//          states: the lane writes its partial (y, ddelta, S) over row j of
//          the state buffer (consumed by then), and after the tile every lane
//          sums the 4 partials of TT/4 (step, channel) pairs and stores dz,
//          ddt, du for them (with 2 states per lane, N = 8, the partials are
//          reduce-scattered over the channel's lanes every step instead); the lane's
//          2*NS values [dB | dC] are reduce-scattered over the 8 channels, and
//          each lane adds its slice of the sums to global memory with one
//          (vector) atomic add.
// dA, dD, ddt_bias accumulate in registers and are added once at the end;
// dh after tile 0 is dh0.  Steps past L in the last tile get delta = 0,
// dy = 0 (the state and the adjoint pass through) and store nothing.
template <typename T, int NS, int TT, int S>
struct BwdLayout {
    static constexpr int G = 4;
    static constexpr int CPW = 32 / G;
    static constexpr int N = G * NS;
    static constexpr int kX = TT * CPW * (int)sizeof(T);  // u / dt / z / dout tile
    static constexpr int kBC = TT * N * 4;                // B / C (fp32) tile
    static constexpr int kBoff = 4 * kX;
    static constexpr int kCoff = kBoff + kBC;
    static constexpr int kStage = 4 * kX + 2 * kBC;
    static constexpr int kTab = S * kStage;               // float4 [TT][CPW]: delta, delta*u, dy, u
    static constexpr int kTab2 = kTab + TT * CPW * 16;    // float2 [TT][CPW]: sigmoid(x), dz slope
    static constexpr int kH = kTab2 + TT * CPW * 8;       // float [TT][NS/HV][32][HV] states
    static constexpr int kBar = kH + TT * 32 * NS * 4;
    static constexpr int kTotal = kBar + S * 8;
    static constexpr int HV = NS >= 4 ? 4 : 2;            // floats per state-buffer vector
    static_assert(kX % 128 == 0 && kBC % 128 == 0, "TMA destinations must stay 128B aligned");
    static_assert(TT % G == 0 && NS % 2 == 0, "tile and state split");
};

// NP = NS/2 state pairs at p (16-byte aligned when NP is even).
template <int NP>
__device__ __forceinline__ void ld_pairs(const float* p, u64 (&v)[NP]) {
    if constexpr (NP % 2 == 0) {
#pragma unroll
        for (int c = 0; c < NP / 2; ++c) {
            const ulonglong2 q = reinterpret_cast<const ulonglong2*>(p)[c];
            v[2 * c] = q.x;
            v[2 * c + 1] = q.y;
        }
    } else {
        v[0] = *reinterpret_cast<const u64*>(p);
    }
}
template <int NP>
__device__ __forceinline__ void st_pairs(float* p, const u64 (&v)[NP]) {
    if constexpr (NP % 2 == 0) {
#pragma unroll
        for (int c = 0; c < NP / 2; ++c)
            reinterpret_cast<ulonglong2*>(p)[c] = make_ulonglong2(v[2 * c], v[2 * c + 1]);
    } else {
        *reinterpret_cast<u64*>(p) = v[0];
    }
}

// The lane's states of step j in the state buffer: NS/HV vectors of HV
// floats, 32 lanes apart, so that a warp's vector access is contiguous.
template <int NS, int HV>
__device__ __forceinline__ void hbuf_st(float* hb, int j, int lane, const u64 (&h)[NS / 2]) {
    constexpr int NC = NS / HV, PV = HV / 2;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        u64 v[PV];
#pragma unroll
        for (int k = 0; k < PV; ++k) v[k] = h[c * PV + k];
        st_pairs<PV>(hb + ((j * NC + c) * 32 + lane) * HV, v);
    }
}
template <int NS, int HV>
__device__ __forceinline__ void hbuf_ld(const float* hb, int j, int lane, u64 (&h)[NS / 2]) {
    constexpr int NC = NS / HV, PV = HV / 2;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        u64 v[PV];
        ld_pairs<PV>(hb + ((j * NC + c) * 32 + lane) * HV, v);
#pragma unroll
        for (int k = 0; k < PV; ++k) h[c * PV + k] = v[k];
    }
}

// Sum of v over the 8 lanes (xor 4, 2, 1) that share lane / 8, scattered:
// at each of the three levels the lane keeps the half of its values that
// the lane bit selects and adds its partner's copy of that half, so that
// it ends with max(F/8, 1) consecutive sums in v[0..], the first of them
// sum number rs8_first<F>(ch) (F < 8: lanes that differ only in the low
// bits end with the same sums).
template <int F>
__device__ __forceinline__ void reduce_scatter8(float (&v)[F], int ch) {
#pragma unroll
    for (int lv = 0; lv < 3; ++lv) {
        const int o = 4 >> lv;
        const int m = F >> lv;  // values still held
        const bool bit = (ch & o) != 0;
        if (m >= 2) {
#pragma unroll
            for (int e = 0; e < m / 2; ++e) {
                const float keep = bit ? v[e + m / 2] : v[e];
                const float send = bit ? v[e] : v[e + m / 2];
                v[e] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
}
template <int F>
__host__ __device__ constexpr int rs8_first(int ch) {
    int e0 = 0;
    for (int lv = 0; lv < 3; ++lv)
        if ((F >> lv) >= 2 && (ch & (4 >> lv))) e0 += (F >> lv) / 2;
    return e0;
}

template <typename T, int NS, int TT, int S>
__global__ void __launch_bounds__(32, NS >= 16 ? 8 : 11)  // the grid's CTAs per SM
scan_bwd_tma_kernel(const __grid_constant__ CUtensorMap tm_u,
                    const __grid_constant__ CUtensorMap tm_dt,
                    const __grid_constant__ CUtensorMap tm_z,
                    const __grid_constant__ CUtensorMap tm_g,
                    const __grid_constant__ CUtensorMap tm_B,
                    const __grid_constant__ CUtensorMap tm_C, const BwdArgs a, const int ntile) {
    using Lay = BwdLayout<T, NS, TT, S>;
    constexpr int G = Lay::G;
    constexpr int CPW = Lay::CPW;
    constexpr int N = Lay::N;
    constexpr int NP = NS / 2;
    constexpr int HV = Lay::HV;
    constexpr int PQ = TT / G;  // prologue (step, channel) pairs per lane and tile
    extern __shared__ __align__(128) unsigned char smem[];

    const int lane = threadIdx.x;
    const int ch = lane % CPW;
    const int g = lane / CPW;
    const int n0 = g * NS;
    const int tile = (int)(blockIdx.x % ntile);
    const int b = (int)(blockIdx.x / ntile);
    const int d0 = tile * CPW;
    const int64_t d = d0 + ch;
    const int nt = (int)a.nseg;
    const int rounds = 2 * nt - 1;
    // with checkpoints from the forward pass the forward rounds are skipped:
    // logical rounds r0 .. rounds-1, ring position q = r - r0
    const int r0 = a.ext_ckpt ? nt - 1 : 0;
    const bool has_z = a.z != nullptr;
    const uint32_t tx_fwd = (uint32_t)(2 * Lay::kX + Lay::kBC);
    const uint32_t tx_rev = (uint32_t)((3 + (has_z ? 1 : 0)) * Lay::kX + 2 * Lay::kBC);

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + Lay::kBar;
    if (lane == 0) {
        for (int s2 = 0; s2 < S; ++s2) mbar_init(bar0 + 8 * s2, 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_u);
        prefetch_tensormap(&tm_dt);
        prefetch_tensormap(&tm_B);
        if (rounds > 0) {
            prefetch_tensormap(&tm_g);
            prefetch_tensormap(&tm_C);
            if (has_z) prefetch_tensormap(&tm_z);
        }
    }
    __syncwarp();
    // round r = r0 + q: forward tile r (r < nt-1), else reverse tile 2nt-2-r;
    // stage q % S
    auto issue = [&](int q) {
        const int r = r0 + q;
        const uint32_t st = sbase + (q % S) * Lay::kStage;
        const uint32_t bar = bar0 + 8 * (q % S);
        const bool fwd = r < nt - 1;
        const int32_t tt = (int32_t)((int64_t)(fwd ? r : 2 * nt - 2 - r) * TT);
        mbar_expect_tx(bar, fwd ? tx_fwd : tx_rev);
        tma_load_3d(st, &tm_u, bar, d0, tt, b);
        tma_load_3d(st + Lay::kX, &tm_dt, bar, d0, tt, b);
        tma_load_3d(st + Lay::kBoff, &tm_B, bar, 0, tt, b);
        if (!fwd) {
            if (has_z) tma_load_3d(st + 2 * Lay::kX, &tm_z, bar, d0, tt, b);
            tma_load_3d(st + 3 * Lay::kX, &tm_g, bar, d0, tt, b);
            tma_load_3d(st + Lay::kCoff, &tm_C, bar, 0, tt, b);
        }
    };
    int issued = min(S, rounds - r0);
    if (lane == 0)
        for (int q = 0; q < issued; ++q) issue(q);

    u64 A2[NP], An[NP], h[NP], dh[NP], dAacc[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        const float* Ar = a.A + d * N + n0 + 2 * i;
        const float a0 = __ldg(Ar), a1 = __ldg(Ar + 1);
        An[i] = pk2(a0, a1);
        A2[i] = pk2(a0 * kLog2e, a1 * kLog2e);
        dAacc[i] = pk2(0.0f, 0.0f);
        dh[i] = pk2(0.0f, 0.0f);
        h[i] = pk2(0.0f, 0.0f);
    }
    if (a.dlast) ld_pairs<NP>(a.dlast + ((int64_t)b * a.d_inner + d) * N + n0, dh);
    const float* h0row = a.h0 ? a.h0 + ((int64_t)b * a.d_inner + d) * N + n0 : nullptr;
    if (h0row) ld_pairs<NP>(h0row, h);
    const float bias = a.dt_bias ? __ldg(a.dt_bias + d) : 0.0f;
    const float Dd = a.D ? __ldg(a.D + d) : 0.0f;
    float dDacc = 0.0f, dbacc = 0.0f;
    float4* const tab = reinterpret_cast<float4*>(smem + Lay::kTab);
    float2* const tab2 = reinterpret_cast<float2*>(smem + Lay::kTab2);
    float* const hb = reinterpret_cast<float*>(smem + Lay::kH);
    // checkpoint rows, (batch, tile, d_inner, N): the state entering tile k
    // (row 0, the state before the sequence, is never read: h0 or zero)
    auto ck_row = [&](int kk) {
        return a.ckpt + (((int64_t)b * nt + kk) * a.d_inner + d) * N + n0;
    };
    // per-lane output of the reverse rounds: g = 0 dz, 1 ddt, 2 du, 3 none
    T* outp = static_cast<T*>(a.du);  // also the (unwritten) address of g = 3
    bool has_out = g < 3;
    if (g == 0) {
        if (a.dz) outp = static_cast<T*>(a.dz);
        else has_out = false;
    }
    if (g == 1) outp = static_cast<T*>(a.ddt);
    outp += (int64_t)b * a.L * a.d_inner + d;
    // the dB / dC sums this lane adds: [dB | dC] values rs8_first .. of its states
    constexpr int MF = 2 * NS >= 8 ? 2 * NS / 8 : 1;
    const int e0 = rs8_first<2 * NS>(ch);
    float* const dbc = (e0 < NS ? a.dB + e0 : a.dC + (e0 - NS)) + (int64_t)b * a.L * N + n0;
    const bool bc_lead = 2 * NS >= 8 || (ch & 1) == 0;
    const bool gb1 = (g & 2) != 0, gb0 = (g & 1) != 0;

    bool ok = true;
    int waited = 0;
    u64 hin[NP];
    for (int q = 0; q < rounds - r0; ++q) {
        const int r = r0 + q;
        ok = __all_sync(0xffffffffu, mbar_wait(bar0 + 8 * (q % S), (q / S) & 1, kWaitLimit));
        if (!ok) break;
        waited = q + 1;
        const unsigned char* st = smem + (q % S) * Lay::kStage;
        const T* su = reinterpret_cast<const T*>(st);
        const T* sdt = reinterpret_cast<const T*>(st + Lay::kX);
        const T* sz = reinterpret_cast<const T*>(st + 2 * Lay::kX);
        const T* sg = reinterpret_cast<const T*>(st + 3 * Lay::kX);
        const float* sB = reinterpret_cast<const float*>(st + Lay::kBoff) + n0;
        const float* sC = reinterpret_cast<const float*>(st + Lay::kCoff) + n0;
        // one recurrence step j of the tile on the state x
        auto step = [&](int j, u64 (&x)[NP]) {
            const float2 t = *reinterpret_cast<const float2*>(tab + j * CPW + ch);
            const u64 dl2 = pk2(t.x, t.x), du2 = pk2(t.y, t.y);
            u64 Bq[NP];
            ld_pairs<NP>(sB + j * N, Bq);
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                const u64 x2 = mul2(dl2, A2[i]);
                const u64 ea = pk2(ex2(lo2(x2)), ex2(hi2(x2)));
                x[i] = fma2(ea, x[i], mul2(du2, Bq[i]));
            }
        };
        if (r < nt - 1) {
            // ---- forward round: tile r is whole (only the last tile can be short)
#pragma unroll
            for (int pq = 0; pq < PQ; ++pq) {
                const int e = lane + 32 * pq;  // step g + 4pq of channel ch
                const float dl = softplus(lds_elem<T>(sdt + e) + bias);
                *reinterpret_cast<float2*>(tab + e) = make_float2(dl, dl * lds_elem<T>(su + e));
            }
            __syncwarp();
#pragma unroll
            for (int j = 0; j < TT; ++j) step(j, h);
            st_pairs<NP>(ck_row(r + 1), h);
        } else {
            // ---- reverse round
            const int it = 2 * nt - 2 - r;
            const int64_t t0 = (int64_t)it * TT;
            const int nst = (int)min((int64_t)TT, a.L - t0);
            if (r == nt - 1) {
                if (a.ext_ckpt && nt >= 2) {
                    ld_pairs<NP>(ck_row(nt - 1), hin);     // from the forward pass
                } else {
#pragma unroll
                    for (int i = 0; i < NP; ++i) hin[i] = h[i];  // the forward walk's last state
                }
            }
            // the entering state of the next (earlier) tile, loaded ahead
            u64 hnext[NP];
#pragma unroll
            for (int i = 0; i < NP; ++i) hnext[i] = pk2(0.0f, 0.0f);
            if (it >= 2) ld_pairs<NP>(ck_row(it - 1), hnext);
            else if (it == 1 && h0row) ld_pairs<NP>(h0row, hnext);
            // (1) per-(step, channel) scalars of the tile
#pragma unroll
            for (int pq = 0; pq < PQ; ++pq) {
                const int e = lane + 32 * pq;
                const int j = g + G * pq;
                const float x = lds_elem<T>(sdt + e) + bias;
                const float uu = lds_elem<T>(su + e);
                const float go = lds_elem<T>(sg + e);
                const bool in = j < nst;  // past L: zero-filled inputs; pass through
                const float dl = in ? softplus(x) : 0.0f;
                const float sx = in ? rcp_approx(1.0f + ex2(-x * kLog2e)) : 0.0f;
                // without z the tile holds stale data: read, then not used
                const float zz = lds_elem<T>(sz + e);
                const float s = rcp_approx(1.0f + ex2(-zz * kLog2e));
                const float dy = has_z ? go * zz * s : go;
                const float dzc = has_z ? go * s * fmaf(zz, 1.0f - s, 1.0f) : 0.0f;
                tab[e] = make_float4(dl, dl * uu, dy, uu);
                tab2[e] = make_float2(sx, dzc);
                dDacc = fmaf(dy, uu, dDacc);
            }
            __syncwarp();
            // (2) the tile's states
            {
                u64 x[NP];
#pragma unroll
                for (int i = 0; i < NP; ++i) x[i] = hin[i];
#pragma unroll
                for (int j = 0; j < TT; ++j) {
                    step(j, x);
                    hbuf_st<NS, HV>(hb, j, lane, x);
                }
            }
            // (3) the adjoint, last step first
            [[maybe_unused]] T* const orow = outp + t0 * a.d_inner;
            float* const brow = dbc + t0 * N;
            u64 ht[NP];  // h of step j; h of step j-1 is loaded once and carried
            hbuf_ld<NS, HV>(hb, TT - 1, lane, ht);
#pragma unroll
            for (int j = TT - 1; j >= 0; --j) {
                const float4 ta = tab[j * CPW + ch];
                u64 hp[NP], Bq[NP], Cq[NP];
                if (j > 0) {
                    hbuf_ld<NS, HV>(hb, j - 1, lane, hp);
                } else {
#pragma unroll
                    for (int i = 0; i < NP; ++i) hp[i] = hin[i];
                }
                ld_pairs<NP>(sB + j * N, Bq);
                ld_pairs<NP>(sC + j * N, Cq);
                const u64 dl2 = pk2(ta.x, ta.x), du2 = pk2(ta.y, ta.y), dy2 = pk2(ta.z, ta.z);
                u64 y2 = pk2(0.0f, 0.0f), ddp = pk2(0.0f, 0.0f), sp = pk2(0.0f, 0.0f);
                u64 dB[NP], dC[NP];
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    y2 = fma2(Cq[i], ht[i], y2);
                    const u64 x2 = mul2(dl2, A2[i]);
                    const u64 ea = pk2(ex2(lo2(x2)), ex2(hi2(x2)));
                    dh[i] = fma2(Cq[i], dy2, dh[i]);
                    dC[i] = mul2(dy2, ht[i]);
                    sp = fma2(dh[i], Bq[i], sp);
                    dB[i] = mul2(dh[i], du2);
                    dh[i] = mul2(dh[i], ea);              // the adjoint carried to step j-1
                    const u64 dae = mul2(dh[i], hp[i]);   // dh * e^{delta A} * h_{j-1}
                    dAacc[i] = fma2(dae, dl2, dAacc[i]);
                    ddp = fma2(dae, An[i], ddp);
                }
                const float ssum = lo2(sp) + hi2(sp);
                const float yp = lo2(y2) + hi2(y2);
                const float dd = fmaf(ta.w, ssum, lo2(ddp) + hi2(ddp));
                if constexpr (HV == 4) {
                    // the lane's partial (y, ddelta, S) into its row j of the state
                    // buffer, whose states were consumed above; summed per
                    // (step, channel) after the tile
                    *reinterpret_cast<float4*>(hb + (j * (NS / HV) * 32 + lane) * HV) =
                        make_float4(yp, dd, ssum, 0.0f);
                } else {
                    const float2 tb = tab2[j * CPW + ch];
                    // (y, ddelta, S) over the channel's 4 lanes: g keeps one of them
                    float k0 = gb1 ? ssum : yp, k1 = gb1 ? 0.0f : dd;
                    const float s0 = gb1 ? yp : ssum, s1 = gb1 ? dd : 0.0f;
                    k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
                    k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
                    float v = gb0 ? k1 : k0;
                    v += __shfl_xor_sync(0xffffffffu, gb0 ? k0 : k1, 8);
                    const float o = g == 0 ? (v + Dd * ta.w) * tb.y
                                           : (g == 1 ? v * tb.x : fmaf(ta.x, v, ta.z * Dd));
                    dbacc += g == 1 ? o : 0.0f;
                    Elem<T>::store_if(has_out && j < nst, orow + j * a.d_inner, o);
                }
                // dB and dC over the warp's 8 channels: reduce-scatter of the
                // lane's 2*NS values [dB | dC], lane ch keeping a slice
                float bc[2 * NS];
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    bc[2 * i] = lo2(dB[i]);
                    bc[2 * i + 1] = hi2(dB[i]);
                    bc[NS + 2 * i] = lo2(dC[i]);
                    bc[NS + 2 * i + 1] = hi2(dC[i]);
                }
                reduce_scatter8<2 * NS>(bc, ch);
                float* const p = brow + j * N;
                const bool lead = bc_lead && j < nst;
                if constexpr (MF == 1) red_add_if(lead, p, bc[0]);
                if constexpr (MF == 2) red_add_v2_if(lead, p, make_float2(bc[0], bc[1]));
                if constexpr (MF == 4)
                    red_add_v4_if(lead, p, make_float4(bc[0], bc[1], bc[2], bc[3]));
#pragma unroll
                for (int i = 0; i < NP; ++i) ht[i] = hp[i];
            }
            if constexpr (HV == 4) {
                // (4) per (step, channel) of the tile, as in the prologue: the
                // channel's four partials summed, then dz, ddt, du stored
                __syncwarp();
                const int64_t o0 = ((int64_t)b * a.L + t0) * a.d_inner + d;
                T* const orow_dz = static_cast<T*>(a.dz ? a.dz : a.du) + o0;
                T* const orow_dt = static_cast<T*>(a.ddt) + o0;
                T* const orow_du = static_cast<T*>(a.du) + o0;
#pragma unroll
                for (int pq = 0; pq < PQ; ++pq) {
                    const int e = lane + 32 * pq;
                    const int j = g + G * pq;
                    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                    for (int g2 = 0; g2 < G; ++g2) {
                        const float4 v = *reinterpret_cast<const float4*>(
                            hb + (j * (NS / HV) * 32 + g2 * CPW + ch) * HV);
                        acc.x += v.x;
                        acc.y += v.y;
                        acc.z += v.z;
                    }
                    const float4 ta = tab[e];
                    const float2 tb = tab2[e];
                    const float ddt = acc.y * tb.x;
                    dbacc += ddt;  // zero past L (sigmoid entry zero)
                    const bool in = j < nst;
                    const int64_t off = (int64_t)j * a.d_inner;
                    Elem<T>::store_if(in, orow_dt + off, ddt);
                    Elem<T>::store_if(in, orow_du + off, fmaf(ta.x, acc.z, ta.z * Dd));
                    Elem<T>::store_if(in && a.dz, orow_dz + off, (acc.x + Dd * ta.w) * tb.y);
                }
            }
#pragma unroll
            for (int i = 0; i < NP; ++i) hin[i] = hnext[i];
        }
        __syncwarp();
        if (q + S < rounds - r0) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(q + S);
            }
            issued = q + S + 1;
        }
    }
    // copies still in flight (after a failed wait) land before exit
    for (int q = waited; q < issued; ++q) mbar_wait(bar0 + 8 * (q % S), (q / S) & 1, kWaitLimit);
    if (!ok) {
        if (lane == 0) atomicOr(&g_scan_error, 1u);
        return;
    }
    if (a.dh0) st_pairs<NP>(a.dh0 + ((int64_t)b * a.d_inner + d) * N + n0, dh);
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        atomicAdd(a.dA + d * N + n0 + 2 * i, lo2(dAacc[i]));
        atomicAdd(a.dA + d * N + n0 + 2 * i + 1, hi2(dAacc[i]));
    }
    dDacc += __shfl_xor_sync(0xffffffffu, dDacc, 8);
    dDacc += __shfl_xor_sync(0xffffffffu, dDacc, 16);
    if (g == 0 && a.dD) atomicAdd(a.dD + d, dDacc);
    if constexpr (HV == 4) {  // per-lane sums of the epilogue's steps
        dbacc += __shfl_xor_sync(0xffffffffu, dbacc, 8);
        dbacc += __shfl_xor_sync(0xffffffffu, dbacc, 16);
        if (g == 0 && a.ddt_bias) atomicAdd(a.ddt_bias + d, dbacc);
    } else {
        if (g == 1 && a.ddt_bias) atomicAdd(a.ddt_bias + d, dbacc);
    }
}

// B and C as fp32 rows for the [TT x N] fp32 TMA boxes; 8 elements per
// thread when the arrays allow 16-byte bf16 reads, element-wise otherwise.
template <typename T>
__global__ void bc_to_f32_kernel(const T* __restrict__ B, const T* __restrict__ C,
                                 float* __restrict__ Bf, float* __restrict__ Cf, int64_t n,
                                 int vec8) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (sizeof(T) == 2 && vec8) {
        for (; i < n / 8; i += stride) {
            const uint4 qb = __ldg(reinterpret_cast<const uint4*>(B) + i);
            const uint4 qc = __ldg(reinterpret_cast<const uint4*>(C) + i);
            float4* ob = reinterpret_cast<float4*>(Bf) + 2 * i;
            float4* oc = reinterpret_cast<float4*>(Cf) + 2 * i;
            ob[0] = make_float4(__uint_as_float(qb.x << 16), __uint_as_float(qb.x & 0xffff0000u),
                                __uint_as_float(qb.y << 16), __uint_as_float(qb.y & 0xffff0000u));
            ob[1] = make_float4(__uint_as_float(qb.z << 16), __uint_as_float(qb.z & 0xffff0000u),
                                __uint_as_float(qb.w << 16), __uint_as_float(qb.w & 0xffff0000u));
            oc[0] = make_float4(__uint_as_float(qc.x << 16), __uint_as_float(qc.x & 0xffff0000u),
                                __uint_as_float(qc.y << 16), __uint_as_float(qc.y & 0xffff0000u));
            oc[1] = make_float4(__uint_as_float(qc.z << 16), __uint_as_float(qc.z & 0xffff0000u),
                                __uint_as_float(qc.w << 16), __uint_as_float(qc.w & 0xffff0000u));
        }
        return;
    }
    for (; i < n; i += stride) {
        Bf[i] = Elem<T>::load(B + i);
        Cf[i] = Elem<T>::load(C + i);
    }
}

// ---- host side ----------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 3-D map over a (batch, L, cols) row-major array, box [box0 cols, box1 steps, 1].
bool make_tensor_map_3d(CUtensorMap* m, CUtensorMapDataType t, int es, const void* base,
                        int64_t cols, int64_t L, int64_t batch, int box0, int box1) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)L, (cuuint64_t)batch};
    cuuint64_t strides[2] = {(cuuint64_t)(cols * es), (cuuint64_t)(L * cols * es)};
    cuuint32_t box[3] = {(cuuint32_t)box0, (cuuint32_t)box1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, t, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tma_scan_supported(int64_t N, int64_t d_inner, msc_dtype dtype, const void* u,
                        const void* dt, const void* z, const void* lam) {
    if (!(N == 8 || N == 16 || N == 32 || N == 64)) return false;
    if (d_inner % 8 != 0) return false;  // whole 8-channel boxes (16 B of bf16)
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    if (!al(u) || !al(dt) || (z && !al(z)) || (lam && !al(lam))) return false;
    (void)dtype;
    return encode_fn() != nullptr;
}

int tma_scan_tile(int64_t N) { return N <= 16 ? 32 : 16; }

template <typename T, int G, int NS, int TT, int S, int DISC>
static cudaError_t launch_tma_d(const ScanArgs& a, const ScanPlan& p, const CUtensorMap& mu,
                                const CUtensorMap& mdt, const CUtensorMap& mz,
                                const CUtensorMap& mB, const CUtensorMap& mC,
                                const CUtensorMap& ml, cudaStream_t s) {
    using Lay = TmaLayout<T, G, NS, TT, S, DISC == 2>;
    const size_t smem = Lay::kTotal;
    if (p.K > 1) {
        auto kern = scan_summary_kernel<T, G, NS, TT, S, DISC>;
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        const int64_t nb = a.batch * (int64_t)(p.K - 1) * p.ntile;
        kern<<<(unsigned)nb, 32, smem, s>>>(mu, mdt, mB, ml, a, p.K - 1);
        const cudaError_t e = launch_carry_prefix(a, s);
        if (e != cudaSuccess) return e;
    }
    const int64_t nb = a.batch * (int64_t)p.K * p.ntile;
    const ProfileMark m = profile_begin(s, MSC_PROF_SCAN);
    // checkpoints for the backward pass: a separate instantiation, so that
    // the plain forward's code is unchanged (Euler only, as the backward)
    auto kern = (DISC == 0 && a.ckpt_out) ? scan_tma_kernel<T, G, NS, TT, S, DISC, kOct, true>
                                          : scan_tma_kernel<T, G, NS, TT, S, DISC, kOct, false>;
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    kern<<<(unsigned)nb, 32, smem, s>>>(mu, mdt, mz, mB, mC, ml, a, p.K);
    profile_end(m, s);
    profile_count(p.K > 1 ? 3 : 1);
    return cudaGetLastError();
}

template <typename T, int G, int NS, int TT, int S>
static cudaError_t launch_tma_ns(const ScanArgs& a, const ScanPlan& p, const float* Bf,
                                 const float* Cf, cudaStream_t s) {
    using Lay = TmaLayout<T, G, NS, TT, S>;
    const CUtensorMapDataType tt =
        sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const int es = (int)sizeof(T);
    CUtensorMap mu, mdt, mz, mB, mC, ml;
    if (!make_tensor_map_3d(&mu, tt, es, a.u, a.d_inner, a.L, a.batch, Lay::CPW, TT) ||
        !make_tensor_map_3d(&mdt, tt, es, a.dt, a.d_inner, a.L, a.batch, Lay::CPW, TT) ||
        !make_tensor_map_3d(&mz, tt, es, a.z ? a.z : a.u, a.d_inner, a.L, a.batch, Lay::CPW, TT) ||
        !make_tensor_map_3d(&ml, tt, es, a.trap ? a.lam : a.u, a.d_inner, a.L, a.batch, Lay::CPW, TT) ||
        !make_tensor_map_3d(&mB, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Bf, a.N, a.L, a.batch, (int)a.N, TT) ||
        !make_tensor_map_3d(&mC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Cf, a.N, a.L, a.batch, (int)a.N, TT))
        return cudaErrorInvalidValue;
    if (a.trap) return launch_tma_d<T, G, NS, TT, S, 2>(a, p, mu, mdt, mz, mB, mC, ml, s);
    if (a.zoh) return launch_tma_d<T, G, NS, TT, S, 1>(a, p, mu, mdt, mz, mB, mC, ml, s);
    return launch_tma_d<T, G, NS, TT, S, 0>(a, p, mu, mdt, mz, mB, mC, ml, s);
}

template <typename T>
static cudaError_t launch_tma_t(const ScanArgs& a, const ScanPlan& p, const float* Bf,
                                const float* Cf, cudaStream_t s) {
    if (p.G == 2) {
        switch (a.N) {
            case 8: return launch_tma_ns<T, 2, 4, 32, 3>(a, p, Bf, Cf, s);
            case 16: return launch_tma_ns<T, 2, 8, 32, 3>(a, p, Bf, Cf, s);
            default: return launch_tma_ns<T, 2, 16, 16, 3>(a, p, Bf, Cf, s);  // 32
        }
    }
    switch (a.N) {
        case 8: return launch_tma_ns<T, 4, 2, 32, 3>(a, p, Bf, Cf, s);
        case 16: return launch_tma_ns<T, 4, 4, 32, 2>(a, p, Bf, Cf, s);  // 2 stages: measured
                                                                          // equal or faster
        case 32: return launch_tma_ns<T, 4, 8, 16, 3>(a, p, Bf, Cf, s);
        default: return launch_tma_ns<T, 4, 16, 16, 2>(a, p, Bf, Cf, s);
    }
}

// B and C rows as fp32 (converted, or realigned copies) for the TMA boxes.
static void convert_bc(const void* B, const void* C, msc_dtype dtype, float* Bf, float* Cf,
                       int64_t n, cudaStream_t s) {
    if (n <= 0) return;
    const int vec8 = dtype == MSC_BF16 && (n % 8 == 0) &&
                     (reinterpret_cast<uintptr_t>(B) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(C) % 16 == 0);
    const int64_t work = vec8 ? n / 8 : n;
    const int64_t nb = (work + 255) / 256;
    const int blocks = (int)(nb < 4096 ? nb : 4096);
    if (dtype == MSC_BF16)
        bc_to_f32_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(B), static_cast<const __nv_bfloat16*>(C), Bf, Cf,
            n, vec8);
    else
        bc_to_f32_kernel<float><<<blocks, 256, 0, s>>>(static_cast<const float*>(B),
                                                       static_cast<const float*>(C), Bf, Cf, n,
                                                       0);
    profile_count(1);
}

cudaError_t launch_scan_tma(const ScanArgs& a, const ScanPlan& p, msc_dtype dtype, float* Bf,
                            float* Cf, cudaStream_t s) {
    const float* Bsrc = static_cast<const float*>(a.B);
    const float* Csrc = static_cast<const float*>(a.C);
    if (Bf && a.batch * a.L * a.N > 0) {
        convert_bc(a.B, a.C, dtype, Bf, Cf, a.batch * a.L * a.N, s);
        Bsrc = Bf;
        Csrc = Cf;
    }
    if (dtype == MSC_BF16) return launch_tma_t<__nv_bfloat16>(a, p, Bsrc, Csrc, s);
    return launch_tma_t<float>(a, p, Bsrc, Csrc, s);
}

cudaError_t scan_error_word(unsigned int* value, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_scan_error, sizeof(unsigned int));
    if (e == cudaSuccess && clear && *value) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_scan_error, &zero, sizeof(unsigned int));
    }
    return e;
}

template <typename T, int NS, int TT>
static cudaError_t launch_bwd_tma_n(const BwdArgs& a, const float* Bf, const float* Cf,
                                    cudaStream_t s) {
    constexpr int S = 2;
    using Lay = BwdLayout<T, NS, TT, S>;
    const CUtensorMapDataType tt =
        sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const int es = (int)sizeof(T);
    CUtensorMap mu, mdt, mz, mg, mB, mC;
    if (!make_tensor_map_3d(&mu, tt, es, a.u, a.d_inner, a.L, a.batch, Lay::CPW, TT) ||
        !make_tensor_map_3d(&mdt, tt, es, a.dt, a.d_inner, a.L, a.batch, Lay::CPW, TT) ||
        !make_tensor_map_3d(&mz, tt, es, a.z ? a.z : a.u, a.d_inner, a.L, a.batch, Lay::CPW, TT) ||
        !make_tensor_map_3d(&mg, tt, es, a.dout, a.d_inner, a.L, a.batch, Lay::CPW, TT) ||
        !make_tensor_map_3d(&mB, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Bf, a.N, a.L, a.batch, (int)a.N, TT) ||
        !make_tensor_map_3d(&mC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Cf, a.N, a.L, a.batch, (int)a.N, TT))
        return cudaErrorInvalidValue;
    auto kern = scan_bwd_tma_kernel<T, NS, TT, S>;
    const size_t smem = Lay::kTotal;
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const int ntile = (int)(a.d_inner / Lay::CPW);
    const ProfileMark m = profile_begin(s, MSC_PROF_SCAN_BWD);
    kern<<<(unsigned)(a.batch * ntile), 32, smem, s>>>(mu, mdt, mz, mg, mB, mC, a, ntile);
    profile_end(m, s);
    profile_count(1);
    return cudaGetLastError();
}

int bwd_tma_tile(int64_t N) { return N <= 16 ? 16 : 8; }

bool bwd_tma_supported(int64_t N, int64_t d_inner, const void* u, const void* dt, const void* z,
                       const void* dout, const void* dB, const void* dC) {
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    return (N == 8 || N == 16 || N == 32 || N == 64) && d_inner % 8 == 0 && al(u) && al(dt) &&
           (!z || al(z)) && al(dout) && al(dB) && al(dC) && encode_fn() != nullptr;
}

static bool bwd_needs_bc(const BwdArgs& a, msc_dtype dtype) {
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    return dtype == MSC_BF16 || !al(a.B) || !al(a.C);
}

size_t scan_bwd_tma_scratch(const BwdArgs& a, msc_dtype dtype) {
    const int64_t TT = bwd_tma_tile(a.N);
    const int64_t nt = (a.L + TT - 1) / TT;
    const size_t ck =
        a.ext_ckpt ? 0 : ((size_t)(a.batch * a.d_inner * a.N * nt) * 4 + 255) / 256 * 256;
    const size_t bc = bwd_needs_bc(a, dtype) ? 2 * (size_t)(a.batch * a.L * a.N) * 4 : 0;
    return ck + bc;
}

cudaError_t launch_scan_bwd_tma(BwdArgs a, msc_dtype dtype, void* scratch, cudaStream_t s) {
    const int64_t TT = bwd_tma_tile(a.N);
    a.nseg = (a.L + TT - 1) / TT;
    const size_t ck =
        a.ext_ckpt ? 0 : ((size_t)(a.batch * a.d_inner * a.N * a.nseg) * 4 + 255) / 256 * 256;
    if (!a.ext_ckpt) a.ckpt = static_cast<float*>(scratch);
    const float* Bf = static_cast<const float*>(a.B);
    const float* Cf = static_cast<const float*>(a.C);
    if (bwd_needs_bc(a, dtype)) {
        float* Bc = reinterpret_cast<float*>(static_cast<char*>(scratch) + ck);
        float* Cc = Bc + a.batch * a.L * a.N;
        convert_bc(a.B, a.C, dtype, Bc, Cc, a.batch * a.L * a.N, s);
        Bf = Bc;
        Cf = Cc;
    }
    const bool bf = dtype == MSC_BF16;
    switch (a.N) {
        case 8:
            return bf ? launch_bwd_tma_n<__nv_bfloat16, 2, 16>(a, Bf, Cf, s)
                      : launch_bwd_tma_n<float, 2, 16>(a, Bf, Cf, s);
        case 16:
            return bf ? launch_bwd_tma_n<__nv_bfloat16, 4, 16>(a, Bf, Cf, s)
                      : launch_bwd_tma_n<float, 4, 16>(a, Bf, Cf, s);
        case 32:
            return bf ? launch_bwd_tma_n<__nv_bfloat16, 8, 8>(a, Bf, Cf, s)
                      : launch_bwd_tma_n<float, 8, 8>(a, Bf, Cf, s);
        default:
            return bf ? launch_bwd_tma_n<__nv_bfloat16, 16, 8>(a, Bf, Cf, s)
                      : launch_bwd_tma_n<float, 16, 8>(a, Bf, Cf, s);
    }
}

}  // namespace msc
