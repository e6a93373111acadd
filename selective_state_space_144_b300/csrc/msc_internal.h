// msc_internal.h -- host-side plan and launcher interfaces between the C ABI
// (msc_api.cu) and the kernel files.  Not installed, not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/msc.h"

namespace msc {

// Everything a scan launch needs.  Pointers are device pointers.
struct ScanArgs {
    const void* u;
    const void* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* dt_bias;
    void* out;
    float* last_state;
    const float* h0;   // initial state (batch, d_inner, N) or nullptr for zero
    int zoh;           // 1: zero-order-hold input matrix, 0: delta*B
    int trap;          // 1: exponential-trapezoid input (lam, u_prev, B_prev below)
    const void* lam;   // trapezoid mixing coefficient (batch, L, d_inner), storage dtype
    const void* u_prev;  // u of the step before t = 0 (batch, d_inner) or nullptr
    const void* B_prev;  // B of the step before t = 0 (batch, N) or nullptr
    float* ws_a;       // chunk transfer coefficients, (batch, K-1, d_inner, N)
    float* ws_b;       // chunk end states from zero,   (batch, K-1, d_inner, N)
    int64_t batch, L, d_inner, N;
    int64_t chunk;     // time steps per chunk (last chunk may be shorter)
    int K;             // number of chunks
    int ntile;         // channel tiles per (batch, chunk)
    int vec;           // 1: B/C rows can be read 4 elements at a time
    uint32_t wait_limit;   // polls before a TMA kernel's wait for a copy gives up
    int starve;            // failure-detection test: 1 = TMA kernels issue no copies
    float* ckpt_out;       // TMA output kernel: the states entering every 2^ckpt_shift
    int ckpt_shift;        //   steps, (batch, ckpt_rows, d_inner, N) fp32, for the
    int64_t ckpt_rows;     //   backward pass (ckpt_shift >= log2 of the octet)
};

// How one scan call is cut up.
struct ScanPlan {
    int tma;           // 1: TMA kernels (8 channels per CTA), 0: element-load kernels
    int G;             // lanes per channel (element-load kernels: 4 states per lane;
                       // TMA kernels: 2 or 4 lanes, N/G states per lane)
    int K;             // time chunks
    int64_t chunk;     // steps per chunk
    int ntile;         // channel tiles per (batch row, chunk)
    size_t ws_carry;   // bytes of chunk summaries (a then b), 0 when K == 1
    size_t ws_bc;      // bytes of fp32 copies of B then C for the TMA boxes
    size_t ws_bytes;   // total workspace (carry, then B/C copies, 256-aligned)
};

struct UpdateArgs {
    float* state;
    const void* u;
    const void* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* dt_bias;
    void* out;
    int64_t batch, d_inner, N;
    int vec;           // 1: state and B/C rows can be read 4 elements at a time
    int zoh;           // 1: zero-order-hold input matrix, 0: delta*B
    int trap;          // 1: exponential-trapezoid input
    const void* lam;   // (batch, d_inner) trapezoid mixing coefficient
    const void* u_prev;  // previous token's u (batch, d_inner) or nullptr
    const void* B_prev;  // previous token's B (batch, N) or nullptr
    int stream_ok;       // 1: the copy-engine streaming kernel may be used
    int sms;             // multiprocessor count of the device
    uint32_t wait_limit; // polls before a bounded wait gives up
    int starve;          // failure-detection test: 1 = the streaming kernel issues no copies
};

// The causal depthwise conv1d before the scan (conv1d.cu).  For the decode
// update, state_out is the conv state updated in place and state_in unused.
struct ConvArgs {
    const void* x;
    const float* w;
    const float* bias;
    const void* state_in;
    void* out;
    void* state_out;
    int64_t batch, L, d_inner, d_conv;
    int silu;          // 1: SiLU on the output
    int vec;           // 1: 8-byte vectors of channels (d_inner and x/out allow)
};
cudaError_t launch_causal_conv1d(const ConvArgs& a, msc_dtype dtype, cudaStream_t s);
cudaError_t launch_conv1d_update(const ConvArgs& a, msc_dtype dtype, cudaStream_t s);

// Backward pass of the scan.  Element-load path (scan_bwd.cu): ckpt is
// (batch, nseg - 1, d_inner, N) fp32, the states entering segments
// 1 .. nseg-1 of the recompute; segment 0 starts from h0 (or zero).  TMA path
// (scan_tma.cu): ckpt is (batch, nseg, d_inner, N) fp32, row k the state
// entering tile k, nseg the tile count -- the kernel's own scratch, or with
// ext_ckpt the rows a checkpointing forward scan wrote (read only).
struct BwdArgs {
    const void* u;
    const void* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* dt_bias;
    const float* h0;
    const void* dout;
    const float* dlast;
    void* du;
    void* ddt;
    float* dA;
    float* dB;
    float* dC;
    float* dD;
    void* dz;
    float* ddt_bias;
    float* dh0;
    float* ckpt;
    int64_t batch, L, d_inner, N, nseg;
    int vec;           // 1: B/C rows can be read 4 elements at a time
    int ext_ckpt;      // TMA path: ckpt holds the forward pass's checkpoints
};
// The element-load checkpoint kernel, then the element-load adjoint (a.ckpt:
// scan_bwd_ckpt_bytes of scratch).
cudaError_t launch_scan_bwd(const BwdArgs& a, msc_dtype dtype, cudaStream_t s);
size_t scan_bwd_ckpt_bytes(int64_t batch, int64_t L, int64_t d_inner, int64_t N);
// The TMA backward (scan_tma.cu): N in {8, 16, 32, 64}, d_inner % 8 == 0,
// 16-byte aligned u / dt / z / dout / dB / dC.  One kernel walks each
// channel group forward (checkpoints every bwd_tma_tile(N) steps) and back;
// `scratch` holds scan_bwd_tma_scratch() bytes (checkpoints, fp32 B / C).
int bwd_tma_tile(int64_t N);
bool bwd_tma_supported(int64_t N, int64_t d_inner, const void* u, const void* dt, const void* z,
                       const void* dout, const void* dB, const void* dC);
size_t scan_bwd_tma_scratch(const BwdArgs& a, msc_dtype dtype);
cudaError_t launch_scan_bwd_tma(BwdArgs a, msc_dtype dtype, void* scratch, cudaStream_t s);
constexpr int64_t kBwdSegment = 32;  // steps per recomputed segment

// Measurement hook (msc_api.cu): while enabled, launchers count kernels and
// bracket their main kernel with an event pair on the launch stream.
struct ProfileMark {
    void* begin;  // cudaEvent_t or nullptr when profiling is off
    int kind;     // MSC_PROF_SCAN, _UPDATE, _CONV or _CONV_UPDATE
};
ProfileMark profile_begin(cudaStream_t s, int kind);
void profile_end(const ProfileMark& m, cudaStream_t s);
void profile_count(int launches);

constexpr int kScanThreads = 128;
constexpr int kUpdateThreads = 256;

int lanes_per_channel(int64_t N);
ScanPlan make_scan_plan(int64_t batch, int64_t L, int64_t d_inner, int64_t N,
                        int sm_count, int64_t force_chunks, int64_t min_chunk);
ScanPlan make_tma_plan(int64_t batch, int64_t L, int64_t d_inner, int64_t N, int sm_count,
                       int64_t force_chunks, int64_t min_chunk, bool need_bc,
                       int64_t force_lanes);

// States entering chunks 1..K-1, written over ws_b (K > 1; h0 or zero first).
cudaError_t launch_carry_prefix(const ScanArgs& a, cudaStream_t s);
cudaError_t launch_scan(const ScanArgs& a, const ScanPlan& p, msc_dtype dtype,
                        cudaStream_t stream);

// Tiled tensor map of a row-major (batch, L, cols) array, box [box0 cols,
// box1 rows, 1] (scan_tma.cu); false when the driver refuses it.
bool make_tensor_map_3d(CUtensorMap* m, CUtensorMapDataType t, int es, const void* base,
                        int64_t cols, int64_t L, int64_t batch, int box0, int box1);

// TMA path (scan_tma.cu): supported shapes, time-tile length, launch, and
// the device word its bounded waits set when a copy never lands.
bool tma_scan_supported(int64_t N, int64_t d_inner, msc_dtype dtype, const void* u,
                        const void* dt, const void* z, const void* lam = nullptr);
int tma_scan_tile(int64_t N);
constexpr uint32_t kWaitLimit = 1u << 22;  // polls of a bounded wait (~1 s at most)
cudaError_t launch_scan_tma(const ScanArgs& a, const ScanPlan& p, msc_dtype dtype, float* Bf,
                            float* Cf, cudaStream_t stream);
cudaError_t scan_error_word(unsigned int* value, bool clear);
cudaError_t launch_state_update(const UpdateArgs& a, msc_dtype dtype,
                                cudaStream_t stream);
cudaError_t update_error_word(unsigned int* value, bool clear);

}  // namespace msc
