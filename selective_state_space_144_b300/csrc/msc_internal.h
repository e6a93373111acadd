// msc_internal.h -- host-side plan and launcher interfaces between the C ABI
// (msc_api.cu) and the kernel files.  Not installed, not part of the ABI.
#pragma once

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
    float* ws_a;       // chunk transfer coefficients, (batch, K-1, d_inner, N)
    float* ws_b;       // chunk end states from zero,   (batch, K-1, d_inner, N)
    int64_t batch, L, d_inner, N;
    int64_t chunk;     // time steps per chunk (last chunk may be shorter)
    int K;             // number of chunks
    int ntile;         // channel tiles per (batch, chunk)
    int vec;           // 1: B/C rows can be read 4 elements at a time
};

// How one scan call is cut up.
struct ScanPlan {
    int G;             // lanes per channel (each lane owns 4 states)
    int K;             // time chunks
    int64_t chunk;     // steps per chunk
    int ntile;         // channel tiles
    size_t ws_bytes;   // carry workspace
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
};

constexpr int kScanThreads = 128;
constexpr int kUpdateThreads = 256;

int lanes_per_channel(int64_t N);
ScanPlan make_scan_plan(int64_t batch, int64_t L, int64_t d_inner, int64_t N,
                        int sm_count, int64_t force_chunks, int64_t min_chunk);

cudaError_t launch_scan(const ScanArgs& a, const ScanPlan& p, msc_dtype dtype,
                        cudaStream_t stream);
cudaError_t launch_state_update(const UpdateArgs& a, msc_dtype dtype,
                                cudaStream_t stream);

}  // namespace msc
