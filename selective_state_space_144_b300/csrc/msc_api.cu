// msc_api.cu -- the extern "C" boundary: argument validation, planning,
// workspace handling and launch.  Declarations and their contracts are in
// include/msc.h.
#include <cstring>
#include <limits>

#include "msc_internal.h"

namespace {

int64_t g_force_chunks = 0;    // "scan_chunks"
int64_t g_min_chunk = 512;     // "scan_min_chunk"

bool aligned(const void* p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

size_t elem_size(msc_dtype t) { return t == MSC_BF16 ? 2 : 4; }

// a * b without int64 overflow; false when it would overflow.
bool mul_ok(int64_t a, int64_t b, int64_t* r) {
    if (a == 0 || b == 0) {
        *r = 0;
        return true;
    }
    if (a > std::numeric_limits<int64_t>::max() / b) return false;
    *r = a * b;
    return true;
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        n <= 0)
        return 148;
    return n;
}

struct ScanCheck {
    msc_status st;
    msc::ScanPlan plan;
    int vec;
};

ScanCheck check_scan(const void* u, const void* dt, const float* A, const void* B,
                     const void* C, const float* D, const void* z, const float* dt_bias,
                     void* out, float* last_state, int64_t batch, int64_t L,
                     int64_t d_inner, int64_t d_state, msc_dtype dtype) {
    ScanCheck r{};
    r.st = MSC_OK;
    if (dtype != MSC_F32 && dtype != MSC_BF16) {
        r.st = MSC_ERR_INVALID_ARG;
        return r;
    }
    if (batch < 0 || L < 0 || d_inner < 0 || d_state < 0) {
        r.st = MSC_ERR_INVALID_ARG;
        return r;
    }
    if (d_state < 1 || d_state > 64) {
        r.st = MSC_ERR_UNSUPPORTED;
        return r;
    }
    int64_t bl, bld, bln, bdn, dn;
    if (!mul_ok(batch, L, &bl) || !mul_ok(bl, d_inner, &bld) || !mul_ok(bl, d_state, &bln) ||
        !mul_ok(batch, d_inner, &bdn) || !mul_ok(bdn, d_state, &dn) ||
        bld > std::numeric_limits<int64_t>::max() / 8 ||
        bln > std::numeric_limits<int64_t>::max() / 8) {
        r.st = MSC_ERR_UNSUPPORTED;
        return r;
    }
    (void)dn;
    const bool empty = (batch == 0 || d_inner == 0);
    if (!empty) {
        if (!A || (L > 0 && (!u || !dt || !B || !C || !out))) {
            r.st = MSC_ERR_INVALID_ARG;
            return r;
        }
    }
    const size_t es = elem_size(dtype);
    const void* typed[] = {u, dt, B, C, z, out};
    for (const void* p : typed)
        if (p && !aligned(p, es)) {
            r.st = MSC_ERR_ALIGNMENT;
            return r;
        }
    const void* f32[] = {A, D, dt_bias, last_state};
    for (const void* p : f32)
        if (p && !aligned(p, 4)) {
            r.st = MSC_ERR_ALIGNMENT;
            return r;
        }
    r.plan = msc::make_scan_plan(batch, L, d_inner, d_state, sm_count(), g_force_chunks,
                                 g_min_chunk);
    const int64_t nblocks = batch * (int64_t)r.plan.K * r.plan.ntile;
    if (nblocks > std::numeric_limits<int>::max()) {
        r.st = MSC_ERR_UNSUPPORTED;
        return r;
    }
    // 4-wide B/C reads: rows of a multiple of 4 elements from an aligned base
    const size_t vec_align = 4 * es;
    r.vec = (d_state % 4 == 0) && (!B || aligned(B, vec_align)) && (!C || aligned(C, vec_align));
    return r;
}

}  // namespace

static msc_status run_scan(const void* u, const void* dt, const float* A, const void* B,
                           const void* C, const float* D, const void* z,
                           const float* dt_bias, void* out, float* last_state, int64_t batch,
                           int64_t L, int64_t d_inner, int64_t d_state, msc_dtype dtype,
                           void* ws, size_t ws_bytes, bool own_ws, msc_stream_t stream) {
    ScanCheck c = check_scan(u, dt, A, B, C, D, z, dt_bias, out, last_state, batch, L, d_inner,
                             d_state, dtype);
    if (c.st != MSC_OK) return c.st;
    if (batch == 0 || d_inner == 0) return MSC_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t need = c.plan.ws_bytes;
    void* w = ws;
    if (need > 0) {
        if (own_ws) {
            if (cudaMallocAsync(&w, need, s) != cudaSuccess) return MSC_ERR_CUDA;
        } else if (!ws || ws_bytes < need || !aligned(ws, 256)) {
            return MSC_ERR_WORKSPACE;
        }
    }
    msc::ScanArgs a{};
    a.u = u; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.dt_bias = dt_bias;
    a.out = out; a.last_state = last_state;
    const size_t half = need / 2 / sizeof(float);
    a.ws_a = need ? static_cast<float*>(w) : nullptr;
    a.ws_b = need ? static_cast<float*>(w) + half : nullptr;
    a.batch = batch; a.L = L; a.d_inner = d_inner; a.N = d_state;
    a.chunk = c.plan.chunk; a.K = c.plan.K; a.ntile = c.plan.ntile; a.vec = c.vec;
    cudaError_t e = msc::launch_scan(a, c.plan, dtype, s);
    if (need > 0 && own_ws) {
        cudaError_t f = cudaFreeAsync(w, s);
        if (e == cudaSuccess) e = f;
    }
    return e == cudaSuccess ? MSC_OK : MSC_ERR_CUDA;
}

extern "C" {

msc_status msc_selective_scan_fwd(const void* u, const void* dt, const float* A, const void* B,
                                  const void* C, const float* D, const void* z,
                                  const float* dt_bias, void* out, float* last_state,
                                  int64_t batch, int64_t L, int64_t d_inner, int64_t d_state,
                                  msc_dtype dtype, msc_stream_t stream) {
    return run_scan(u, dt, A, B, C, D, z, dt_bias, out, last_state, batch, L, d_inner, d_state,
                    dtype, nullptr, 0, true, stream);
}

msc_status msc_selective_scan_fwd_ws(const void* u, const void* dt, const float* A,
                                     const void* B, const void* C, const float* D,
                                     const void* z, const float* dt_bias, void* out,
                                     float* last_state, int64_t batch, int64_t L,
                                     int64_t d_inner, int64_t d_state, msc_dtype dtype,
                                     void* workspace, size_t workspace_bytes,
                                     msc_stream_t stream) {
    return run_scan(u, dt, A, B, C, D, z, dt_bias, out, last_state, batch, L, d_inner, d_state,
                    dtype, workspace, workspace_bytes, false, stream);
}

msc_status msc_selective_scan_workspace_size(int64_t batch, int64_t L, int64_t d_inner,
                                             int64_t d_state, msc_dtype dtype, size_t* bytes) {
    if (!bytes) return MSC_ERR_INVALID_ARG;
    if (dtype != MSC_F32 && dtype != MSC_BF16) return MSC_ERR_INVALID_ARG;
    if (batch < 0 || L < 0 || d_inner < 0 || d_state < 0) return MSC_ERR_INVALID_ARG;
    if (d_state < 1 || d_state > 64) return MSC_ERR_UNSUPPORTED;
    int64_t bl, bld;
    if (!mul_ok(batch, L, &bl) || !mul_ok(bl, d_inner, &bld)) return MSC_ERR_UNSUPPORTED;
    if (batch == 0 || d_inner == 0) {
        *bytes = 0;
        return MSC_OK;
    }
    msc::ScanPlan p =
        msc::make_scan_plan(batch, L, d_inner, d_state, sm_count(), g_force_chunks, g_min_chunk);
    *bytes = p.ws_bytes;
    return MSC_OK;
}

msc_status msc_selective_state_update(float* state, const void* u, const void* dt,
                                      const float* A, const void* B, const void* C,
                                      const float* D, const void* z, const float* dt_bias,
                                      void* out, int64_t batch, int64_t d_inner,
                                      int64_t d_state, msc_dtype dtype, msc_stream_t stream) {
    if (dtype != MSC_F32 && dtype != MSC_BF16) return MSC_ERR_INVALID_ARG;
    if (batch < 0 || d_inner < 0 || d_state < 0) return MSC_ERR_INVALID_ARG;
    if (d_state < 1 || d_state > 64) return MSC_ERR_UNSUPPORTED;
    int64_t bd, bdn;
    if (!mul_ok(batch, d_inner, &bd) || !mul_ok(bd, d_state, &bdn) ||
        bdn > std::numeric_limits<int64_t>::max() / 8)
        return MSC_ERR_UNSUPPORTED;
    if (batch == 0 || d_inner == 0) return MSC_OK;
    if (!state || !u || !dt || !A || !B || !C || !out) return MSC_ERR_INVALID_ARG;
    const int G = msc::lanes_per_channel(d_state);
    if ((bd * G + msc::kUpdateThreads - 1) / msc::kUpdateThreads >
        std::numeric_limits<int>::max())
        return MSC_ERR_UNSUPPORTED;
    const size_t es = elem_size(dtype);
    const void* typed[] = {u, dt, B, C, z, out};
    for (const void* p : typed)
        if (p && !aligned(p, es)) return MSC_ERR_ALIGNMENT;
    const void* f32[] = {state, A, D, dt_bias};
    for (const void* p : f32)
        if (p && !aligned(p, 4)) return MSC_ERR_ALIGNMENT;
    msc::UpdateArgs a{};
    a.state = state; a.u = u; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z;
    a.dt_bias = dt_bias; a.out = out; a.batch = batch; a.d_inner = d_inner; a.N = d_state;
    a.vec = (d_state % 4 == 0) && aligned(state, 16) && aligned(B, 4 * es) && aligned(C, 4 * es);
    cudaError_t e = msc::launch_state_update(a, dtype, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MSC_OK : MSC_ERR_CUDA;
}

msc_status msc_tuning_set(const char* key, int64_t value) {
    if (!key || value < 0) return MSC_ERR_INVALID_ARG;
    if (std::strcmp(key, "scan_chunks") == 0) {
        g_force_chunks = value;
        return MSC_OK;
    }
    if (std::strcmp(key, "scan_min_chunk") == 0) {
        g_min_chunk = value > 0 ? value : 1;
        return MSC_OK;
    }
    return MSC_ERR_INVALID_ARG;
}

const char* msc_status_string(msc_status s) {
    switch (s) {
        case MSC_OK: return "ok";
        case MSC_ERR_INVALID_ARG: return "invalid argument";
        case MSC_ERR_UNSUPPORTED: return "unsupported size";
        case MSC_ERR_ALIGNMENT: return "pointer not aligned to its element size";
        case MSC_ERR_CUDA: return "CUDA runtime error";
        case MSC_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    }
    return "unknown status";
}

int msc_version(void) { return 100; }

}  // extern "C"
