// msc_api.cu -- the extern "C" boundary: argument validation, planning,
// workspace handling and launch.  Declarations and their contracts are in
// include/msc.h.
#include <cstring>
#include <limits>
#include <mutex>
#include <vector>

#include "msc_internal.h"

namespace {

int64_t g_force_chunks = 0;    // "scan_chunks"
int64_t g_min_chunk = 512;     // "scan_min_chunk"
int64_t g_scan_path = 0;       // "scan_path": 0 auto, 1 element-load kernels only
int64_t g_scan_lanes = 0;      // "scan_lanes": TMA kernels' lanes per channel, 0 auto
int64_t g_starve = 0;          // "debug_starve_copies": poll limit of starved waits, 0 off
int64_t g_update_path = 0;     // "update_path": 0 auto, 1 thread-per-channel kernels only

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

// Multiprocessor count of the current device, queried once per device.
int sm_count() {
    static int counts[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev >= 0 && dev < 64 && counts[dev] > 0) return counts[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        n <= 0)
        return 148;
    if (dev >= 0 && dev < 64) counts[dev] = n;
    return n;
}

// Stream-ordered scratch comes from a memory pool of the library's own on
// each device, which keeps the memory it has reserved between calls (release
// threshold at the maximum): with the device's default pool, whose threshold
// is zero, every synchronisation returns the memory and the next call maps it
// afresh (about 0.2 ms for the 100 MB of a backward call).  The memory stays
// reserved for the process until msc_scratch_release.
constexpr int kMaxDevices = 64;
std::mutex g_pool_mu;
cudaMemPool_t g_pools[kMaxDevices] = {};

cudaMemPool_t scratch_pool() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_pool_mu);
    if (!g_pools[dev]) {
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        if (cudaMemPoolCreate(&p, &props) != cudaSuccess) return nullptr;
        uint64_t keep = std::numeric_limits<uint64_t>::max();
        cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
        g_pools[dev] = p;
    }
    return g_pools[dev];
}

cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t s) {
    cudaMemPool_t pool = scratch_pool();
    return pool ? cudaMallocFromPoolAsync(p, bytes, pool, s) : cudaMallocAsync(p, bytes, s);
}

// Longest sequence the TMA kernels take: their box coordinates are int32.
constexpr int64_t kTmaMaxExtent = (int64_t{1} << 31) - 1024;

struct ScanCheck {
    msc_status st;
    msc::ScanPlan plan;
    int vec;
};

ScanCheck check_scan(const void* u, const void* dt, const float* A, const void* B,
                     const void* C, const float* D, const void* z, const float* dt_bias,
                     void* out, float* last_state, int64_t batch, int64_t L,
                     int64_t d_inner, int64_t d_state, msc_dtype dtype,
                     const float* h0 = nullptr, const void* lam = nullptr,
                     const void* u_prev = nullptr, const void* B_prev = nullptr) {
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
    const void* typed[] = {u, dt, B, C, z, out, lam, u_prev, B_prev};
    for (const void* p : typed)
        if (p && !aligned(p, es)) {
            r.st = MSC_ERR_ALIGNMENT;
            return r;
        }
    const void* f32[] = {A, D, dt_bias, last_state, h0};
    for (const void* p : f32)
        if (p && !aligned(p, 4)) {
            r.st = MSC_ERR_ALIGNMENT;
            return r;
        }
    // TMA box coordinates are 32-bit: longer sequences take the element-load
    // kernels, whose indices are 64-bit
    if (g_scan_path == 0 && L > 0 && L < kTmaMaxExtent &&
        msc::tma_scan_supported(d_state, d_inner, dtype, u, dt, z, lam)) {
        // fp32 B/C copies unless fp32 inputs already suit 16-byte TMA boxes
        const bool need_bc = dtype == MSC_BF16 || !aligned(B, 16) || !aligned(C, 16);
        r.plan = msc::make_tma_plan(batch, L, d_inner, d_state, sm_count(), g_force_chunks,
                                    g_min_chunk, need_bc, g_scan_lanes);
    } else {
        r.plan = msc::make_scan_plan(batch, L, d_inner, d_state, sm_count(), g_force_chunks,
                                     g_min_chunk);
    }
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

// ---- measurement hook ------------------------------------------------------
bool g_profile = false;
int64_t g_prof_launches = 0;
struct ProfPair {
    cudaEvent_t a, b;
    int kind;
};
std::vector<ProfPair> g_prof_pairs;                              // recorded, unread
std::vector<cudaEvent_t> g_prof_free;                            // reusable events

cudaEvent_t prof_event() {
    if (!g_prof_free.empty()) {
        cudaEvent_t e = g_prof_free.back();
        g_prof_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

}  // namespace

namespace msc {

ProfileMark profile_begin(cudaStream_t s, int kind) {
    ProfileMark m{nullptr, kind};
    if (!g_profile) return m;
    cudaEvent_t e = prof_event();
    if (e && cudaEventRecord(e, s) == cudaSuccess) m.begin = e;
    return m;
}

void profile_end(const ProfileMark& m, cudaStream_t s) {
    if (!m.begin) return;
    cudaEvent_t e = prof_event();
    if (e && cudaEventRecord(e, s) == cudaSuccess)
        g_prof_pairs.push_back({static_cast<cudaEvent_t>(m.begin), e, m.kind});
}

void profile_count(int launches) {
    if (g_profile) g_prof_launches += launches;
}

}  // namespace msc

static msc_status run_scan(const void* u, const void* dt, const float* A, const void* B,
                           const void* C, const float* D, const void* z,
                           const float* dt_bias, void* out, float* last_state, int64_t batch,
                           int64_t L, int64_t d_inner, int64_t d_state, msc_dtype dtype,
                           void* ws, size_t ws_bytes, bool own_ws, msc_stream_t stream,
                           const float* h0 = nullptr, int zoh = 0, const void* lam = nullptr,
                           const void* u_prev = nullptr, const void* B_prev = nullptr,
                           float* ckpt_out = nullptr) {
    ScanCheck c = check_scan(u, dt, A, B, C, D, z, dt_bias, out, last_state, batch, L, d_inner,
                             d_state, dtype, h0, lam, u_prev, B_prev);
    if (c.st != MSC_OK) return c.st;
    if (batch == 0 || d_inner == 0) return MSC_OK;
    // backward checkpoints: written by the TMA output kernel only, at octet
    // starts, so the interval must divide every time chunk
    const int ck_tt = msc::bwd_tma_tile(d_state);
    if (ckpt_out && L > 0 && (!c.plan.tma || c.plan.chunk % ck_tt != 0 || zoh || lam))
        return MSC_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t need = c.plan.ws_bytes;
    void* w = ws;
    if (need > 0) {
        if (own_ws) {
            if (scratch_alloc(&w, need, s) != cudaSuccess) return MSC_ERR_CUDA;
        } else if (!ws || ws_bytes < need || !aligned(ws, 256)) {
            return MSC_ERR_WORKSPACE;
        }
    }
    msc::ScanArgs a{};
    a.u = u; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.dt_bias = dt_bias;
    a.out = out; a.last_state = last_state; a.h0 = h0; a.zoh = zoh;
    a.trap = lam != nullptr; a.lam = lam; a.u_prev = u_prev; a.B_prev = B_prev;
    const size_t half = c.plan.ws_carry / 2 / sizeof(float);
    a.ws_a = c.plan.ws_carry ? static_cast<float*>(w) : nullptr;
    a.ws_b = c.plan.ws_carry ? static_cast<float*>(w) + half : nullptr;
    a.batch = batch; a.L = L; a.d_inner = d_inner; a.N = d_state;
    a.chunk = c.plan.chunk; a.K = c.plan.K; a.ntile = c.plan.ntile; a.vec = c.vec;
    a.wait_limit = g_starve > 0 ? (uint32_t)g_starve : msc::kWaitLimit;
    a.starve = g_starve > 0;
    if (ckpt_out && L > 0) {
        a.ckpt_out = ckpt_out;
        a.ckpt_shift = ck_tt == 16 ? 4 : 3;
        a.ckpt_rows = (L + ck_tt - 1) / ck_tt;
    }
    cudaError_t e;
    if (c.plan.tma) {
        float* Bf = nullptr;
        float* Cf = nullptr;
        if (c.plan.ws_bc) {
            Bf = reinterpret_cast<float*>(static_cast<char*>(w) + c.plan.ws_carry);
            Cf = reinterpret_cast<float*>(static_cast<char*>(w) + c.plan.ws_carry +
                                          c.plan.ws_bc / 2);
        }
        e = msc::launch_scan_tma(a, c.plan, dtype, Bf, Cf, s);
    } else {
        e = msc::launch_scan(a, c.plan, dtype, s);
    }
    if (need > 0 && own_ws) {
        cudaError_t f = cudaFreeAsync(w, s);
        if (e == cudaSuccess) e = f;
    }
    return e == cudaSuccess ? MSC_OK : MSC_ERR_CUDA;
}

// ---- allocation-free scan: scratch in a file-scope device array ------------
// Callers that may not allocate device memory (a runtime whose allocator owns
// the device, no allocation while requests are served) get the scan with its
// scratch here.  Host code must not use the array's name as an address: its
// device address comes from cudaGetSymbolAddress with the device current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MSC_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoallocMaxDevices] = {};

// Device address of the scratch array on the current device.  Looked up
// afresh on every call whose stream is not being captured (cheap once the
// module is loaded, and correct again after a device reset reloaded the
// module at another address); while the stream is being captured the
// address found by the last such lookup on this device is used, and a
// capture before any lookup is refused.
cudaError_t noalloc_scratch(cudaStream_t s, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kNoallocMaxDevices) return cudaErrorInvalidDevice;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(s, &cap);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (e == cudaSuccess && cap == cudaStreamCaptureStatusNone) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (!p) return cudaErrorInvalidSymbol;
        g_noalloc_addr[dev] = p;
    } else if (!g_noalloc_addr[dev]) {
        return e != cudaSuccess ? e : cudaErrorStreamCaptureUnsupported;
    }
    *out = g_noalloc_addr[dev];
    return cudaSuccess;
}
}  // namespace

extern "C" {

msc_status msc_selective_scan_fwd_noalloc(const void* u, const void* dt, const float* A,
                                          const void* B, const void* C, const float* D,
                                          const void* z, const float* dt_bias, void* out,
                                          float* last_state, int64_t batch, int64_t L,
                                          int64_t d_inner, int64_t d_state, msc_dtype dtype,
                                          msc_stream_t stream) {
    ScanCheck c = check_scan(u, dt, A, B, C, D, z, dt_bias, out, last_state, batch, L, d_inner,
                             d_state, dtype);
    if (c.st != MSC_OK) return c.st;
    if (batch == 0 || d_inner == 0) return MSC_OK;
    if (c.plan.ws_bytes > MSC_NOALLOC_SCRATCH_BYTES) return MSC_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    if (c.plan.ws_bytes > 0 &&
        noalloc_scratch(reinterpret_cast<cudaStream_t>(stream), &scratch) != cudaSuccess)
        return MSC_ERR_CUDA;
    return run_scan(u, dt, A, B, C, D, z, dt_bias, out, last_state, batch, L, d_inner, d_state,
                    dtype, scratch, MSC_NOALLOC_SCRATCH_BYTES, false, stream);
}

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

msc_status msc_selective_scan_fwd_ex(const void* u, const void* dt, const float* A,
                                     const void* B, const void* C, const float* D,
                                     const void* z, const float* dt_bias, const float* h0,
                                     void* out, float* last_state, int64_t batch, int64_t L,
                                     int64_t d_inner, int64_t d_state, msc_dtype dtype,
                                     msc_discretization disc, void* workspace,
                                     size_t workspace_bytes, msc_stream_t stream) {
    if (disc != MSC_DISC_EULER && disc != MSC_DISC_ZOH) return MSC_ERR_INVALID_ARG;
    return run_scan(u, dt, A, B, C, D, z, dt_bias, out, last_state, batch, L, d_inner, d_state,
                    dtype, workspace, workspace_bytes, workspace == nullptr, stream, h0,
                    disc == MSC_DISC_ZOH ? 1 : 0);
}

msc_status msc_scan_checkpoint_size(int64_t batch, int64_t L, int64_t d_inner, int64_t d_state,
                                    int64_t* interval, size_t* bytes) {
    if (!interval || !bytes) return MSC_ERR_INVALID_ARG;
    if (batch < 0 || L < 0 || d_inner < 0 || d_state < 0) return MSC_ERR_INVALID_ARG;
    if (!(d_state == 8 || d_state == 16 || d_state == 32 || d_state == 64))
        return MSC_ERR_UNSUPPORTED;
    const int64_t tt = msc::bwd_tma_tile(d_state);
    const int64_t rows = (L + tt - 1) / tt;
    int64_t br, brd, n;
    if (!mul_ok(batch, rows, &br) || !mul_ok(br, d_inner, &brd) || !mul_ok(brd, d_state, &n) ||
        n > std::numeric_limits<int64_t>::max() / 4)
        return MSC_ERR_UNSUPPORTED;
    *interval = tt;
    *bytes = (size_t)n * sizeof(float);
    return MSC_OK;
}

msc_status msc_selective_scan_fwd_ckpt(const void* u, const void* dt, const float* A,
                                       const void* B, const void* C, const float* D,
                                       const void* z, const float* dt_bias, const float* h0,
                                       void* out, float* last_state, float* ckpt, int64_t batch,
                                       int64_t L, int64_t d_inner, int64_t d_state,
                                       msc_dtype dtype, void* workspace, size_t workspace_bytes,
                                       msc_stream_t stream) {
    int64_t tt = 0;
    size_t bytes = 0;
    const msc_status st = msc_scan_checkpoint_size(batch < 0 ? 0 : batch, L < 0 ? 0 : L,
                                                   d_inner < 0 ? 0 : d_inner,
                                                   d_state < 0 ? 0 : d_state, &tt, &bytes);
    if (st == MSC_ERR_INVALID_ARG) return st;
    if (batch > 0 && L > 0 && d_inner > 0) {
        if (st != MSC_OK) return st;
        if (!ckpt) return MSC_ERR_INVALID_ARG;
        if (!aligned(ckpt, 16)) return MSC_ERR_ALIGNMENT;
    }
    return run_scan(u, dt, A, B, C, D, z, dt_bias, out, last_state, batch, L, d_inner, d_state,
                    dtype, workspace, workspace_bytes, workspace == nullptr, stream, h0, 0,
                    nullptr, nullptr, nullptr, ckpt);
}

msc_status msc_selective_scan_trap_fwd(const void* u, const void* dt, const void* lam,
                                       const float* A, const void* B, const void* C,
                                       const float* D, const void* z, const float* dt_bias,
                                       const float* h0, const void* u_prev, const void* B_prev,
                                       void* out, float* last_state, int64_t batch, int64_t L,
                                       int64_t d_inner, int64_t d_state, msc_dtype dtype,
                                       void* workspace, size_t workspace_bytes,
                                       msc_stream_t stream) {
    if (!lam && batch > 0 && L > 0 && d_inner > 0) return MSC_ERR_INVALID_ARG;
    return run_scan(u, dt, A, B, C, D, z, dt_bias, out, last_state, batch, L, d_inner, d_state,
                    dtype, workspace, workspace_bytes, workspace == nullptr, stream, h0, 0,
                    L > 0 ? lam : nullptr, u_prev, B_prev);
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
    // the plan also depends on pointer alignment, unknown here: the larger of
    // the two kernel families' needs covers either choice
    const int sms = sm_count();
    msc::ScanPlan p =
        msc::make_scan_plan(batch, L, d_inner, d_state, sms, g_force_chunks, g_min_chunk);
    size_t need = p.ws_bytes;
    if (g_scan_path == 0 && msc::tma_scan_supported(d_state, d_inner, dtype, nullptr, nullptr,
                                                    nullptr)) {
        msc::ScanPlan q = msc::make_tma_plan(batch, L, d_inner, d_state, sms, g_force_chunks,
                                             g_min_chunk, true, g_scan_lanes);
        need = need > q.ws_bytes ? need : q.ws_bytes;
    }
    *bytes = need;
    return MSC_OK;
}

static msc_status run_update(float* state, const void* u, const void* dt, const float* A,
                             const void* B, const void* C, const float* D, const void* z,
                             const float* dt_bias, void* out, int64_t batch, int64_t d_inner,
                             int64_t d_state, msc_dtype dtype, int zoh, msc_stream_t stream,
                             const void* lam = nullptr, const void* u_prev = nullptr,
                             const void* B_prev = nullptr) {
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
    const void* typed[] = {u, dt, B, C, z, out, lam, u_prev, B_prev};
    for (const void* p : typed)
        if (p && !aligned(p, es)) return MSC_ERR_ALIGNMENT;
    const void* f32[] = {state, A, D, dt_bias};
    for (const void* p : f32)
        if (p && !aligned(p, 4)) return MSC_ERR_ALIGNMENT;
    msc::UpdateArgs a{};
    a.state = state; a.u = u; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z;
    a.dt_bias = dt_bias; a.out = out; a.batch = batch; a.d_inner = d_inner; a.N = d_state;
    a.vec = (d_state % 4 == 0) && aligned(state, 16) && aligned(B, 4 * es) && aligned(C, 4 * es);
    a.zoh = zoh;
    a.trap = lam != nullptr; a.lam = lam; a.u_prev = u_prev; a.B_prev = B_prev;
    a.stream_ok = g_update_path == 0;
    a.sms = sm_count();
    a.wait_limit = g_starve > 0 ? (uint32_t)g_starve : msc::kWaitLimit;
    a.starve = g_starve > 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    msc::ProfileMark m = msc::profile_begin(s, MSC_PROF_UPDATE);
    cudaError_t e = msc::launch_state_update(a, dtype, s);
    msc::profile_end(m, s);
    msc::profile_count(1);
    return e == cudaSuccess ? MSC_OK : MSC_ERR_CUDA;
}

msc_status msc_selective_state_update(float* state, const void* u, const void* dt,
                                      const float* A, const void* B, const void* C,
                                      const float* D, const void* z, const float* dt_bias,
                                      void* out, int64_t batch, int64_t d_inner,
                                      int64_t d_state, msc_dtype dtype, msc_stream_t stream) {
    return run_update(state, u, dt, A, B, C, D, z, dt_bias, out, batch, d_inner, d_state, dtype,
                      0, stream);
}

msc_status msc_selective_state_update_ex(float* state, const void* u, const void* dt,
                                         const float* A, const void* B, const void* C,
                                         const float* D, const void* z, const float* dt_bias,
                                         void* out, int64_t batch, int64_t d_inner,
                                         int64_t d_state, msc_dtype dtype,
                                         msc_discretization disc, msc_stream_t stream) {
    if (disc != MSC_DISC_EULER && disc != MSC_DISC_ZOH) return MSC_ERR_INVALID_ARG;
    return run_update(state, u, dt, A, B, C, D, z, dt_bias, out, batch, d_inner, d_state, dtype,
                      disc == MSC_DISC_ZOH ? 1 : 0, stream);
}

msc_status msc_selective_state_update_trap(float* state, const void* u_prev, const void* B_prev,
                                           const void* u, const void* dt, const void* lam,
                                           const float* A, const void* B, const void* C,
                                           const float* D, const void* z, const float* dt_bias,
                                           void* out, int64_t batch, int64_t d_inner,
                                           int64_t d_state, msc_dtype dtype,
                                           msc_stream_t stream) {
    if (!lam && batch > 0 && d_inner > 0) return MSC_ERR_INVALID_ARG;
    return run_update(state, u, dt, A, B, C, D, z, dt_bias, out, batch, d_inner, d_state, dtype,
                      0, stream, lam, u_prev, B_prev);
}

static msc_status run_bwd(const void* u, const void* dt, const float* A, const void* B,
                          const void* C, const float* D, const void* z, const float* dt_bias,
                          const float* h0, const void* dout, const float* dlast, void* du,
                          void* ddt, float* dA, float* dB, float* dC, float* dD, void* dz,
                          float* ddt_bias, float* dh0, int64_t batch, int64_t L,
                          int64_t d_inner, int64_t d_state, msc_dtype dtype,
                          msc_stream_t stream, const float* ckpt) {
    if (dtype != MSC_F32 && dtype != MSC_BF16) return MSC_ERR_INVALID_ARG;
    if (batch < 0 || L < 0 || d_inner < 0 || d_state < 0) return MSC_ERR_INVALID_ARG;
    if (d_state < 1 || d_state > 64) return MSC_ERR_UNSUPPORTED;
    int64_t bl, bld, bln, dn;
    if (!mul_ok(batch, L, &bl) || !mul_ok(bl, d_inner, &bld) || !mul_ok(bl, d_state, &bln) ||
        !mul_ok(d_inner, d_state, &dn) || bld > std::numeric_limits<int64_t>::max() / 8 ||
        bln > std::numeric_limits<int64_t>::max() / 8)
        return MSC_ERR_UNSUPPORTED;
    if (batch == 0 || d_inner == 0) return MSC_OK;
    if (!A || !dA || (L > 0 && (!u || !dt || !B || !C || !dout || !du || !ddt || !dB || !dC)))
        return MSC_ERR_INVALID_ARG;
    if (batch > 65535) return MSC_ERR_UNSUPPORTED;
    const size_t es = elem_size(dtype);
    const void* typed[] = {u, dt, B, C, z, dout, du, ddt, dz};
    for (const void* p : typed)
        if (p && !aligned(p, es)) return MSC_ERR_ALIGNMENT;
    const void* f32[] = {A, D, dt_bias, h0, dlast, dA, dB, dC, dD, ddt_bias, dh0};
    for (const void* p : f32)
        if (p && !aligned(p, 4)) return MSC_ERR_ALIGNMENT;
    if (ckpt && !aligned(ckpt, 16)) return MSC_ERR_ALIGNMENT;  // read as 16-byte vectors
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    msc::BwdArgs a{};
    a.u = u; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.dt_bias = dt_bias;
    a.h0 = h0; a.dout = dout; a.dlast = dlast; a.du = du; a.ddt = ddt; a.dA = dA; a.dB = dB;
    a.dC = dC; a.dD = dD; a.dz = dz; a.ddt_bias = ddt_bias; a.dh0 = dh0;
    a.batch = batch; a.L = L; a.d_inner = d_inner; a.N = d_state;
    // the TMA backward (checkpoints and adjoint in one kernel) where the shape
    // allows, else the element-load checkpoint and adjoint kernels
    const bool v2 = g_scan_path == 0 && L > 0 && L < kTmaMaxExtent &&
                    msc::bwd_tma_supported(d_state, d_inner, u, dt, z, dout, dB, dC);
    // the forward's checkpoints are read by the TMA backward only
    const bool ext = ckpt != nullptr && L > 0;
    if (ext && !v2) return MSC_ERR_UNSUPPORTED;
    a.ext_ckpt = ext ? 1 : 0;
    if (ext) a.ckpt = const_cast<float*>(ckpt);  // read only when ext_ckpt
    a.nseg = (L + msc::kBwdSegment - 1) / msc::kBwdSegment;
    a.vec = (d_state % 4 == 0) && (!B || aligned(B, 4 * es)) && (!C || aligned(C, 4 * es));
    // the accumulated gradients start from zero
    cudaError_t e = cudaMemsetAsync(dA, 0, (size_t)dn * sizeof(float), s);
    if (e == cudaSuccess && L > 0) e = cudaMemsetAsync(dB, 0, (size_t)bln * sizeof(float), s);
    if (e == cudaSuccess && L > 0) e = cudaMemsetAsync(dC, 0, (size_t)bln * sizeof(float), s);
    if (e == cudaSuccess && dD) e = cudaMemsetAsync(dD, 0, (size_t)d_inner * sizeof(float), s);
    if (e == cudaSuccess && ddt_bias)
        e = cudaMemsetAsync(ddt_bias, 0, (size_t)d_inner * sizeof(float), s);
    if (e != cudaSuccess) return MSC_ERR_CUDA;
    void* ck = nullptr;
    size_t ck_bytes = v2 ? msc::scan_bwd_tma_scratch(a, dtype)
                         : msc::scan_bwd_ckpt_bytes(batch, L, d_inner, d_state);
    if (ck_bytes == 0 && !ext) ck_bytes = 256;
    if (ck_bytes > 0 && scratch_alloc(&ck, ck_bytes, s) != cudaSuccess) return MSC_ERR_CUDA;
    if (v2) {
        e = msc::launch_scan_bwd_tma(a, dtype, ck, s);
    } else {
        a.ckpt = static_cast<float*>(ck);
        e = msc::launch_scan_bwd(a, dtype, s);
    }
    if (ck) {
        const cudaError_t f = cudaFreeAsync(ck, s);
        if (e == cudaSuccess) e = f;
    }
    return e == cudaSuccess ? MSC_OK : MSC_ERR_CUDA;
}

msc_status msc_selective_scan_bwd(const void* u, const void* dt, const float* A, const void* B,
                                  const void* C, const float* D, const void* z,
                                  const float* dt_bias, const float* h0, const void* dout,
                                  const float* dlast, void* du, void* ddt, float* dA, float* dB,
                                  float* dC, float* dD, void* dz, float* ddt_bias, float* dh0,
                                  int64_t batch, int64_t L, int64_t d_inner, int64_t d_state,
                                  msc_dtype dtype, msc_stream_t stream) {
    return run_bwd(u, dt, A, B, C, D, z, dt_bias, h0, dout, dlast, du, ddt, dA, dB, dC, dD, dz,
                   ddt_bias, dh0, batch, L, d_inner, d_state, dtype, stream, nullptr);
}

msc_status msc_selective_scan_bwd_ckpt(const void* u, const void* dt, const float* A,
                                       const void* B, const void* C, const float* D,
                                       const void* z, const float* dt_bias, const float* h0,
                                       const float* ckpt, const void* dout, const float* dlast,
                                       void* du, void* ddt, float* dA, float* dB, float* dC,
                                       float* dD, void* dz, float* ddt_bias, float* dh0,
                                       int64_t batch, int64_t L, int64_t d_inner,
                                       int64_t d_state, msc_dtype dtype, msc_stream_t stream) {
    if (!ckpt && batch > 0 && L > 0 && d_inner > 0) return MSC_ERR_INVALID_ARG;
    return run_bwd(u, dt, A, B, C, D, z, dt_bias, h0, dout, dlast, du, ddt, dA, dB, dC, dD, dz,
                   ddt_bias, dh0, batch, L, d_inner, d_state, dtype, stream, ckpt);
}

static msc_status run_conv(const void* x, const float* w, const float* bias,
                           const void* state_in, void* out, void* state, int64_t batch,
                           int64_t L, int64_t d_inner, int64_t d_conv, int silu,
                           msc_dtype dtype, bool update, msc_stream_t stream) {
    if (dtype != MSC_F32 && dtype != MSC_BF16) return MSC_ERR_INVALID_ARG;
    if (batch < 0 || L < 0 || d_inner < 0 || d_conv < 0 || (silu != 0 && silu != 1))
        return MSC_ERR_INVALID_ARG;
    if (d_conv < 1 || d_conv > 8) return MSC_ERR_UNSUPPORTED;
    int64_t bl, bld, bdk;
    if (!mul_ok(batch, L, &bl) || !mul_ok(bl, d_inner, &bld) || !mul_ok(batch, d_inner, &bdk) ||
        !mul_ok(bdk, d_conv, &bdk) || bld > std::numeric_limits<int64_t>::max() / 8)
        return MSC_ERR_UNSUPPORTED;
    if (batch == 0 || d_inner == 0) return MSC_OK;
    if (!w || ((update || L > 0) && (!x || !out)) || (update && d_conv > 1 && !state))
        return MSC_ERR_INVALID_ARG;
    if (batch > 65535 || (!update && (L + 63) / 64 > 65535)) return MSC_ERR_UNSUPPORTED;
    const size_t es = elem_size(dtype);
    const void* typed[] = {x, out, state_in, state};
    for (const void* p : typed)
        if (p && !aligned(p, es)) return MSC_ERR_ALIGNMENT;
    if (!aligned(w, 4) || (bias && !aligned(bias, 4))) return MSC_ERR_ALIGNMENT;
    msc::ConvArgs a{};
    a.x = x; a.w = w; a.bias = bias; a.state_in = update ? nullptr : state_in;
    a.out = out; a.state_out = state;
    a.batch = batch; a.L = update ? 1 : L; a.d_inner = d_inner; a.d_conv = d_conv;
    a.silu = silu;
    a.vec = !update && (d_inner % (int64_t)(8 / es) == 0) && (!x || aligned(x, 8)) &&
            (!out || aligned(out, 8));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = update ? msc::launch_conv1d_update(a, dtype, s)
                           : msc::launch_causal_conv1d(a, dtype, s);
    msc::profile_count(1);
    return e == cudaSuccess ? MSC_OK : MSC_ERR_CUDA;
}

msc_status msc_causal_conv1d_fwd(const void* x, const float* w, const float* bias,
                                 const void* state_in, void* out, void* state_out,
                                 int64_t batch, int64_t L, int64_t d_inner, int64_t d_conv,
                                 int silu, msc_dtype dtype, msc_stream_t stream) {
    return run_conv(x, w, bias, state_in, out, state_out, batch, L, d_inner, d_conv, silu,
                    dtype, false, stream);
}

msc_status msc_causal_conv1d_update(void* state, const void* x, const float* w,
                                    const float* bias, void* out, int64_t batch,
                                    int64_t d_inner, int64_t d_conv, int silu, msc_dtype dtype,
                                    msc_stream_t stream) {
    return run_conv(x, w, bias, nullptr, out, state, batch, 1, d_inner, d_conv, silu, dtype,
                    true, stream);
}

msc_status msc_tuning_set(const char* key, int64_t value) {
    if (!key || value < 0) return MSC_ERR_INVALID_ARG;
    if (std::strcmp(key, "scan_chunks") == 0) {
        g_force_chunks = value;
        return MSC_OK;
    }
    if (std::strcmp(key, "scan_lanes") == 0) {
        if (value != 0 && value != 2 && value != 4) return MSC_ERR_INVALID_ARG;
        g_scan_lanes = value;
        return MSC_OK;
    }
    if (std::strcmp(key, "scan_path") == 0) {
        if (value > 1) return MSC_ERR_INVALID_ARG;
        g_scan_path = value;
        return MSC_OK;
    }
    if (std::strcmp(key, "update_path") == 0) {
        if (value > 1) return MSC_ERR_INVALID_ARG;
        g_update_path = value;
        return MSC_OK;
    }
    if (std::strcmp(key, "debug_starve_copies") == 0) {
        if (value > (int64_t)msc::kWaitLimit) return MSC_ERR_INVALID_ARG;
        g_starve = value;
        return MSC_OK;
    }
    if (std::strcmp(key, "scan_min_chunk") == 0) {
        g_min_chunk = value > 0 ? value : 1;
        return MSC_OK;
    }
    return MSC_ERR_INVALID_ARG;
}

msc_status msc_profile_enable(int on) {
    g_profile = on != 0;
    return MSC_OK;
}

msc_status msc_profile_read(int64_t* launches, int64_t* timed, double* total_ms) {
    double ms[MSC_PROF_KINDS] = {};
    int64_t n[MSC_PROF_KINDS] = {};
    msc_status st = MSC_OK;
    for (auto& pr : g_prof_pairs) {
        float t = 0.0f;
        if (cudaEventSynchronize(pr.b) != cudaSuccess ||
            cudaEventElapsedTime(&t, pr.a, pr.b) != cudaSuccess)
            st = MSC_ERR_CUDA;
        ms[pr.kind] += t;
        n[pr.kind] += 1;
        g_prof_free.push_back(pr.a);
        g_prof_free.push_back(pr.b);
    }
    if (launches) *launches = g_prof_launches;
    for (int k = 0; k < MSC_PROF_KINDS; ++k) {
        if (timed) timed[k] = n[k];
        if (total_ms) total_ms[k] = ms[k];
    }
    g_prof_pairs.clear();
    g_prof_launches = 0;
    return st;
}

msc_status msc_check_device_error(int clear) {
    unsigned int v = 0, w = 0;
    if (msc::scan_error_word(&v, clear != 0) != cudaSuccess) return MSC_ERR_CUDA;
    if (msc::update_error_word(&w, clear != 0) != cudaSuccess) return MSC_ERR_CUDA;
    return (v | w) ? MSC_ERR_TIMEOUT : MSC_OK;
}

msc_status msc_scratch_release(void) {
    std::lock_guard<std::mutex> lock(g_pool_mu);
    for (cudaMemPool_t p : g_pools)
        if (p && cudaMemPoolTrimTo(p, 0) != cudaSuccess) return MSC_ERR_CUDA;
    return MSC_OK;
}

const char* msc_status_string(msc_status s) {
    switch (s) {
        case MSC_OK: return "ok";
        case MSC_ERR_INVALID_ARG: return "invalid argument";
        case MSC_ERR_UNSUPPORTED: return "unsupported size";
        case MSC_ERR_ALIGNMENT: return "pointer not aligned to its element size";
        case MSC_ERR_CUDA: return "CUDA runtime error";
        case MSC_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case MSC_ERR_TIMEOUT: return "a kernel's bounded wait for a data copy gave up";
        case MSC_ERR_SCRATCH_LIMIT:
            return "problem needs more scratch than the allocation-free entry point holds";
    }
    return "unknown status";
}

int msc_version(void) { return 100; }

}  // extern "C"
