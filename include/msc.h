/*
 * msc.h -- C ABI of the Mamba selective scan (S6) for NVIDIA B300 (sm_103a).
 *
 * Two operations, both defined by the web pages on the subject (and the
 * causal conv1d that produces the scan's input, declared further down):
 *
 *   msc_selective_scan_fwd   -- the selective scan forward of "Deep dive into
 *     Mamba: architecture and implementation of selective state-space models"
 *     (aiattnstudio.link/posts/mamba), sections 4.4 and 5.2, with the step
 *     size delta = softplus(dt + dt_bias) and the output gate y * silu(z) of
 *     the MambaBlock in "State space models and Mamba"
 *     (metaphor-xennon.pages.dev):
 *         delta = softplus(dt[b,t,d] + dt_bias[d])
 *         h[n]  = exp(delta * A[d,n]) * h[n] + delta * B[b,t,n] * u[b,t,d]
 *         y     = sum_n C[b,t,n] * h[n] + D[d] * u[b,t,d]
 *         out[b,t,d] = y * silu(z[b,t,d])             (silu(z) = z*sigmoid(z))
 *     with h = 0 before t = 0, the state h held in fp32, and the state after
 *     the last step written to last_state.
 *
 *   msc_selective_state_update -- one decode step of the same recurrence
 *     (the "Mamba decoding" example of "State space models and Mamba":
 *     constant memory per token), reading and writing the fp32 state in
 *     place.
 *
 *   The _ex forms add an initial state h0 (split prefill: a long prompt
 *   scanned in pieces, each seeded with the previous piece's last_state)
 *   and a choice of discretisation of B: delta*B as above (the form every
 *   listing on the pages uses), or the zero-order hold that the formulas of
 *   "State space models and Mamba" (section on discretisation) and "Deep
 *   dive into Mamba" (section 12) give, Bbar = A^-1 (exp(delta*A) - I) B,
 *   i.e. per state (exp(delta*A[d,n]) - 1) / A[d,n] * B[b,t,n] (delta*B
 *   where A[d,n] = 0).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers to contiguous row-major arrays.
 *     The caller owns every buffer; the library never frees caller memory.
 *   - `dtype` gives the storage type of u, dt, z, B, C and out (fp32 or
 *     bf16).  A, D, dt_bias, state and last_state are always fp32.  All
 *     arithmetic is fp32; out is rounded once, to nearest even.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     Argument errors are returned synchronously, before anything is
 *     launched; launch failures return MSC_ERR_CUDA.  Faults inside a
 *     kernel surface at the caller's next synchronisation.
 *   - out must not overlap any input.  Inputs are never written.
 *   - Pointers must be aligned to their element size; wider alignment
 *     (16 bytes) selects vector loads, any other alignment still runs on the
 *     GPU with element loads.  There is no CPU fallback.
 *   - Supported sizes: batch, L, d_inner >= 0; 1 <= d_state <= 64; every
 *     array's element count must fit in int64 and the launch grid in 2^31-1
 *     blocks.  Empty batches are valid and launch nothing.
 */
#ifndef MSC_H
#define MSC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* msc_stream_t;

typedef enum msc_dtype {
    MSC_F32 = 0,  /* float */
    MSC_BF16 = 1  /* bfloat16 (1 sign, 8 exponent, 7 mantissa bits) */
} msc_dtype;

typedef enum msc_status {
    MSC_OK = 0,
    MSC_ERR_INVALID_ARG = 1,  /* NULL required pointer, negative size, bad dtype */
    MSC_ERR_UNSUPPORTED = 2,  /* d_state outside [1, 64], or sizes overflow */
    MSC_ERR_ALIGNMENT = 3,    /* a pointer not aligned to its element size */
    MSC_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    MSC_ERR_WORKSPACE = 5,    /* workspace NULL, smaller than required or misaligned */
    MSC_ERR_TIMEOUT = 6,      /* a kernel gave up waiting for a data copy (see
                                 msc_check_device_error) */
    MSC_ERR_SCRATCH_LIMIT = 7 /* msc_selective_scan_fwd_noalloc: the problem needs
                                 more scratch than MSC_NOALLOC_SCRATCH_BYTES */
} msc_status;

/*
 * Selective scan forward.
 *   u, dt, z, out : (batch, L, d_inner), `dtype`       z nullable: no gate
 *   B, C          : (batch, L, d_state), `dtype`
 *   A             : (d_inner, d_state) fp32            any real values
 *   D, dt_bias    : (d_inner) fp32                     nullable: 0
 *   last_state    : (batch, d_inner, d_state) fp32     nullable: not written
 * With L == 0 last_state is set to zero.  Scratch for the inter-chunk carry,
 * when the plan needs it, is taken stream-ordered on `stream` from the
 * library's memory pool (see msc_scratch_release); use
 * msc_selective_scan_fwd_ws to pass it in.
 */
msc_status msc_selective_scan_fwd(
    const void* u, const void* dt, const float* A, const void* B,
    const void* C, const float* D, const void* z, const float* dt_bias,
    void* out, float* last_state, int64_t batch, int64_t L, int64_t d_inner,
    int64_t d_state, msc_dtype dtype, msc_stream_t stream);

/*
 * Bytes of device workspace msc_selective_scan_fwd_ws needs for these sizes
 * on the current device (0 when the plan runs in one pass).  The plan, and
 * so the size, depends on the device's SM count and on msc_tuning_set.
 */
msc_status msc_selective_scan_workspace_size(
    int64_t batch, int64_t L, int64_t d_inner, int64_t d_state,
    msc_dtype dtype, size_t* bytes);

/*
 * As msc_selective_scan_fwd, with caller-owned device workspace of at least
 * msc_selective_scan_workspace_size bytes, 256-byte aligned (NULL allowed
 * when that size is 0).  Nothing is allocated.  The workspace is scratch:
 * its contents on entry do not matter, and two calls that share one
 * workspace must not run concurrently.
 */
msc_status msc_selective_scan_fwd_ws(
    const void* u, const void* dt, const float* A, const void* B,
    const void* C, const float* D, const void* z, const float* dt_bias,
    void* out, float* last_state, int64_t batch, int64_t L, int64_t d_inner,
    int64_t d_state, msc_dtype dtype, void* workspace,
    size_t workspace_bytes, msc_stream_t stream);

/*
 * Allocation-free variant of msc_selective_scan_fwd (the pages have no
 * counterpart: this is a deployment facility of this library).
 *
 * Some callers cannot call cudaMalloc or cudaMallocAsync on the path that
 * runs the scan: a serving runtime that reserves all device memory through
 * its own allocator at start-up and forbids allocation while requests are
 * in flight, or a host application whose memory manager owns the device.
 * This entry point takes the same arguments as msc_selective_scan_fwd and
 * allocates nothing.  The scratch the scan needs (chunk carries, fp32 copies
 * of B and C) lives in one file-scope device array of
 * MSC_NOALLOC_SCRATCH_BYTES (16 MiB), which every GPU that loads the library
 * holds until the process exits.
 *   - A problem whose plan needs more scratch than that returns
 *     MSC_ERR_SCRATCH_LIMIT before anything is launched (query the need with
 *     msc_selective_scan_workspace_size).
 *   - Every call whose stream is not being captured looks up the array's
 *     device address with cudaGetSymbolAddress on the current device (so
 *     the address is right again after a device reset, which reloads the
 *     module, possibly at another address); a call on a capturing stream
 *     uses the address the last uncaptured call on that device found, and
 *     fails with MSC_ERR_CUDA when there was none.  Make the first call on
 *     each device before any stream capture on it.
 *   - With CUDA's default lazy module loading, the array is mapped on a
 *     device by the first call into this library on that device, and that
 *     mapping is a device allocation.  A caller that may not allocate while
 *     serving makes one call into the library on each device at start-up
 *     (a scan of any size will do), before serving begins.
 *   - All calls share the one array, and it keeps the last call's contents;
 *     nothing in it needs to start at zero (every byte a call reads was
 *     written earlier in the same call).  Calls whose executions overlap on
 *     the GPU (different streams, no ordering between them) race on it.
 * Other behaviour, layouts and errors are those of msc_selective_scan_fwd.
 */
#define MSC_NOALLOC_SCRATCH_BYTES (16u << 20)
msc_status msc_selective_scan_fwd_noalloc(
    const void* u, const void* dt, const float* A, const void* B,
    const void* C, const float* D, const void* z, const float* dt_bias,
    void* out, float* last_state, int64_t batch, int64_t L, int64_t d_inner,
    int64_t d_state, msc_dtype dtype, msc_stream_t stream);

/*
 * Causal depthwise conv1d (+ SiLU) that produces the scan's input u from the
 * block's projected input x ("Deep dive into Mamba", section 3.2: Conv1d
 * with kernel d_conv, padding d_conv - 1, one group per channel, bias;
 * section 5.2 and the MambaBlock of "State space models and Mamba": the
 * first L outputs, then SiLU):
 *     out[b,t,d] = silu(bias[d] + sum_k w[d,k] * x[b, t - (d_conv-1) + k, d])
 *   x, out        : (batch, L, d_inner), `dtype`
 *   w             : (d_inner, d_conv) fp32;  bias: (d_inner) fp32, nullable
 *   state_in      : (batch, d_inner, d_conv-1), `dtype`, nullable: the
 *                   d_conv-1 inputs before t = 0, oldest first (zero if NULL)
 *   state_out     : same layout, nullable: receives the last d_conv-1
 *                   inputs (the state msc_causal_conv1d_update continues
 *                   from); with L < d_conv-1 it includes state_in's tail
 *   silu          : 1 apply SiLU, 0 return the linear conv; else
 *                   MSC_ERR_INVALID_ARG
 * 1 <= d_conv <= 8 (MSC_ERR_UNSUPPORTED otherwise); batch <= 65535 and
 * L <= 4,194,240.  out must not overlap x or the states; state_in and
 * state_out must not overlap each other.  Arithmetic fp32, out rounded once.
 */
msc_status msc_causal_conv1d_fwd(
    const void* x, const float* w, const float* bias, const void* state_in,
    void* out, void* state_out, int64_t batch, int64_t L, int64_t d_inner,
    int64_t d_conv, int silu, msc_dtype dtype, msc_stream_t stream);

/*
 * One decode token of the same conv: the window is the d_conv-1 inputs in
 * `state` followed by x; out = (SiLU of) bias + sum_k w[d,k] * window[k];
 * then `state` drops its oldest input and appends x, in place.
 *   state         : (batch, d_inner, d_conv-1), `dtype` (NULL allowed only
 *                   for d_conv == 1)
 *   x, out        : (batch, d_inner), `dtype`;  w, bias as above.
 */
msc_status msc_causal_conv1d_update(
    void* state, const void* x, const float* w, const float* bias, void* out,
    int64_t batch, int64_t d_inner, int64_t d_conv, int silu, msc_dtype dtype,
    msc_stream_t stream);

/*
 * Backward pass of msc_selective_scan_fwd (the Euler form): the gradients of
 * a loss J(out, last_state) given dout = dJ/dout and dlast_state =
 * dJ/dlast_state.  The states are recomputed from checkpoints (one per 32
 * steps), not read from the forward -- the pages' chunk + recompute scheme
 * ("Deep dive into Mamba" section 7.3) -- and the adjoint
 *     dh_t = C_t * dy_t + exp(delta_{t+1}*A) * dh_{t+1},  dy_t = dout_t * silu(z_t)
 * runs backwards through the sequence.
 *   forward inputs: as msc_selective_scan_fwd (h0 nullable: zero)
 *   dout          : (batch, L, d_inner), `dtype`
 *   dlast_state   : (batch, d_inner, d_state) fp32, nullable: zero
 *   du, ddt, dz   : (batch, L, d_inner), `dtype` (ddt is d/d dt, before the
 *                   softplus); dz nullable (not written), zeros when z is NULL
 *   dA            : (d_inner, d_state) fp32
 *   dB, dC        : (batch, L, d_state) fp32 (sums over the channels)
 *   dD, ddt_bias  : (d_inner) fp32, nullable (not written)
 *   dh0           : (batch, d_inner, d_state) fp32, nullable (not written)
 * dA, dB, dC, dD, ddt_bias are accumulated with atomic adds after being
 * zeroed by the call: their last bits depend on the order of the adds.
 * Scratch, taken stream-ordered: the checkpoints, batch * d_inner * d_state
 * * 4 bytes per 16 steps (d_state <= 16 on the TMA path) or 8 steps
 * (d_state 32, 64) or 32 steps (element-load path), plus fp32 copies of B
 * and C for bf16 storage.  batch <= 65535.  Errors as msc_selective_scan_fwd.
 */
msc_status msc_selective_scan_bwd(
    const void* u, const void* dt, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* dt_bias, const float* h0,
    const void* dout, const float* dlast_state, void* du, void* ddt, float* dA,
    float* dB, float* dC, float* dD, void* dz, float* ddt_bias, float* dh0,
    int64_t batch, int64_t L, int64_t d_inner, int64_t d_state, msc_dtype dtype,
    msc_stream_t stream);

/* Discretisation of the input matrix B (the _ex entry points). */
typedef enum msc_discretization {
    MSC_DISC_EULER = 0,  /* delta * B                                    */
    MSC_DISC_ZOH = 1     /* (exp(delta*A) - 1) / A * B  (zero-order hold) */
} msc_discretization;

/*
 * The scan of msc_selective_scan_fwd with two additions:
 *   h0   : (batch, d_inner, d_state) fp32, the state before t = 0.
 *          Nullable: zero.  Must not overlap last_state or out (every time
 *          chunk of the plan reads it).  With L == 0, last_state = h0.
 *   disc : MSC_DISC_EULER or MSC_DISC_ZOH; anything else is
 *          MSC_ERR_INVALID_ARG.
 * workspace: NULL takes the scratch stream-ordered as msc_selective_scan_fwd
 * does; otherwise as msc_selective_scan_fwd_ws (size from
 * msc_selective_scan_workspace_size, which does not depend on h0 or disc).
 * Other arguments, layouts and errors as msc_selective_scan_fwd.
 */
msc_status msc_selective_scan_fwd_ex(
    const void* u, const void* dt, const float* A, const void* B,
    const void* C, const float* D, const void* z, const float* dt_bias,
    const float* h0, void* out, float* last_state, int64_t batch, int64_t L,
    int64_t d_inner, int64_t d_state, msc_dtype dtype,
    msc_discretization disc, void* workspace, size_t workspace_bytes,
    msc_stream_t stream);

/*
 * Training without the backward's re-walk.  msc_selective_scan_bwd recomputes
 * the states at the start of every tile of its own by walking the sequence
 * forward again (one exponential per state update, about a fifth of its
 * work).  A forward scan that is followed by a backward can write those
 * states as it goes -- the pages' "save the states at chunk boundaries,
 * recompute inside the chunk" scheme ("Deep dive into Mamba", section 7.3) --
 * and the backward then starts at once from the last tile.
 *
 * msc_scan_checkpoint_size: the interval (steps between checkpoints: 16 for
 * d_state 8 and 16, 8 for 32 and 64) and the bytes of the checkpoint array,
 *     (batch, rows, d_inner, d_state) fp32, rows = ceil(L / interval),
 * row k = the state entering step k * interval (row 0 = h0, or zero).
 * d_state other than 8, 16, 32, 64 is MSC_ERR_UNSUPPORTED; negative sizes
 * MSC_ERR_INVALID_ARG; sizes whose byte count overflows MSC_ERR_UNSUPPORTED.
 */
msc_status msc_scan_checkpoint_size(int64_t batch, int64_t L, int64_t d_inner,
                                    int64_t d_state, int64_t* interval,
                                    size_t* bytes);

/*
 * msc_selective_scan_fwd_ex (Euler form, optional h0) that also writes the
 * checkpoint array `ckpt` (caller-owned device memory, 16-byte aligned,
 * msc_scan_checkpoint_size bytes; every row is written).  Other arguments,
 * the workspace and the results as msc_selective_scan_fwd_ex: out and
 * last_state are bit-identical to that call's.  The checkpoints are written
 * by the TMA-staged kernel only: d_state 8, 16, 32 or 64, d_inner a multiple
 * of 8, u, dt, z 16-byte aligned; other shapes are MSC_ERR_UNSUPPORTED (use
 * msc_selective_scan_bwd, which recomputes them).  ckpt NULL with work to do:
 * MSC_ERR_INVALID_ARG.
 */
msc_status msc_selective_scan_fwd_ckpt(
    const void* u, const void* dt, const float* A, const void* B,
    const void* C, const float* D, const void* z, const float* dt_bias,
    const float* h0, void* out, float* last_state, float* ckpt, int64_t batch,
    int64_t L, int64_t d_inner, int64_t d_state, msc_dtype dtype,
    void* workspace, size_t workspace_bytes, msc_stream_t stream);

/*
 * msc_selective_scan_bwd reading the checkpoints `ckpt` that
 * msc_selective_scan_fwd_ckpt wrote for the same inputs (and h0) instead of
 * recomputing them; nothing of ckpt is written.  Arguments, results and
 * errors as msc_selective_scan_bwd, plus: the TMA backward is required
 * (d_state 8, 16, 32, 64, d_inner a multiple of 8, u, dt, z, dout, dB, dC
 * 16-byte aligned), else MSC_ERR_UNSUPPORTED; ckpt 16-byte aligned, else
 * MSC_ERR_ALIGNMENT; NULL with work to do, MSC_ERR_INVALID_ARG.  When the
 * forward ran in one time chunk, its checkpoints are the states the backward
 * would recompute, bit for bit, and du, ddt, dz, dh0 equal
 * msc_selective_scan_bwd's bit for bit (the atomically summed gradients up to
 * the order of their adds); when it split time into chunks (long sequences
 * over few channels), the rows at chunk starts carry the chunked scan's
 * rounding.  Scratch: only the fp32 copies of B and C for bf16 storage (or
 * unaligned fp32).
 */
msc_status msc_selective_scan_bwd_ckpt(
    const void* u, const void* dt, const float* A, const void* B, const void* C,
    const float* D, const void* z, const float* dt_bias, const float* h0,
    const float* ckpt, const void* dout, const float* dlast_state, void* du,
    void* ddt, float* dA, float* dB, float* dC, float* dD, void* dz,
    float* ddt_bias, float* dh0, int64_t batch, int64_t L, int64_t d_inner,
    int64_t d_state, msc_dtype dtype, msc_stream_t stream);

/*
 * The Mamba-3 exponential-trapezoid scan ("State space models and the Mamba
 * series", section 2.1), in the S6 layout: the input term mixes the previous
 * and the current step with a data-dependent lambda in [0, 1],
 *     h_t = exp(delta_t*A) h_{t-1} + (1 - lambda_t)*delta_t * B_{t-1} u_{t-1}
 *                                  + lambda_t*delta_t * B_t u_t
 * (the formula as the page prints it: no decay on the t-1 term); the rest as
 * msc_selective_scan_fwd (softplus step size, y = C.h + D*u, gate).
 *   lam           : (batch, L, d_inner), `dtype`, values in [0, 1]; required
 *   u_prev        : (batch, d_inner), `dtype`, nullable: u of the step before
 *                   t = 0 (split prefill: the previous piece's last u)
 *   B_prev        : (batch, d_state), `dtype`, nullable: its B; the t = 0
 *                   previous-step term is zero unless both are given
 *   h0, workspace : as msc_selective_scan_fwd_ex
 * lambda = 1 everywhere gives the msc_selective_scan_fwd result bit for bit.
 * Errors as msc_selective_scan_fwd; lam NULL is MSC_ERR_INVALID_ARG.
 */
msc_status msc_selective_scan_trap_fwd(
    const void* u, const void* dt, const void* lam, const float* A,
    const void* B, const void* C, const float* D, const void* z,
    const float* dt_bias, const float* h0, const void* u_prev,
    const void* B_prev, void* out, float* last_state, int64_t batch,
    int64_t L, int64_t d_inner, int64_t d_state, msc_dtype dtype,
    void* workspace, size_t workspace_bytes, msc_stream_t stream);

/*
 * Single-token selective state update (decode).
 *   state         : (batch, d_inner, d_state) fp32, read and written in place
 *   u, dt, z, out : (batch, d_inner), `dtype`          z nullable: no gate
 *   B, C          : (batch, d_state), `dtype`
 *   A             : (d_inner, d_state) fp32
 *   D, dt_bias    : (d_inner) fp32                     nullable: 0
 * out must not overlap state or any input.
 */
msc_status msc_selective_state_update(
    float* state, const void* u, const void* dt, const float* A,
    const void* B, const void* C, const float* D, const void* z,
    const float* dt_bias, void* out, int64_t batch, int64_t d_inner,
    int64_t d_state, msc_dtype dtype, msc_stream_t stream);

/*
 * msc_selective_state_update with a choice of discretisation (`disc` as in
 * msc_selective_scan_fwd_ex); a ZOH scan's last_state continues with ZOH
 * decode steps.  Same arguments and errors otherwise.
 */
msc_status msc_selective_state_update_ex(
    float* state, const void* u, const void* dt, const float* A,
    const void* B, const void* C, const float* D, const void* z,
    const float* dt_bias, void* out, int64_t batch, int64_t d_inner,
    int64_t d_state, msc_dtype dtype, msc_discretization disc,
    msc_stream_t stream);

/*
 * One decode token of the exponential-trapezoid scan: u_prev / B_prev are
 * the previous token's u (batch, d_inner) and B (batch, d_state) (nullable:
 * zero term); lam (batch, d_inner).  Other arguments as
 * msc_selective_state_update.
 */
msc_status msc_selective_state_update_trap(
    float* state, const void* u_prev, const void* B_prev, const void* u,
    const void* dt, const void* lam, const float* A, const void* B,
    const void* C, const float* D, const void* z, const float* dt_bias,
    void* out, int64_t batch, int64_t d_inner, int64_t d_state,
    msc_dtype dtype, msc_stream_t stream);

/*
 * Kernels never spin without bound: every wait for an asynchronous copy
 * gives up after a fixed number of polls, records the event in a device
 * word, and the kernel exits early (its outputs are then incomplete).  This
 * reads that word -- call it after synchronising the streams the library
 * was used on -- and returns MSC_ERR_TIMEOUT when it is set, MSC_OK
 * otherwise; a nonzero `clear` resets it.  MSC_ERR_CUDA if the read fails.
 * Each device has its own word and this reads the CURRENT device's only: a
 * caller that runs the library on several devices calls it once per device,
 * with that device current.
 */
msc_status msc_check_device_error(int clear);

/*
 * Calls that take scratch stream-ordered (msc_selective_scan_fwd,
 * msc_selective_scan_fwd_ex without a workspace, the trapezoid scan and
 * msc_selective_scan_bwd) draw it from a memory pool that the library keeps
 * on each device and that holds on to the memory it has reserved, so that
 * repeated calls do not map memory again.  This returns the pools' unused
 * memory to the device (cudaMemPoolTrimTo); memory of calls still in flight
 * on some stream stays reserved.  MSC_ERR_CUDA if a trim fails.
 */
msc_status msc_scratch_release(void);

/*
 * Plan overrides, for measurement and tuning.  Keys:
 *   "scan_chunks"   number of time chunks the scan is cut into (0 = auto)
 *   "scan_min_chunk" shortest chunk the automatic plan will make (steps)
 *   "scan_path"     0 = automatic, 1 = element-load kernels only (no TMA)
 *   "scan_lanes"    lanes per channel of the TMA kernels: 0 = automatic, 2, 4
 *   "update_path"   0 = automatic (d_state 16, 32, 64: the copy-engine
 *                   streaming decode kernel where sizes and alignment
 *                   allow), 1 = the thread-per-channel and general decode
 *                   kernels only
 *   "debug_starve_copies"  failure-detection test, 0 (default) = off; n > 0:
 *                   the forward scan's TMA kernels and the streaming decode
 *                   kernel issue none of their data copies and give up each
 *                   wait after n polls, so every such launch ends through the
 *                   bounded-wait exit (device word set, msc_check_device_error
 *                   -> MSC_ERR_TIMEOUT, outputs and state not written).  No
 *                   copy is in flight when the kernel returns and nothing
 *                   faults.
 * Process-wide and not thread-safe; returns MSC_ERR_INVALID_ARG for an
 * unknown key or a negative value.
 */
msc_status msc_tuning_set(const char* key, int64_t value);

/*
 * Measurement hook.  While enabled, every call records a CUDA event pair
 * on its stream around its main kernel (the kinds below) and counts every
 * kernel it launches.  msc_profile_read synchronises those events and
 * returns, since the last read: the number of kernels launched, and per
 * kind the number of timed main kernels and their summed device time in
 * milliseconds (arrays of MSC_PROF_KINDS, indexed by kind; NULL outputs are
 * skipped);
 * then it resets.  Process-wide and not thread-safe.  Disabled by default.
 */
enum {
    MSC_PROF_SCAN = 0,         /* scan output kernel                 */
    MSC_PROF_UPDATE = 1,       /* decode state-update kernel         */
    MSC_PROF_CONV = 2,         /* causal conv1d prefill kernel       */
    MSC_PROF_CONV_UPDATE = 3,  /* causal conv1d decode-update kernel */
    MSC_PROF_SCAN_BWD = 4,     /* scan backward (adjoint) kernel      */
    MSC_PROF_KINDS = 5
};
msc_status msc_profile_enable(int on);
msc_status msc_profile_read(int64_t* launches, int64_t* timed, double* total_ms);

/* Static description of a status code (never NULL). */
const char* msc_status_string(msc_status status);

/* Library version, as major*10000 + minor*100 + patch. */
int msc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MSC_H */
