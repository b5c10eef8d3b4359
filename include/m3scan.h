/*
 * m3scan.h -- C ABI of the GB300 selective-scan layer core (Mamba-1).
 *
 * The layer core, forward (the per-layer loop of
 * gpu_forward_mamba_backbone_mixed on the mamba-rs 0.3.1 page
 * src/mamba_ssm/gpu/forward_mixed.rs, steps F4a conv1d, F4c softplus,
 * F4d selective scan, F4e gating):
 *
 *   c[t]     = conv_b + sum_{k<4} conv_w[k] * x[t-3+k]
 *              (x = 0 for t < 0, or a carried conv state, m3scan_fwd_state)
 *   u[t]     = c[t] * sigmoid(c[t])
 *   delta[t] = softplus(delta_raw[t] + dt_bias)
 *   A[n]     = -exp(a_log[n])                 (trainer.rs 0.7.3, recompute_a_neg_all)
 *   h_t[n]   = exp(delta[t] * A[n]) * h_{t-1}[n] + delta[t] * B_t[n] * u[t],
 *              h_{-1} = 0 (or a carried state, m3scan_fwd_state)
 *   y[t]     = sum_n C_t[n] * h_t[n] + D * u[t]
 *   gated[t] = y[t] * z[t] * sigmoid(z[t])
 *
 * per (batch b, channel d); B_t and C_t are shared by every channel of a
 * token.  The backward is the reverse-time derivative of
 * L = sum gated * d_gated, giving the gradients the backward scratch of the
 * same page names (d_u, d_delta, d_B, d_C reduced over d_inner, d_D, d_a_log,
 * softplus and conv1d backward).
 *
 * Layouts (row-major, channel fastest; every pointer is a DEVICE pointer):
 *   x, delta_raw, z, gated, y_dbg, d_gated, d_x, d_delta_raw, dz, du_dbg
 *                       : [batch, seq_len, d_inner]  activation dtype
 *   Bm, Cm              : [batch, seq_len, d_state]  activation dtype
 *   dB, dC              : [batch, seq_len, d_state]  float32
 *   conv_w, d_conv_w    : [d_inner, d_conv]          float32
 *   a_log, d_a_log      : [d_inner, d_state]         float32
 *   conv_b, dt_bias, D and their grads : [d_inner]   float32
 *   ckpt                : [batch, n_chunks, d_state, d_inner] float32, where
 *                         ckpt[b, c, n, d] is h before step c * chunk.
 *
 * Ownership: the caller allocates and frees every buffer, including the
 * workspace sized by m3scan_plan.  The library never allocates, frees or
 * synchronises; all work is enqueued on `stream` in order.  Buffers must
 * stay valid until that work completes.  Calls on one workspace must not
 * overlap on the GPU.
 *
 * Errors: arguments are validated before anything is enqueued; a failed
 * validation returns a status and enqueues nothing.  A failed launch
 * returns M3_ERR_CUDA (the CUDA error is cleared with cudaGetLastError).
 * Unsupported shapes return M3_ERR_UNSUPPORTED; there is no fallback path.
 * (The mamba-rs 0.4.0 page src/mamba3_siso/gpu/backward_mixed.rs states the
 * same rules in its module header: labelled errors, never a silent
 * fallback.)  Errors that only the GPU can see -- a kernel that gave up
 * waiting for a tile copy (every such wait is bounded to about a second, so
 * the GPU cannot hang) -- are recorded on the device: in the status block at
 * the start of the call's workspace, read with m3scan_get_status, and in a
 * per-device word read with m3scan_device_status.
 *
 * Workspace status block: the first M3SCAN_STATUS_BYTES of every workspace
 * belong to the library.  They must be zero when a workspace is first used
 * (allocate it zeroed, or clear those bytes); kernels only ever set bits in
 * them, and m3scan_get_status reads and clears them.
 */
#ifndef M3SCAN_H
#define M3SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st* m3_stream_t;

typedef enum {
    M3_F32 = 0,  /* activations stored as float32 */
    M3_BF16 = 1  /* activations stored as bfloat16 (state, params, grads f32) */
} m3_dtype;

typedef enum {
    M3_OK = 0,
    M3_ERR_NULL = 1,        /* a required pointer is NULL */
    M3_ERR_DIMS = 2,        /* a size is negative or out of range */
    M3_ERR_UNSUPPORTED = 3, /* d_state not 16/32/64, d_conv != 4, d_inner % 8 != 0, dtype */
    M3_ERR_ALIGN = 4,       /* a pointer is not aligned as required */
    M3_ERR_WORKSPACE = 5,   /* workspace missing or smaller than planned */
    M3_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed */
    M3_ERR_TIMEOUT = 7      /* reported by m3scan_get_status: a kernel of an earlier call
                               gave up waiting for a tile copy; that call's outputs are
                               incomplete */
} m3_status;

/* Bytes at the start of every workspace that hold the status block. */
#define M3SCAN_STATUS_BYTES 256

typedef struct {
    int64_t batch, seq_len, d_inner, d_state, d_conv;
    /* Checkpoint interval K in steps: the forward writes the state before
       every K-th step, the backward recomputes from there.  0 = library
       default (8).  1..8, or a multiple of 8 up to 256 (other values:
       M3_ERR_UNSUPPORTED; above 256: M3_ERR_DIMS).  The backward recomputes
       at most 8 steps on chip at a time: with K > 8 it first runs each chunk
       forward from its checkpoint to the start of every 8-step tile, keeping
       those states in the workspace (m3scan_plan sizes it), so a longer
       chunk moves fewer checkpoint bytes through HBM for more arithmetic. */
    int64_t chunk;
    /* Number of time segments scanned in parallel (each segment is a run of
       whole chunks); 0 = chosen from the shape and the current device. */
    int64_t segments;
    /* 1: param grads are added to the output buffers; 0: overwritten. */
    int32_t accumulate_param_grads;
    /* Kernel variant of the forward's and the backward's main passes:
       1 = one thread per channel (16 state lanes each, the most channels per
       SM; d_state 16 only), 2 = the split kernels (8 lanes per thread,
       d_state / 8 threads per channel: half the per-thread work at d_state
       16, for grids that fill less than one wave), 0 = chosen per pass
       (d_state 32 and 64 always take the split kernels).  The plan reports
       the threads per channel chosen.  Same results up to the order of f32
       sums. */
    int32_t threads_per_channel;
    /* Row strides, in elements, between consecutive (batch, step) rows of
       Bm and Cm, and of dB and dC; 0 = d_state (dense).  A stride > d_state
       lets Bm/Cm be column slices of the x_proj output [batch, seq_len,
       dt_rank + 2 d_state] and dB/dC slices of its gradient, with no copy
       (the x_proj step F4b of forward_mixed.rs splits one GEMM output into
       dt_low, B and C).  bc_stride times the activation size must be a
       multiple of 16 bytes (M3_ERR_ALIGN otherwise).  Only the d_state
       columns of each row are read or written. */
    int64_t bc_stride;
    int64_t dbc_stride;
    /* dB and dC are sums over all channels, the parameter gradients
       (d_a_log, dD, d_dt_bias, d_conv_w, d_conv_b) sums over batch and
       time.  0: blocks add their shares of dB and dC with float atomics,
       and so do the clusters of the split backward over 2-8 time segments
       for the parameter gradients (fastest; the order of the additions, and
       so the last bits of these outputs, may differ between runs).  1: every
       block writes its shares to the workspace and the backward's last
       kernels add them in a fixed order, so repeated calls give identical
       bits for every output.  The workspace then also holds
       batch * seq_len * 2 * d_state floats per channel block and the
       per-(batch, segment) parameter partials.  d_x, d_delta_raw, dz and du
       are the same bits either way. */
    int32_t deterministic;
    int32_t reserved0;  /* must be 0 */
} m3_dims;

typedef struct {
    int64_t chunk;              /* K actually used */
    int64_t n_chunks;           /* ceil(seq_len / K) */
    int64_t fwd_segments;       /* time segments of the forward */
    int64_t bwd_segments;       /* time segments of the backward */
    int64_t ckpt_bytes;         /* size of ckpt */
    int64_t workspace_bytes;    /* size of the workspace both calls need */
    int32_t fwd_launches;       /* kernels one m3scan_fwd enqueues */
    int32_t bwd_launches;       /* kernels one m3scan_bwd enqueues (memsets excluded) */
    int32_t fwd_threads_per_channel;  /* 1, or d_state / 8 for the split kernels */
    int32_t bwd_threads_per_channel;
} m3_plan;

/*
 * Resolve defaults and size the caller-owned buffers.  With
 * dims->segments == 0 it queries the current CUDA device (SM count and
 * kernel occupancy); with an explicit segment count it touches no device.
 * Returns M3_OK and fills *plan, or a validation status.
 */
m3_status m3scan_plan(const m3_dims* dims, m3_dtype act, m3_plan* plan);

/*
 * Forward.  Writes gated (and y_dbg = y when non-NULL) and the chunk
 * checkpoints ckpt that m3scan_bwd reads.  Activation pointers and ckpt
 * must be 16-byte aligned; the other float32 pointers 4-byte aligned;
 * workspace 256-byte aligned with workspace_bytes >= plan.workspace_bytes.
 */
m3_status m3scan_fwd(const m3_dims* dims, m3_dtype act,
                     const void* x, const void* delta_raw, const void* z,
                     const void* Bm, const void* Cm,
                     const float* conv_w, const float* conv_b,
                     const float* dt_bias, const float* a_log, const float* D,
                     void* gated, void* y_dbg, float* ckpt,
                     void* workspace, size_t workspace_bytes,
                     m3_stream_t stream);

/*
 * Backward of L = sum(gated * d_gated), from the forward's inputs and its
 * checkpoints.  Writes d_x, d_delta_raw, dz (and du_dbg = dL/du through the
 * D skip and the recurrence, when non-NULL) in the activation dtype;
 * overwrites dB and dC (float32, reduced over d_inner); writes or adds the
 * float32 parameter grads d_conv_w, d_conv_b, d_dt_bias, d_a_log, dD per
 * dims->accumulate_param_grads.  dims->chunk must equal the chunk the
 * forward that wrote ckpt used; the segment counts of the two calls are
 * independent of each other.
 */
m3_status m3scan_bwd(const m3_dims* dims, m3_dtype act,
                     const void* x, const void* delta_raw, const void* z,
                     const void* Bm, const void* Cm,
                     const float* conv_w, const float* conv_b,
                     const float* dt_bias, const float* a_log, const float* D,
                     const float* ckpt, const void* d_gated,
                     void* d_x, void* d_delta_raw, void* dz, void* du_dbg,
                     float* dB, float* dC,
                     float* d_conv_w, float* d_conv_b, float* d_dt_bias,
                     float* d_a_log, float* dD,
                     void* workspace, size_t workspace_bytes,
                     m3_stream_t stream);

/*
 * Carried state.  The mamba-rs pages carry two pieces of recurrent state
 * from one call to the next: the conv1d of step F4a reads and updates a
 * per-layer conv state (the last d_conv-1 conv inputs of each channel), and
 * the selective scan of step F4d reads and writes the SSM state h through a
 * state pointer (forward_mixed.rs 0.3.1, the per-layer loop of
 * gpu_forward_mamba_backbone_mixed); the trainer (trainer.rs 0.7.3) keeps
 * them between windows of a long sequence and zeroes them in reset_state.
 * With these structs a window starts from a given state and returns its
 * final one, so that running a sequence window by window, each window from
 * the previous one's outputs, gives the results of one call over the whole
 * sequence (and the backward chains the same way, in reverse order).
 *
 * Layouts (DEVICE pointers, channel fastest):
 *   ssm_state, ssm_state_out, d_ssm_state, d_ssm_state_out
 *        : [batch, d_state, d_inner] float32; ssm_state is h_{-1} (the state
 *          before step 0), ssm_state_out is h_{seq_len-1};
 *   conv_state, conv_state_out, d_conv_state, d_conv_state_out
 *        : [batch, d_conv-1, d_inner] activation dtype, oldest step first;
 *          conv_state row r is the conv input x of step r-(d_conv-1), and
 *          conv_state_out row r that of step seq_len-(d_conv-1)+r (taken
 *          from conv_state where that step is negative).
 * Every pointer may be NULL: a NULL input state means zero (the
 * reset_state case), a NULL upstream gradient means zero, a NULL output is
 * not written.  float32 pointers must be 4-byte aligned, activation-dtype
 * ones aligned to their element.  A window of seq_len 0 copies each state
 * input to its output (and each upstream gradient to the state gradient).
 */
typedef struct {
    const float* ssm_state;      /* in, nullable */
    const void* conv_state;      /* in, nullable */
    float* ssm_state_out;        /* out, nullable */
    void* conv_state_out;        /* out, nullable */
} m3_fwd_state;

typedef struct {
    const void* conv_state;        /* in: the conv_state the forward used */
    const float* d_ssm_state_out;  /* in: dL/d ssm_state_out, nullable */
    const void* d_conv_state_out;  /* in: dL/d conv_state_out, nullable */
    float* d_ssm_state;            /* out: dL/d ssm_state, nullable */
    void* d_conv_state;            /* out: dL/d conv_state, nullable */
} m3_bwd_state;

/*
 * m3scan_fwd starting from a carried state and writing the final one.  The
 * checkpoints it writes start at ssm_state (ckpt[:, 0] = ssm_state), so
 * m3scan_bwd_state needs only the conv_state among the state inputs.
 * state must not be NULL (M3_ERR_NULL).
 */
m3_status m3scan_fwd_state(const m3_dims* dims, m3_dtype act,
                           const void* x, const void* delta_raw, const void* z,
                           const void* Bm, const void* Cm,
                           const float* conv_w, const float* conv_b,
                           const float* dt_bias, const float* a_log, const float* D,
                           void* gated, void* y_dbg, float* ckpt,
                           const m3_fwd_state* state,
                           void* workspace, size_t workspace_bytes,
                           m3_stream_t stream);

/*
 * m3scan_bwd of the loss
 *   L = sum gated * d_gated + sum ssm_state_out * d_ssm_state_out
 *       + sum conv_state_out * d_conv_state_out,
 * from a forward made by m3scan_fwd_state.  Besides m3scan_bwd's outputs
 * it writes d_ssm_state and d_conv_state when they are non-NULL (the
 * latter in the activation dtype).  state must not be NULL (M3_ERR_NULL).
 */
m3_status m3scan_bwd_state(const m3_dims* dims, m3_dtype act,
                           const void* x, const void* delta_raw, const void* z,
                           const void* Bm, const void* Cm,
                           const float* conv_w, const float* conv_b,
                           const float* dt_bias, const float* a_log, const float* D,
                           const float* ckpt, const void* d_gated,
                           void* d_x, void* d_delta_raw, void* dz, void* du_dbg,
                           float* dB, float* dC,
                           float* d_conv_w, float* d_conv_b, float* d_dt_bias,
                           float* d_a_log, float* dD,
                           const m3_bwd_state* state,
                           void* workspace, size_t workspace_bytes,
                           m3_stream_t stream);

/*
 * Two-phase backward, for a layer whose u also feeds the x_proj GEMM.  In
 * the mamba-rs backward (forward_mixed.rs 0.3.1, GpuMambaMixedTrainScratch)
 * the x_proj input gradient is added into d_u before the SiLU and conv1d
 * backward; that gradient needs dB, dC and d_delta_raw (through dt_proj)
 * of this same backward, so the layer core's backward runs in two calls
 * with the caller's GEMMs between them:
 *
 *   1. m3scan_bwd_scan: everything of m3scan_bwd_state up to u -- dz,
 *      d_delta_raw, dB, dC, d_dt_bias, d_a_log, dD, d_ssm_state -- and du
 *      (dL/du through the D skip and the recurrence, activation dtype,
 *      required).  d_x, d_conv_w, d_conv_b and d_conv_state are not
 *      touched.  From the state struct it reads conv_state and
 *      d_ssm_state_out and writes d_ssm_state.
 *   2. the caller forms d_x_dbl = [d_delta_raw W_dt, dB, dC] and
 *      du_extra = d_x_dbl W_xproj (its GEMMs);
 *   3. m3scan_conv_bwd: dc = (du + du_extra) silu'(c) with c recomputed
 *      from x (and conv_state), then d_x, d_conv_w, d_conv_b (written or
 *      added per dims->accumulate_param_grads) and, from the state struct,
 *      d_conv_state (using conv_state and d_conv_state_out).  du_extra may
 *      be NULL (zero).
 *
 * With du_extra = NULL the two calls give the results of m3scan_bwd_state.
 * Both take the same dims (the plan's workspace_bytes covers either call;
 * one workspace may serve both, in stream order).  Pointer rules as in
 * m3scan_bwd; state may be NULL.
 */
m3_status m3scan_bwd_scan(const m3_dims* dims, m3_dtype act,
                          const void* x, const void* delta_raw, const void* z,
                          const void* Bm, const void* Cm,
                          const float* conv_w, const float* conv_b,
                          const float* dt_bias, const float* a_log, const float* D,
                          const float* ckpt, const void* d_gated,
                          void* du, void* d_delta_raw, void* dz,
                          float* dB, float* dC,
                          float* d_dt_bias, float* d_a_log, float* dD,
                          const m3_bwd_state* state,
                          void* workspace, size_t workspace_bytes,
                          m3_stream_t stream);

m3_status m3scan_conv_bwd(const m3_dims* dims, m3_dtype act,
                          const void* x, const float* conv_w, const float* conv_b,
                          const void* du, const void* du_extra,
                          void* d_x, float* d_conv_w, float* d_conv_b,
                          const m3_bwd_state* state,
                          void* workspace, size_t workspace_bytes,
                          m3_stream_t stream);

/*
 * Decode: the forward of a short window -- typically one new token per
 * sequence (dims->seq_len == 1) -- from the carried state, which is
 * updated in place: on return ssm_state holds h after the window's last
 * step and conv_state the conv inputs of the window's last d_conv-1 steps
 * (the m3_fwd_state layouts; the mamba-rs trainer carries the same two
 * states between calls, see m3_fwd_state above).  Same arithmetic as
 * m3scan_fwd_state with both state pointers given and the outputs written
 * over the inputs; no checkpoints are written, no workspace is used and
 * time is not split, so the cost grows with seq_len step by step: use it
 * for decoding and short verification windows, and m3scan_fwd_state for
 * long prompts.
 *
 * dims->d_state may be 16, 32 or 64 here (a_log [d_inner, d_state],
 * Bm/Cm [batch, seq_len, d_state], ssm_state [batch, d_state, d_inner]);
 * dims->chunk, segments and accumulate_param_grads are ignored; d_inner
 * may be any size.  Activation pointers (x, delta_raw, z, Bm, Cm,
 * conv_state, gated, y_dbg) must be aligned to their element, float32
 * pointers to 4 bytes.  seq_len == 0 leaves the state unchanged.
 */
m3_status m3scan_decode(const m3_dims* dims, m3_dtype act,
                        const void* x, const void* delta_raw, const void* z,
                        const void* Bm, const void* Cm,
                        const float* conv_w, const float* conv_b,
                        const float* dt_bias, const float* a_log, const float* D,
                        float* ssm_state, void* conv_state,
                        void* gated, void* y_dbg,
                        m3_stream_t stream);

/*
 * Size in bytes of the scratch array the library keeps on every GPU that
 * loads it, for m3scan_bwd_noalloc.
 */
#define M3SCAN_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * The paper has no counterpart to this entry point: it is an addition for
 * callers that cannot allocate device memory -- for example a plugin or host
 * application that hands the library a fixed device-memory budget and
 * forbids allocation inside its execution path, or a latency-critical caller
 * that cannot accept the implicit device synchronisation of cudaMalloc and
 * cudaFree.
 *
 * Same computation, arguments and results as m3scan_bwd, without the
 * workspace arguments: the scratch is a fixed array of
 * M3SCAN_NOALLOC_SCRATCH_BYTES inside the library.  Neither this call nor
 * anything it calls allocates or frees memory.  The caller still passes
 * (and owns) every input and output.
 *
 * - A shape whose plan needs more scratch than M3SCAN_NOALLOC_SCRATCH_BYTES
 *   (m3scan_plan's workspace_bytes) is rejected with M3_ERR_WORKSPACE before
 *   anything is enqueued; use m3scan_bwd with a workspace for it.
 * - The first call on a device, with that device current, looks up the
 *   array's device address (cudaGetSymbolAddress) and caches it for that
 *   device's CUDA context; make that first call before any stream capture on
 *   that device.  A new context on the device (after cudaDeviceReset) has the
 *   array elsewhere: the first call in it looks the address up again, so it
 *   too must come before any capture.
 * - Every call on a device shares the one array, and the array keeps what
 *   the last call left in it (nothing in it needs to start at zero).  Calls
 *   that overlap on the GPU -- on different streams, or from different host
 *   threads without ordering -- race on it and give wrong results; order
 *   them on one stream or with events.
 */
m3_status m3scan_bwd_noalloc(const m3_dims* dims, m3_dtype act,
                             const void* x, const void* delta_raw, const void* z,
                             const void* Bm, const void* Cm,
                             const float* conv_w, const float* conv_b,
                             const float* dt_bias, const float* a_log, const float* D,
                             const float* ckpt, const void* d_gated,
                             void* d_x, void* d_delta_raw, void* dz, void* du_dbg,
                             float* dB, float* dC,
                             float* d_conv_w, float* d_conv_b, float* d_dt_bias,
                             float* d_a_log, float* dD,
                             m3_stream_t stream);

/* A static, human-readable name for a status code. */
const char* m3scan_status_string(m3_status status);

/* Name of the last CUDA error this thread's calls into the library met
 * (the detail behind M3_ERR_CUDA), e.g. "cudaErrorInvalidValue";
 * "cudaSuccess" if none. */
const char* m3scan_last_cuda_error(void);

/* Library version as major * 10000 + minor * 100 + patch. */
int32_t m3scan_version(void);

/* Device-side status of the calls made with `workspace`: waits for `stream`
 * (the stream those calls were enqueued on), reads the workspace's status
 * block and clears it (on `stream`).  *device_status = M3_OK if every kernel
 * of those calls since the last query ran normally, M3_ERR_TIMEOUT if one of
 * them gave up waiting for a tile copy (its call's outputs are incomplete).
 * Calls on other workspaces and streams are neither seen nor waited for.
 * Calls that were given no workspace (a forward over one time segment with
 * workspace NULL, m3scan_decode) report only to m3scan_device_status.
 * Returns M3_ERR_NULL for a NULL workspace or device_status, M3_ERR_CUDA if
 * waiting or reading fails.  Synchronous for the host. */
m3_status m3scan_get_status(const void* workspace, m3_stream_t stream, m3_status* device_status);

/* Device-side status of the calling thread's current device since the last
 * query, then cleared: *out = 0 if every kernel ran normally; nonzero if a
 * kernel of any call on that device gave up waiting for a tile copy into
 * shared memory (each such wait is bounded to about a second so the GPU
 * cannot hang; that call's outputs are then incomplete).  One word per
 * device, shared by every caller: prefer m3scan_get_status, which reports
 * the calls of one workspace only.  Synchronous: it waits for the device's
 * queued work.  Returns M3_ERR_NULL for a NULL out, M3_ERR_CUDA if reading
 * fails. */
m3_status m3scan_device_status(int32_t* out);

/* Diagnostic of the bounded waits: enqueues one block on `stream` that waits
 * for a tile copy it never issues.  The wait gives up after about a second
 * and the block sets the device status word and, when `workspace` is not
 * NULL, that workspace's status block, so m3scan_device_status and
 * m3scan_get_status then report the failure (and clear it).  Nothing else is
 * touched. */
m3_status m3scan_selftest_wait_timeout(void* workspace, m3_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* M3SCAN_H */
