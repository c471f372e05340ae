/*
 * ssd.h - C ABI of the GB300 (sm_103a) Mamba-2 SSD chunked-scan prefill forward.
 *
 * One call computes, for every batch b and head h, the selective state-space
 * recurrence over the whole sequence:
 *
 *   dt_t = softplus(dt_raw[b,t,h] + dt_bias[h])
 *   h_t  = exp(dt_t * A[h]) * h_{t-1} + dt_t * x[b,t,h,:] (outer) B[b,t,g,:]
 *   y[b,t,h,:] = h_t . C[b,t,g,:] + D[h] * x[b,t,h,:]
 *   final_states[b,h] = h_{L-1},  h_{-1} = init_states[b,h] (zeros if NULL)
 *
 * with g = h / (nheads / ngroups). The recurrence is the one of "Mamba-2
 * state space model compiler optimisation" (bxzpzcl.cn) section 1.1, computed
 * the way "Accelerating Mamba2 with Kernel Fusion" (section on the SSD core
 * operations) splits it: chunk cumsum, BMM, chunk state, state passing and
 * chunk scan, here fused into one persistent kernel launch.
 *
 * Layouts (row-major, last index contiguous, no padding):
 *   x, y            [batch, seqlen, nheads, headdim]        io dtype
 *   dt_raw          [batch, seqlen, nheads]                 io dtype
 *   B, C            [batch, seqlen, ngroups, dstate]        io dtype
 *   dt_bias, A, D   [nheads]                                fp32
 *   init_states,
 *   final_states    [batch, nheads, headdim, dstate]        state dtype
 *   (the state layout is the decode-cache layout of the compiler-optimisation
 *   page, section 2.2)
 *
 * Ownership: the caller owns every buffer, including the workspace; the
 * library allocates no device memory and keeps no per-call global state
 * (ssd_fwd_host keeps two copy streams per device for the process's life).
 * Tensor pointers are device pointers, except the host tensors of
 * ssd_fwd_host.
 *
 * Errors: argument errors are detected on the host, return immediately and
 * launch nothing. The launch itself is asynchronous on `stream`; a device-side
 * failure (a state-passing wait that ran past its time limit) is recorded in
 * the workspace and reported by ssd_fwd_check().
 */
#ifndef MAMBA_SSD_H
#define MAMBA_SSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSD_API __attribute__((visibility("default")))

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1, /* bad shape, NULL or misaligned pointer, bad enum */
    SSD_ERR_UNSUPPORTED = 2, /* valid problem, but no kernel instance for it */
    SSD_ERR_WORKSPACE = 3,   /* workspace NULL, too small or misaligned */
    SSD_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, copy) */
    SSD_ERR_TIMEOUT = 5,     /* device: a state-passing wait ran out of time */
    SSD_ERR_DEVICE = 6       /* device: an internal pipeline wait gave up */
} ssd_status_t;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1, SSD_F16 = 2 } ssd_dtype_t;

/* Which kernel runs the problem. AUTO picks the single-token step kernel for
 * seqlen == 1 (decode: the recurrence advanced by one token; init_states is the
 * cached state and final_states, which may be the same buffer, receives the
 * advanced one; the workspace is only its 256-byte header). STEP also accepts
 * seqlen 0 and is rejected (SSD_ERR_UNSUPPORTED) for longer sequences.
 * Otherwise AUTO picks the tensor-core kernel where it
 * has an instance (bf16/fp16 I/O, headdim 64, dstate 128, chunk_size a
 * multiple of 128) and the fp32 SIMT kernel otherwise. The tensor-core kernel
 * passes states every 128 tokens whatever multiple of 128 is requested: the
 * chunked method reaches the recurrence's result exactly for any chunk size
 * ("Mamba hardware-aware algorithms", structured state space duality), so only
 * the rounding depends on it. */
typedef enum { SSD_KERNEL_AUTO = 0, SSD_KERNEL_SIMT = 1, SSD_KERNEL_TC = 2, SSD_KERNEL_STEP = 3 } ssd_kernel_t;

typedef struct {
    int64_t batch;      /* >= 0                                              */
    int64_t seqlen;     /* >= 0; any length, the last chunk may be ragged    */
    int64_t nheads;     /* >= 1                                              */
    int64_t headdim;    /* P                                                 */
    int64_t dstate;     /* N                                                 */
    int64_t ngroups;    /* G, divides nheads                                 */
    int64_t chunk_size; /* Q: tokens per state-passing step                  */
    int32_t io_dtype;   /* ssd_dtype_t of x, dt_raw, B, C, y                 */
    int32_t state_dtype;/* SSD_F32 or SSD_F16: init/final and passed states  */
    int32_t kernel;     /* ssd_kernel_t                                      */
    int32_t reserved;   /* must be 0                                         */
} ssd_problem_t;

/* Bytes of workspace ssd_fwd needs for `prob` (written to *bytes). The
 * workspace must be zero-filled once before its first use; after that each
 * call leaves it ready for the next one (launches on one stream may reuse it
 * back to back; concurrent launches need separate workspaces). State-passing
 * tags carry the workspace's launch count modulo 2^22 (fp16 states) or 2^32:
 * zero-fill a workspace again before its 2^22-th launch. */
SSD_API ssd_status_t ssd_fwd_workspace_size(const ssd_problem_t *prob, size_t *bytes);

/* Launch the fused SSD prefill forward on `stream` (a cudaStream_t, NULL for
 * the legacy default stream).
 *  x, dt_raw, B, C, y   required, 16-byte aligned
 *  dt_bias, A           required
 *  D                    optional (NULL: no skip term)
 *  init_states          optional (NULL: zero initial state)
 *  final_states         optional (NULL: not written)
 *  workspace            required, 256-byte aligned, >= ssd_fwd_workspace_size
 *                       (for long sequences that size includes two-level
 *                       state passing; a workspace too small for it but large
 *                       enough for one state chain per sequence runs without
 *                       it, with the same results up to rounding)
 * Returns SSD_OK once the launch is queued. */
SSD_API ssd_status_t ssd_fwd(const ssd_problem_t *prob, const void *x, const void *dt_raw,
                             const float *dt_bias, const float *A, const void *B, const void *C,
                             const float *D, const void *init_states, void *y, void *final_states,
                             void *workspace, size_t workspace_bytes, void *stream);

/* Variable-length batch ("Mamba hardware-aware algorithms": sequences of
 * different lengths packed along one token axis, each restarting the
 * recurrence from its own initial state; chunks never cross a sequence
 * boundary).
 *  prob         batch must be 1 and seqlen the total token count T; the other
 *               fields as for ssd_fwd (STEP is not offered here)
 *  cu_seqlens   device int32 [nseq + 1]: sequence s holds tokens
 *               cu_seqlens[s] .. cu_seqlens[s+1] (0 = first, T = last,
 *               non-decreasing; zero-length sequences allowed)
 *  x, dt_raw, B, C, y   [1, T, ...] as for ssd_fwd
 *  init_states, final_states   [nseq, nheads, headdim, dstate] (optional)
 * The offsets are read on the device: malformed ones are reported by
 * ssd_fwd_check as SSD_ERR_INVALID_ARG and nothing is computed. Workspace: as
 * for ssd_fwd, sized by ssd_fwd_varlen_workspace_size for this nseq. */
SSD_API ssd_status_t ssd_fwd_varlen_workspace_size(const ssd_problem_t *prob, int64_t nseq, size_t *bytes);
SSD_API ssd_status_t ssd_fwd_varlen(const ssd_problem_t *prob, const int32_t *cu_seqlens, int64_t nseq,
                                    const void *x, const void *dt_raw, const float *dt_bias, const float *A,
                                    const void *B, const void *C, const float *D, const void *init_states, void *y,
                                    void *final_states, void *workspace, size_t workspace_bytes, void *stream);

/* Activation after the depthwise convolution of ssd_fwd_conv. */
typedef enum { SSD_ACT_NONE = 0, SSD_ACT_SILU = 1 } ssd_activation_t;

/* The SSD forward on the output of a causal depthwise convolution over the
 * tokens ("Accelerating Mamba2 with Kernel Fusion", Mamba-2 core operations
 * item 3; "Mamba-2 compiler optimisation" section 2.2 for the conv cache):
 *   xbc_out[t, ch] = act(conv_bias[ch] + sum_j conv_weight[ch, j] * xbc[t - (k-1) + j, ch])
 * then x, B, C are the column slices [0, H*P), [H*P, H*P + G*N), [H*P + G*N, D)
 * of xbc_out and the rest is ssd_fwd.
 *  prob             as for ssd_fwd (regular batch); D = H*P + 2*G*N channels,
 *                   H*P and G*N multiples of 16 bytes of the I/O dtype
 *  conv_width       k, 1 .. 8;  activation  ssd_activation_t (SiLU: v * sigmoid(v))
 *  xbc              [batch, seqlen, D] raw inputs (I/O dtype), 16-byte aligned
 *  conv_weight      [D, k] fp32 (tap k-1 on the current token); conv_bias [D] or NULL
 *  conv_state       [batch, D, k-1] I/O dtype: the k-1 inputs before each sequence
 *                   (NULL: zeros, a fresh sequence)
 *  conv_state_out   [batch, D, k-1] or NULL: the last k-1 inputs, to continue the
 *                   sequences (by prefill or by seqlen-1 decode steps); may alias
 *                   conv_state
 *  xbc_out          [batch, seqlen, D] buffer for the convolved rows, or NULL:
 *                   - NULL: the convolution is fused into the tensor-core kernel,
 *                     which convolves the raw rows as it loads them (no activation
 *                     buffer, one write and one read of [b, L, D] saved); needs
 *                     that kernel, conv_width 4 and 16-byte aligned conv_weight and
 *                     conv_bias, else SSD_ERR_UNSUPPORTED;
 *                   - a buffer: a convolution kernel writes it (it must not alias
 *                     xbc) and the SSD reads x, B, C from it (any kernel, width)
 *  the rest         as for ssd_fwd (y, init/final states are unchanged in layout)
 * The cache is written by one more small kernel after the others. */
SSD_API ssd_status_t ssd_fwd_conv(const ssd_problem_t *prob, int32_t conv_width, int32_t activation, const void *xbc,
                                  const float *conv_weight, const float *conv_bias, const void *conv_state,
                                  void *conv_state_out, void *xbc_out, const void *dt_raw, const float *dt_bias,
                                  const float *A, const float *D, const void *init_states, void *y, void *final_states,
                                  void *workspace, size_t workspace_bytes, void *stream);

/* Synchronise `stream`, read the device status recorded in `workspace` by the
 * calls queued before, clear it, and return it (SSD_OK when none failed). */
SSD_API ssd_status_t ssd_fwd_check(void *workspace, void *stream);

/* Test hooks, written into the workspace header on `stream`:
 *  timeout_ns     limit of every device-side wait (0 restores the 2 s default)
 *  skip_publish   chunk index whose state publish is skipped, so that the next
 *                 chunk's wait runs out (-1 disables). Host-armed fault
 *                 injection: no memory fault, no trap, the kernel returns.
 *                 -2 instead arms the probe of the bounds-checked debug build
 *                 (compiled with SSD_BOUNDS_CHECK): the tensor-core kernel's
 *                 dt_raw indices are planted one extent past the end, the
 *                 check redirects them to the buffer's start and records the
 *                 violation, and ssd_fwd_check returns SSD_ERR_DEVICE; release
 *                 builds ignore it.
 * In the bounds-checked build every kernel compares its global indices with
 * the buffers' extents; an index outside is never used (the access goes to
 * the buffer's first element) and ssd_fwd_check reports SSD_ERR_DEVICE. */
SSD_API ssd_status_t ssd_debug_set(void *workspace, uint64_t timeout_ns, int64_t skip_publish, void *stream);

/* Process-wide test hooks that force a kernel's launch configuration, for
 * tests that compare each form with the default one and with the oracle. Every
 * argument is -1 for the library's own choice (the state at load time); any
 * other value must be valid for its field, else SSD_ERR_INVALID_ARG and
 * nothing changes:
 *  tc_heads_per_unit  tensor-core kernel: heads per work unit, 1 .. 8 (used only
 *                     when it divides nheads / ngroups)
 *  tc_late_ticket     tensor-core kernel: 0 = every next work ticket taken one
 *                     unit ahead, 1 = only when the unit before nears its end
 *  simt_two_pass      fp32 SIMT kernel: 0 = one pass per unit, 1 = the chunk
 *                     state before the entering state is awaited, then y
 *  conv_tma           depthwise convolution: 0 = the 16-byte-copy pipeline
 *                     (the form for rows that are not 16-byte multiples),
 *                     1 = the TMA-fed one where the rows allow it
 *  tc_segment_chunks  tensor-core kernel, regular batches: 0 = one state
 *                     chain per sequence, n >= 1 = two-level state passing
 *                     with segments of n chunks (of 128 tokens); used only
 *                     when it cuts a sequence into two or more segments.
 *                     It changes the workspace size: set it before
 *                     ssd_fwd_workspace_size.
 *  tc_head_flags      tensor-core kernel: 0 = states passed the default way
 *                     (fp32: every row behind its own release flag, stored by
 *                     its chain thread; fp16: tagged words), 1 = one release
 *                     flag per head, stored by the C.S warp once all rows are
 *                     written (fp16 states then as plain halves). The library
 *                     chooses 1 only for fp32 states.
 * The values are read by later calls on any host thread (not by calls already
 * queued). The library reads no environment variable. */
SSD_API ssd_status_t ssd_debug_knobs(int32_t tc_heads_per_unit, int32_t tc_late_ticket, int32_t simt_two_pass,
                                     int32_t conv_tma, int32_t tc_segment_chunks, int32_t tc_head_flags);

/* ssd_fwd without a workspace argument, for callers that cannot allocate
 * device memory (no counterpart on the pages; it is a library convenience).
 * Some callers hand a kernel only its inputs and outputs: host applications or
 * plugin frameworks that own every byte of device memory, or latency-critical
 * loops that cannot afford a cudaMalloc, which may synchronise the device.
 * This entry point takes its scratch from a 16 MiB array compiled into the
 * library (every GPU that loads the library holds it until the process exits)
 * and allocates nothing.
 *  - Problems whose ssd_fwd_workspace_size() exceeds 16 MiB are rejected with
 *    SSD_ERR_WORKSPACE (at headdim 64, d_state 128 this is roughly 250 (batch x
 *    head) chains with fp32 states, 500 with fp16 states).
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any
 *    stream capture.
 *  - All calls share the one array. Each call zero-fills the part it uses on
 *    `stream` before launching, so earlier contents do not matter, but calls
 *    that overlap on the GPU (unordered streams or host threads) race on it.
 *  - A device-side wait that gives up is not reported (there is no workspace
 *    to pass to ssd_fwd_check); it needs a device malfunction to happen.
 * Arguments, layouts and the other errors are those of ssd_fwd. */
SSD_API ssd_status_t ssd_fwd_static_scratch(const ssd_problem_t *prob, const void *x, const void *dt_raw,
                                            const float *dt_bias, const float *A, const void *B, const void *C,
                                            const float *D, const void *init_states, void *y, void *final_states,
                                            void *stream);

/* The forward pass on host-resident tensors, streamed through the GPU in
 * pieces so that the host<->device copies overlap the computation (no
 * counterpart on the pages; a library convenience for batches that live in
 * host memory).
 *  pieces       number of pieces (0: the library's choice, about 256 MiB of
 *               copies per piece and from 8 to 32 pieces; at most one per
 *               chunk). The batch is cut along its tokens at multiples of
 *               chunk_size, each piece holding the same token range of every
 *               sequence; the states leaving one piece enter the next (the
 *               same chunks, in the same order and precision, as one call).
 *               From 8 pieces on, the first and the last piece are a quarter
 *               of an even piece's size (a shorter pipeline fill and drain)
 *               and the others share the rest evenly.
 *  x, dt_raw, B, C, init_states (optional): host inputs, and y, final_states
 *               (optional): host outputs, in the layouts of ssd_fwd. Page-locked
 *               memory lets the copies overlap; pageable memory also works,
 *               without the overlap.
 *  dt_bias, A, D   device pointers, as for ssd_fwd.
 *  scratch      device memory of ssd_fwd_host_scratch_size(prob, pieces)
 *               bytes, 256-byte aligned, zero-filled once before its first use;
 *               it begins with the workspace that ssd_fwd_check reads. Calls
 *               on one stream may reuse it back to back; calls that may overlap
 *               (other streams, other host threads) need separate scratch.
 *               Such calls share the device's two copy streams, so their
 *               copies queue behind each other.
 * The computation runs on `stream`; the copies run on two streams the library
 * creates once per device and keeps, ordered after the work queued on `stream`
 * before the call, and `stream` waits for all of them before any later work:
 * once `stream` is synchronised the outputs are in host memory. The host
 * buffers must stay valid until then. Problem checks and errors: those of
 * ssd_fwd. */
SSD_API ssd_status_t ssd_fwd_host_scratch_size(const ssd_problem_t *prob, int32_t pieces, size_t *bytes);
SSD_API ssd_status_t ssd_fwd_host(const ssd_problem_t *prob, int32_t pieces, const void *x, const void *dt_raw,
                                  const float *dt_bias, const float *A, const void *B, const void *C, const float *D,
                                  const void *init_states, void *y, void *final_states, void *scratch,
                                  size_t scratch_bytes, void *stream);

/* Which kernel ssd_fwd would run for `prob` (SSD_KERNEL_SIMT or _TC), or a
 * negative ssd_status_t if the problem is rejected. */
SSD_API int ssd_fwd_kernel_for(const ssd_problem_t *prob);

/* What ssd_fwd plans for `prob` (a regular batch; host only, no CUDA call but
 * the SM count): the kernel, the kernel launches one call makes, and the
 * state passing. With two-level state passing (long sequences on the
 * tensor-core path) every sequence is cut into `segments` segments of
 * `segment_chunks` chunks of 128 tokens ("Accelerating Mamba2 with Kernel
 * Fusion", state passing step, regrouped): a block kernel and a combine kernel
 * compute the states entering the segments before the fused kernel, whose
 * chunk-to-chunk state chain then restarts at every segment. segments == 1:
 * one chain per sequence. head_flags == 1: the tensor-core kernel publishes
 * each head's passed state behind one release flag, stored by the warp that
 * issues the head's C.S once every state row is written (fp16 states then as
 * plain halves); 0: fp32 rows each behind their own flag, fp16 states in tagged
 * words. The struct grew head_flags in ABI 1.1 (ssd_version() >= 10100). */
typedef struct {
    int32_t kernel;          /* ssd_kernel_t (SSD_KERNEL_SIMT, _TC or _STEP)  */
    int32_t launches;        /* kernel launches per ssd_fwd call              */
    int64_t segments;        /* per sequence (1: no two-level state passing)  */
    int64_t segment_chunks;  /* chunks per segment                             */
    size_t workspace_bytes;  /* = ssd_fwd_workspace_size                       */
    int32_t head_flags;      /* tensor-core kernel: one release flag per head */
    int32_t reserved;        /* 0                                              */
} ssd_plan_t;
SSD_API ssd_status_t ssd_fwd_plan(const ssd_problem_t *prob, ssd_plan_t *plan);

/* Static text for a status code. */
SSD_API const char *ssd_status_string(ssd_status_t status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
SSD_API int ssd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA_SSD_H */
