/*
 * ssd_scan.h -- C ABI of libssdscan.so: the Mamba-2 state-space-duality (SSD)
 * selective scan, its one-token decode step, and the Mamba-1 diagonal
 * selective scan, as hand-written CUDA kernels for NVIDIA GB300 (sm_103a).
 *
 * What is computed (per batch b and head h, group g = h / (nheads/ngroups)):
 *
 *     h_t[p,n] = exp(dt_t * A_h) * h_{t-1}[p,n] + dt_t * x_t[p] * B_t[n]
 *     y_t[p]   = sum_n C_t[n] * h_t[p,n] + D_h * x_t[p]
 *
 * the generic selective update h_t = A_t h_{t-1} + B_t x_t, y_t = C_t h_t +
 * D_t x_t of "COREY: Entropy-Guided Runtime Chunk Scheduling for Selective
 * Scan Kernels" (section 3.1) with the scalar per-head decay of the SSD layer
 * ("Compiler-First State Space Duality and Portable O(1) Autoregressive
 * Caching for Inference", abstract: diagonal per-head dynamics, fixed-size
 * chunking). y uses the updated state h_t. dt is used as given: no softplus
 * and no bias are applied inside.
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers of the current CUDA device,
 *    dense, row-major with the innermost dimension last, and 16-byte aligned.
 *    The caller owns every buffer (inputs, outputs, workspace); the library
 *    allocates nothing and never frees.
 *  - Calls are asynchronous on `stream` (0 = legacy default stream): they
 *    validate their arguments on the host, enqueue kernels and return. There
 *    is no host synchronisation and no exception crosses the ABI.
 *  - The tensor-core prefill, decode, decode-layer and Mamba-1 kernels are
 *    launched as programmatic dependents of the kernel before them in the
 *    stream (CUDA programmatic dependent launch): they may be placed on the
 *    GPU while it drains, but each waits for its completion before touching
 *    memory, so stream order means what it means for ordinary launches (a
 *    kernel of another library before a call has completed before the call
 *    reads its inputs).
 *  - Validation happens before any CUDA call: an invalid argument returns
 *    SSD_ERR_INVALID_ARG (or SSD_ERR_UNSUPPORTED for a valid but unbuilt
 *    shape) and enqueues nothing. SSD_ERR_CUDA reports a failed launch.
 *    ssd_last_error() then describes the failure (thread-local text).
 *  - Results are deterministic: no atomics in any reduction, so runs are
 *    bitwise reproducible and a batch of sequences gives bitwise the same
 *    rows as each sequence alone.
 *  - io_dtype selects the element type of x, dt, B, C and y (float32 or
 *    bfloat16). A, D and every state are float32 in all cases; decays,
 *    cumulative sums and exponentials are always evaluated in float32
 *    ("Compiler-First State Space Duality ...", Table 8: decay kept in
 *    float32).
 */
#ifndef SSD_SCAN_H
#define SSD_SCAN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad alignment, short workspace */
    SSD_ERR_UNSUPPORTED = 2, /* valid arguments, shape outside what the kernels handle */
    SSD_ERR_CUDA = 3,        /* a CUDA launch or runtime call failed */
    SSD_ERR_TIMEOUT = 4,     /* a bounded in-kernel wait gave up (see ssd_workspace_status) */
    SSD_ERR_BOUNDS = 5       /* debug builds: a kernel's bounds check failed (see ssd_debug_bounds_status) */
} ssd_status;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

/* Option bits for ssd_dims.flags. */
#define SSD_FLAG_SIMT 1   /* bf16 prefill: use the CUDA-core kernels instead of the tensor-core ones */
#define SSD_FLAG_FUSED 2  /* bf16 prefill: the single-pass tensor-core kernel (chunk 128 only; else
                             SSD_ERR_UNSUPPORTED) whatever the shape */
#define SSD_FLAG_STAGED 4 /* bf16 prefill: the three-kernel tensor-core path whatever the shape */

typedef struct {
    int64_t batch;    /* B >= 0                                   */
    int64_t seqlen;   /* L >= 0 (prefill); ignored by the decode step */
    int64_t nheads;   /* H >= 1                                   */
    int64_t headdim;  /* P >= 1                                   */
    int64_t dstate;   /* N >= 1                                   */
    int64_t ngroups;  /* G >= 1, H % G == 0; head h reads B/C group h/(H/G) */
    int32_t io_dtype; /* ssd_dtype of x, dt, B, C, y              */
    int32_t flags;    /* SSD_FLAG_* bits, 0 by default            */
} ssd_dims;

/*
 * Bytes of device workspace ssd_scan_chunked needs for these sizes and chunk
 * size; 0 if the arguments are invalid. The workspace holds the per-chunk
 * states [B, ceil(L/Q), H, P, N] (float32, plus a bfloat16 copy on the
 * tensor-core path), the per-chunk decay totals and a status word.
 */
size_t ssd_workspace_size(const ssd_dims *dims, int chunk_size);

/*
 * The chunk size (64, 128 or 256) a static policy picks for these sizes: the
 * fastest measured on GB300 for the nearest shape of a sweep over batch 1-8,
 * length 512-8192 and 24-80 heads (bf16, P = 64, N = 128), after the pages'
 * static-oracle / table policies ("COREY ...", section 5.2). Shapes outside
 * the tensor-core path get 128. Host-only, no CUDA call; 0 if the dims are
 * invalid.
 */
int ssd_best_chunk(const ssd_dims *dims);

/* Kernel paths of ssd_scan_chunked (return values of ssd_scan_path). */
#define SSD_PATH_SIMT 0   /* CUDA cores, float32: chunk state, state passing, chunk scan */
#define SSD_PATH_STAGED 1 /* tensor cores: the same three steps as three kernels */
#define SSD_PATH_FUSED 2  /* tensor cores: one persistent kernel (and a kernel that clears its flags) */

/*
 * The kernel path ssd_scan_chunked takes for these sizes, chunk size and
 * dims->flags on the current device (SSD_PATH_*), or -1 if the arguments are
 * invalid or SSD_FLAG_FUSED is set for sizes the single pass does not take.
 * Without flags the single pass is taken for bf16, headdim 64, dstate 128,
 * chunk 128 and an even number of heads per group when batch * nheads / 2 is
 * at least 0.6 times the SM count: it runs at least one whole chain (b, head
 * pair) of chunks per SM, and a chain split between two SMs hands its
 * carried state over once.
 * Host-only: no launch, no synchronisation.
 */
int ssd_scan_path(const ssd_dims *dims, int chunk_size);

/*
 * Chunked SSD prefill over a whole sequence (the SSD scan run "chunk by chunk,
 * each chunk continuing from the previous chunk's state", "Recurrence Scan",
 * first section; fixed-size chunking, "Compiler-First State Space Duality
 * ...", abstract).
 *
 *   x          [B, L, H, P]  io_dtype
 *   dt         [B, L, H]     io_dtype, used as given (already positive)
 *   A          [H]           float32, the per-head decay rate (normally < 0)
 *   B, C       [B, L, G, N]  io_dtype
 *   D          [H]           float32, may be NULL (no skip term)
 *   init_state [B, H, P, N]  float32, may be NULL (zero initial state)
 *   chunk_size Q in {64, 128, 256}; L need not be a multiple of Q. The result
 *              does not depend on Q beyond float32 rounding.
 *   y          [B, L, H, P]  io_dtype, written
 *   final_state[B, H, P, N]  float32, the state after token L-1 (init_state,
 *              or zero, when L = 0); may be NULL (not written). It may be the
 *              same buffer as init_state (the state is then updated in place).
 *   workspace  device buffer of at least ssd_workspace_size(dims, Q) bytes,
 *              256-byte aligned; contents on entry are ignored. Two calls in
 *              flight at once need two workspaces.
 *
 * bf16 inputs with P = 64 and N = 128 run on the tensor cores (tcgen05 MMAs
 * with float32 accumulation in tensor memory, operands staged by TMA) unless
 * dims->flags has SSD_FLAG_SIMT; every other case, and all float32 inputs,
 * run on the CUDA cores in float32 (limit: nheads * ceil(P/64) * ceil(N/64)
 * <= 65535).
 */
ssd_status ssd_scan_chunked(const ssd_dims *dims, const void *x, const void *dt, const float *A,
                            const void *B, const void *C, const float *D, const float *init_state,
                            int chunk_size, void *y, float *final_state, void *workspace,
                            size_t workspace_bytes, cudaStream_t stream);

/*
 * ssd_scan_chunked without a caller-provided workspace, for callers that
 * cannot allocate device memory where they run the scan: plug-ins whose host
 * framework owns all device memory and forbids allocating inside its enqueue
 * call, and latency-critical loops that cannot take the device-wide
 * synchronisation a cudaMalloc/cudaFree pair brings. The pages have no
 * counterpart of this call; it exists for such callers only.
 *
 * Same arguments and results as ssd_scan_chunked, minus the workspace: the
 * per-chunk states live in a 64 MiB scratch array compiled into the library
 * (a file-scope __device__ array that every GPU loading it holds until the
 * process exits). Sizes whose ssd_workspace_size() exceeds 64 MiB return
 * SSD_ERR_UNSUPPORTED and launch nothing. The first call on each device looks
 * up the scratch address with that device current; make it before any stream
 * capture begins. Nothing here allocates. All calls on a device share the
 * scratch: calls whose kernels may overlap on the GPU (e.g. on two unordered
 * streams) race on it and must be serialised by the caller. A bounded in-kernel
 * wait that gives up records SSD_ERR_TIMEOUT in the scratch's status word,
 * which ssd_scan_chunked_noalloc_status reads.
 */
ssd_status ssd_scan_chunked_noalloc(const ssd_dims *dims, const void *x, const void *dt, const float *A,
                                    const void *B, const void *C, const float *D,
                                    const float *init_state, int chunk_size, void *y,
                                    float *final_state, cudaStream_t stream);

/*
 * Status of the latest ssd_scan_chunked_noalloc call on the current device:
 * waits for `stream` (host synchronisation, like ssd_workspace_status), then
 * reads the status word at the start of the built-in scratch. Returns SSD_OK,
 * or SSD_ERR_TIMEOUT when a bounded wait of that call gave up (its y and
 * final_state are then not valid). When scratch_addr is not NULL it receives
 * the scratch's device address on the current device (for example to run
 * ssd_selftest_bounded_wait on its status word). Allocates nothing; like the
 * scan, its first use on a device looks the scratch address up.
 */
ssd_status ssd_scan_chunked_noalloc_status(cudaStream_t stream, void **scratch_addr);

/*
 * One decode token for a batch of sequences, state updated in place (the
 * O(1) cached decode of "Compiler-First State Space Duality ...", Figure 1;
 * the state is laid out [B, H, P, N] with N contiguous, so a warp streams one
 * (b, h, p) row with coalesced 128-bit accesses -- the opposite of the
 * one-thread-per-channel mapping whose uncoalesced state reads the
 * "Mamba-2 SSD fused layer via VGpuWarp" log diagnoses).
 *
 *   state [B, H, P, N] float32, read and overwritten with the new state
 *   x     [B, H, P]    io_dtype      dt [B, H] io_dtype
 *   A     [H]          float32       B, C [B, G, N] io_dtype
 *   D     [H]          float32, may be NULL
 *   y     [B, H, P]    io_dtype, written
 * dims->seqlen is ignored. Equivalent to ssd_scan_chunked with L = 1 and
 * init_state = final_state = state.
 */
ssd_status ssd_decode_step(const ssd_dims *dims, float *state, const void *x, const void *dt,
                           const float *A, const void *B, const void *C, const float *D, void *y,
                           cudaStream_t stream);

/*
 * Mamba-1 selective scan with a per-channel diagonal A (the selective_scan_fn
 * workload of "COREY ...", section 5.1 and appendix A.9; d_state 16):
 *
 *     h_t[n] = exp(dt_t[d] * A[d,n]) * h_{t-1}[n] + dt_t[d] * x_t[d] * B_t[n]
 *     y_t[d] = sum_n C_t[n] * h_t[n] + D[d] * x_t[d]
 *
 *   x, dt      [batch, seqlen, dim]  io_dtype (dt used as given)
 *   A          [dim, dstate]         float32
 *   B, C       [batch, seqlen, dstate] io_dtype
 *   D          [dim]                 float32, may be NULL
 *   init_state [batch, dim, dstate]  float32, may be NULL
 *   chunk_size tokens per pass, a multiple of 32, >= 32: the kernel walks the
 *              sequence chunk by chunk carrying the state exactly in
 *              registers, so the output is bitwise independent of it
 *              (runtime chunk routing preserves outputs bitwise, "COREY ...",
 *              section 5.4).
 *   y          [batch, seqlen, dim]  io_dtype, written
 *   final_state[batch, dim, dstate]  float32, may be NULL
 * Limits: 1 <= dstate <= 64.
 */
ssd_status selective_scan_diag(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                               int32_t io_dtype, const void *x, const void *dt, const float *A,
                               const void *B, const void *C, const float *D,
                               const float *init_state, int chunk_size, void *y,
                               float *final_state, cudaStream_t stream);

/*
 * The same scan with selective_scan_fn's options (the kernel-level timing of
 * "COREY ...", section 7, runs selective_scan_fn with delta_softplus set):
 *
 *     dt'_t[d] = dt_t[d] + delta_bias[d]           (delta_bias may be NULL: 0)
 *     dt''_t[d] = softplus(dt'_t[d]) = log(1 + exp(dt'_t[d]))  if delta_softplus
 *                 dt'_t[d]                                      otherwise
 *     the recurrence above with dt'' in place of dt
 *     out_t[d] = y_t[d] * z_t[d] / (1 + exp(-z_t[d]))   (z may be NULL: no gate)
 *
 *   z          [batch, seqlen, dim]  io_dtype, may be NULL
 *   delta_bias [dim]                 float32, may be NULL
 *   delta_softplus 0 or 1 (else SSD_ERR_INVALID_ARG)
 * The gate multiplies the finished output, D term included; the carried
 * state is not gated. The kernel evaluates softplus(v) as v for v > 20, where
 * the two agree in float32.
 *
 *   workspace  device scratch of selective_scan_diag_workspace_size() bytes,
 *              256-byte aligned, owned by the caller, or NULL. When the batch
 *              and dim leave most of the GPU idle (one pass per sequence gives
 *              fewer than ~39k threads) and a workspace is given, the sequence
 *              is cut into time segments of a multiple of 32 tokens, scanned in
 *              parallel from a zero state, chained by one segment pass
 *              (decay over a segment = exp(A * sum of its steps)), then
 *              rescanned from their entering states to form y. The result
 *              equals the one-pass scan up to float32 rounding. The split
 *              depends on the shape only, so the output stays bitwise
 *              independent of chunk_size. A workspace smaller than the size
 *              query (or not 256-byte aligned) is SSD_ERR_INVALID_ARG; NULL
 *              runs one pass per sequence.
 * Other arguments, limits, ownership and errors as for selective_scan_diag,
 * which is this call with z = delta_bias = workspace = NULL and
 * delta_softplus = 0.
 */
ssd_status selective_scan_diag_ex(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                                  int32_t io_dtype, const void *x, const void *dt, const float *A,
                                  const void *B, const void *C, const float *D, const void *z,
                                  const float *delta_bias, int32_t delta_softplus,
                                  const float *init_state, int chunk_size, void *y,
                                  float *final_state, void *workspace, size_t ws_bytes,
                                  cudaStream_t stream);

/*
 * Workspace bytes selective_scan_diag_ex needs for its time-segmented scan of
 * this shape; 0 when the shape runs one pass per sequence (or the arguments
 * are invalid). Host-only, no CUDA call.
 */
size_t selective_scan_diag_workspace_size(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                                          int32_t io_dtype);

/*
 * Status word of a workspace: waits for `stream`, then reports SSD_OK or the
 * first error a kernel recorded there during the last ssd_scan_chunked call
 * that used it (SSD_ERR_TIMEOUT when a bounded wait gave up). Every bounded
 * wait in the kernels records its failure here and returns instead of
 * spinning forever.
 */
ssd_status ssd_workspace_status(const void *workspace, cudaStream_t stream);

/*
 * Self-test of the bounded-wait machinery: launches one kernel that waits on a
 * shared-memory barrier nothing will ever complete, with a budget of
 * `spin_limit` polls, records SSD_ERR_TIMEOUT in the workspace status word
 * and exits. The caller then reads ssd_workspace_status(workspace, stream),
 * which must report SSD_ERR_TIMEOUT while the context stays usable.
 * workspace: at least 256 bytes. spin_limit: 1 .. 1<<20.
 */
ssd_status ssd_selftest_bounded_wait(void *workspace, int spin_limit, cudaStream_t stream);

/*
 * Per-stage timing of the next ssd_scan_chunked call made on this thread.
 * `events` points to 4 CUDA events created by the caller (timing enabled, on
 * the device of the call); that call records them on its stream before its
 * first kernel and after each stage -- chunk state, state passing, chunk scan
 * -- so that cudaEventElapsedTime(e[i], e[i+1]) is the device time of stage i.
 * Inside stream capture they are recorded as external event nodes. The request
 * is consumed by that one call; the stages are then launched without
 * programmatic overlap. count must be 4; events = NULL cancels a request.
 */
ssd_status ssd_record_stage_events(cudaEvent_t *events, int count);

/*
 * Bounds checks of a debug build. A library compiled with -DSSD_DEBUG_BOUNDS
 * (python -m mamba_ssd_selective_gb300.build --debug-bounds, which writes
 * lib/libssdscan_dbg.so) checks the raw global-memory accesses of its decode,
 * Mamba-1, state-pass and single-pass prefill kernels against the extents of
 * their buffers: a failing access is skipped (never a trap) and the first
 * failure is recorded. This call waits for the device, then returns SSD_OK if
 * no check has failed, or SSD_ERR_BOUNDS with *site (a site number of
 * csrc/debug_bounds.cuh) and *index (the first element of the failing
 * access) filled in; clear != 0 resets the record. site and index may be
 * NULL. A release build returns SSD_ERR_UNSUPPORTED.
 */
ssd_status ssd_debug_bounds_status(int *site, int64_t *index, int clear);

/*
 * Backward of ssd_scan_chunked (the training step's backward; "Compiler-First
 * State Space Duality ...", appendix Table 13): the gradients of
 *     L = <dy, y> + <dfinal_state, final_state>
 * with respect to every input, for the recurrence of ssd_scan_chunked. It
 * recomputes the forward entering states chunk by chunk, runs the adjoint
 * chunk states and a reverse state pass, then one CTA per (b, chunk, head)
 * forms every gradient of that chunk. bf16 inputs with headdim 64 and dstate
 * 128 on a GB300-class device take chunks of 128 tokens with every product
 * on the tensor cores (bf16 operands, float32 accumulation and elementwise
 * steps); everything else, or flags containing SSD_FLAG_SIMT, takes chunks of
 * 64 tokens in float32 on the CUDA cores. Deterministic (fixed-order sums,
 * no atomics).
 *   dims      as for ssd_scan_chunked (seqlen L, io_dtype of x, dt, B, C, dy;
 *             of the flags only SSD_FLAG_SIMT is read). Limits: headdim <= 64,
 *             dstate <= 128 (else SSD_ERR_UNSUPPORTED).
 *   x, dt, A, B, C, D, init_state   the forward's inputs (D, init_state may be NULL)
 *   dy          [B, L, H, P]  io_dtype: cotangent of y
 *   dfinal_state[B, H, P, N]  float32, may be NULL (0)
 *   dx [B,L,H,P], ddt [B,L,H], dA [H], dB, dC [B,L,G,N]   float32, written
 *   dD [H], dinit_state [B,H,P,N]                         float32, may be NULL
 *   workspace   ssd_scan_chunked_bwd_workspace_size(dims) bytes, 256-byte aligned
 */
size_t ssd_scan_chunked_bwd_workspace_size(const ssd_dims *dims);
ssd_status ssd_scan_chunked_bwd(const ssd_dims *dims, const void *x, const void *dt, const float *A, const void *B,
                                const void *C, const float *D, const float *init_state, const void *dy,
                                const float *dfinal_state, float *dx, float *ddt, float *dA, float *dB, float *dC,
                                float *dD, float *dinit_state, void *workspace, size_t ws_bytes,
                                cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Decode-layer neighbours of ssd_decode_step: the pieces of a Mamba-2 decode
 * layer body that must run on the device so that a token's layer stays
 * resident and can be replayed as one CUDA graph ("Mamba-2 SSD fused layer via
 * VGpuWarp — design sketch", section "What has to become a device op",
 * items 1 and 2, and section "The concrete mechanism").
 * ------------------------------------------------------------------------- */

typedef enum { SSD_ACT_NONE = 0, SSD_ACT_SILU = 1 } ssd_activation;

/*
 * One step of a causal depthwise convolution with a rolling window, per
 * (b, c): the window holds the last `width` inputs, oldest first; x shifts in
 * (the oldest value drops out), then
 *     out[b,c] = act(sum_k weight[c,k] * window[b,c,k] + bias[c]).
 *   x          [batch, channels]          io_dtype
 *   conv_state [batch, channels, width]   float32, updated in place
 *   weight     [channels, width]          float32
 *   bias       [channels]                 float32, may be NULL (0)
 *   activation SSD_ACT_NONE or SSD_ACT_SILU (v * sigmoid(v))
 *   out        [batch, channels]          io_dtype, written (may not alias x)
 * Limits: 1 <= width <= 8. Pointers 16-byte aligned. Errors as for the scans.
 */
ssd_status ssd_conv1d_step(int64_t batch, int64_t channels, int64_t width, int32_t io_dtype, const void *x,
                           float *conv_state, const float *weight, const float *bias, int32_t activation,
                           void *out, cudaStream_t stream);

/*
 * Gated RMS norm over groups of `group` consecutive channels:
 *     g = y * silu(z)                 (z NULL: g = y)
 *     out = g / sqrt(mean over the group of g^2 + eps) * weight
 *   y, z, out  [batch, dim]  io_dtype (out may alias y)
 *   weight     [dim]         float32
 * Limits: dim % group == 0, eps >= 0. One CTA per (b, group).
 */
ssd_status ssd_gated_rmsnorm(int64_t batch, int64_t dim, int64_t group, int32_t io_dtype, const void *y,
                             const void *z, const float *weight, float eps, void *out, cudaStream_t stream);

/*
 * One token of the decode layer body, in three kernels on `stream`:
 *     xBC' = silu(causal conv step of xBC)          (conv_state updated)
 *     x, B, C = the H*P, G*N and G*N channels of xBC'
 *     y = ssd_decode_step(x, dt, B, C)              (ssm_state updated)
 *     out = gated RMS norm of y with gate z over groups of norm_group
 *   dims       batch, nheads H, headdim P, dstate N, ngroups G, io_dtype
 *              (seqlen and flags ignored); conv channels Cc = H*P + 2*G*N
 *   xBC        [batch, Cc] io_dtype        conv_state [batch, Cc, conv_width] f32
 *   conv_weight [Cc, conv_width] f32       conv_bias [Cc] f32, may be NULL
 *   dt         [batch, H] io_dtype (used as given)   A [H] f32   D [H] f32, may be NULL
 *   ssm_state  [batch, H, P, N] f32        z [batch, H*P] io_dtype, may be NULL
 *   norm_weight [H*P] f32                  out [batch, H*P] io_dtype
 *   workspace  ssd_decode_layer_workspace_size(dims) bytes, 256-byte aligned:
 *              holds x, B, C and y of the step in io_dtype.
 */
size_t ssd_decode_layer_workspace_size(const ssd_dims *dims);
ssd_status ssd_decode_layer_step(const ssd_dims *dims, int64_t conv_width, const void *xBC, float *conv_state,
                                 const float *conv_weight, const float *conv_bias, const void *dt, const float *A,
                                 const float *D, float *ssm_state, const void *z, const float *norm_weight,
                                 int64_t norm_group, float eps, void *out, void *workspace, size_t ws_bytes,
                                 cudaStream_t stream);

/*
 * A decode loop of `steps` layer steps captured once as a CUDA graph and
 * replayed with one launch. Step s reads xBC + s*batch*Cc, dt + s*batch*H and
 * z + s*batch*H*P (elements of io_dtype) and writes out + s*batch*H*P; the
 * states carry from step to step. Arguments as for ssd_decode_layer_step; all
 * buffers must stay valid while the graph exists. Creation allocates the
 * graph (host and driver resources) and captures on a private stream; launch
 * allocates nothing; destroy releases the graph.
 */
typedef struct ssd_decode_graph ssd_decode_graph;
ssd_status ssd_decode_graph_create(const ssd_dims *dims, int64_t conv_width, int32_t steps, const void *xBC,
                                   float *conv_state, const float *conv_weight, const float *conv_bias,
                                   const void *dt, const float *A, const float *D, float *ssm_state, const void *z,
                                   const float *norm_weight, int64_t norm_group, float eps, void *out,
                                   void *workspace, size_t ws_bytes, ssd_decode_graph **graph);
ssd_status ssd_decode_graph_launch(ssd_decode_graph *graph, cudaStream_t stream);
ssd_status ssd_decode_graph_destroy(ssd_decode_graph *graph);

/* Thread-local description of the last error returned on this thread. */
const char *ssd_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* SSD_SCAN_H */
