// Internal host-side launchers shared between the C-ABI layer (ssd_api.cu)
// and the kernel translation units. Not part of the public ABI.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace ssd {

// Kernel attributes (maximum dynamic shared memory, carveout) are kept per
// device, so a launcher that sets them once remembers it per device ordinal:
// one bit per device, for ordinals below 64 (others are set on every call).
class DeviceOnce {
  public:
    // true when the current device still needs the attribute calls; *dev gets
    // the ordinal to pass to done()
    bool pending(int *dev, cudaError_t *err) {
        *err = cudaGetDevice(dev);
        if (*err != cudaSuccess) return false;
        return *dev < 0 || *dev >= 64 || !((bits_.load(std::memory_order_acquire) >> *dev) & 1ull);
    }
    void done(int dev) {
        if (dev >= 0 && dev < 64) bits_.fetch_or(1ull << dev, std::memory_order_release);
    }

  private:
    std::atomic<unsigned long long> bits_{0};
};

// Streaming multiprocessors of the current device, queried once per device
// ordinal (below 64). Returns `fallback` when no device can be queried (host
// code on a machine without a GPU, e.g. a workspace-size query).
int sm_count(int fallback = 1);

enum IoType { IO_F32 = 0, IO_BF16 = 1 };

// Sizes and pointers of one chunked SSD prefill call (layouts as in ssd_scan.h).
struct ChunkedArgs {
    int64_t B, L, H, P, N, G;
    int Q;       // chunk size
    int64_t nc;  // number of chunks, ceil(L / Q)
    int io;      // IoType
    const void *x, *dt, *Bm, *Cm;
    const float *A, *D, *init_state;
    void *y;
    float *final_state;
    // workspace carve
    int *status;             // device status word
    float *states;           // [B, nc, H, P, N] float32: chunk states, then entering states
    uint16_t *states_bf16;   // [B, nc, H, P, N] bfloat16 entering states (tensor-core path)
    float *chunk_sum;        // [B, H, nc] float32: decay over each chunk, exp(sum of dt*A)
    // optional stage timing: events[0..3] recorded before stage 1 and after
    // stages 1, 2, 3 (all NULL when not requested)
    cudaEvent_t stage_ev[4];
};

// Records stage event i of `a` on `stream` if requested (external node when
// the stream is being captured).
cudaError_t mark_stage(const ChunkedArgs &a, int i, cudaStream_t stream);

// Workspace layout (byte offsets from the workspace base).
struct WorkspaceLayout {
    size_t status, states, states_bf16, chunk_sum, total;
};
WorkspaceLayout workspace_layout(int64_t B, int64_t L, int64_t H, int64_t P, int64_t N, int Q);

cudaError_t launch_decode(int io, int64_t B, int64_t H, int64_t P, int64_t N, int64_t G, float *state,
                          const void *x, const void *dt, const float *A, const void *Bm, const void *Cm,
                          const float *D, void *y, cudaStream_t stream);

// CUDA-core (float32 arithmetic) chunked path: chunk-state, state passing, chunk scan.
cudaError_t launch_chunked_simt(const ChunkedArgs &a, cudaStream_t stream);

// Tensor-core path (bf16 operands, tcgen05 MMAs). Returns cudaErrorNotSupported
// when the shape is outside what it handles.
bool chunked_tc_supported(const ChunkedArgs &a);
cudaError_t launch_chunked_tc(const ChunkedArgs &a, cudaStream_t stream);

// Single-pass tensor-core path (chunk 128, bf16, P = 64, N = 128, an even
// number of heads per B/C group): one persistent kernel (plus a kernel that
// clears its chain flags) carrying the state across chunks in float32.
bool chunked_fused_supported(const ChunkedArgs &a);
cudaError_t launch_chunked_fused(const ChunkedArgs &a, cudaStream_t stream);
// Whether the automatic path choice takes the single-pass kernel for this shape.
bool chunked_fused_preferred(const ChunkedArgs &a);

// State passing across chunks (shared by both paths).
// bf16_in: the chunk states are bfloat16 in states_bf16 (tensor-core path) and
// the entering states replace them in place; otherwise they are float32 in
// states.
cudaError_t launch_state_pass(const ChunkedArgs &a, bool write_f32_inplace, bool write_bf16,
                              cudaStream_t stream, bool programmatic, bool bf16_in = false);

// Arguments of one Mamba-1 diagonal scan (layouts as in selective_scan_diag_ex);
// z, delta_bias, D, init and final_state may be null. With nseg > 1 the
// sequence is split into nseg time segments of seg_len tokens (a multiple of
// 32) scanned in parallel; ws_h [nseg][B][Dm][N] and ws_s [nseg][B][Dm] (float32)
// hold the per-segment states and step sums.
struct DiagArgs {
    int64_t B, L, Dm;
    int N, chunk, softplus;
    const void *x, *dt, *z, *Bm, *Cm;
    const float *A, *D, *delta_bias, *init;
    void *y;
    float *final_state;
    int nseg;
    int64_t seg_len;
    float *ws_h, *ws_s;
};
// Time segments the scan of this shape is split into (1: one pass per
// sequence); the workspace the split needs is diag_workspace_bytes.
int diag_segments(int64_t B, int64_t L, int64_t Dm, int64_t N, int io);
size_t diag_workspace_bytes(int64_t B, int64_t L, int64_t Dm, int64_t N, int io);
cudaError_t launch_diag(int io, const DiagArgs &a, cudaStream_t stream);

// Causal depthwise convolution step (layouts as in ssd_conv1d_step). The
// output of channel c goes to out[s] for the first segment s with
// c < seg_end[s]; seg_end[2] == C. One segment: seg_end = {C, C, C}.
struct ConvArgs {
    int64_t B, C;
    int W, act;
    const void *x;
    float *state;
    const float *w, *bias;
    void *out[3];
    int64_t seg_end[3];
};
cudaError_t launch_conv1d_step(int io, const ConvArgs &a, cudaStream_t stream);

// Gated RMS norm over groups of `group` channels (layouts as in ssd_gated_rmsnorm).
struct NormArgs {
    int64_t B, D, group;
    float eps;
    const void *y, *z;
    const float *w;
    void *out;
};
cudaError_t launch_gated_rmsnorm(int io, const NormArgs &a, cudaStream_t stream);

// Forward chunk states and entering states only (CUDA-core chunk state, then
// the float32 state pass in place): a.states holds h_in(c), a.chunk_sum the
// chunk decays. Used by the backward to recompute the forward.
cudaError_t launch_forward_states(const ChunkedArgs &a, cudaStream_t stream);

// Backward of the chunked scan (layouts as in ssd_scan_chunked_bwd).
struct BwdArgs {
    static constexpr int kChunk = 64, kMaxP = 64, kMaxN = 128;
    int64_t B, L, H, P, N, G, nc;
    int io;
    int Q;                    // tokens per chunk: 64 (CUDA cores) or 128 (tensor-core gradients)
    int *status;              // SSD_OK, or SSD_ERR_TIMEOUT when a bounded wait gave up
    const void *x, *dt, *Bm, *Cm, *dy;
    const float *A, *D, *dfinal;
    float *hin;               // [B, nc, H, P, N] state entering each chunk (forward recompute)
    const float *init;        // [B, H, P, N] or null: state before the first chunk (tensor-core path)
    float *adj;               // [B, nc, H, P, N] adjoint chunk states, then leaving cotangents
    const float *chunk_sum;   // [B, H, nc] exp(sum of dt*A over the chunk)
    float *dB_part, *dC_part; // [B, L, H, N] per-head parts
    float *dA_part, *dD_part; // [B, nc, H]
    float *dx, *ddt, *dB, *dC, *dA, *dD, *dinit;
};
size_t bwd_chunk_smem_bytes(int64_t P, int64_t N);
cudaError_t launch_ssd_bwd(const BwdArgs &a, cudaStream_t stream);
// The per-chunk gradients on the tensor cores (chunks of 128 tokens, bf16
// inputs, P = 64, N = 128, a GB300-class device); the other steps as above.
bool chunk_bwd_tc_supported(int io, int64_t P, int64_t N);
cudaError_t launch_chunk_bwd_tc(const BwdArgs &a, cudaStream_t stream);
// The backward's float32 chunk states for those chunks on the tensor cores
// (forward recompute into hin with chunk_sum, adjoint into adj; one launch),
// then both passes over the chunks in place (one launch; writes dinit).
cudaError_t launch_bwd_states_tc(const BwdArgs &a, cudaStream_t stream);

cudaError_t launch_selftest_wait(int *status, int spin_limit, cudaStream_t stream);

// The bounds-check record of each translation unit with checked kernels (0
// when nothing failed or in a release build); clear resets it.
cudaError_t bounds_word_decode(unsigned long long *out, bool clear);
cudaError_t bounds_word_diag(unsigned long long *out, bool clear);
cudaError_t bounds_word_fused(unsigned long long *out, bool clear);
cudaError_t bounds_word_simt(unsigned long long *out, bool clear);

// Sets the thread-local text returned by ssd_last_error() and returns `status`.
int set_error(int status, const char *fmt, ...);

}  // namespace ssd
