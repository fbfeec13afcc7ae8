// C ABI of libssdscan.so (declared in include/ssd_scan.h): argument
// validation, workspace carving and kernel launch order. No allocation, no
// host synchronisation (except ssd_workspace_status, which exists to wait).
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "launch.h"
#include "ssd_scan.h"

namespace {

thread_local char g_err[512] = "";
thread_local cudaEvent_t g_stage_ev[4] = {nullptr, nullptr, nullptr, nullptr};

ssd_status fail(ssd_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

ssd_status ok() {
    g_err[0] = '\0';
    return SSD_OK;
}

ssd_status cuda_fail(cudaError_t e, const char *where) {
    return fail(SSD_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t round256(size_t v) { return (v + 255) & ~(size_t)255; }

// Returns SSD_OK and fills nothing on success; validates the sizes of a dims block.
ssd_status check_dims(const ssd_dims *d, bool need_seqlen) {
    if (!d) return fail(SSD_ERR_INVALID_ARG, "dims is NULL");
    if (d->batch < 0) return fail(SSD_ERR_INVALID_ARG, "batch must be >= 0 (got %lld)", (long long)d->batch);
    if (need_seqlen && d->seqlen < 0)
        return fail(SSD_ERR_INVALID_ARG, "seqlen must be >= 0 (got %lld)", (long long)d->seqlen);
    if (d->nheads < 1 || d->headdim < 1 || d->dstate < 1 || d->ngroups < 1)
        return fail(SSD_ERR_INVALID_ARG, "nheads, headdim, dstate and ngroups must be >= 1");
    if (d->nheads % d->ngroups != 0)
        return fail(SSD_ERR_INVALID_ARG, "nheads (%lld) must be a multiple of ngroups (%lld)",
                    (long long)d->nheads, (long long)d->ngroups);
    if (d->io_dtype != SSD_F32 && d->io_dtype != SSD_BF16)
        return fail(SSD_ERR_INVALID_ARG, "io_dtype must be SSD_F32 or SSD_BF16 (got %d)", d->io_dtype);
    if (d->flags & ~SSD_FLAG_SIMT) return fail(SSD_ERR_INVALID_ARG, "unknown flags 0x%x", d->flags);
    if (d->nheads > 65535 || d->batch > 65535)
        return fail(SSD_ERR_UNSUPPORTED, "nheads and batch must be <= 65535");
    return SSD_OK;
}

bool valid_chunk(int q) { return q == 64 || q == 128 || q == 256; }

}  // namespace

namespace ssd {
int set_error(int status, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return status;
}

cudaError_t mark_stage(const ChunkedArgs &a, int i, cudaStream_t stream) {
    if (!a.stage_ev[i]) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return e;
    if (cs == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(a.stage_ev[i], stream, cudaEventRecordExternal);
    return cudaEventRecord(a.stage_ev[i], stream);
}

WorkspaceLayout workspace_layout(int64_t B, int64_t L, int64_t H, int64_t P, int64_t N, int Q) {
    WorkspaceLayout w{};
    const int64_t nc = (L + Q - 1) / Q;
    const size_t n_state = (size_t)B * nc * H * P * N;
    w.status = 0;
    w.states = 256;
    w.states_bf16 = w.states + round256(n_state * sizeof(float));
    w.chunk_sum = w.states_bf16 + round256(n_state * sizeof(uint16_t));
    w.total = w.chunk_sum + round256((size_t)B * H * nc * sizeof(float));
    return w;
}
}  // namespace ssd

extern "C" {

const char *ssd_last_error(void) { return g_err; }

size_t ssd_workspace_size(const ssd_dims *dims, int chunk_size) {
    if (check_dims(dims, true) != SSD_OK || !valid_chunk(chunk_size)) return 0;
    return ssd::workspace_layout(dims->batch, dims->seqlen, dims->nheads, dims->headdim, dims->dstate,
                                 chunk_size)
        .total;
}

ssd_status ssd_scan_chunked(const ssd_dims *dims, const void *x, const void *dt, const float *A, const void *B,
                            const void *C, const float *D, const float *init_state, int chunk_size, void *y,
                            float *final_state, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    ssd_status s = check_dims(dims, true);
    if (s != SSD_OK) return s;
    if (!valid_chunk(chunk_size))
        return fail(SSD_ERR_INVALID_ARG, "chunk_size must be 64, 128 or 256 (got %d)", chunk_size);
    const int64_t Bsz = dims->batch, L = dims->seqlen;
    const bool has_tokens = Bsz > 0 && L > 0;
    if (has_tokens && (!x || !dt || !A || !B || !C || !y))
        return fail(SSD_ERR_INVALID_ARG, "x, dt, A, B, C and y must be non-NULL");
    const void *ptrs[] = {x, dt, A, B, C, D, init_state, y, final_state};
    const char *names[] = {"x", "dt", "A", "B", "C", "D", "init_state", "y", "final_state"};
    for (int i = 0; i < 9; ++i)
        if (ptrs[i] && !aligned(ptrs[i], 16)) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    const ssd::WorkspaceLayout w =
        ssd::workspace_layout(Bsz, L, dims->nheads, dims->headdim, dims->dstate, chunk_size);
    if (Bsz > 0) {
        if (!workspace) return fail(SSD_ERR_INVALID_ARG, "workspace is NULL");
        if (!aligned(workspace, 256)) return fail(SSD_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
        if (workspace_bytes < w.total)
            return fail(SSD_ERR_INVALID_ARG, "workspace too small: %zu bytes given, %zu needed", workspace_bytes,
                        w.total);
    }
    if (Bsz == 0) return ok();

    ssd::ChunkedArgs a{};
    a.B = Bsz; a.L = L; a.H = dims->nheads; a.P = dims->headdim; a.N = dims->dstate; a.G = dims->ngroups;
    a.Q = chunk_size;
    a.nc = (L + chunk_size - 1) / chunk_size;
    a.io = dims->io_dtype == SSD_BF16 ? ssd::IO_BF16 : ssd::IO_F32;
    a.x = x; a.dt = dt; a.Bm = B; a.Cm = C; a.A = A; a.D = D; a.init_state = init_state;
    a.y = y; a.final_state = final_state;
    char *ws = static_cast<char *>(workspace);
    a.status = reinterpret_cast<int *>(ws + w.status);
    a.states = reinterpret_cast<float *>(ws + w.states);
    a.states_bf16 = reinterpret_cast<uint16_t *>(ws + w.states_bf16);
    a.chunk_sum = reinterpret_cast<float *>(ws + w.chunk_sum);
    for (int i = 0; i < 4; ++i) {
        a.stage_ev[i] = g_stage_ev[i];
        g_stage_ev[i] = nullptr;  // consumed by this call
    }

    const int64_t tilesP = (a.P + 63) / 64, tilesN = (a.N + 63) / 64;
    // the status word reports this call only: the first kernel of either path
    // clears it (thread 0 of its first CTA) before any wait of this call can
    // give up, which takes seconds
    cudaError_t e;
    if (a.io == ssd::IO_BF16 && !(dims->flags & SSD_FLAG_SIMT) && has_tokens && ssd::chunked_tc_supported(a)) {
        e = ssd::launch_chunked_tc(a, stream);
        if (e != cudaSuccess) return cuda_fail(e, "ssd_scan_chunked (tensor-core path)");
        return ok();
    }
    if (a.H * tilesP * tilesN > 65535) return fail(SSD_ERR_UNSUPPORTED, "nheads * tiles of P and N too large");
    e = ssd::launch_chunked_simt(a, stream);
    if (e != cudaSuccess) return cuda_fail(e, "ssd_scan_chunked");
    return ok();
}

ssd_status ssd_decode_step(const ssd_dims *dims, float *state, const void *x, const void *dt, const float *A,
                           const void *B, const void *C, const float *D, void *y, cudaStream_t stream) {
    ssd_status s = check_dims(dims, false);
    if (s != SSD_OK) return s;
    if (dims->batch > 0 && (!state || !x || !dt || !A || !B || !C || !y))
        return fail(SSD_ERR_INVALID_ARG, "state, x, dt, A, B, C and y must be non-NULL");
    const void *ptrs[] = {state, x, dt, A, B, C, D, y};
    const char *names[] = {"state", "x", "dt", "A", "B", "C", "D", "y"};
    for (int i = 0; i < 8; ++i)
        if (ptrs[i] && !aligned(ptrs[i], 16)) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    if (dims->batch * dims->nheads > 0x7fffffffLL) return fail(SSD_ERR_UNSUPPORTED, "batch * nheads too large");
    if (dims->batch == 0) return ok();
    cudaError_t e = ssd::launch_decode(dims->io_dtype == SSD_BF16 ? ssd::IO_BF16 : ssd::IO_F32, dims->batch,
                                       dims->nheads, dims->headdim, dims->dstate, dims->ngroups, state, x, dt, A,
                                       B, C, D, y, stream);
    if (e != cudaSuccess) return cuda_fail(e, "ssd_decode_step");
    return ok();
}

ssd_status selective_scan_diag_ex(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int32_t io_dtype,
                                  const void *x, const void *dt, const float *A, const void *B, const void *C,
                                  const float *D, const void *z, const float *delta_bias, int32_t delta_softplus,
                                  const float *init_state, int chunk_size, void *y, float *final_state,
                                  void *workspace, size_t ws_bytes, cudaStream_t stream) {
    if (batch < 0 || seqlen < 0) return fail(SSD_ERR_INVALID_ARG, "batch and seqlen must be >= 0");
    if (dim < 1) return fail(SSD_ERR_INVALID_ARG, "dim must be >= 1");
    if (dstate < 1) return fail(SSD_ERR_INVALID_ARG, "dstate must be >= 1");
    if (dstate > 64) return fail(SSD_ERR_UNSUPPORTED, "dstate must be <= 64 (got %lld)", (long long)dstate);
    if (io_dtype != SSD_F32 && io_dtype != SSD_BF16)
        return fail(SSD_ERR_INVALID_ARG, "io_dtype must be SSD_F32 or SSD_BF16 (got %d)", io_dtype);
    if (chunk_size < 32 || chunk_size % 32 != 0)
        return fail(SSD_ERR_INVALID_ARG, "chunk_size must be a positive multiple of 32 (got %d)", chunk_size);
    if (delta_softplus != 0 && delta_softplus != 1)
        return fail(SSD_ERR_INVALID_ARG, "delta_softplus must be 0 or 1 (got %d)", delta_softplus);
    if (batch > 65535) return fail(SSD_ERR_UNSUPPORTED, "batch must be <= 65535");
    const bool has_tokens = batch > 0 && seqlen > 0;
    if (has_tokens && (!x || !dt || !A || !B || !C || !y))
        return fail(SSD_ERR_INVALID_ARG, "x, dt, A, B, C and y must be non-NULL");
    if (batch > 0 && !A) return fail(SSD_ERR_INVALID_ARG, "A must be non-NULL");
    const void *ptrs[] = {x, dt, A, B, C, D, z, delta_bias, init_state, y, final_state};
    const char *names[] = {"x", "dt", "A", "B", "C", "D", "z", "delta_bias", "init_state", "y", "final_state"};
    for (int i = 0; i < 11; ++i)
        if (ptrs[i] && !aligned(ptrs[i], 16)) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    if (batch == 0) return ok();
    const int io = io_dtype == SSD_BF16 ? ssd::IO_BF16 : ssd::IO_F32;
    ssd::DiagArgs a{};
    a.nseg = 1;
    if (workspace) {
        if (!aligned(workspace, 256)) return fail(SSD_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
        const size_t need = ssd::diag_workspace_bytes(batch, seqlen, dim, dstate, io);
        if (ws_bytes < need)
            return fail(SSD_ERR_INVALID_ARG, "workspace too small: %zu bytes, need %zu", ws_bytes, need);
        a.nseg = ssd::diag_segments(batch, seqlen, dim, dstate, io);
        if (a.nseg > 1) {
            a.ws_h = static_cast<float *>(workspace);
            const size_t h = (size_t)a.nseg * batch * dim * dstate * sizeof(float);
            a.ws_s = reinterpret_cast<float *>(static_cast<char *>(workspace) + (h + 255) / 256 * 256);
        }
    }
    a.B = batch;
    a.L = seqlen;
    a.Dm = dim;
    a.N = (int)dstate;
    a.chunk = chunk_size;
    a.softplus = delta_softplus;
    a.x = x;
    a.dt = dt;
    a.z = z;
    a.Bm = B;
    a.Cm = C;
    a.A = A;
    a.D = D;
    a.delta_bias = delta_bias;
    a.init = init_state;
    a.y = y;
    a.final_state = final_state;
    cudaError_t e = ssd::launch_diag(io, a, stream);
    if (e != cudaSuccess) return cuda_fail(e, "selective_scan_diag");
    return ok();
}

ssd_status selective_scan_diag(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int32_t io_dtype,
                               const void *x, const void *dt, const float *A, const void *B, const void *C,
                               const float *D, const float *init_state, int chunk_size, void *y,
                               float *final_state, cudaStream_t stream) {
    return selective_scan_diag_ex(batch, seqlen, dim, dstate, io_dtype, x, dt, A, B, C, D, nullptr, nullptr, 0,
                                  init_state, chunk_size, y, final_state, nullptr, 0, stream);
}

size_t selective_scan_diag_workspace_size(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                                          int32_t io_dtype) {
    if (batch < 1 || seqlen < 1 || dim < 1 || dstate < 1 || dstate > 64) return 0;
    if (io_dtype != SSD_F32 && io_dtype != SSD_BF16) return 0;
    return ssd::diag_workspace_bytes(batch, seqlen, dim, dstate, io_dtype == SSD_BF16 ? ssd::IO_BF16 : ssd::IO_F32);
}

ssd_status ssd_record_stage_events(cudaEvent_t *events, int count) {
    if (!events) {
        for (int i = 0; i < 4; ++i) g_stage_ev[i] = nullptr;
        return ok();
    }
    if (count != 4) return fail(SSD_ERR_INVALID_ARG, "count must be 4 (got %d)", count);
    for (int i = 0; i < 4; ++i)
        if (!events[i]) return fail(SSD_ERR_INVALID_ARG, "event %d is NULL", i);
    for (int i = 0; i < 4; ++i) g_stage_ev[i] = events[i];
    return ok();
}

ssd_status ssd_workspace_status(const void *workspace, cudaStream_t stream) {
    if (!workspace) return fail(SSD_ERR_INVALID_ARG, "workspace is NULL");
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "ssd_workspace_status: stream");
    int word = 0;
    e = cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "ssd_workspace_status: read");
    if (word == SSD_OK) return ok();
    if (word == SSD_ERR_TIMEOUT) return fail(SSD_ERR_TIMEOUT, "a bounded in-kernel wait timed out");
    return fail((ssd_status)word, "kernel recorded status %d", word);
}

ssd_status ssd_selftest_bounded_wait(void *workspace, int spin_limit, cudaStream_t stream) {
    if (!workspace) return fail(SSD_ERR_INVALID_ARG, "workspace is NULL");
    if (!aligned(workspace, 16)) return fail(SSD_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
    if (spin_limit < 1 || spin_limit > (1 << 20))
        return fail(SSD_ERR_INVALID_ARG, "spin_limit must be in [1, 2^20] (got %d)", spin_limit);
    cudaError_t e = ssd::launch_selftest_wait(static_cast<int *>(workspace), spin_limit, stream);
    if (e != cudaSuccess) return cuda_fail(e, "ssd_selftest_bounded_wait");
    return ok();
}

}  // extern "C"
