// C ABI of libssdscan.so (declared in include/ssd_scan.h): argument
// validation, workspace carving and kernel launch order. No allocation, no
// host synchronisation (except ssd_workspace_status, which exists to wait).
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

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
    if (d->flags & ~(SSD_FLAG_SIMT | SSD_FLAG_FUSED | SSD_FLAG_STAGED))
        return fail(SSD_ERR_INVALID_ARG, "unknown flags 0x%x", d->flags);
    if ((d->flags & SSD_FLAG_FUSED) && (d->flags & (SSD_FLAG_STAGED | SSD_FLAG_SIMT)))
        return fail(SSD_ERR_INVALID_ARG, "SSD_FLAG_FUSED excludes SSD_FLAG_STAGED and SSD_FLAG_SIMT");
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

int ssd_scan_path(const ssd_dims *dims, int chunk_size) {
    if (check_dims(dims, true) != SSD_OK || !valid_chunk(chunk_size)) return -1;
    ssd::ChunkedArgs a{};
    a.B = dims->batch; a.L = dims->seqlen; a.H = dims->nheads; a.P = dims->headdim; a.N = dims->dstate;
    a.G = dims->ngroups; a.Q = chunk_size;
    a.nc = (a.L + chunk_size - 1) / chunk_size;
    a.io = dims->io_dtype == SSD_BF16 ? ssd::IO_BF16 : ssd::IO_F32;
    const bool has_tokens = a.B > 0 && a.L > 0;
    if (dims->flags & SSD_FLAG_FUSED) return ssd::chunked_fused_supported(a) ? SSD_PATH_FUSED : -1;
    if (a.io == ssd::IO_BF16 && !(dims->flags & (SSD_FLAG_SIMT | SSD_FLAG_STAGED)) && has_tokens &&
        ssd::chunked_fused_supported(a) && ssd::chunked_fused_preferred(a))
        return SSD_PATH_FUSED;
    if (a.io == ssd::IO_BF16 && !(dims->flags & SSD_FLAG_SIMT) && has_tokens && ssd::chunked_tc_supported(a))
        return SSD_PATH_STAGED;
    return SSD_PATH_SIMT;
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
    if (dims->flags & SSD_FLAG_FUSED) {
        if (!has_tokens) return ok();  // nothing to compute; validated above
        if (!ssd::chunked_fused_supported(a))
            return fail(SSD_ERR_UNSUPPORTED,
                        "SSD_FLAG_FUSED needs bf16, headdim 64, dstate 128, chunk 128 and an even number of heads "
                        "per group on an sm_100-family GPU");
        e = ssd::launch_chunked_fused(a, stream);
        if (e != cudaSuccess) return cuda_fail(e, "ssd_scan_chunked (single-pass path)");
        return ok();
    }
    if (a.io == ssd::IO_BF16 && !(dims->flags & (SSD_FLAG_SIMT | SSD_FLAG_STAGED)) && has_tokens &&
        ssd::chunked_fused_supported(a) && ssd::chunked_fused_preferred(a)) {
        e = ssd::launch_chunked_fused(a, stream);
        if (e != cudaSuccess) return cuda_fail(e, "ssd_scan_chunked (single-pass path)");
        return ok();
    }
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

// ------------------------------------------------------------- backward

namespace {

struct BwdWs {
    size_t status, hin, adj, chunk_sum, dB_part, dC_part, dA_part, dD_part, total;
};
BwdWs bwd_ws(const ssd_dims *d) {
    const int64_t Q = ssd::BwdArgs::kChunk, nc = (d->seqlen + Q - 1) / Q;
    const size_t st = (size_t)(d->batch * nc * d->nheads * d->headdim * d->dstate) * sizeof(float);
    const size_t part = (size_t)(d->batch * d->seqlen * d->nheads * d->dstate) * sizeof(float);
    const size_t small = (size_t)(d->batch * nc * d->nheads) * sizeof(float);
    BwdWs w{};
    w.status = 0;
    w.hin = 256;
    w.adj = w.hin + round256(st);
    w.chunk_sum = w.adj + round256(st);
    w.dB_part = w.chunk_sum + round256(small);
    w.dC_part = w.dB_part + round256(part);
    w.dA_part = w.dC_part + round256(part);
    w.dD_part = w.dA_part + round256(small);
    w.total = w.dD_part + round256(small);
    return w;
}

}  // namespace

size_t ssd_scan_chunked_bwd_workspace_size(const ssd_dims *dims) {
    if (!dims || dims->batch < 0 || dims->seqlen < 0 || dims->nheads < 1 || dims->headdim < 1 ||
        dims->dstate < 1 || dims->ngroups < 1 || dims->nheads % dims->ngroups != 0 ||
        (dims->io_dtype != SSD_F32 && dims->io_dtype != SSD_BF16) || dims->headdim > ssd::BwdArgs::kMaxP ||
        dims->dstate > ssd::BwdArgs::kMaxN)
        return 0;
    return bwd_ws(dims).total;
}

ssd_status ssd_scan_chunked_bwd(const ssd_dims *dims, const void *x, const void *dt, const float *A, const void *B,
                                const void *C, const float *D, const float *init_state, const void *dy,
                                const float *dfinal_state, float *dx, float *ddt, float *dA, float *dB, float *dC,
                                float *dD, float *dinit_state, void *workspace, size_t ws_bytes,
                                cudaStream_t stream) {
    ssd_status s = check_dims(dims, true);
    if (s != SSD_OK) return s;
    if (dims->headdim > ssd::BwdArgs::kMaxP || dims->dstate > ssd::BwdArgs::kMaxN)
        return fail(SSD_ERR_UNSUPPORTED, "backward supports headdim <= %d and dstate <= %d", ssd::BwdArgs::kMaxP,
                    ssd::BwdArgs::kMaxN);
    if (!A || !dA) return fail(SSD_ERR_INVALID_ARG, "A and dA must be non-NULL");
    const bool has_tokens = dims->batch > 0 && dims->seqlen > 0;
    if (has_tokens && (!x || !dt || !B || !C || !dy || !dx || !ddt || !dB || !dC))
        return fail(SSD_ERR_INVALID_ARG, "x, dt, B, C, dy, dx, ddt, dB and dC must be non-NULL");
    const void *ptrs[] = {x, dt, A, B, C, D, init_state, dy, dfinal_state, dx, ddt, dA, dB, dC, dD, dinit_state};
    const char *names[] = {"x", "dt", "A", "B", "C", "D", "init_state", "dy", "dfinal_state", "dx", "ddt", "dA",
                           "dB", "dC", "dD", "dinit_state"};
    for (int i = 0; i < 16; ++i)
        if (ptrs[i] && !aligned(ptrs[i], 16)) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    const BwdWs w = bwd_ws(dims);
    if (!workspace) return fail(SSD_ERR_INVALID_ARG, "workspace is NULL");
    if (!aligned(workspace, 256)) return fail(SSD_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
    if (ws_bytes < w.total) return fail(SSD_ERR_INVALID_ARG, "workspace too small: %zu bytes, need %zu", ws_bytes, w.total);
    const int io = dims->io_dtype == SSD_BF16 ? ssd::IO_BF16 : ssd::IO_F32;
    char *ws = static_cast<char *>(workspace);
    cudaError_t e = cudaSuccess;
    if (!has_tokens) {
        // no tokens: dinit = dfinal, every other gradient zero
        const size_t hpn = (size_t)(dims->batch * dims->nheads * dims->headdim * dims->dstate) * sizeof(float);
        if (dinit_state && hpn)
            e = dfinal_state ? cudaMemcpyAsync(dinit_state, dfinal_state, hpn, cudaMemcpyDeviceToDevice, stream)
                             : cudaMemsetAsync(dinit_state, 0, hpn, stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(dA, 0, (size_t)dims->nheads * sizeof(float), stream);
        if (e == cudaSuccess && dD) e = cudaMemsetAsync(dD, 0, (size_t)dims->nheads * sizeof(float), stream);
        if (e != cudaSuccess) return cuda_fail(e, "ssd_scan_chunked_bwd");
        return ok();
    }
    // chunks of 128 tokens with the per-chunk gradients on the tensor cores
    // (bf16, P 64, N 128, unless SSD_FLAG_SIMT), else 64 on the CUDA cores;
    // the workspace is sized for 64
    const bool tc = !(dims->flags & SSD_FLAG_SIMT) && ssd::chunk_bwd_tc_supported(io, dims->headdim, dims->dstate);
    ssd::ChunkedArgs f{};
    f.B = dims->batch;
    f.L = dims->seqlen;
    f.H = dims->nheads;
    f.P = dims->headdim;
    f.N = dims->dstate;
    f.G = dims->ngroups;
    f.Q = tc ? 128 : ssd::BwdArgs::kChunk;
    f.nc = (f.L + f.Q - 1) / f.Q;
    f.io = io;
    f.x = x;
    f.dt = dt;
    f.Bm = B;
    f.Cm = C;
    f.A = A;
    f.D = D;
    f.init_state = init_state;
    f.status = reinterpret_cast<int *>(ws + w.status);
    f.states = reinterpret_cast<float *>(ws + w.hin);
    f.chunk_sum = reinterpret_cast<float *>(ws + w.chunk_sum);
    // the tensor-core path recomputes the forward states inside launch_ssd_bwd
    if (!tc && (e = ssd::launch_forward_states(f, stream)) != cudaSuccess)
        return cuda_fail(e, "ssd_scan_chunked_bwd: forward states");
    ssd::BwdArgs a{};
    a.B = f.B;
    a.L = f.L;
    a.H = f.H;
    a.P = f.P;
    a.N = f.N;
    a.G = f.G;
    a.nc = f.nc;
    a.io = io;
    a.Q = f.Q;
    a.status = f.status;
    a.x = x;
    a.dt = dt;
    a.Bm = B;
    a.Cm = C;
    a.dy = dy;
    a.A = A;
    a.D = D;
    a.dfinal = dfinal_state;
    a.hin = f.states;
    a.init = init_state;
    a.adj = reinterpret_cast<float *>(ws + w.adj);
    a.chunk_sum = f.chunk_sum;
    a.dB_part = reinterpret_cast<float *>(ws + w.dB_part);
    a.dC_part = reinterpret_cast<float *>(ws + w.dC_part);
    a.dA_part = reinterpret_cast<float *>(ws + w.dA_part);
    a.dD_part = reinterpret_cast<float *>(ws + w.dD_part);
    a.dx = dx;
    a.ddt = ddt;
    a.dB = dB;
    a.dC = dC;
    a.dA = dA;
    a.dD = dD;
    a.dinit = dinit_state;
    e = ssd::launch_ssd_bwd(a, stream);
    if (e != cudaSuccess) return cuda_fail(e, "ssd_scan_chunked_bwd");
    return ok();
}

// ------------------------------------------------------ decode-layer pieces

namespace {

size_t io_size(int32_t io) { return io == SSD_BF16 ? 2 : 4; }

struct LayerWs {
    size_t x, b, c, y, total;
};
LayerWs layer_ws(const ssd_dims *d) {
    const size_t e = io_size(d->io_dtype), hp = (size_t)(d->batch * d->nheads * d->headdim);
    const size_t gn = (size_t)(d->batch * d->ngroups * d->dstate);
    LayerWs w{};
    w.x = 0;
    w.b = round256(hp * e);
    w.c = w.b + round256(gn * e);
    w.y = w.c + round256(gn * e);
    w.total = w.y + round256(hp * e);
    return w;
}

// Validation shared by the layer step and the graph capture.
ssd_status check_layer(const ssd_dims *dims, int64_t conv_width, const void *xBC, const float *conv_state,
                       const float *conv_weight, const float *conv_bias, const void *dt, const float *A,
                       const float *D, const float *ssm_state, const void *z, const float *norm_weight,
                       int64_t norm_group, float eps, const void *out, const void *workspace, size_t ws_bytes) {
    ssd_status s = check_dims(dims, false);
    if (s != SSD_OK) return s;
    if (conv_width < 1 || conv_width > 8)
        return fail(SSD_ERR_INVALID_ARG, "conv_width must be 1..8 (got %lld)", (long long)conv_width);
    const int64_t hp = dims->nheads * dims->headdim;
    if (norm_group < 1 || hp % norm_group != 0)
        return fail(SSD_ERR_INVALID_ARG, "norm_group must divide nheads*headdim (got %lld)", (long long)norm_group);
    if (!(eps >= 0.f)) return fail(SSD_ERR_INVALID_ARG, "eps must be >= 0");
    if (dims->batch == 0) return SSD_OK;
    if (!xBC || !conv_state || !conv_weight || !dt || !A || !ssm_state || !norm_weight || !out || !workspace)
        return fail(SSD_ERR_INVALID_ARG,
                    "xBC, conv_state, conv_weight, dt, A, ssm_state, norm_weight, out and workspace must be non-NULL");
    const void *ptrs[] = {xBC, conv_state, conv_weight, conv_bias, dt, A, D, ssm_state, z, norm_weight, out};
    const char *names[] = {"xBC", "conv_state", "conv_weight", "conv_bias", "dt", "A", "D", "ssm_state", "z",
                           "norm_weight", "out"};
    for (int i = 0; i < 11; ++i)
        if (ptrs[i] && !aligned(ptrs[i], 16)) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    if (!aligned(workspace, 256)) return fail(SSD_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
    const size_t need = layer_ws(dims).total;
    if (ws_bytes < need) return fail(SSD_ERR_INVALID_ARG, "workspace too small: %zu bytes, need %zu", ws_bytes, need);
    return SSD_OK;
}

cudaError_t layer_launch(const ssd_dims *d, int64_t conv_width, const void *xBC, float *conv_state,
                         const float *conv_weight, const float *conv_bias, const void *dt, const float *A,
                         const float *D, float *ssm_state, const void *z, const float *norm_weight,
                         int64_t norm_group, float eps, void *out, void *workspace, cudaStream_t stream) {
    const int io = d->io_dtype == SSD_BF16 ? ssd::IO_BF16 : ssd::IO_F32;
    const LayerWs w = layer_ws(d);
    char *ws = static_cast<char *>(workspace);
    const int64_t hp = d->nheads * d->headdim, gn = d->ngroups * d->dstate;
    ssd::ConvArgs c{};
    c.B = d->batch;
    c.C = hp + 2 * gn;
    c.W = (int)conv_width;
    c.act = 1;
    c.x = xBC;
    c.state = conv_state;
    c.w = conv_weight;
    c.bias = conv_bias;
    c.out[0] = ws + w.x;
    c.out[1] = ws + w.b;
    c.out[2] = ws + w.c;
    c.seg_end[0] = hp;
    c.seg_end[1] = hp + gn;
    c.seg_end[2] = hp + 2 * gn;
    cudaError_t e = ssd::launch_conv1d_step(io, c, stream);
    if (e != cudaSuccess) return e;
    e = ssd::launch_decode(io, d->batch, d->nheads, d->headdim, d->dstate, d->ngroups, ssm_state, ws + w.x, dt, A,
                           ws + w.b, ws + w.c, D, ws + w.y, stream);
    if (e != cudaSuccess) return e;
    ssd::NormArgs n{};
    n.B = d->batch;
    n.D = hp;
    n.group = norm_group;
    n.eps = eps;
    n.y = ws + w.y;
    n.z = z;
    n.w = norm_weight;
    n.out = out;
    return ssd::launch_gated_rmsnorm(io, n, stream);
}

}  // namespace

ssd_status ssd_conv1d_step(int64_t batch, int64_t channels, int64_t width, int32_t io_dtype, const void *x,
                           float *conv_state, const float *weight, const float *bias, int32_t activation,
                           void *out, cudaStream_t stream) {
    if (batch < 0) return fail(SSD_ERR_INVALID_ARG, "batch must be >= 0");
    if (channels < 1) return fail(SSD_ERR_INVALID_ARG, "channels must be >= 1");
    if (width < 1 || width > 8) return fail(SSD_ERR_INVALID_ARG, "width must be 1..8 (got %lld)", (long long)width);
    if (io_dtype != SSD_F32 && io_dtype != SSD_BF16)
        return fail(SSD_ERR_INVALID_ARG, "io_dtype must be SSD_F32 or SSD_BF16 (got %d)", io_dtype);
    if (activation != SSD_ACT_NONE && activation != SSD_ACT_SILU)
        return fail(SSD_ERR_INVALID_ARG, "activation must be SSD_ACT_NONE or SSD_ACT_SILU (got %d)", activation);
    if (batch * channels > ((int64_t)1 << 38)) return fail(SSD_ERR_UNSUPPORTED, "batch * channels too large");
    if (batch == 0) return ok();
    if (!x || !conv_state || !weight || !out)
        return fail(SSD_ERR_INVALID_ARG, "x, conv_state, weight and out must be non-NULL");
    const void *ptrs[] = {x, conv_state, weight, bias, out};
    const char *names[] = {"x", "conv_state", "weight", "bias", "out"};
    for (int i = 0; i < 5; ++i)
        if (ptrs[i] && !aligned(ptrs[i], 16)) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    if (x == out) return fail(SSD_ERR_INVALID_ARG, "out may not alias x");
    ssd::ConvArgs c{};
    c.B = batch;
    c.C = channels;
    c.W = (int)width;
    c.act = activation;
    c.x = x;
    c.state = conv_state;
    c.w = weight;
    c.bias = bias;
    c.out[0] = c.out[1] = c.out[2] = out;
    c.seg_end[0] = c.seg_end[1] = c.seg_end[2] = channels;
    cudaError_t e = ssd::launch_conv1d_step(io_dtype == SSD_BF16 ? ssd::IO_BF16 : ssd::IO_F32, c, stream);
    if (e != cudaSuccess) return cuda_fail(e, "ssd_conv1d_step");
    return ok();
}

ssd_status ssd_gated_rmsnorm(int64_t batch, int64_t dim, int64_t group, int32_t io_dtype, const void *y,
                             const void *z, const float *weight, float eps, void *out, cudaStream_t stream) {
    if (batch < 0) return fail(SSD_ERR_INVALID_ARG, "batch must be >= 0");
    if (dim < 1 || group < 1 || dim % group != 0)
        return fail(SSD_ERR_INVALID_ARG, "dim must be a positive multiple of group (dim %lld, group %lld)",
                    (long long)dim, (long long)group);
    if (io_dtype != SSD_F32 && io_dtype != SSD_BF16)
        return fail(SSD_ERR_INVALID_ARG, "io_dtype must be SSD_F32 or SSD_BF16 (got %d)", io_dtype);
    if (!(eps >= 0.f)) return fail(SSD_ERR_INVALID_ARG, "eps must be >= 0");
    if (batch * (dim / group) > 0x7fffffffLL) return fail(SSD_ERR_UNSUPPORTED, "batch * dim / group too large");
    if (batch == 0) return ok();
    if (!y || !weight || !out) return fail(SSD_ERR_INVALID_ARG, "y, weight and out must be non-NULL");
    const void *ptrs[] = {y, z, weight, out};
    const char *names[] = {"y", "z", "weight", "out"};
    for (int i = 0; i < 4; ++i)
        if (ptrs[i] && !aligned(ptrs[i], 16)) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    ssd::NormArgs n{};
    n.B = batch;
    n.D = dim;
    n.group = group;
    n.eps = eps;
    n.y = y;
    n.z = z;
    n.w = weight;
    n.out = out;
    cudaError_t e = ssd::launch_gated_rmsnorm(io_dtype == SSD_BF16 ? ssd::IO_BF16 : ssd::IO_F32, n, stream);
    if (e != cudaSuccess) return cuda_fail(e, "ssd_gated_rmsnorm");
    return ok();
}

size_t ssd_decode_layer_workspace_size(const ssd_dims *dims) {
    if (!dims || dims->batch < 1 || dims->nheads < 1 || dims->headdim < 1 || dims->dstate < 1 ||
        dims->ngroups < 1 || dims->nheads % dims->ngroups != 0 ||
        (dims->io_dtype != SSD_F32 && dims->io_dtype != SSD_BF16))
        return 0;
    return layer_ws(dims).total;
}

ssd_status ssd_decode_layer_step(const ssd_dims *dims, int64_t conv_width, const void *xBC, float *conv_state,
                                 const float *conv_weight, const float *conv_bias, const void *dt, const float *A,
                                 const float *D, float *ssm_state, const void *z, const float *norm_weight,
                                 int64_t norm_group, float eps, void *out, void *workspace, size_t ws_bytes,
                                 cudaStream_t stream) {
    ssd_status s = check_layer(dims, conv_width, xBC, conv_state, conv_weight, conv_bias, dt, A, D, ssm_state, z,
                               norm_weight, norm_group, eps, out, workspace, ws_bytes);
    if (s != SSD_OK) return s;
    if (dims->batch == 0) return ok();
    cudaError_t e = layer_launch(dims, conv_width, xBC, conv_state, conv_weight, conv_bias, dt, A, D, ssm_state, z,
                                 norm_weight, norm_group, eps, out, workspace, stream);
    if (e != cudaSuccess) return cuda_fail(e, "ssd_decode_layer_step");
    return ok();
}

struct ssd_decode_graph {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

ssd_status ssd_decode_graph_create(const ssd_dims *dims, int64_t conv_width, int32_t steps, const void *xBC,
                                   float *conv_state, const float *conv_weight, const float *conv_bias,
                                   const void *dt, const float *A, const float *D, float *ssm_state, const void *z,
                                   const float *norm_weight, int64_t norm_group, float eps, void *out,
                                   void *workspace, size_t ws_bytes, ssd_decode_graph **graph) {
    if (!graph) return fail(SSD_ERR_INVALID_ARG, "graph is NULL");
    *graph = nullptr;
    if (steps < 1) return fail(SSD_ERR_INVALID_ARG, "steps must be >= 1 (got %d)", steps);
    ssd_status s = check_layer(dims, conv_width, xBC, conv_state, conv_weight, conv_bias, dt, A, D, ssm_state, z,
                               norm_weight, norm_group, eps, out, workspace, ws_bytes);
    if (s != SSD_OK) return s;
    if (dims->batch == 0) return fail(SSD_ERR_INVALID_ARG, "batch must be >= 1 for a decode graph");
    const size_t e = io_size(dims->io_dtype);
    const int64_t hp = dims->nheads * dims->headdim, cc = hp + 2 * dims->ngroups * dims->dstate;
    const size_t step_xbc = (size_t)(dims->batch * cc) * e, step_dt = (size_t)(dims->batch * dims->nheads) * e;
    const size_t step_hp = (size_t)(dims->batch * hp) * e;
    if (step_xbc % 16 || step_dt % 16 || step_hp % 16)
        return fail(SSD_ERR_INVALID_ARG, "per-step slices of xBC, dt, z and out must be multiples of 16 bytes");
    cudaStream_t st = nullptr;
    cudaError_t ce = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (ce != cudaSuccess) return cuda_fail(ce, "ssd_decode_graph_create: stream");
    cudaGraph_t g = nullptr;
    ce = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal);
    if (ce == cudaSuccess) {
        cudaError_t le = cudaSuccess;
        for (int32_t k = 0; k < steps && le == cudaSuccess; ++k)
            le = layer_launch(dims, conv_width, static_cast<const char *>(xBC) + k * step_xbc, conv_state,
                              conv_weight, conv_bias, static_cast<const char *>(dt) + k * step_dt, A, D, ssm_state,
                              z ? static_cast<const char *>(z) + k * step_hp : nullptr, norm_weight, norm_group,
                              eps, static_cast<char *>(out) + k * step_hp, workspace, st);
        ce = cudaStreamEndCapture(st, &g);
        if (le != cudaSuccess) ce = le;
    }
    cudaStreamDestroy(st);
    if (ce != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        return cuda_fail(ce, "ssd_decode_graph_create: capture");
    }
    cudaGraphExec_t ex = nullptr;
    ce = cudaGraphInstantiate(&ex, g, 0);
    if (ce != cudaSuccess) {
        cudaGraphDestroy(g);
        return cuda_fail(ce, "ssd_decode_graph_create: instantiate");
    }
    auto *h = new (std::nothrow) ssd_decode_graph{g, ex};
    if (!h) {
        cudaGraphExecDestroy(ex);
        cudaGraphDestroy(g);
        return fail(SSD_ERR_CUDA, "ssd_decode_graph_create: out of host memory");
    }
    *graph = h;
    return ok();
}

ssd_status ssd_decode_graph_launch(ssd_decode_graph *graph, cudaStream_t stream) {
    if (!graph) return fail(SSD_ERR_INVALID_ARG, "graph is NULL");
    cudaError_t e = cudaGraphLaunch(graph->exec, stream);
    if (e != cudaSuccess) return cuda_fail(e, "ssd_decode_graph_launch");
    return ok();
}

ssd_status ssd_decode_graph_destroy(ssd_decode_graph *graph) {
    if (!graph) return ok();
    cudaError_t e1 = cudaGraphExecDestroy(graph->exec);
    cudaError_t e2 = cudaGraphDestroy(graph->graph);
    delete graph;
    if (e1 != cudaSuccess) return cuda_fail(e1, "ssd_decode_graph_destroy");
    if (e2 != cudaSuccess) return cuda_fail(e2, "ssd_decode_graph_destroy");
    return ok();
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

ssd_status ssd_debug_bounds_status(int *site, int64_t *index, int clear) {
#ifndef SSD_DEBUG_BOUNDS
    (void)site;
    (void)index;
    (void)clear;
    return fail(SSD_ERR_UNSUPPORTED, "this library was built without SSD_DEBUG_BOUNDS: no bounds checks run");
#else
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "ssd_debug_bounds_status: synchronize");
    cudaError_t (*readers[])(unsigned long long *, bool) = {ssd::bounds_word_decode, ssd::bounds_word_diag,
                                                            ssd::bounds_word_fused, ssd::bounds_word_simt};
    unsigned long long first = 0;
    for (auto rd : readers) {
        unsigned long long w = 0;
        if ((e = rd(&w, clear != 0)) != cudaSuccess) return cuda_fail(e, "ssd_debug_bounds_status: read");
        if (!first) first = w;
    }
    if (!first) {
        if (site) *site = 0;
        if (index) *index = -1;
        return ok();
    }
    const int st = (int)((first >> 48) & 0xff);
    const int64_t idx = (int64_t)(first & 0xffffffffffffull);
    if (site) *site = st;
    if (index) *index = idx;
    return fail(SSD_ERR_BOUNDS, "bounds check failed at site %d, element %lld", st, (long long)idx);
#endif
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
