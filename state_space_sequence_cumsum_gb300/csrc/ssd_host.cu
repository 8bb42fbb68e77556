// ssd_fwd_host: the SSD forward from host memory to host memory, with the
// host <-> device copies overlapped with the computation.
//
// The sequence is cut into parts of whole chunks.  Each part runs the same
// forward as ssd_fwd on its own tokens, starting from the state the previous
// part ended with ("Kernel 2: fwd_pass_state" carries the state across chunk
// boundaries, so cutting at a chunk boundary and carrying the state computes
// the same function).  Part k's inputs go up on a copy stream while part k-1
// computes and part k-2's output comes down on a second copy stream: the two
// copy directions and the kernels run at the same time.  Two slots of device
// buffers alternate between parts.
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kTargetParts = 4;
constexpr int64_t kMinPartTokens = 512;

// Copy streams and events of one device, made on first use and kept.
struct HostPipe {
    bool ready = false;
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t entry = nullptr, done = nullptr, in[2] = {}, comp[2] = {}, out[2] = {};
};
std::mutex g_pipe_mu;  // one pipelined call issues at a time (the events are shared)
HostPipe g_pipe[kMaxDevices];

cudaError_t pipe_for_device(HostPipe **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    HostPipe &p = g_pipe[dev];
    if (!p.ready) {
        const unsigned ef = cudaEventDisableTiming;
        if ((e = cudaStreamCreateWithFlags(&p.up, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&p.down, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&p.entry, ef)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&p.done, ef)) != cudaSuccess)
            return e;
        for (int s = 0; s < 2; ++s)
            if ((e = cudaEventCreateWithFlags(&p.in[s], ef)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&p.comp[s], ef)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&p.out[s], ef)) != cudaSuccess)
                return e;
        p.ready = true;
    }
    *out = &p;
    return cudaSuccess;
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// The parts and the device workspace they need.
struct HostPlan {
    int T = 0, n_parts = 0;
    int64_t Lp = 0;  // tokens per part (the last part may be shorter)
    size_t esz = 0;
    // byte offsets in the workspace
    size_t off_A = 0, off_D = 0, off_st[2] = {}, off_slot[2] = {}, off_fws = 0;
    // within a slot
    size_t off_x = 0, off_dt = 0, off_b = 0, off_c = 0, off_y = 0;
    size_t fws_bytes = 0, bytes = 0;
};

ssd_status_t make_host_plan(const ssd_dims_t &d, ssd_dtype_t dtype, int chunk_size, HostPlan *pl)
{
    if (dtype != SSD_BF16 && dtype != SSD_F32)
        return SSD_ERR_INVALID_ARG;
    if (d.batch < 1 || d.seqlen < 0 || d.nheads < 1 || d.headdim < 1 || d.dstate < 1 ||
        d.ngroups < 1 || chunk_size < 0 || chunk_size > 256)
        return SSD_ERR_INVALID_ARG;
    HostPlan p;
    p.esz = dtype == SSD_BF16 ? 2 : 4;
    p.T = chunk_size ? chunk_size : chunk_size_peek(d, dtype);
    if (p.T <= 0)
        return SSD_ERR_INVALID_ARG;
    const int64_t L = d.seqlen;
    // parts of whole chunks, about kTargetParts of them, none shorter than
    // kMinPartTokens unless the sequence itself is
    int64_t per = (L + kTargetParts - 1) / kTargetParts;
    if (per < kMinPartTokens)
        per = kMinPartTokens;
    p.Lp = L > 0 ? (per + p.T - 1) / p.T * p.T : p.T;
    p.n_parts = L > 0 ? (int)((L + p.Lp - 1) / p.Lp) : 0;
    const int64_t lens[2] = {p.Lp, L - (int64_t)(p.n_parts - 1) * p.Lp};
    for (int k = 0; k < 2; ++k) {
        if (lens[k] <= 0 || p.n_parts == 0)
            continue;
        ssd_dims_t dp = d;
        dp.seqlen = lens[k];
        const size_t w = ssd_fwd_workspace_size(dp, dtype, p.T, 0);
        if (w == 0)
            return SSD_ERR_INVALID_ARG;
        if (w > p.fws_bytes)
            p.fws_bytes = w;
    }
    const size_t B = (size_t)d.batch, H = (size_t)d.nheads, P = (size_t)d.headdim,
                 S = (size_t)d.dstate, G = (size_t)d.ngroups, Lp = (size_t)p.Lp;
    const size_t state = B * H * P * S * 4;
    size_t off = 0;
    p.off_A = off;
    off = up256(off + H * 4);
    p.off_D = off;
    off = up256(off + H * 4);
    for (int s = 0; s < 2; ++s) {
        p.off_st[s] = off;
        off = up256(off + state);
    }
    p.off_x = 0;
    size_t so = up256(B * Lp * H * P * p.esz);
    p.off_dt = so;
    so = up256(so + B * Lp * H * 4);
    p.off_b = so;
    so = up256(so + B * Lp * G * S * p.esz);
    p.off_c = so;
    so = up256(so + B * Lp * G * S * p.esz);
    p.off_y = so;
    so = up256(so + B * Lp * H * P * p.esz);
    for (int s = 0; s < 2; ++s) {
        p.off_slot[s] = off;
        off += so;
    }
    p.off_fws = off;
    off = up256(off + p.fws_bytes);
    p.bytes = off;
    *pl = p;
    return SSD_OK;
}

// rows of `width` bytes, one per batch row, `spitch` / `dpitch` apart
cudaError_t copy_rows(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width,
                      size_t rows, cudaMemcpyKind kind, cudaStream_t st)
{
    if (width == 0 || rows == 0)
        return cudaSuccess;
    if (rows == 1 || (dpitch == width && spitch == width))
        return cudaMemcpyAsync(dst, src, width * rows, kind, st);
    constexpr size_t kMaxPitch = (size_t(1) << 31) - 1;  // beyond it: one copy per row
    if (dpitch <= kMaxPitch && spitch <= kMaxPitch)
        return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, st);
    for (size_t r = 0; r < rows; ++r) {
        const cudaError_t e = cudaMemcpyAsync(static_cast<char *>(dst) + r * dpitch,
                                              static_cast<const char *>(src) + r * spitch, width, kind, st);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

size_t ssd_fwd_host_workspace_size(ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size)
{
    HostPlan p;
    if (make_host_plan(dims, dtype, chunk_size, &p) != SSD_OK)
        return 0;
    return p.bytes;
}

ssd_status_t ssd_fwd_host(const void *x, const float *dt, const float *A, const void *Bm,
                          const void *Cm, const float *D, const float *init_state, void *y,
                          float *final_state, ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size,
                          void *workspace, size_t workspace_bytes, void *stream)
{
    HostPlan pl;
    ssd_status_t s0 = make_host_plan(dims, dtype, chunk_size, &pl);
    if (s0 != SSD_OK)
        return s0;
    const bool ne = dims.seqlen > 0;
    if ((ne && (!x || !dt || !Bm || !Cm || !y)) || !A || !D)
        return SSD_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < pl.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return SSD_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    const size_t B = (size_t)dims.batch, H = (size_t)dims.nheads, P = (size_t)dims.headdim,
                 S = (size_t)dims.dstate, G = (size_t)dims.ngroups, L = (size_t)dims.seqlen;
    const size_t state_bytes = B * H * P * S * 4;
    float *A_d = reinterpret_cast<float *>(ws + pl.off_A);
    float *D_d = reinterpret_cast<float *>(ws + pl.off_D);
    float *st_d[2] = {reinterpret_cast<float *>(ws + pl.off_st[0]),
                      reinterpret_cast<float *>(ws + pl.off_st[1])};

    std::lock_guard<std::mutex> lk(g_pipe_mu);
    HostPipe *pp = nullptr;
    cudaError_t e = pipe_for_device(&pp);
    if (e != cudaSuccess)
        return SSD_ERR_CUDA;
    // On a failure after work was issued, `stream` still waits for the copy
    // streams before the error is returned, so the caller's stream order
    // covers every copy that did start.
    auto join = [&]() {
        if (cudaEventRecord(pp->done, pp->up) == cudaSuccess)
            cudaStreamWaitEvent(st, pp->done, 0);
        if (cudaEventRecord(pp->done, pp->down) == cudaSuccess)
            cudaStreamWaitEvent(st, pp->done, 0);
    };
#define HOST_TRY(expr)                  \
    do {                                \
        if ((expr) != cudaSuccess) {    \
            join();                     \
            return SSD_ERR_CUDA;        \
        }                               \
    } while (0)
    // everything already on `stream` comes first
    HOST_TRY(cudaEventRecord(pp->entry, st));
    HOST_TRY(cudaStreamWaitEvent(pp->up, pp->entry, 0));
    HOST_TRY(cudaStreamWaitEvent(pp->down, pp->entry, 0));
    HOST_TRY(cudaMemcpyAsync(A_d, A, H * 4, cudaMemcpyHostToDevice, pp->up));
    HOST_TRY(cudaMemcpyAsync(D_d, D, H * 4, cudaMemcpyHostToDevice, pp->up));
    // part 0 starts from st_d[1] (the initial state, or zeros)
    if (init_state)
        HOST_TRY(cudaMemcpyAsync(st_d[1], init_state, state_bytes, cudaMemcpyHostToDevice, pp->up));
    else if (!ne)
        HOST_TRY(cudaMemsetAsync(st_d[1], 0, state_bytes, pp->up));

    const size_t rx = H * P * pl.esz, rdt = H * 4, rbc = G * S * pl.esz;  // bytes per token
    const char *xh = static_cast<const char *>(x), *dth = reinterpret_cast<const char *>(dt);
    const char *bh = static_cast<const char *>(Bm), *ch = static_cast<const char *>(Cm);
    char *yh = static_cast<char *>(y);
    int last_slot = 1;
    for (int k = 0; k < pl.n_parts; ++k) {
        const int s = k & 1;
        const size_t l0 = (size_t)k * (size_t)pl.Lp;
        const size_t lk = (size_t)((int64_t)L - (int64_t)l0 < pl.Lp ? (int64_t)L - (int64_t)l0 : pl.Lp);
        char *slot = ws + pl.off_slot[s];
        // slot s is free once part k-2's output has come down
        if (k >= 2)
            HOST_TRY(cudaStreamWaitEvent(pp->up, pp->out[s], 0));
        HOST_TRY(copy_rows(slot + pl.off_x, lk * rx, xh + l0 * rx, L * rx, lk * rx, B,
                           cudaMemcpyHostToDevice, pp->up));
        HOST_TRY(copy_rows(slot + pl.off_dt, lk * rdt, dth + l0 * rdt, L * rdt, lk * rdt, B,
                           cudaMemcpyHostToDevice, pp->up));
        HOST_TRY(copy_rows(slot + pl.off_b, lk * rbc, bh + l0 * rbc, L * rbc, lk * rbc, B,
                           cudaMemcpyHostToDevice, pp->up));
        HOST_TRY(copy_rows(slot + pl.off_c, lk * rbc, ch + l0 * rbc, L * rbc, lk * rbc, B,
                           cudaMemcpyHostToDevice, pp->up));
        HOST_TRY(cudaEventRecord(pp->in[s], pp->up));
        HOST_TRY(cudaStreamWaitEvent(st, pp->in[s], 0));
        ssd_dims_t dp = dims;
        dp.seqlen = (int64_t)lk;
        const float *init_k = k == 0 ? (init_state ? st_d[1] : nullptr) : st_d[(k - 1) & 1];
        const ssd_status_t sk =
            ssd_fwd(slot + pl.off_x, reinterpret_cast<const float *>(slot + pl.off_dt), A_d,
                    slot + pl.off_b, slot + pl.off_c, D_d, init_k, slot + pl.off_y, st_d[k & 1],
                    nullptr, dp, dtype, pl.T, ws + pl.off_fws, pl.fws_bytes, st);
        if (sk != SSD_OK) {
            join();
            return sk;
        }
        HOST_TRY(cudaEventRecord(pp->comp[s], st));
        HOST_TRY(cudaStreamWaitEvent(pp->down, pp->comp[s], 0));
        HOST_TRY(copy_rows(yh + l0 * rx, L * rx, slot + pl.off_y, lk * rx, lk * rx, B,
                           cudaMemcpyDeviceToHost, pp->down));
        HOST_TRY(cudaEventRecord(pp->out[s], pp->down));
        last_slot = k & 1;
    }
    if (final_state) {
        // after the last part's computation (the down stream waited for it),
        // or the initial state / zeros when there are no tokens
        if (!ne) {
            HOST_TRY(cudaEventRecord(pp->in[0], pp->up));
            HOST_TRY(cudaStreamWaitEvent(pp->down, pp->in[0], 0));
        }
        HOST_TRY(cudaMemcpyAsync(final_state, st_d[ne ? last_slot : 1], state_bytes,
                                 cudaMemcpyDeviceToHost, pp->down));
    }
    // the caller's stream waits for both copy streams
    if (cudaEventRecord(pp->done, pp->up) != cudaSuccess ||
        cudaStreamWaitEvent(st, pp->done, 0) != cudaSuccess ||
        cudaEventRecord(pp->done, pp->down) != cudaSuccess ||
        cudaStreamWaitEvent(st, pp->done, 0) != cudaSuccess)
        return SSD_ERR_CUDA;
#undef HOST_TRY
    return SSD_OK;
}

}  // extern "C"
