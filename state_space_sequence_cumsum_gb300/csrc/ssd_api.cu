// C ABI of the SSD forward library: argument validation, workspace layout,
// stage orchestration and the kernel status word.  See include/ssd.h for the
// contract of every entry point.
#include <algorithm>
#include <atomic>
#include <initializer_list>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>

#include "common.cuh"
#include "ssd_internal.h"

namespace ssd {

// Kernel-side error word.  Kernels OR bit 0 into it when a bounded wait runs
// out; ssd_stream_status() reads and clears it.
__device__ unsigned int g_ssd_status_word;

namespace {
std::atomic<uint64_t> g_launches{0};
}  // namespace

void note_launch(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int *g_status_addr[kMaxDevices];
}  // namespace

unsigned int *device_status_word()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ssd_status_word) != cudaSuccess)
            return nullptr;
        g_status_addr[dev] = static_cast<unsigned int *>(p);
    }
    return g_status_addr[dev];
}

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validates dims and chunk size; fills g.  T == 0 is accepted only when
// allow_auto (ssd_fwd), and then g.T stays 0 for the caller to choose.
ssd_status_t make_geom(const ssd_dims_t &d, int T, bool allow_auto, Geom *g)
{
    if (d.batch < 1 || d.seqlen < 0 || d.nheads < 1 || d.headdim < 1 || d.dstate < 1 ||
        d.ngroups < 1)
        return SSD_ERR_INVALID_ARG;
    if (d.nheads % d.ngroups != 0)
        return SSD_ERR_INVALID_ARG;
    if (T < 0 || (T == 0 && !allow_auto))
        return SSD_ERR_INVALID_ARG;
    if (T > 256 || d.headdim > 256 || d.dstate > 512 || d.batch > 65535 ||
        d.batch * d.nheads > 65535LL * 64 || d.seqlen > (1LL << 40))
        return SSD_ERR_UNSUPPORTED;
    // keep every element count far from int64 overflow
    const double elems = (double)d.batch * (double)d.seqlen * (double)d.nheads * (double)d.headdim;
    const double st = (double)d.batch * d.nheads * d.headdim * d.dstate *
                      (double)((d.seqlen + (T ? T : 64) - 1) / (T ? T : 64) + 1);
    if (elems > 4e15 || st > 4e15)
        return SSD_ERR_UNSUPPORTED;
    g->B = d.batch;
    g->L = d.seqlen;
    g->H = d.nheads;
    g->P = d.headdim;
    g->S = d.dstate;
    g->G = d.ngroups;
    g->T = T;
    g->nc = T ? (d.seqlen + T - 1) / T : 0;
    g->hpg = (int)(d.nheads / d.ngroups);
    return SSD_OK;
}

// A required pointer may be NULL only when the tensor it names is empty.
ssd_status_t need(const void *p, bool nonempty)
{
    if (!p)
        return nonempty ? SSD_ERR_INVALID_ARG : SSD_OK;
    return aligned16(p) ? SSD_OK : SSD_ERR_ALIGNMENT;
}

ssd_status_t opt(const void *p) { return (!p || aligned16(p)) ? SSD_OK : SSD_ERR_ALIGNMENT; }

// A required pointer aligned to its element size.
ssd_status_t need_elem(const void *p, size_t esz)
{
    if (!p)
        return SSD_ERR_INVALID_ARG;
    return (reinterpret_cast<uintptr_t>(p) % esz == 0) ? SSD_OK : SSD_ERR_ALIGNMENT;
}

#define SSD_TRY(expr)                                  \
    do {                                               \
        ssd_status_t _s = (expr);                      \
        if (_s != SSD_OK)                              \
            return _s;                                 \
    } while (0)

ssd_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Stage 3 dispatch: tcgen05 kernel for bf16 shapes it serves, else CUDA cores.
cudaError_t run_chunk_out(const void *x, const void *Bm, const void *Cm, const float *dtT,
                          const float *Gc, const float *states, const float *D, void *y,
                          const Geom &g, bool bf16, cudaStream_t st)
{
    if (bf16 && chunk_tc_supported(g))
        return launch_chunk_out_tc(x, Bm, Cm, dtT, Gc, states, D, y, g, st);
    if (bf16 && chunk_out_big_supported(g))
        return launch_chunk_out_big(x, Bm, Cm, dtT, Gc, states, D, y, g, st);
    return launch_chunk_out_simt(x, Bm, Cm, dtT, Gc, states, D, y, g, bf16, st);
}

// ssd_fwd's choice of kernels.  SSD_FWD_PATH=staged|fused overrides the
// default for the tensor-core shapes (a debugging / measurement switch).
ssd_path_t choose_path(const Geom &g, ssd_dtype_t t, bool want_states)
{
    if (t != SSD_BF16 || !fused_tc_supported(g))
        return (t == SSD_BF16 && state_pass_tc_supported(g)) ? SSD_PATH_STAGED_TENSOR_CORES
                                                             : SSD_PATH_STAGED_CUDA_CORES;
    const char *env = getenv("SSD_FWD_PATH");
    if (env && strcmp(env, "staged") == 0)
        return SSD_PATH_STAGED_TENSOR_CORES;
    // dstate 384 / 512 with every chunk state asked for: the staged path's
    // state pass writes them as part of its work, and there it is the faster
    // one (B 1, L 262144, H 32, S 512: 4.98 ms staged, 5.20 ms fused)
    const bool force_fused = env && strcmp(env, "fused") == 0;
    if (want_states && !force_fused && !chunk_tc_supported(g) && state_pass_tc_supported(g) &&
        chunk_out_big_supported(g))
        return SSD_PATH_STAGED_TENSOR_CORES;
    return fused_pair_enabled(g) ? SSD_PATH_FUSED_PAIR_TENSOR_CORES : SSD_PATH_FUSED_TENSOR_CORES;
}

// Stage 2 dispatch: tcgen05 kernel for bf16 shapes it serves (split into
// parallel segments when the (batch, head) units cannot fill the GPU), else
// CUDA cores.  SSD_STATE_PASS=plain keeps the unsplit pass (a measurement and
// test switch).
cudaError_t run_state_pass(const void *x, const void *Bm, const float *dtT, const float *Gc,
                           const float *init, float *states, float *final_state, const Geom &g,
                           bool bf16, cudaStream_t st)
{
    if (bf16 && state_pass_tc_supported(g)) {
        const char *env = getenv("SSD_STATE_PASS");
        if (states && !(env && strcmp(env, "plain") == 0)) {
            const cudaError_t e =
                launch_state_pass_tc_segmented(x, Bm, dtT, Gc, init, states, final_state, g, st);
            if (e != cudaErrorNotSupported)
                return e;
        }
        return launch_state_pass_tc(x, Bm, dtT, Gc, init, states, final_state, g, st);
    }
    return launch_state_pass_simt(x, Bm, dtT, Gc, init, states, final_state, g, bf16, st);
}

// The chunk size used for chunk_size == 0 before (or instead of) timing.
// bf16: the tensor-core kernels walk 128-token tiles; 128 keeps the chunk
// states (when requested) as fine as the tiles.  f32: short chunks keep the
// CUDA-core score tile small.
int static_chunk_size(const Geom &g, ssd_dtype_t t)
{
    if (t == SSD_BF16)
        return 128;
    return g.L <= 64 ? 64 : 128;
}

// ---------------------------------------------------------------------------
// chunk_size == 0: the per-shape choice ("Accelerating Mamba-2 forward-pass
// kernels with CUDA Tile (cuTile)", section "Mamba-2 性能优化": the best
// configuration is searched per shape).  The candidates are the chunk sizes
// {64, 128, 256} and, on the head-pair path where the prefilled-segment plan
// applies, that plan or the hand-off plan.  A choice is fixed once per
// (B, L, H, P, S, G, dtype) and process, by whichever comes first:
//   * the first ssd_fwd(chunk_size = 0) call without chunk states, outside
//     stream capture and with no output overlapping an input: it runs every
//     candidate whose workspace fits the one passed (once untimed, then twice
//     between CUDA events on the caller's stream, keeping the faster time) and
//     keeps the fastest; a candidate must beat the current best by 2% to
//     replace it, so near-ties keep the static choice;
//   * ssd_fwd_chosen_chunk_size, or any other ssd_fwd(chunk_size = 0) call:
//     the static choice above.
// The choice never changes afterwards, so a caller can size chunk_states from
// ssd_fwd_chosen_chunk_size.  The cache is guarded by a mutex; two threads
// tuning one shape at once both time it and the first to finish wins.
struct TuneKey {
    int64_t B, L, H, P, S, G;
    int dtype;
    bool operator<(const TuneKey &o) const
    {
        const int64_t a[7] = {B, L, H, P, S, G, dtype}, b[7] = {o.B, o.L, o.H, o.P, o.S, o.G, o.dtype};
        return std::lexicographical_compare(a, a + 7, b, b + 7);
    }
};
struct TuneChoice {
    int T;
    bool allow_prefill;  // head-pair path: the prefilled plan where it applies
    bool timed;
};
std::mutex g_tune_mu;
std::map<TuneKey, TuneChoice> g_tune;

TuneKey tune_key(const Geom &g, ssd_dtype_t t) { return TuneKey{g.B, g.L, g.H, g.P, g.S, g.G, (int)t}; }

bool tune_lookup(const Geom &g, ssd_dtype_t t, TuneChoice *c)
{
    std::lock_guard<std::mutex> lk(g_tune_mu);
    const auto it = g_tune.find(tune_key(g, t));
    if (it == g_tune.end())
        return false;
    *c = it->second;
    return true;
}

// Fixes c unless a choice is already there; returns the one that stands.
TuneChoice tune_fix(const Geom &g, ssd_dtype_t t, const TuneChoice &c)
{
    std::lock_guard<std::mutex> lk(g_tune_mu);
    return g_tune.emplace(tune_key(g, t), c).first->second;
}

// The current choice without fixing it: the cached one, else the static one.
TuneChoice tune_peek(const Geom &g, ssd_dtype_t t)
{
    TuneChoice c;
    if (tune_lookup(g, t, &c))
        return c;
    return TuneChoice{static_chunk_size(g, t), true, false};
}

Geom with_chunk(const Geom &g0, int T)
{
    Geom g = g0;
    g.T = T;
    g.nc = (g.L + T - 1) / T;
    return g;
}

struct Workspace {
    float *Gc, *dtT, *states;
    char *fused_scratch;
    size_t fused_scratch_bytes;
    size_t bytes;      // what ssd_fwd_workspace_size reports
    size_t min_bytes;  // the least the call runs with (head pairs: the hand-off plan)
};

// ssd_fwd's workspace: G_cum and dt_t, then either the chunk states the
// staged path keeps between stages (when the caller does not want them) or
// the fused path's segment hand-off scratch.  The head-pair fused path forms
// G itself and needs only its hand-off scratch.
Workspace layout(const Geom &g, ssd_path_t path, bool caller_states, char *base)
{
    const size_t bhl = (size_t)(g.B * g.H * g.L) * sizeof(float);
    size_t off = 0;
    Workspace w{};
    if (path == SSD_PATH_FUSED_PAIR_TENSOR_CORES) {
        w.fused_scratch_bytes = pair_tc_scratch_bytes(g);
        w.fused_scratch = base;
        w.bytes = round_up(w.fused_scratch_bytes, 256);
        // the hand-off plan's scratch may be the smaller one or not (it has
        // more segments, but no G / dt^T)
        w.min_bytes = std::min(w.bytes, round_up(pair_tc_scratch_bytes(g, false), 256));
        if (!base)
            w.fused_scratch = nullptr;
        return w;
    }
    const bool fused = path == SSD_PATH_FUSED_TENSOR_CORES;
    w.Gc = reinterpret_cast<float *>(base + off);
    off = round_up(off + bhl, 256);
    w.dtT = reinterpret_cast<float *>(base + off);
    off = round_up(off + bhl, 256);
    if (fused) {
        w.fused_scratch_bytes = fused_tc_scratch_bytes(g);
        w.fused_scratch = base + off;
        off = round_up(off + w.fused_scratch_bytes, 256);
    } else if (!caller_states) {
        w.states = reinterpret_cast<float *>(base + off);
        off = round_up(off + (size_t)(g.B * g.H * g.nc * g.P * g.S) * sizeof(float), 256);
    }
    w.bytes = off;
    w.min_bytes = off;
    if (!base) {
        w.Gc = w.dtT = w.states = nullptr;
        w.fused_scratch = nullptr;
    }
    return w;
}

// Workspace of ssd_bwd: G and dt^T [B,H,L], the forward chunk states and
// their gradients [B,H,nc,P,S], the dB / dC f32 accumulators [B,L,G,S].
struct BwdWs {
    float *Gc, *dtT, *states, *dstates, *dB, *dC;
    size_t bytes;
};
BwdWs bwd_layout(const Geom &g, char *base)
{
    BwdWs w{};
    size_t off = 0;
    auto take = [&](size_t n) {
        char *p = base ? base + off : nullptr;
        off += round_up(n * sizeof(float), 256);
        return reinterpret_cast<float *>(p);
    };
    w.Gc = take((size_t)(g.B * g.H * g.L));
    w.dtT = take((size_t)(g.B * g.H * g.L));
    w.states = take((size_t)(g.B * g.H * g.nc * g.P * g.S));
    w.dstates = take((size_t)(g.B * g.H * g.nc * g.P * g.S));
    w.dB = take((size_t)(g.B * g.L * g.G * g.S));
    w.dC = take((size_t)(g.B * g.L * g.G * g.S));
    w.bytes = off;
    return w;
}
}  // namespace

// The least workspace ssd_fwd runs with for these arguments (0: invalid).
size_t fwd_workspace_min_size(ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size,
                              int want_chunk_states)
{
    Geom g;
    if (make_geom(dims, chunk_size, true, &g) != SSD_OK)
        return 0;
    if (dtype != SSD_BF16 && dtype != SSD_F32)
        return 0;
    if (g.T == 0)
        g = with_chunk(g, tune_peek(g, dtype).T);
    const size_t b = layout(g, choose_path(g, dtype, want_chunk_states != 0),
                            want_chunk_states != 0, nullptr).min_bytes;
    return b ? b : 256;
}

int chunk_size_peek(ssd_dims_t dims, ssd_dtype_t dtype)
{
    Geom g;
    if (make_geom(dims, 0, true, &g) != SSD_OK || (dtype != SSD_BF16 && dtype != SSD_F32))
        return 0;
    return tune_peek(g, dtype).T;
}

}  // namespace ssd

using namespace ssd;

extern "C" {

uint64_t ssd_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *ssd_status_string(ssd_status_t s)
{
    switch (s) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID_ARG: return "invalid argument";
    case SSD_ERR_UNSUPPORTED: return "unsupported size";
    case SSD_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case SSD_ERR_CUDA: return "CUDA error";
    case SSD_ERR_TIMEOUT: return "device-side wait timed out";
    case SSD_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

ssd_status_t ssd_chunk_cumsum(const float *dt, const float *A, float *G_cum, float *dt_t,
                              ssd_dims_t dims, int chunk_size, void *stream)
{
    Geom g;
    SSD_TRY(make_geom(dims, chunk_size, false, &g));
    const bool ne = g.L > 0;
    SSD_TRY(need(dt, ne));
    SSD_TRY(need(A, true));
    SSD_TRY(need(G_cum, ne));
    SSD_TRY(opt(dt_t));
    return cuda_status(launch_chunk_cumsum(dt, A, G_cum, dt_t, g, (cudaStream_t)stream));
}

ssd_status_t ssd_state_pass(const void *x, const void *Bm, const float *dt_t, const float *G_cum,
                            const float *init_state, float *chunk_states, float *final_state,
                            ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size, void *stream)
{
    Geom g;
    SSD_TRY(make_geom(dims, chunk_size, false, &g));
    if (dtype != SSD_BF16 && dtype != SSD_F32)
        return SSD_ERR_INVALID_ARG;
    const bool ne = g.L > 0;
    SSD_TRY(need(x, ne));
    SSD_TRY(need(Bm, ne));
    SSD_TRY(need(dt_t, ne));
    SSD_TRY(need(G_cum, ne));
    SSD_TRY(opt(init_state));
    SSD_TRY(opt(chunk_states));
    SSD_TRY(opt(final_state));
    cudaStream_t st = (cudaStream_t)stream;
    if (g.L == 0) {
        if (!final_state)
            return SSD_OK;
        const size_t bytes = (size_t)(g.B * g.H * g.P * g.S) * sizeof(float);
        return cuda_status(init_state
                               ? cudaMemcpyAsync(final_state, init_state, bytes,
                                                 cudaMemcpyDeviceToDevice, st)
                               : cudaMemsetAsync(final_state, 0, bytes, st));
    }
    return cuda_status(run_state_pass(x, Bm, dt_t, G_cum, init_state, chunk_states, final_state,
                                      g, dtype == SSD_BF16, st));
}

ssd_status_t ssd_chunk_out(const void *x, const void *Bm, const void *Cm, const float *dt_t,
                           const float *G_cum, const float *chunk_states, const float *D, void *y,
                           ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size, void *stream)
{
    Geom g;
    SSD_TRY(make_geom(dims, chunk_size, false, &g));
    if (dtype != SSD_BF16 && dtype != SSD_F32)
        return SSD_ERR_INVALID_ARG;
    const bool ne = g.L > 0;
    SSD_TRY(need(x, ne));
    SSD_TRY(need(Bm, ne));
    SSD_TRY(need(Cm, ne));
    SSD_TRY(need(dt_t, ne));
    SSD_TRY(need(G_cum, ne));
    SSD_TRY(need(chunk_states, ne));
    SSD_TRY(need(D, true));
    SSD_TRY(need(y, ne));
    if (!ne)
        return SSD_OK;
    return cuda_status(run_chunk_out(x, Bm, Cm, dt_t, G_cum, chunk_states, D, y, g,
                                     dtype == SSD_BF16, (cudaStream_t)stream));
}

size_t ssd_state_out_workspace_size(ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size)
{
    Geom g;
    if (make_geom(dims, chunk_size, false, &g) != SSD_OK || (dtype != SSD_BF16 && dtype != SSD_F32))
        return 0;
    const size_t b = (dtype == SSD_BF16 && fused_tc_supported(g)) ? fused_tc_scratch_bytes(g) : 0;
    return b ? b : 256;
}

ssd_status_t ssd_state_out(const void *x, const void *Bm, const void *Cm, const float *dt_t,
                           const float *G_cum, const float *D, const float *init_state, void *y,
                           float *final_state, float *chunk_states, ssd_dims_t dims,
                           ssd_dtype_t dtype, int chunk_size, void *workspace,
                           size_t workspace_bytes, void *stream)
{
    Geom g;
    SSD_TRY(make_geom(dims, chunk_size, false, &g));
    if (dtype != SSD_BF16 && dtype != SSD_F32)
        return SSD_ERR_INVALID_ARG;
    const bool ne = g.L > 0;
    SSD_TRY(need(x, ne));
    SSD_TRY(need(Bm, ne));
    SSD_TRY(need(Cm, ne));
    SSD_TRY(need(dt_t, ne));
    SSD_TRY(need(G_cum, ne));
    SSD_TRY(need(D, true));
    SSD_TRY(need(y, ne));
    SSD_TRY(opt(init_state));
    SSD_TRY(opt(final_state));
    SSD_TRY(opt(chunk_states));
    if (!ne)
        return ssd_state_pass(x, Bm, dt_t, G_cum, init_state, chunk_states, final_state, dims,
                              dtype, chunk_size, stream);
    if (dtype != SSD_BF16 || !fused_tc_supported(g))
        return SSD_ERR_UNSUPPORTED;
    const size_t need_ws = fused_tc_scratch_bytes(g);
    if (need_ws && (!workspace || workspace_bytes < need_ws ||
                    (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return SSD_ERR_WORKSPACE;
    return cuda_status(launch_fused_tc(x, Bm, Cm, dt_t, G_cum, D, init_state, chunk_states,
                                       final_state, y, g, workspace, workspace_bytes,
                                       (cudaStream_t)stream));
}

ssd_path_t ssd_fwd_path(ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size, int want_chunk_states)
{
    Geom g;
    if (make_geom(dims, chunk_size, true, &g) != SSD_OK ||
        (dtype != SSD_BF16 && dtype != SSD_F32))
        return SSD_PATH_INVALID;
    if (g.T == 0)
        g = with_chunk(g, tune_peek(g, dtype).T);
    return choose_path(g, dtype, want_chunk_states != 0);
}

int ssd_fwd_chosen_chunk_size(ssd_dims_t dims, ssd_dtype_t dtype)
{
    Geom g;
    if (make_geom(dims, 0, true, &g) != SSD_OK || (dtype != SSD_BF16 && dtype != SSD_F32))
        return 0;
    return tune_fix(g, dtype, tune_peek(g, dtype)).T;
}

int ssd_fwd_chunk_size_was_timed(ssd_dims_t dims, ssd_dtype_t dtype)
{
    Geom g;
    TuneChoice c;
    if (make_geom(dims, 0, true, &g) != SSD_OK || (dtype != SSD_BF16 && dtype != SSD_F32) ||
        !tune_lookup(g, dtype, &c))
        return 0;
    return c.timed ? 1 : 0;
}

size_t ssd_fwd_workspace_size(ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size,
                              int want_chunk_states)
{
    Geom g;
    if (make_geom(dims, chunk_size, true, &g) != SSD_OK)
        return 0;
    if (dtype != SSD_BF16 && dtype != SSD_F32)
        return 0;
    const bool ws = want_chunk_states != 0;
    TuneChoice c;
    if (g.T == 0 && !ws && !tune_lookup(g, dtype, &c)) {
        // not fixed yet: room for every candidate the tuner may time, leaving
        // out CUDA-core candidates where another candidate runs on tensor cores
        // (they cannot win, and the staged CUDA-core path keeps every chunk
        // state in the workspace)
        size_t b_tc = 0, b_all = 0;
        for (int T : {64, 128, 256}) {
            Geom gt;
            if (make_geom(dims, T, false, &gt) != SSD_OK)
                continue;
            const ssd_path_t p = choose_path(gt, dtype, false);
            const size_t b = layout(gt, p, false, nullptr).bytes;
            b_all = std::max(b_all, b);
            if (p != SSD_PATH_STAGED_CUDA_CORES)
                b_tc = std::max(b_tc, b);
        }
        const size_t b = b_tc ? b_tc : b_all;
        return b ? b : 256;
    }
    if (g.T == 0)
        g = with_chunk(g, tune_peek(g, dtype).T);
    const size_t b = layout(g, choose_path(g, dtype, ws), ws, nullptr).bytes;
    return b ? b : 256;
}

}  // extern "C"

namespace ssd {
namespace {

struct FwdArgs {
    const void *x;
    const float *dt, *A;
    const void *Bm, *Cm;
    const float *D, *init_state;
    void *y;
    float *final_state, *chunk_states;
    ssd_dims_t dims;
    ssd_dtype_t dtype;
    void *workspace;
    size_t workspace_bytes;
    cudaStream_t st;
};

// The forward with the chunk size fixed (g.T > 0); pointers already validated.
ssd_status_t fwd_impl(const FwdArgs &a, const Geom &g, bool allow_prefill)
{
    const bool ne = g.L > 0;
    if (!ne)
        return ssd_state_pass(a.x, a.Bm, nullptr, nullptr, a.init_state, a.chunk_states,
                              a.final_state, a.dims, a.dtype, g.T, a.st);
    const ssd_path_t path = choose_path(g, a.dtype, a.chunk_states != nullptr);
    const bool fused = path == SSD_PATH_FUSED_TENSOR_CORES;
    const Workspace need_ws = layout(g, path, a.chunk_states != nullptr, nullptr);
    if (need_ws.min_bytes && (!a.workspace || a.workspace_bytes < need_ws.min_bytes ||
                              (reinterpret_cast<uintptr_t>(a.workspace) & 255u)))
        return SSD_ERR_WORKSPACE;
    const Workspace w = layout(g, path, a.chunk_states != nullptr, static_cast<char *>(a.workspace));
    // the head-pair kernel takes the plan the whole workspace holds
    if (path == SSD_PATH_FUSED_PAIR_TENSOR_CORES)
        return cuda_status(launch_fused_pair_tc(a.x, a.Bm, a.Cm, a.dt, a.A, a.D, a.init_state,
                                                a.chunk_states, a.final_state, a.y, g,
                                                w.fused_scratch,
                                                a.workspace ? a.workspace_bytes : 0, a.st,
                                                allow_prefill));
    float *states = a.chunk_states ? a.chunk_states : w.states;
    const bool bf16 = a.dtype == SSD_BF16;

    SSD_TRY(cuda_status(launch_chunk_cumsum(a.dt, a.A, w.Gc, w.dtT, g, a.st)));
    if (fused)
        return cuda_status(launch_fused_tc(a.x, a.Bm, a.Cm, w.dtT, w.Gc, a.D, a.init_state,
                                           a.chunk_states, a.final_state, a.y, g, w.fused_scratch,
                                           w.fused_scratch_bytes, a.st));
    SSD_TRY(cuda_status(run_state_pass(a.x, a.Bm, w.dtT, w.Gc, a.init_state, states,
                                       a.final_state, g, bf16, a.st)));
    return cuda_status(run_chunk_out(a.x, a.Bm, a.Cm, w.dtT, w.Gc, states, a.D, a.y, g, bf16, a.st));
}

bool overlaps(const void *p, size_t np, const void *q, size_t nq)
{
    if (!p || !q || !np || !nq)
        return false;
    const char *a = static_cast<const char *>(p), *b = static_cast<const char *>(q);
    return a < b + nq && b < a + np;
}

// Repeated runs are harmless only when no output overlaps an input.
bool outputs_disjoint(const FwdArgs &a, const Geom &g)
{
    const size_t e = a.dtype == SSD_BF16 ? 2 : 4;
    const size_t nx = (size_t)(g.B * g.L * g.H * g.P) * e, nbc = (size_t)(g.B * g.L * g.G * g.S) * e;
    const size_t ndt = (size_t)(g.B * g.L * g.H) * 4, nh = (size_t)g.H * 4;
    const size_t nst = (size_t)(g.B * g.H * g.P * g.S) * 4;
    const void *in[7] = {a.x, a.dt, a.A, a.Bm, a.Cm, a.D, a.init_state};
    const size_t nin[7] = {nx, ndt, nh, nbc, nbc, nh, nst};
    const void *out[2] = {a.y, a.final_state};
    const size_t nout[2] = {nx, nst};
    for (int o = 0; o < 2; ++o)
        for (int i = 0; i < 7; ++i)
            if (overlaps(out[o], nout[o], in[i], nin[i]))
                return false;
    return !overlaps(a.y, nx, a.final_state, nst);
}

// Times every candidate (see the note at tune_key) and fixes the fastest.
TuneChoice tune_and_fix(const FwdArgs &a, const Geom &g0)
{
    const TuneChoice fallback{static_chunk_size(g0, a.dtype), true, false};
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        if (e0)
            cudaEventDestroy(e0);
        cudaGetLastError();
        return tune_fix(g0, a.dtype, fallback);
    }
    // the static choice first, so that near-ties keep it
    int order[3] = {fallback.T, 0, 0}, n_order = 1;
    for (int T : {64, 128, 256})
        if (T != fallback.T)
            order[n_order++] = T;
    float best = 0.f;
    TuneChoice best_c = fallback;
    bool have = false, failed = false;
    auto run_once = [&](const Geom &g, bool pre, float *ms) {
        if (cudaEventRecord(e0, a.st) != cudaSuccess)
            return false;
        if (fwd_impl(a, g, pre) != SSD_OK)
            return false;
        if (cudaEventRecord(e1, a.st) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess)
            return false;
        return cudaEventElapsedTime(ms, e0, e1) == cudaSuccess;
    };
    for (int k = 0; k < n_order && !failed; ++k) {
        Geom g;
        if (make_geom(a.dims, order[k], false, &g) != SSD_OK)
            continue;
        const ssd_path_t path = choose_path(g, a.dtype, false);
        if (layout(g, path, false, nullptr).min_bytes > (a.workspace ? a.workspace_bytes : 0))
            continue;
        // the hand-off plan as a second candidate where the prefilled one runs
        const bool two_plans = path == SSD_PATH_FUSED_PAIR_TENSOR_CORES &&
                               pair_tc_prefers_prefill(g) &&
                               a.workspace_bytes >= pair_tc_scratch_bytes(g, true) &&
                               a.workspace_bytes >= pair_tc_scratch_bytes(g, false);
        for (int pl = 0; pl < (two_plans ? 2 : 1); ++pl) {
            const bool pre = pl == 0;
            float t_warm = 0.f, t1 = 0.f, t2 = 0.f;
            if (!run_once(g, pre, &t_warm)) {
                failed = true;  // a launch failed: stop timing, keep what stands
                break;
            }
            if (have && t_warm > 1.5f * best)
                continue;  // far behind: not worth timing
            if (!run_once(g, pre, &t1) || !run_once(g, pre, &t2)) {
                failed = true;
                break;
            }
            const float t = std::min(t1, t2);
            if (!have || t < 0.98f * best) {
                best = t;
                best_c = TuneChoice{order[k], pre, true};
                have = true;
            }
        }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (failed)
        cudaGetLastError();  // the caller's own run reports any sticky error
    return tune_fix(g0, a.dtype, have ? best_c : fallback);
}

}  // namespace
}  // namespace ssd

extern "C" {

ssd_status_t ssd_fwd(const void *x, const float *dt, const float *A, const void *Bm,
                     const void *Cm, const float *D, const float *init_state, void *y,
                     float *final_state, float *chunk_states, ssd_dims_t dims,
                     ssd_dtype_t dtype, int chunk_size, void *workspace, size_t workspace_bytes,
                     void *stream)
{
    Geom g;
    SSD_TRY(make_geom(dims, chunk_size, true, &g));
    if (dtype != SSD_BF16 && dtype != SSD_F32)
        return SSD_ERR_INVALID_ARG;
    const bool ne = g.L > 0;
    SSD_TRY(need(x, ne));
    SSD_TRY(need(dt, ne));
    SSD_TRY(need(A, true));
    SSD_TRY(need(Bm, ne));
    SSD_TRY(need(Cm, ne));
    SSD_TRY(need(D, true));
    SSD_TRY(need(y, ne));
    SSD_TRY(opt(init_state));
    SSD_TRY(opt(final_state));
    SSD_TRY(opt(chunk_states));
    const FwdArgs a{x, dt, A, Bm, Cm, D, init_state, y, final_state, chunk_states, dims, dtype,
                    workspace, workspace_bytes, (cudaStream_t)stream};
    bool allow_prefill = true;
    if (g.T == 0) {
        TuneChoice c;
        if (!tune_lookup(g, dtype, &c)) {
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            const bool capturing =
                cudaStreamIsCapturing(a.st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone;
            if (capturing)
                cudaGetLastError();
            c = (!ne || chunk_states || capturing || !outputs_disjoint(a, g))
                    ? tune_fix(g, dtype, tune_peek(g, dtype))
                    : tune_and_fix(a, g);
        }
        g = with_chunk(g, c.T);
        allow_prefill = c.allow_prefill;
    }
    return fwd_impl(a, g, allow_prefill);
}

size_t ssd_bwd_workspace_size(ssd_dims_t dims, ssd_dtype_t dtype)
{
    Geom g;
    if (make_geom(dims, bwd_chunk_size(), false, &g) != SSD_OK ||
        (dtype != SSD_BF16 && dtype != SSD_F32))
        return 0;
    // the 64-token-chunk layout is the larger of the two paths' layouts
    return bwd_layout(g, nullptr).bytes;
}

ssd_status_t ssd_bwd(const void *x, const float *dt, const float *A, const void *Bm,
                     const void *Cm, const float *D, const float *init_state, const void *dy,
                     const float *dfinal, void *dx, float *ddt, float *dA, void *dB, void *dC,
                     float *dD, float *dinit, ssd_dims_t dims, ssd_dtype_t dtype,
                     void *workspace, size_t workspace_bytes, void *stream)
{
    Geom g;
    SSD_TRY(make_geom(dims, bwd_chunk_size(), false, &g));
    if (dtype != SSD_BF16 && dtype != SSD_F32)
        return SSD_ERR_INVALID_ARG;
    if (!bwd_supported(g))
        return SSD_ERR_UNSUPPORTED;
    const bool ne = g.L > 0;
    for (const void *p : std::initializer_list<const void *>{x, dt, Bm, Cm, dy, dx, ddt, dB, dC})
        SSD_TRY(need(p, ne));
    SSD_TRY(need(A, true));
    SSD_TRY(need(D, true));
    SSD_TRY(need(dA, true));
    SSD_TRY(need(dD, true));
    SSD_TRY(opt(init_state));
    SSD_TRY(opt(dfinal));
    SSD_TRY(opt(dinit));
    const BwdWs need_ws = bwd_layout(g, nullptr);
    if (ne && (!workspace || workspace_bytes < need_ws.bytes ||
               (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return SSD_ERR_WORKSPACE;
    // every argument is valid: nothing was launched before this point
    cudaStream_t st = (cudaStream_t)stream;
    SSD_TRY(cuda_status(cudaMemsetAsync(dA, 0, (size_t)g.H * sizeof(float), st)));
    SSD_TRY(cuda_status(cudaMemsetAsync(dD, 0, (size_t)g.H * sizeof(float), st)));
    const size_t sbytes = (size_t)(g.B * g.H * g.P * g.S) * sizeof(float);
    if (!ne) {  // no tokens: the initial state is the final state
        if (!dinit)
            return SSD_OK;
        return cuda_status(dfinal ? cudaMemcpyAsync(dinit, dfinal, sbytes, cudaMemcpyDeviceToDevice, st)
                                  : cudaMemsetAsync(dinit, 0, sbytes, st));
    }
    const bool bf16 = dtype == SSD_BF16;
    // tensor-core path: 128-token chunks, the forward and reverse state passes
    // and the chunk gradients on tcgen05 (SSD_BWD_KERNEL=cuda-cores forces the
    // CUDA-core path)
    Geom gt;
    const char *force = std::getenv("SSD_BWD_KERNEL");
    const bool tc = bf16 && !(force && std::strcmp(force, "cuda-cores") == 0) &&
                    make_geom(dims, 128, false, &gt) == SSD_OK && bwd_tc_supported(gt) &&
                    state_pass_tc_supported(gt) && reverse_state_pass_tc_supported(gt);
    if (tc) {
        const BwdWs w = bwd_layout(gt, static_cast<char *>(workspace));
        SSD_TRY(cuda_status(launch_chunk_cumsum(dt, A, w.Gc, w.dtT, gt, st)));
        SSD_TRY(cuda_status(launch_state_pass_tc(x, Bm, w.dtT, w.Gc, init_state, w.states, nullptr, gt, st)));
        SSD_TRY(cuda_status(launch_reverse_state_pass_tc(dy, Cm, w.Gc, dfinal, w.dstates, dinit, gt, st)));
        const size_t bct = (size_t)(gt.B * gt.L * gt.G * gt.S) * sizeof(float);
        SSD_TRY(cuda_status(cudaMemsetAsync(w.dB, 0, bct, st)));
        SSD_TRY(cuda_status(cudaMemsetAsync(w.dC, 0, bct, st)));
        SSD_TRY(cuda_status(launch_bwd_chunk_tc(x, Bm, Cm, dy, w.dtT, w.Gc, A, D, w.states, w.dstates, dx,
                                                ddt, dA, dD, w.dB, w.dC, gt, st)));
        const int64_t nbc = gt.B * gt.L * gt.G * gt.S;
        SSD_TRY(cuda_status(launch_convert_f32(w.dB, dB, nbc, true, st)));
        return cuda_status(launch_convert_f32(w.dC, dC, nbc, true, st));
    }
    const BwdWs w = bwd_layout(g, static_cast<char *>(workspace));
    SSD_TRY(cuda_status(launch_chunk_cumsum(dt, A, w.Gc, w.dtT, g, st)));
    SSD_TRY(cuda_status(run_state_pass(x, Bm, w.dtT, w.Gc, init_state, w.states, nullptr, g, bf16, st)));
    const size_t bc = (size_t)(g.B * g.L * g.G * g.S) * sizeof(float);
    SSD_TRY(cuda_status(cudaMemsetAsync(w.dB, 0, bc, st)));
    SSD_TRY(cuda_status(cudaMemsetAsync(w.dC, 0, bc, st)));
    return cuda_status(launch_bwd(x, Bm, Cm, dy, w.dtT, w.Gc, A, D, w.states, dfinal, w.dstates,
                                  dx, ddt, dA, dD, w.dB, w.dC, dB, dC, dinit, g, bf16, st));
}

ssd_status_t ssd_gated_rmsnorm(const void *y, const void *z, const float *weight, void *out,
                               int64_t ntokens, int64_t dim, int64_t group_size, float eps,
                               ssd_dtype_t dtype, void *stream)
{
    if (dtype != SSD_BF16 && dtype != SSD_F32)
        return SSD_ERR_INVALID_ARG;
    if (ntokens < 0 || dim < 1 || group_size < 1 || dim % group_size != 0 || !(eps >= 0.f) ||
        eps > 1e30f)
        return SSD_ERR_INVALID_ARG;
    if (group_size > (1 << 30) || ntokens > (1LL << 40) || (double)ntokens * (double)dim > 4e15)
        return SSD_ERR_UNSUPPORTED;
    const size_t esz = dtype == SSD_BF16 ? 2 : 4;
    if (ntokens > 0) {
        for (const void *p : std::initializer_list<const void *>{y, z, out})
            SSD_TRY(need_elem(p, esz));
        SSD_TRY(need_elem(weight, 4));
    }
    return cuda_status(launch_gated_rmsnorm(y, z, weight, out, ntokens, dim, group_size, eps,
                                            dtype == SSD_BF16, (cudaStream_t)stream));
}

ssd_status_t ssd_decode_step(const void *x, const float *dt, const float *A, const void *Bm,
                             const void *Cm, const float *D, const float *state_in,
                             float *state_out, void *y, ssd_dims_t dims, ssd_dtype_t dtype,
                             void *stream)
{
    if (dims.seqlen != 1)
        return SSD_ERR_INVALID_ARG;
    Geom g;
    SSD_TRY(make_geom(dims, 1, false, &g));
    if (dtype != SSD_BF16 && dtype != SSD_F32)
        return SSD_ERR_INVALID_ARG;
    // one token's slices of larger tensors are rarely 16-byte aligned, so this
    // entry point asks only for element alignment (the kernel picks its vector
    // width from the actual alignment)
    const size_t esz = dtype == SSD_BF16 ? 2 : 4;
    for (const void *p : {x, static_cast<const void *>(Bm), static_cast<const void *>(Cm),
                          static_cast<const void *>(y)})
        SSD_TRY(need_elem(p, esz));
    for (const void *p : {static_cast<const void *>(dt), static_cast<const void *>(A),
                          static_cast<const void *>(D), static_cast<const void *>(state_in),
                          static_cast<const void *>(state_out)})
        SSD_TRY(need_elem(p, 4));
    // the state may be updated in place, but not through partly overlapping buffers
    const size_t sb = (size_t)g.B * g.H * g.P * g.S * sizeof(float);
    const char *si = reinterpret_cast<const char *>(state_in);
    const char *so = reinterpret_cast<const char *>(state_out);
    if (si != so && si < so + sb && so < si + sb)
        return SSD_ERR_INVALID_ARG;
    return cuda_status(launch_decode_step(x, dt, A, Bm, Cm, D, state_in, state_out, y, g,
                                          dtype == SSD_BF16, (cudaStream_t)stream));
}

ssd_status_t ssd_stream_status(void *stream)
{
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return SSD_ERR_CUDA;
    unsigned int *w = device_status_word();
    if (!w)
        return SSD_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (v && cudaMemset(w, 0, sizeof(v)) != cudaSuccess)
        return SSD_ERR_CUDA;
    return (v & 1u) ? SSD_ERR_TIMEOUT : SSD_OK;
}

}  // extern "C"
