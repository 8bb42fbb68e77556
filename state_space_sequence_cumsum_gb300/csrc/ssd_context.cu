// Sequence-sharded (context-parallel) forward: the two pieces that run on
// each rank around one exchange of per-segment summaries.
//
// "Accelerating Mamba-2 forward-pass kernels with CUDA Tile (cuTile)",
// section "Kernel 2: fwd_pass_state": the state at the end of one call is the
// initial state of the next, and the chunk-to-chunk update is
//     h <- exp2(G_last) h + (contribution of the chunk's tokens),
// which is linear in h.  So a sequence cut into segments k = 0..R-1 (one per
// rank, in sequence order) runs as:
//   1. every rank: its segment from a zero state -> end state s_k, and the
//      segment's total decay D_k = sum of A dt over its tokens (log2 units);
//   2. an all-gather of (s_k, D_k) (the caller's collective);
//   3. rank r: its carried-in state h_r = exp2(D_{r-1}) h_{r-1} + s_{r-1},
//      h_0 = the sequence's initial state (or zero);
//   4. rank r: the ordinary forward of its segment from h_r.
// ssd_segment_summary is step 1 and ssd_carry_in step 3.
#include <initializer_list>

#include "common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

// D[bh] = sum over chunks c of G[bh, last valid token of c] (log2 units):
// G restarts at every chunk start, so its value at a chunk's last token is
// that chunk's whole decay.  One warp per (batch, head); lanes stride over
// the chunks, then a shuffle reduction (fixed order: deterministic).
__global__ void __launch_bounds__(256)
segment_decay_kernel(const float *__restrict__ Gc, float *__restrict__ decay, int64_t nbh,
                     int64_t L, int T)
{
    const int64_t bh = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (bh >= nbh)
        return;
    const int64_t nc = (L + T - 1) / T;
    float d = 0.f;
    for (int64_t c = lane; c < nc; c += 32)
        d += Gc[bh * L + min64(L, (c + 1) * T) - 1];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        d += __shfl_xor_sync(0xffffffffu, d, o);
    if (lane == 0)
        decay[bh] = d;
}

// h[e] = exp2(D_{upto-1}) (... (exp2(D_0) init[e] + s_0[e]) ...) + s_{upto-1}[e]
// for every state element e of every (batch, head).  One thread per element;
// the segments' states are independent of the chain, so each thread loads
// them eight at a time ahead of it.
__global__ void __launch_bounds__(256)
carry_in_kernel(const float *__restrict__ seg_states, const float *__restrict__ seg_decays,
                const float *__restrict__ init, float *__restrict__ h_in, int64_t nbh, int64_t ps,
                int upto)
{
    const int64_t n = nbh * ps;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= n)
        return;
    const int64_t bh = e / ps;
    float h = init ? init[e] : 0.f;
    for (int k0 = 0; k0 < upto; k0 += 8) {
        float v[8], w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const bool in = k0 + j < upto;
            v[j] = in ? seg_states[(int64_t)(k0 + j) * n + e] : 0.f;
            w[j] = in ? exp2f(seg_decays[(int64_t)(k0 + j) * nbh + bh]) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (k0 + j < upto)
                h = fmaf(w[j], h, v[j]);
    }
    h_in[e] = h;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

size_t ssd_segment_summary_workspace_size(ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size)
{
    if (dtype != SSD_BF16 && dtype != SSD_F32)
        return 0;
    if (dims.batch < 1 || dims.seqlen < 0 || dims.nheads < 1 || dims.headdim < 1 ||
        dims.dstate < 1 || dims.ngroups < 1 || chunk_size < 1 || chunk_size > 256)
        return 0;
    const size_t bhl = (size_t)(dims.batch * dims.nheads * dims.seqlen) * sizeof(float);
    const size_t b = 2 * round256(bhl);
    return b ? b : 256;
}

ssd_status_t ssd_segment_summary(const void *x, const float *dt, const float *A, const void *Bm,
                                 float *seg_state, float *seg_decay, ssd_dims_t dims,
                                 ssd_dtype_t dtype, int chunk_size, void *workspace,
                                 size_t workspace_bytes, void *stream)
{
    const size_t need = ssd_segment_summary_workspace_size(dims, dtype, chunk_size);
    // every size check of the forward, before anything is launched
    if (need == 0 || ssd_fwd_workspace_size(dims, dtype, chunk_size, 0) == 0)
        return SSD_ERR_INVALID_ARG;
    const bool ne = dims.seqlen > 0;
    if (!seg_state || !seg_decay || !A || (ne && (!x || !dt || !Bm)))
        return SSD_ERR_INVALID_ARG;
    for (const void *p : {x, static_cast<const void *>(dt), static_cast<const void *>(A), Bm,
                          static_cast<const void *>(seg_state), static_cast<const void *>(seg_decay)})
        if (p && !aligned16(p))
            return SSD_ERR_ALIGNMENT;
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t nbh = dims.batch * dims.nheads;
    if (dims.seqlen == 0) {
        // an empty segment: zero state, zero decay (the state pass validates the rest)
        const ssd_status_t s = ssd_state_pass(x, Bm, nullptr, nullptr, nullptr, nullptr, seg_state,
                                              dims, dtype, chunk_size, stream);
        if (s != SSD_OK)
            return s;
        return cudaMemsetAsync(seg_decay, 0, (size_t)nbh * sizeof(float), st) == cudaSuccess
                   ? SSD_OK
                   : SSD_ERR_CUDA;
    }
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return SSD_ERR_WORKSPACE;
    float *Gc = static_cast<float *>(workspace);
    float *dtT = reinterpret_cast<float *>(static_cast<char *>(workspace) + need / 2);
    ssd_dims_t d1 = dims;
    d1.headdim = 1;
    d1.dstate = 1;
    d1.ngroups = 1;
    ssd_status_t s = ssd_chunk_cumsum(dt, A, Gc, dtT, d1, chunk_size, stream);
    if (s != SSD_OK)
        return s;
    s = ssd_state_pass(x, Bm, dtT, Gc, nullptr, nullptr, seg_state, dims, dtype, chunk_size,
                       stream);
    if (s != SSD_OK)
        return s;
    segment_decay_kernel<<<(unsigned)((nbh + 7) / 8), 256, 0, st>>>(Gc, seg_decay, nbh,
                                                                     dims.seqlen, chunk_size);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status_t ssd_carry_in(const float *seg_states, const float *seg_decays,
                          const float *init_state, int n_segments, int upto, float *h_in,
                          ssd_dims_t dims, void *stream)
{
    if (dims.batch < 1 || dims.nheads < 1 || dims.headdim < 1 || dims.dstate < 1 ||
        n_segments < 1 || upto < 0 || upto > n_segments || !h_in)
        return SSD_ERR_INVALID_ARG;
    if (dims.headdim > 256 || dims.dstate > 512 || dims.batch * dims.nheads > 65535LL * 64)
        return SSD_ERR_UNSUPPORTED;
    if (upto > 0 && (!seg_states || !seg_decays))
        return SSD_ERR_INVALID_ARG;
    for (const void *p : {static_cast<const void *>(seg_states), static_cast<const void *>(seg_decays),
                          static_cast<const void *>(init_state), static_cast<const void *>(h_in)})
        if (p && !aligned16(p))
            return SSD_ERR_ALIGNMENT;
    const int64_t nbh = dims.batch * dims.nheads, ps = dims.headdim * dims.dstate;
    const int64_t n = nbh * ps;
    // h_in may not partly overlap what it is computed from
    const char *o = reinterpret_cast<const char *>(h_in);
    const size_t nb = (size_t)n * sizeof(float);
    auto clash = [&](const void *p, size_t len) {
        const char *q = static_cast<const char *>(p);
        return p && q < o + nb && o < q + len;
    };
    if (clash(seg_states, (size_t)upto * nb) || clash(seg_decays, (size_t)upto * nbh * sizeof(float)) ||
        (init_state && init_state != h_in && clash(init_state, nb)))
        return SSD_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    carry_in_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(seg_states, seg_decays,
                                                                  init_state, h_in, nbh, ps, upto);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
