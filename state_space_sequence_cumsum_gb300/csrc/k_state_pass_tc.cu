// Stage 2 on tensor cores: the chunk-to-chunk state pass for bf16 inputs.
//
// "Accelerating Mamba-2 forward-pass kernels with CUDA Tile (cuTile)",
// section "Kernel 2: fwd_pass_state": per (batch, head) the state h [P, S] is
// carried serially across chunks; at every chunk start it is stored, then
//     h <- exp2(G_last) h + X^T (B * dt * exp2(G_last - G))
// as one tensor-core contraction over the chunk's tokens.
//
// GB300 mapping
//   * CTA = (128-wide dstate slice sigma, batch*head).  The state slice
//     h^T [128 s, P] is the tcgen05 accumulator itself and stays in TMEM for
//     the whole sequence (lane = s, column = p); each step scales it by
//     exp2(G_last) in place and the MMA accumulates the jump onto it.
//   * Tokens are walked in 128-token tiles (the MMA K extent).  For
//     chunk_size 256 a chunk is two tiles; the decay of the first tile is
//     G at its last token, of the second G_last - G at the first tile's last
//     token, so the product of the two steps is the chunk's exp2(G_last).
//   * x [128 t, P] and B [128 t, 128 s] tiles arrive by TMA (128-byte
//     swizzle) into a 3-stage ring; both are token-major, so the contraction
//     over tokens uses MN-major operands: A = B^T (M = s), B = X_hat (N = p).
//   * The pages scale B by dt * exp2(G_last - G) (b_dt_d); here the same
//     per-token weight w_t is applied to x instead (X_hat = w * X, P < S so
//     fewer elements), written back to shared memory in the swizzled layout.
//     w_t <= dt_t because G is non-increasing, so nothing can overflow.
//   * X_hat is split into two bf16 operands, hi = bf16(w x) and
//     lo = bf16(w x - hi), and both are contracted (two MMA passes): the jump
//     then carries ~16 mantissa bits instead of bf16's 8, so the carried
//     state does not accumulate bf16 rounding of the weighted inputs.
//   * Roles: warps 0-3 (one thread per token row / state row) build X_hat,
//     store chunk states and rescale the accumulator; one thread of warp 4
//     issues TMA loads and MMAs.  Every mbarrier wait is bounded; a timeout
//     sets the kernel status word and the CTA leaves its loop.
#include "common.cuh"
#include "ssd_internal.h"
#include "tc05.cuh"

namespace ssd {
namespace {
using namespace tc;

constexpr int kTile = 128;
constexpr int kThreads = 160;
constexpr int kMaxSeg = 64;  // segments of one sequence in the segmented pass
constexpr uint32_t kRegion = 128 * 128;  // one 128-row x 128-byte swizzled region

template <int P>
struct SpLayout {
    static constexpr int kStages = P <= 64 ? 3 : 2;
    static constexpr int kXRegions = P / 64;
    static constexpr uint32_t kX = kXRegions * kRegion;
    static constexpr uint32_t kB = 2 * kRegion;
    static constexpr uint32_t kStage = kX + kB;
    static constexpr uint32_t off_xh = kStages * kStage;  // X_hat hi, then lo
    static constexpr uint32_t bytes = off_xh + 2 * kX;
    static constexpr uint32_t kTmemCols = P < 32 ? 32 : P;
    static_assert(bytes + 1024 + 256 <= 232448, "shared memory budget");
};

// (w * a pair of bf16) as hi = bf16(value) and lo = bf16(value - hi), packed.
__device__ __forceinline__ void split_scaled(uint32_t v, float w, uint32_t &hi, uint32_t &lo)
{
    const float a = __uint_as_float(v << 16) * w;
    const float b = __uint_as_float(v & 0xffff0000u) * w;
    hi = pack_bf16x2(a, b);
    const float ah = __uint_as_float(hi << 16), bh = __uint_as_float(hi & 0xffff0000u);
    lo = pack_bf16x2(a - ah, b - bh);
}

__device__ __forceinline__ void tma_load_4d(void *dst, const void *tmap, uint64_t *bar, int c0,
                                            int c1, int c2, int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Segments of a sequence, all run at once (blockIdx.z = segment).  Mode 1:
// each segment from a zero state, no chunk states, its end state into
// slot(seg) (seg < n_seg - 1).  Mode 2: segment k > 0 from slot(k - 1),
// chunk states emitted, the final state from the last segment.  Mode 0: one
// segment, the whole sequence (the plain pass).  slot(k) of (batch, head) bh
// is slot_base + bh * slot_bh + k * slot_k floats, a [P, S] state.
struct SpSeg {
    int mode, seg_tiles, n_seg;
    float *slot_base;
    int64_t slot_bh, slot_k;
};

template <int P, bool REV>
__global__ void __launch_bounds__(kThreads, 1)
state_pass_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_b, const float *__restrict__ dtT,
                     const float *__restrict__ Gc, const float *__restrict__ init,
                     float *__restrict__ states, float *__restrict__ final_state, Geom g,
                     unsigned int *status, SpSeg sg)
{
    using Lay = SpLayout<P>;
    constexpr int kStages = Lay::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_full[kStages], bar_empty[kStages], bar_ready, bar_mma;
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5;
    const int sigma = blockIdx.x;
    const int64_t bh = blockIdx.y, b = bh / g.H, h = bh % g.H, grp = h / g.hpg;
    const int64_t n_all = (g.L + kTile - 1) / kTile;
    const int seg = blockIdx.z;
    const int64_t t_begin = sg.mode ? (int64_t)seg * sg.seg_tiles : 0;
    const int64_t t_end = sg.mode ? min64(n_all, t_begin + sg.seg_tiles) : n_all;
    const int64_t n_tiles = t_end - t_begin;  // tiles of this CTA
    float *slot_prev = (sg.mode == 2 && seg > 0)
                           ? sg.slot_base + bh * sg.slot_bh + (int64_t)(seg - 1) * sg.slot_k
                           : nullptr;
    float *slot_out = (sg.mode == 1 && seg < sg.n_seg - 1)
                          ? sg.slot_base + bh * sg.slot_bh + (int64_t)seg * sg.slot_k
                          : nullptr;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], 4);  // one arrival per compute warp
        }
        mbar_init(&bar_ready, 4);
        mbar_init(&bar_mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, Lay::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (tid == 128) {
        // ---------------- TMA producer + MMA issuer (one thread)
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_b);
        auto issue = [&](int64_t i) {
            const int s = (int)(i % kStages);
            uint8_t *stage = smem + s * Lay::kStage;
            mbar_arrive_expect_tx(&bar_full[s], Lay::kStage);
            const int tok = (int)((REV ? t_end - 1 - i : t_begin + i) * kTile);
            for (int r = 0; r < Lay::kXRegions; ++r)
                tma_load_4d(stage + r * kRegion, &tm_x, &bar_full[s], r * 64, (int)h, tok, (int)b);
            for (int r = 0; r < 2; ++r)
                tma_load_4d(stage + Lay::kX + r * kRegion, &tm_b, &bar_full[s],
                            sigma * 128 + r * 64, (int)grp, tok, (int)b);
        };
        for (int64_t i = 0; i < kStages && i < n_tiles; ++i)
            issue(i);
        const uint32_t idesc = idesc_bf16(128, P, true, true);
        const uint32_t xh = smem_u32(smem + Lay::off_xh);
        for (int64_t i = 0; i < n_tiles; ++i) {
            const int s = (int)(i % kStages);
            if (!mbar_wait(&bar_ready, (uint32_t)(i & 1))) {
                atomicOr(status, 1u);
                break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(smem + s * Lay::kStage + Lay::kX);
#pragma unroll
            for (int part = 0; part < 2; ++part)  // X_hat hi, then lo
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks)
                    mma_ss(tmem, smem_desc(a0 + ks * 2048, kRegion, 1024),
                           smem_desc(xh + part * Lay::kX + ks * 2048, kRegion, 1024), idesc, 1u);
            mma_commit(&bar_mma);
            if (i + kStages < n_tiles) {
                const uint32_t par = (uint32_t)((i / kStages) & 1);
                if (!mbar_wait(&bar_empty[s], par) || !mbar_wait(&bar_mma, (uint32_t)(i & 1))) {
                    atomicOr(status, 1u);
                    break;
                }
                issue(i + kStages);
            }
        }
    } else if (tid < 128) {
        // ---------------- compute threads: token row `tid`, state row s = sigma*128 + tid
        const int row = tid;
        const int64_t s_idx = (int64_t)sigma * 128 + row;
        const bool s_ok = s_idx < g.S;
        const uint32_t lane_base = tmem_at(tmem, (uint32_t)(warp * 32), 0);
#pragma unroll
        for (int c0 = 0; c0 < P; c0 += 16) {
            uint32_t r[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float v = 0.f;
                if (s_ok && sg.mode != 1) {
                    if (slot_prev)
                        v = slot_prev[(int64_t)(c0 + j) * g.S + s_idx];
                    else if (init)
                        v = init[(bh * g.P + c0 + j) * g.S + s_idx];
                }
                r[j] = __float_as_uint(v);
            }
            tmem_st16(lane_base + c0, r);
        }
        tmem_st_wait();

        const float *grow = Gc + bh * g.L;
        const float *drow = dtT + bh * g.L;
        uint8_t *sxh = smem + Lay::off_xh;
        for (int64_t i = 0; i < n_tiles; ++i) {
            const int s = (int)(i % kStages);
            const int64_t tau = (REV ? t_end - 1 - i : t_begin + i) * kTile;
            const int n = (int)min64(kTile, g.L - tau);
            // tile-local log2 decay: G restarts at chunk starts, so a tile in
            // the middle of a chunk subtracts G at the token before it
            const float base = (tau % g.T == 0) ? 0.f : grow[tau - 1];
            const float gL = grow[tau + n - 1] - base;
            // forward: dt_t exp2(G_last - G_t); reverse (tile = chunk): exp2(G_t)
            const float w = row < n ? (REV ? exp2f(grow[tau + row] - base)
                                           : drow[tau + row] * exp2f(gL - (grow[tau + row] - base)))
                                    : 0.f;
            const float decay = exp2f(gL);

            if (!mbar_wait(&bar_full[s], (uint32_t)((i / kStages) & 1))) {
                atomicOr(status, 1u);
                break;
            }
            const uint8_t *sx = smem + s * Lay::kStage;
#pragma unroll
            for (int r = 0; r < Lay::kXRegions; ++r) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t off = r * kRegion + sw128_offset(row, c);
                    const uint4 v = *reinterpret_cast<const uint4 *>(sx + off);
                    uint4 hi, lo;
                    split_scaled(v.x, w, hi.x, lo.x);
                    split_scaled(v.y, w, hi.y, lo.y);
                    split_scaled(v.z, w, hi.z, lo.z);
                    split_scaled(v.w, w, hi.w, lo.w);
                    *reinterpret_cast<uint4 *>(sxh + off) = hi;
                    *reinterpret_cast<uint4 *>(sxh + Lay::kX + off) = lo;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if ((tid & 31) == 0)
                mbar_arrive(&bar_empty[s]);

            // chunk start: store h (the state before this chunk), then decay it
            const bool emit = states && s_ok && sg.mode != 1 && (tau % g.T == 0);
            float *dst = emit ? states + ((bh * g.nc + tau / g.T) * g.P) * g.S + s_idx : nullptr;
#pragma unroll
            for (int c0 = 0; c0 < P; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(lane_base + c0, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float v = __uint_as_float(r[j]);
                    if (emit)
                        dst[(int64_t)(c0 + j) * g.S] = v;
                    r[j] = __float_as_uint(v * decay);
                }
                tmem_st16(lane_base + c0, r);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if ((tid & 31) == 0)
                mbar_arrive(&bar_ready);
            if (!mbar_wait(&bar_mma, (uint32_t)(i & 1))) {
                atomicOr(status, 1u);
                break;
            }
            tc_fence_after();
        }
        // the end state: a segment's (mode 1) or the sequence's final state
        float *end_dst = slot_out ? slot_out
                                  : ((final_state && sg.mode != 1 && (sg.mode == 0 || seg == sg.n_seg - 1))
                                         ? final_state + bh * g.P * g.S
                                         : nullptr);
        if (end_dst && s_ok) {
#pragma unroll
            for (int c0 = 0; c0 < P; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(lane_base + c0, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    end_dst[(int64_t)(c0 + j) * g.S + s_idx] = __uint_as_float(r[j]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, Lay::kTmemCols);
    }
}

template <int P, bool REV>
cudaError_t launch_p(const CUtensorMap &tx, const CUtensorMap &tb, const float *dtT,
                     const float *Gc, const float *init, float *states, float *final_state,
                     const Geom &g, unsigned int *status, cudaStream_t st, const SpSeg &sg = SpSeg{})
{
    const size_t smem = SpLayout<P>::bytes + 1024;
    auto k = state_pass_tc_kernel<P, REV>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    dim3 grid((unsigned)((g.S + 127) / 128), (unsigned)(g.B * g.H), (unsigned)(sg.mode ? sg.n_seg : 1));
    k<<<grid, kThreads, smem, st>>>(tx, tb, dtT, Gc, init, states, final_state, g, status, sg);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

bool state_pass_tc_supported(const Geom &g)
{
    return (g.P == 64 || g.P == 128) && g.S % 64 == 0 && g.T % kTile == 0 && g.L > 0 &&
           g.H <= 65535 && g.G <= 65535 && g.L < (1LL << 31) && g.B * g.H <= 65535;
}

cudaError_t launch_state_pass_tc(const void *x, const void *Bm, const float *dtT,
                                 const float *Gc, const float *init, float *states,
                                 float *final_state, const Geom &g, cudaStream_t st)
{
    if (!state_pass_tc_supported(g))
        return cudaErrorNotSupported;
    unsigned int *status = device_status_word();
    if (!status)
        return cudaErrorUnknown;
    CUtensorMap tx, tb;
    if (!make_tmap_tokens_heads(&tx, x, g) || !make_tmap_tokens_groups(&tb, Bm, g))
        return cudaErrorInvalidValue;
    if (g.P == 64)
        return launch_p<64, false>(tx, tb, dtT, Gc, init, states, final_state, g, status, st);
    return launch_p<128, false>(tx, tb, dtT, Gc, init, states, final_state, g, status, st);
}

// Start states of the segments from their local end states (mode 1):
// slot(k) <- exp2(D_k) slot(k-1) + slot(k), slot(-1) = init (or 0), where D_k
// is segment k's total log2 decay, the sum of G at each of its chunks' last
// valid tokens.  One thread per state element; the first n_seg - 1 threads
// of each block form the decay factors.  The slot loads are independent of
// the carried state, so they are issued eight at a time ahead of the chain.
__global__ void __launch_bounds__(256)
seg_combine_kernel(const float *__restrict__ Gc, const float *__restrict__ init, Geom g, SpSeg sg)
{
    __shared__ float sdec[kMaxSeg];
    const int64_t bh = blockIdx.y;
    const int chunks_per_seg = sg.seg_tiles * kTile / g.T;
    for (int k = threadIdx.x; k < sg.n_seg - 1; k += blockDim.x) {
        float d = 0.f;
        for (int c = k * chunks_per_seg; c < (k + 1) * chunks_per_seg && c < g.nc; ++c)
            d += Gc[bh * g.L + min64(g.L, (int64_t)(c + 1) * g.T) - 1];
        sdec[k] = exp2f(d);
    }
    __syncthreads();
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= g.P * g.S)
        return;
    float h = init ? init[bh * g.P * g.S + e] : 0.f;
    float *slot = sg.slot_base + bh * sg.slot_bh + e;
    for (int k0 = 0; k0 < sg.n_seg - 1; k0 += 8) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            v[j] = k0 + j < sg.n_seg - 1 ? slot[(int64_t)(k0 + j) * sg.slot_k] : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (k0 + j < sg.n_seg - 1) {
                h = fmaf(sdec[k0 + j], h, v[j]);
                slot[(int64_t)(k0 + j) * sg.slot_k] = h;
            }
        }
    }
}

// The reverse pass of the backward: the same contraction run from the last
// 128-token chunk to the first, on dy and C with the weights exp2(G_t), so
// the carried matrix is the state gradient:
//     dstates[c] = dS (gradient of chunk c's end state);  dS <- exp2(G_last) dS + dy^T (C * exp2(G))
// starting from dfinal (NULL: zero); dinit receives dS after chunk 0.
bool reverse_state_pass_tc_supported(const Geom &g) { return state_pass_tc_supported(g) && g.T == kTile; }

cudaError_t launch_reverse_state_pass_tc(const void *dy, const void *Cm, const float *Gc,
                                         const float *dfinal, float *dstates, float *dinit,
                                         const Geom &g, cudaStream_t st)
{
    if (!reverse_state_pass_tc_supported(g))
        return cudaErrorNotSupported;
    unsigned int *status = device_status_word();
    if (!status)
        return cudaErrorUnknown;
    CUtensorMap tx, tb;
    if (!make_tmap_tokens_heads(&tx, dy, g) || !make_tmap_tokens_groups(&tb, Cm, g))
        return cudaErrorInvalidValue;
    if (g.P == 64)
        return launch_p<64, true>(tx, tb, Gc, Gc, dfinal, dstates, dinit, g, status, st);
    return launch_p<128, true>(tx, tb, Gc, Gc, dfinal, dstates, dinit, g, status, st);
}

}  // namespace ssd

namespace ssd {

// Segment plan of the segmented state pass.  The kernel holds one CTA per SM
// and the split runs the sequence twice, so it pays only when the (batch,
// head, dstate slice) units fill a third of the SMs or less: then n segments
// per unit, units * n <= SMs (one wave), cost 2/n of the unsplit pass.
// Segments are at least four tiles and a whole number of chunks.  n_seg 1
// means "not worth it".
void state_pass_seg_plan(const Geom &g, int sms, int *seg_tiles, int *n_seg)
{
    const int64_t n_tiles = (g.L + kTile - 1) / kTile;
    const int64_t units = g.B * g.H * ((g.S + 127) / 128);
    const int tpc = g.T / kTile;  // tiles per chunk
    int64_t want = sms / units;
    if (want > kMaxSeg)
        want = kMaxSeg;
    if (want * 4 > n_tiles)
        want = n_tiles / 4;
    if (want < 3) {
        *n_seg = 1;
        *seg_tiles = (int)n_tiles;
        return;
    }
    int64_t st = (n_tiles + want - 1) / want;
    st = (st + tpc - 1) / tpc * tpc;
    *seg_tiles = (int)st;
    *n_seg = (int)((n_tiles + st - 1) / st);
}

// Long sequences with few (batch, head) units: pass 1 (every segment's end
// state from zero, in parallel), the short serial combine, pass 2 (every
// segment from its true start state, emitting chunk states).  The segment
// start states are kept in the chunk-state array at the segments' first
// chunks, so no other scratch is needed.  Returns cudaErrorNotSupported when
// the plain pass should be used.
cudaError_t launch_state_pass_tc_segmented(const void *x, const void *Bm, const float *dtT,
                                           const float *Gc, const float *init, float *states,
                                           float *final_state, const Geom &g, cudaStream_t st)
{
    if (!state_pass_tc_supported(g) || !states)
        return cudaErrorNotSupported;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorNotSupported;
    SpSeg sg{};
    state_pass_seg_plan(g, sms, &sg.seg_tiles, &sg.n_seg);
    if (sg.n_seg < 2)
        return cudaErrorNotSupported;
    unsigned int *status = device_status_word();
    if (!status)
        return cudaErrorUnknown;
    CUtensorMap tx, tb;
    if (!make_tmap_tokens_heads(&tx, x, g) || !make_tmap_tokens_groups(&tb, Bm, g))
        return cudaErrorInvalidValue;
    // slot(k) = the chunk state at segment k+1's first chunk
    const int64_t chunks_per_seg = (int64_t)sg.seg_tiles * kTile / g.T;
    sg.slot_base = states + chunks_per_seg * g.P * g.S;
    sg.slot_bh = g.nc * g.P * g.S;
    sg.slot_k = chunks_per_seg * g.P * g.S;
    cudaError_t e;
    sg.mode = 1;
    e = g.P == 64 ? launch_p<64, false>(tx, tb, dtT, Gc, nullptr, nullptr, nullptr, g, status, st, sg)
                  : launch_p<128, false>(tx, tb, dtT, Gc, nullptr, nullptr, nullptr, g, status, st, sg);
    if (e != cudaSuccess)
        return e;
    const dim3 cgrid((unsigned)((g.P * g.S + 255) / 256), (unsigned)(g.B * g.H));
    seg_combine_kernel<<<cgrid, 256, 0, st>>>(Gc, init, g, sg);
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    sg.mode = 2;
    return g.P == 64 ? launch_p<64, false>(tx, tb, dtT, Gc, init, states, final_state, g, status, st, sg)
                     : launch_p<128, false>(tx, tb, dtT, Gc, init, states, final_state, g, status, st, sg);
}

}  // namespace ssd
