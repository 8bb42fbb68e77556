// Stage 2 on tensor cores: the chunk-to-chunk state pass for bf16 inputs.
//
// "Accelerating Mamba-2 forward-pass kernels with CUDA Tile (cuTile)",
// section "Kernel 2: fwd_pass_state": per (batch, head) the state h [P, S] is
// carried serially across chunks; at every chunk start it is stored, then
//     h <- exp2(G_last) h + X^T (B * dt * exp2(G_last - G))
// as one tensor-core contraction over the chunk's tokens.
//
// GB300 mapping
//   * CTA = (128-wide dstate slice sigma, batch*head[, segment]).  State row
//     s = sigma*128 + row, h^T[s, 0..P), lives in registers for the whole
//     sequence, split between the two compute threads of that row.
//   * Tokens are walked in 128-token tiles (the MMA K extent).  For
//     chunk_size 256 a chunk is two tiles; the decay of the first tile is
//     G at its last token, of the second G_last - G at the first tile's last
//     token, so the product of the two steps is the chunk's exp2(G_last).
//   * Per tile the tensor core computes the jump J = B^T X_hat [128 s, P]
//     into one of two TMEM buffers (a fresh accumulation, not onto h), and
//     the compute threads fold it in, h <- exp2(G_last) h + J, in f32
//     registers.  With two jump buffers and two X_hat buffers, the MMAs of
//     tile i+1 run while tile i is folded in and stored: the carried state
//     is not a round trip through the tensor core per tile.
//   * x [128 t, P] and B [128 t, 128 s] tiles arrive by TMA (128-byte
//     swizzle) into a ring of stages; both are token-major, so the
//     contraction over tokens uses MN-major operands: A = B^T (M = s),
//     B = X_hat (N = p).
//   * The pages scale B by dt * exp2(G_last - G) (b_dt_d); here the same
//     per-token weight w_t is applied to x instead (X_hat = w * X, P < S so
//     fewer elements), written over x in place in the stage.  w_t <= dt_t
//     because G is non-increasing, so nothing can overflow.
//   * X_hat is split into two bf16 operands, hi (over x in the stage) and
//     lo (its own buffer) with hi + lo = w x to ~2^-16, and both are
//     contracted: the jump then
//     carries ~16 mantissa bits instead of bf16's 8, so the carried state
//     does not accumulate bf16 rounding of the weighted inputs.
//   * Roles: warps 0-7, two warpgroups over the same 128 rows, each with half
//     of every row, build X_hat (thread = token row), fold the jumps in and
//     store chunk states (thread = state row); one thread of warp 8 issues
//     the MMAs; warp 9 issues the TMA loads (one lane) and forms each tile's
//     per-token weights and decay from G and dt (loaded a tile ahead) into
//     the stage, off the compute warps' path.  Every mbarrier
//     wait is bounded; a timeout sets the kernel status word and the role
//     leaves its loop.
#include "common.cuh"
#include "ssd_internal.h"
#include "tc05.cuh"

namespace ssd {
namespace {
using namespace tc;

constexpr int kTile = 128;
constexpr int kCompute = 256;  // warps 0-7: two warpgroups over the same 128 rows
constexpr int kThreads = kCompute + 64;  // + warp 8 (MMA issue), warp 9 (TMA)
constexpr int kMaxSeg = 64;  // segments of one sequence in the segmented pass
constexpr uint32_t kRegion = 128 * 128;  // one 128-row x 128-byte swizzled region

template <int P>
struct SpLayout {
    static constexpr int kStages = P <= 64 ? 3 : 2;
    static constexpr int kXRegions = P / 64;
    static constexpr uint32_t kX = kXRegions * kRegion;  // x tile, then X_hat hi over it
    static constexpr uint32_t kB = 2 * kRegion;          // B tile [128 t, 128 s]
    static constexpr uint32_t off_b = kX;
    static constexpr uint32_t kStage = kX + kB;          // what TMA brings per stage
    static constexpr uint32_t kTxBytes = kStage;
    // X_hat lo, two buffers (tile parity): tile i+1's is written while the
    // MMAs of tile i read the other one
    static constexpr uint32_t off_lo = kStages * kStage;
    // chunk states leave through a [P, 128] f32 staging box and a TMA store
    // (P = 64; P = 128 has no room and stores from registers)
    static constexpr bool kTmaEmit = P <= 64;
    static constexpr uint32_t off_stg = off_lo + 2 * kX;
    // weights of each stage's tile (128 f32) and its decay, by the load warp
    static constexpr uint32_t off_gd = off_stg + (kTmaEmit ? P * 128 * 4 : 0);
    static constexpr uint32_t bytes = off_gd + kStages * 1024;
    static constexpr uint32_t kTmemCols = 2 * P;         // two jump buffers
    static_assert(bytes + 1024 + 256 <= 232448, "shared memory budget");
};

// w * (a pair of bf16) as hi + lo, two packed bf16 pairs, with w = w_hi + w_lo
// (w_hi = bf16(w)): hi = bf16(x w_hi); the residual x w_hi - hi is exact in
// bf16 (x and w_hi carry 8 significant bits each), so lo = bf16(x w_lo +
// residual) and hi + lo is within ~2^-16 of x w.
__device__ __forceinline__ void split_scaled(uint32_t v, uint32_t whi, uint32_t wlo, uint32_t &hi,
                                             uint32_t &lo)
{
    hi = bf2_mul(v, whi);
    lo = bf2_fma(v, wlo, bf2_fma(v, whi, hi ^ 0x80008000u));
}

// the 256 compute threads (named barrier 1; warps 8 and 9 never join it)
__device__ __forceinline__ void compute_sync()
{
    asm volatile("barrier.sync 1, %0;" ::"n"(kCompute) : "memory");
}

// TMA store of an unswizzled box, marked evict-first in L2: chunk states are
// written once and not read by this kernel, so they should not push x, B and
// G out of L2
__device__ __forceinline__ void tma_store_2d(const void *tmap, const void *src, int c0, int c1)
{
    asm volatile(
        "{\n\t.reg .b64 pol;\n\t"
        "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], pol;\n\t}" ::"l"(tmap),
        "r"(smem_u32(src)), "r"(c0), "r"(c1)
        : "memory");
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
                     const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ CUtensorMap tm_st, const float *__restrict__ dtT,
                     const float *__restrict__ Gc, const float *__restrict__ init,
                     float *__restrict__ states, float *__restrict__ final_state, Geom g,
                     unsigned int *status, SpSeg sg, int tma_emit)
{
    using Lay = SpLayout<P>;
    constexpr int kStages = Lay::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_full[kStages], bar_xready[kStages], bar_empty[kStages];
    __shared__ uint64_t bar_jfull[2], bar_jfree[2], bar_end;
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sigma = blockIdx.x;
    const int64_t bh = blockIdx.y, b = bh / g.H, h = bh % g.H, grp = h / g.hpg;
    const int64_t n_all = (g.L + kTile - 1) / kTile;
    const int seg = blockIdx.z;
    const int64_t t_begin = sg.mode ? (int64_t)seg * sg.seg_tiles : 0;
    const int64_t t_end = sg.mode ? min64(n_all, t_begin + sg.seg_tiles) : n_all;
    const int n_tiles = (int)(t_end - t_begin);  // tiles of this CTA
    // first token of the i-th tile this CTA walks
    auto tile_tau = [&](int i) -> int64_t { return (REV ? t_end - 1 - i : t_begin + i) * kTile; };
    // chunks are one or two tiles (T = 128 or 256): chunk index and chunk
    // start by shift and mask, no 64-bit division in the tile loop
    const int tpc_shift = g.T == 2 * kTile ? 1 : 0;
    auto tile_index = [&](int i) -> int { return (int)(REV ? t_end - 1 - i : t_begin + i); };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_xready[s], kCompute / 32);  // one arrival per compute warp
            mbar_init(&bar_empty[s], 1);   // MMA commit
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&bar_jfull[j], 1);
            mbar_init(&bar_jfree[j], kCompute / 32);
        }
        mbar_init(&bar_end, 1);
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

    if (warp == kCompute / 32 + 1) {
        // ---------------- load warp: x and B by TMA (lane 0); G and dt of the
        // tile by the whole warp, loaded a tile ahead into registers so their
        // latency overlaps the wait for a free stage, turned into the tile's
        // weights here
        const float *grow = Gc + bh * g.L;
        const float *drow = dtT + bh * g.L;
        float pg0 = 0.f, pg1 = 0.f, pg2 = 0.f, pg3 = 0.f;  // G of tokens 4 lane + 0..3
        float pd0 = 0.f, pd1 = 0.f, pd2 = 0.f, pd3 = 0.f;  // dt of the same tokens
        float gl_prev = 0.f;  // G at the previous tile's last token (forward walk)
        auto gload = [&](int i) {
            const int64_t tau = tile_tau(i);
            const int n = (int)min64(kTile, g.L - tau);
            const int t = 4 * lane;
            const float *gp = grow + tau + t, *dp = drow + tau + t;
            pg0 = t < n ? gp[0] : 0.f;
            pg1 = t + 1 < n ? gp[1] : 0.f;
            pg2 = t + 2 < n ? gp[2] : 0.f;
            pg3 = t + 3 < n ? gp[3] : 0.f;
            pd0 = (!REV && t < n) ? dp[0] : 0.f;
            pd1 = (!REV && t + 1 < n) ? dp[1] : 0.f;
            pd2 = (!REV && t + 2 < n) ? dp[2] : 0.f;
            pd3 = (!REV && t + 3 < n) ? dp[3] : 0.f;
        };
        if (lane == 0) {
            prefetch_tmap(&tm_x);
            prefetch_tmap(&tm_b);
        }
        if (n_tiles > 0)
            gload(0);
        for (int i = 0; i < n_tiles; ++i) {
            const int s = (int)(i % kStages);
            if (i >= kStages &&
                !__all_sync(0xffffffffu, mbar_wait(&bar_empty[s], (uint32_t)((i / kStages - 1) & 1)))) {
                if (lane == 0)
                    atomicOr(status, 1u);
                break;
            }
            // the tile's per-token weights and its decay, into the stage's
            // slot: forward w = dt_t exp2(G_last - G_t), reverse exp2(G_t),
            // with G relative to the tile start (G restarts at chunk starts; a
            // tile in the middle of a chunk subtracts G before it)
            {
                const int n = (int)min64(kTile, g.L - tile_tau(i));
                const float gb = (tile_index(i) & tpc_shift) == 0 ? 0.f : gl_prev;
                const int e = (n - 1) & 3;
                const float mine = e == 0 ? pg0 : (e == 1 ? pg1 : (e == 2 ? pg2 : pg3));
                const float gl = __shfl_sync(0xffffffffu, mine, (n - 1) >> 2);
                const float gL = gl - gb;
                float *sw = reinterpret_cast<float *>(smem + Lay::off_gd + s * 1024);
                auto wt = [&](int t, float gv, float dv) {
                    return t < n ? (REV ? exp2f(gv - gb) : dv * exp2f(gL - (gv - gb))) : 0.f;
                };
                const int t = 4 * lane;
                *reinterpret_cast<float4 *>(sw + t) =
                    make_float4(wt(t, pg0, pd0), wt(t + 1, pg1, pd1), wt(t + 2, pg2, pd2), wt(t + 3, pg3, pd3));
                if (lane == 0)
                    sw[128] = exp2f(gL);
                gl_prev = gl;
            }
            if (i + 1 < n_tiles)
                gload(i + 1);
            __syncwarp();  // the warp's weight stores precede lane 0's arrival
            if (lane == 0) {
                uint8_t *stage = smem + s * Lay::kStage;
                mbar_arrive_expect_tx(&bar_full[s], Lay::kTxBytes);
                const int tok = (int)tile_tau(i);
                for (int r = 0; r < Lay::kXRegions; ++r)
                    tma_load_4d(stage + r * kRegion, &tm_x, &bar_full[s], r * 64, (int)h, tok, (int)b);
                for (int r = 0; r < 2; ++r)
                    tma_load_4d(stage + Lay::off_b + r * kRegion, &tm_b, &bar_full[s],
                                sigma * 128 + r * 64, (int)grp, tok, (int)b);
            }
        }
    } else if (warp == kCompute / 32) {
        // ---------------- MMA issuer: J[i & 1] = B^T (X_hat hi + X_hat lo)
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, P, true, true);
            for (int i = 0; i < n_tiles; ++i) {
                const int s = (int)(i % kStages), jb = (int)(i & 1);
                if (!mbar_wait(&bar_xready[s], (uint32_t)((i / kStages) & 1)) ||
                    (i >= 2 && !mbar_wait(&bar_jfree[jb], (uint32_t)(((i - 2) >> 1) & 1)))) {
                    atomicOr(status, 1u);
                    break;
                }
                tc_fence_after();
                const uint32_t st = smem_u32(smem + s * Lay::kStage);
                const uint32_t lo = smem_u32(smem + Lay::off_lo + jb * Lay::kX);
                const uint32_t d = tmem + (uint32_t)(jb * P);
#pragma unroll
                for (int part = 0; part < 2; ++part)  // X_hat hi, then lo
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks)
                        mma_ss(d, smem_desc(st + Lay::off_b + ks * 2048, kRegion, 1024),
                               smem_desc(part ? lo + ks * 2048 : st + ks * 2048, kRegion, 1024),
                               idesc, (part | ks) ? 1u : 0u);
                mma_commit(&bar_jfull[jb]);
                mma_commit(&bar_empty[s]);
            }
            // every MMA this thread issued has completed before TMEM is freed
            // (the compute warps wait for each jump only while nothing failed)
            mma_commit(&bar_end);
            if (!mbar_wait(&bar_end, 0))
                atomicOr(status, 1u);
        }
    } else {
        // ---------------- compute threads: token row `row` for X_hat, state row
        // s = sigma*128 + row for the carried state.  Warpgroup wg takes half
        // of each row: X_hat chunks and state columns p0 .. p0 + P/2.
        constexpr int PH = P / 2;
        constexpr int NQ = Lay::kXRegions * 4;  // 16-byte X_hat chunks per row per warpgroup
        const int row = tid & 127, wg = tid >> 7;
        const int p0 = wg * PH;
        const int64_t s_idx = (int64_t)sigma * 128 + row;
        const bool s_ok = s_idx < g.S;
        const uint32_t lane_base = tmem_at(tmem, (uint32_t)((warp & 3) * 32), 0);
        float *stg = reinterpret_cast<float *>(smem + Lay::off_stg);
        const int bw = g.S < 128 ? (int)g.S : 128;  // staging box width (state rows)
        const float *slot_prev = (sg.mode == 2 && seg > 0)
                                     ? sg.slot_base + bh * sg.slot_bh + (int64_t)(seg - 1) * sg.slot_k
                                     : nullptr;
        float hs[PH];
#pragma unroll
        for (int p = 0; p < PH; ++p) {
            float v = 0.f;
            if (s_ok && sg.mode != 1) {
                if (slot_prev)
                    v = slot_prev[(int64_t)(p0 + p) * g.S + s_idx];
                else if (init)
                    v = init[(bh * g.P + p0 + p) * g.S + s_idx];
            }
            hs[p] = v;
        }

        // weight of this thread's token row and decay of tile i, formed by the
        // load warp in the stage's slot
        auto weights = [&](int i, float &w, float &decay) {
            const float *sw = reinterpret_cast<const float *>(smem + Lay::off_gd + (i % kStages) * 1024);
            w = sw[row];
            decay = sw[128];
        };
        // this warpgroup's half of X_hat of tile i: hi over x, lo in buffer i & 1
        auto build = [&](int i, float &decay) -> bool {
            const int s = (int)(i % kStages);
            if (!__all_sync(0xffffffffu, mbar_wait(&bar_full[s], (uint32_t)((i / kStages) & 1))))
                return false;
            float w;
            weights(i, w, decay);
            const uint32_t whi = pack_bf16x2(w, w);
            const float w_lo = w - __uint_as_float(whi << 16);
            const uint32_t wlo = pack_bf16x2(w_lo, w_lo);
            uint8_t *stage = smem + s * Lay::kStage;
            uint8_t *slo = smem + Lay::off_lo + (uint32_t)(i & 1) * Lay::kX;
            // every load before the first store: the stores go over the same
            // buffer, so the compiler would otherwise keep each chunk's load
            // behind the previous chunk's store
            uint32_t off[NQ];
            uint4 v[NQ];
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const int qq = wg * NQ + q;
                off[q] = (qq >> 3) * kRegion + sw128_offset(row, qq & 7);
                v[q] = *reinterpret_cast<const uint4 *>(stage + off[q]);
            }
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                uint4 hi, lo;
                split_scaled(v[q].x, whi, wlo, hi.x, lo.x);
                split_scaled(v[q].y, whi, wlo, hi.y, lo.y);
                split_scaled(v[q].z, whi, wlo, hi.z, lo.z);
                split_scaled(v[q].w, whi, wlo, hi.w, lo.w);
                *reinterpret_cast<uint4 *>(stage + off[q]) = hi;
                *reinterpret_cast<uint4 *>(slo + off[q]) = lo;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bar_xready[s]);
            return true;
        };

        // A warp whose wait gives up (ok false) keeps walking the tiles without
        // work: the chunk-state stores below synchronise all compute warps, so
        // leaving the loop early would hold the others at that barrier.
        bool ok = true;
        float d_cur = 1.f, d_next = 1.f;
        if (n_tiles > 0)
            ok = build(0, d_cur);
        for (int i = 0; i < n_tiles; ++i) {
            // chunk start: store h, the state before this chunk
            const int ti = tile_index(i);
            if (states && sg.mode != 1 && (ti & tpc_shift) == 0) {
                const int64_t row0 = (bh * g.nc + (ti >> tpc_shift)) * g.P;  // row of p = 0 in [.., S]
                if (Lay::kTmaEmit && tma_emit) {
                    // the staging box is free once the previous store has read it
                    if (tid == 0)
                        bulk_wait_read();
                    compute_sync();
                    if (row < bw) {
#pragma unroll
                        for (int p = 0; p < PH; ++p)
                            stg[(p0 + p) * bw + row] = hs[p];
                    }
                    fence_proxy_async_smem();
                    compute_sync();
                    if (tid == 0) {
                        tma_store_2d(&tm_st, stg, sigma * 128, (int)row0);
                        bulk_commit();
                    }
                } else if (s_ok) {
                    float *dst = states + (row0 + p0) * g.S + s_idx;
#pragma unroll
                    for (int p = 0; p < PH; ++p)
                        dst[(int64_t)p * g.S] = hs[p];
                }
            }
            if (ok && i + 1 < n_tiles)
                ok = build(i + 1, d_next);
            // fold in this warpgroup's columns of the jump of tile i
            const int jb = (int)(i & 1);
            if (ok)
                ok = __all_sync(0xffffffffu, mbar_wait(&bar_jfull[jb], (uint32_t)((i >> 1) & 1)));
            if (!ok)
                continue;
            tc_fence_after();
            constexpr int kQ = PH / 16 < 4 ? PH / 16 : 4;  // 16-column loads in flight
#pragma unroll
            for (int c0 = 0; c0 < PH; c0 += 16 * kQ) {
                uint32_t r[kQ][16];
#pragma unroll
                for (int q = 0; q < kQ; ++q)
                    tmem_ld16(lane_base + (uint32_t)(jb * P + p0 + c0 + 16 * q), r[q]);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < kQ; ++q)
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        hs[c0 + 16 * q + j] = fmaf(d_cur, hs[c0 + 16 * q + j], __uint_as_float(r[q][j]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bar_jfree[jb]);
            d_cur = d_next;
        }
        if (!ok) {
            if (lane == 0)
                atomicOr(status, 1u);
        } else {
            // the end state: a segment's (mode 1) or the sequence's final state
            float *end_dst = nullptr;
            if (sg.mode == 1) {
                if (seg < sg.n_seg - 1)
                    end_dst = sg.slot_base + bh * sg.slot_bh + (int64_t)seg * sg.slot_k;
            } else if (final_state && (sg.mode == 0 || seg == sg.n_seg - 1)) {
                end_dst = final_state + bh * g.P * g.S;
            }
            if (end_dst && s_ok) {
#pragma unroll
                for (int p = 0; p < PH; ++p)
                    end_dst[(int64_t)(p0 + p) * g.S + s_idx] = hs[p];
            }
        }
        if (Lay::kTmaEmit && tma_emit && tid == 0)
            bulk_wait_all();  // the staging box must outlive its last store
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
    // chunk states [B, H, nc, P, S] as f32 rows of S; box {min(S, 128), P}
    CUtensorMap tst;
    memset(&tst, 0, sizeof(tst));
    const int64_t rows = g.B * g.H * g.nc * g.P;
    const int tma_emit = SpLayout<P>::kTmaEmit && states && rows < (1LL << 31) &&
                         make_tmap_f32_rows(&tst, states, (uint64_t)g.S, (uint64_t)rows,
                                            (uint32_t)(g.S < 128 ? g.S : 128), (uint32_t)P);
    const size_t smem = SpLayout<P>::bytes + 1024;
    auto k = state_pass_tc_kernel<P, REV>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    dim3 grid((unsigned)((g.S + 127) / 128), (unsigned)(g.B * g.H), (unsigned)(sg.mode ? sg.n_seg : 1));
    k<<<grid, kThreads, smem, st>>>(tx, tb, tst, dtT, Gc, init, states, final_state, g, status, sg,
                                    tma_emit);
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
// valid tokens.  One thread per state element; each warp of the block sums
// the decays of some segments, its lanes striding over the segment's chunks.
// The slot loads are independent of the carried state, so they are issued
// eight at a time ahead of the chain.
__global__ void __launch_bounds__(256)
seg_combine_kernel(const float *__restrict__ Gc, const float *__restrict__ init, Geom g, SpSeg sg)
{
    __shared__ float sdec[kMaxSeg];
    const int64_t bh = blockIdx.y;
    const int chunks_per_seg = sg.seg_tiles * kTile / g.T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int k = warp; k < sg.n_seg - 1; k += blockDim.x >> 5) {
        float d = 0.f;
        for (int c = k * chunks_per_seg + lane; c < (k + 1) * chunks_per_seg && c < g.nc; c += 32)
            d += Gc[bh * g.L + min64(g.L, (int64_t)(c + 1) * g.T) - 1];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            d += __shfl_xor_sync(0xffffffffu, d, o);
        if (lane == 0)
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

// Start states of n_seg segments of seg_tiles tiles each (a whole number of
// chunks): pass 1 and the combine of the segmented pass, with
// slots[(bh * n_seg + k) * P * S ..] receiving the state at the start of
// segment k + 1 (k < n_seg - 1).  For kernels that then run every segment at
// once from these states.
cudaError_t launch_segment_starts_tc(const void *x, const void *Bm, const float *dtT,
                                     const float *Gc, const float *init, float *slots,
                                     int seg_tiles, int n_seg, const Geom &g, cudaStream_t st)
{
    if (!state_pass_tc_supported(g) || n_seg < 2 || n_seg > kMaxSeg ||
        (seg_tiles * kTile) % g.T != 0)
        return cudaErrorNotSupported;
    unsigned int *status = device_status_word();
    if (!status)
        return cudaErrorUnknown;
    CUtensorMap tx, tb;
    if (!make_tmap_tokens_heads(&tx, x, g) || !make_tmap_tokens_groups(&tb, Bm, g))
        return cudaErrorInvalidValue;
    SpSeg sg{};
    sg.mode = 1;
    sg.seg_tiles = seg_tiles;
    sg.n_seg = n_seg;
    sg.slot_base = slots;
    sg.slot_k = g.P * g.S;
    sg.slot_bh = (int64_t)n_seg * sg.slot_k;
    cudaError_t e =
        g.P == 64 ? launch_p<64, false>(tx, tb, dtT, Gc, nullptr, nullptr, nullptr, g, status, st, sg)
                  : launch_p<128, false>(tx, tb, dtT, Gc, nullptr, nullptr, nullptr, g, status, st, sg);
    if (e != cudaSuccess)
        return e;
    const dim3 cgrid((unsigned)((g.P * g.S + 255) / 256), (unsigned)(g.B * g.H));
    seg_combine_kernel<<<cgrid, 256, 0, st>>>(Gc, init, g, sg);
    note_launch();
    return cudaGetLastError();
}

}  // namespace ssd
