// Fused SSD forward (state pass + chunk output) for TWO heads of one B/C
// group per CTA, on tensor cores, bf16 inputs, headdim 64, dstate 64 or 128.
//
// "Accelerating Mamba-2 forward-pass kernels with CUDA Tile (cuTile)",
// section "Kernel 2: fwd_pass_state" (state jump) and section
// "Kernel 3: compute_out":
//     Y = exp2(G) * (C h_c^T) + (exp2(G_i - G_j) * (C B^T) * M)(dt * X) + D X,
//     h <- exp2(G_last) h + X^T (B * dt * exp2(G_last - G)).
//
// Heads of one group share B and C, so a CTA that carries two of them loads
// each B / C tile once and computes C B^T once.  Per 128-token tile and head,
// with g = G relative to the chunk start (non-increasing) and a reference
// g_ref inside the tile's range,
//     exp2(g_i - g_j) dt_j = exp2(g_i - g_ref) * [dt_j exp2(g_ref - g_j)]
// splits the decay into a row factor and a column factor.  While both factors
// stay within 2^kRefRange (log2 units) the score matrix is the masked C B^T
// itself -- the same for both heads -- and
//     Y_k   = D x / r  +  C H_k^T  +  (M * C B^T) X_hat_k      (one accumulator)
//     y_k,i = r_i Y_k,i,      r_i = exp2(g_i - g_ref)
// with X_hat_k = dt exp2(g_ref - g) x_k and H_k = bf16(exp2(g_ref) h_k).  The
// state jump uses the same X_hat: h_end = exp2(g_L - g_ref) [exp2(g_ref) h +
// B^T X_hat].  The state is stored as S with h = exp2(lp) S and the reference
// is normally g_ref = -lp: then exp2(g_ref) h = S, so H = bf16(S) and the
// stored state needs no rescaling -- the jump adds B^T X_hat to S and the
// tile's decay goes into lp (lp <- lp + g_L).  Only when an exponent would
// leave 2^(+-kRefRange) is the scale folded into S, with g_ref at the middle
// of the tile's range (S <- exp2(g_ref) h, lp <- g_L - g_ref).  Both heads' contractions then run as
// single N = 128 MMAs: C [H_0 | H_1]^T, B^T [X_hat_0 | X_hat_1] (bf16 hi + lo
// passes, so the carried state keeps ~16 mantissa bits) and
// (M * C B^T) [X_hat_0 | X_hat_1].
//
// A tile whose decay exceeds kRefRange for a head (a very fast-decaying head)
// takes the exact per-element form for that head: its scores
// CB_ij exp2(g_i - g_j) dt_j are built in a TMEM region of their own and
// multiply the raw x, the state reference is g_L, and its Y accumulator is
// rescaled by exp2(g_i) (plus D x) before the score product is added.
//
// Roles (one CTA per SM, persistent over (batch, head pair, segment) items):
//   warps 0-3 / 4-7  warpgroup k owns head k of the pair: thread i owns tile
//                    row / TMEM lane i for X_hat, the state, and the output;
//                    the shared scores are split between the warpgroups by keys;
//   warp 8           TMA loads: x of each head as soon as its X_hat is built,
//                    B and C as soon as the tile's MMAs that read them are done
//                    (single-buffered: the loads overlap the rest of the tile);
//   warp 9           MMA issue;
//   warp 10          TMA store of y (staged in the H buffers).
// Every wait is bounded; a timeout sets the kernel status word and the role
// leaves its loop.
#include "common.cuh"
#include "ssd_internal.h"
#include "tc05.cuh"

namespace ssd {
namespace {
using namespace tc;

constexpr int kTile = 128;
constexpr int kWarps = 8;  // compute warps; warpgroup k owns head k
constexpr int kThreads = kWarps * 32 + 96;
constexpr uint32_t kRegion = 128 * 128;  // 128 rows of 128 bytes (64 bf16)
// The factorized form is used while every row and column factor stays within
// 2^(+-kRefRange) (log2 units); a tile whose decay range exceeds 2 kRefRange
// takes the exact per-element form.  Scale products are never formed as one
// scalar (2^-100 * 2^-100 is below the f32 range); each factor is applied in turn.
constexpr float kRefRange = 100.f;

template <int S>
struct PairLayout {
    static constexpr int kSReg = S / 64;  // 64-wide dstate regions of B / C
    static constexpr uint32_t kB = kSReg * kRegion;
    static constexpr uint32_t off_b = 0, off_c = kB;
    static constexpr uint32_t off_x = 2 * kB;                // x of head 0, head 1
    static constexpr uint32_t off_xh = off_x + 2 * kRegion;  // X_hat hi0, hi1, lo0, lo1
    static constexpr uint32_t off_h = off_xh + 4 * kRegion;  // H0, H1 (MN-major [s][p]); y staging
    static constexpr uint32_t off_g = off_h + 2 * kRegion;   // [parity][head][g 128 | dt 128] f32
    // the next tile's dt of both heads: [parity][128 rows][2 heads] f32
    static constexpr uint32_t off_raw = off_g + 2 * 2 * 256 * 4;
    static constexpr uint32_t bytes = off_raw + 2 * 128 * 2 * 4;
    // TMEM columns: CB (f32), shared masked scores (bf16 pairs), Y of both
    // heads, the f32 states h^T [S, P] of both heads, one wide-score region
    static constexpr uint32_t t_cb = 0, t_sc = 128, t_y = 192, t_st = 320, t_wide = 448;
    static_assert(S == 64 || S == 128, "state rows fit one 128-lane TMEM block");
    static_assert(bytes + 1024 + 512 <= 232448, "shared memory budget");
};

struct PairParams {
    const float *dt, *A, *D, *init;  // dt in the input layout [B, L, H]
    float *states_out, *final_state;
    Geom g;
    int n_items, n_tiles, tpc_shift;
    int batch, H, npairs, hpg;
    // Work assignment, one of:
    //  wrap  -- (at least as many head pairs as CTAs) all pairs' tiles laid end
    //           to end and cut into one contiguous piece per CTA; a CTA first
    //           runs the start of the sequence crossing its upper cut (handing
    //           its state off), then its whole sequences, then the rest of the
    //           sequence crossing its lower cut, which its neighbour started
    //           first.  A piece is at least one sequence long, so the hand-off
    //           is always complete before it is needed.
    //  segments -- each sequence is split into n_seg segments of seg_tiles
    //           tiles, items (pair, segment) dealt round-robin, segment-major.
    // Segment k > 0 starts from the state segment k-1 leaves in seg_state,
    // published by seg_count reaching 4 (one count per warp) -- unless
    // `prefilled`: then a state pass has already put every segment's start
    // state in seg_state, all items are independent and none hands off.
    int wrap, prefilled;
    long long wrap_units;  // B * H/2 * n_tiles
    int seg_tiles, n_seg;
    float *seg_state;         // [B*H*n_seg][P][S]
    unsigned int *seg_count;  // [B*H*n_seg], zero at launch
    unsigned int *status;
    // Bounded waits give up after wait_ns.  Fault injection (a host-set debug
    // parameter, off by default): with fault_skip_arrive, compute warp 0 of
    // every CTA skips its X_hat-barrier arrival on the CTA's first tile, so
    // the waits on that barrier run out and every role leaves its loop with
    // no copy or MMA in flight (see the launcher).
    unsigned long long wait_ns;
    int fault_skip_arrive;
};

struct PItem {
    int b, h0, grp, t0, t1, seg;
};

__device__ __forceinline__ PItem pair_item(const PairParams &p, unsigned q, int t0, int t1, int seg)
{
    PItem w;
    w.b = (int)(q / (unsigned)p.npairs);
    w.h0 = 2 * (int)(q % (unsigned)p.npairs);
    w.grp = (int)((unsigned)w.h0 / (unsigned)p.hpg);
    w.t0 = t0;
    w.t1 = t1;
    w.seg = seg;
    return w;
}

// This CTA's share of the work, worked out once per CTA (the 64-bit
// arithmetic of the wrap plan stays out of the per-item code).
struct Plan {
    int count;               // items of this CTA
    int head;                // wrap: the first item starts the sequence crossing the upper cut
    int hi_q, hi_t;          //   that sequence and the tile where the cut falls
    int first_full, n_full;  //   whole sequences [first_full, first_full + n_full)
    int lo_q, lo_t;          //   the sequence crossing the lower cut, from tile lo_t on
};

__device__ __noinline__ void make_plan(const PairParams &p, Plan &pl)
{
    if (!p.wrap) {
        pl.count = (int)blockIdx.x < p.n_items ? (p.n_items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
        pl.head = pl.hi_q = pl.hi_t = pl.first_full = pl.n_full = pl.lo_q = pl.lo_t = 0;
        return;
    }
    // this CTA's piece [lo, hi) of the pair-major tile sequence
    const long long lo = (long long)blockIdx.x * p.wrap_units / gridDim.x;
    const long long hi = (long long)(blockIdx.x + 1) * p.wrap_units / gridDim.x;
    const long long n = p.n_tiles;
    const long long first_full = (lo + n - 1) / n, end_full = hi / n;
    pl.head = hi % n != 0;
    pl.hi_q = (int)(hi / n);
    pl.hi_t = (int)(hi % n);
    pl.first_full = (int)first_full;
    pl.n_full = (int)(end_full - first_full);
    pl.lo_q = (int)(lo / n);
    pl.lo_t = (int)(lo % n);
    pl.count = pl.head + pl.n_full + (lo % n != 0);
}

// The j-th item of this CTA, in the order it runs them.
__device__ __forceinline__ PItem my_item(const PairParams &p, const Plan &pl, int j)
{
    unsigned q;
    int t0, t1, seg;
    if (!p.wrap) {
        // segment-major: every segment k of every head pair comes before any
        // segment k+1, so a segment's predecessor is always an earlier item
        const unsigned item = blockIdx.x + (unsigned)j * gridDim.x;
        const unsigned per_seg = (unsigned)(p.batch * p.npairs);
        const unsigned sg = item / per_seg;
        q = item - sg * per_seg;
        seg = (int)sg;
        t0 = seg * p.seg_tiles;
        t1 = min(t0 + p.seg_tiles, p.n_tiles);
    } else if (pl.head && j == 0) {
        // start of the sequence crossing the upper cut: hands its state off
        q = (unsigned)pl.hi_q;
        t0 = 0;
        t1 = pl.hi_t;
        seg = 0;
    } else if (j - pl.head < pl.n_full) {
        q = (unsigned)(pl.first_full + j - pl.head);
        t0 = 0;
        t1 = p.n_tiles;
        seg = 0;
    } else {
        // rest of the sequence crossing the lower cut, from its neighbour's state
        q = (unsigned)pl.lo_q;
        t0 = pl.lo_t;
        t1 = p.n_tiles;
        seg = 1;
    }
    return pair_item(p, q, t0, t1, seg);
}

template <int S>
__global__ void __launch_bounds__(kThreads, 1)
pair_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_y,
               const PairParams prm)
{
    using Lay = PairLayout<S>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // TMA landed: B and C; x of head k
    __shared__ uint64_t bar_bc, bar_x[2];
    // MMA completions: CB; Y2; Y2 + state jump (B / C / X_hat free); Y1 (Y complete)
    __shared__ uint64_t bar_cb, bar_y2, bar_ds, bar_y, bar_end;
    // compute warps (8 arrivals): X_hat + D x + modes; H + decayed state;
    // scores (+ wide rescale); y staged
    __shared__ uint64_t bar_xh, bar_h, bar_sc, bar_ys;
    // the y store has read the H buffers
    __shared__ uint64_t bar_hfree;
    __shared__ uint32_t tmem_slot;
    __shared__ int s_mode[2][2];  // [tile parity][head]: 1 = factorized
    __shared__ Plan s_plan;

    const Geom &g = prm.g;
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint64_t wait_ns = prm.wait_ns;

    if (tid == 0) {
        mbar_init(&bar_bc, 1);
        mbar_init(&bar_x[0], 1);
        mbar_init(&bar_x[1], 1);
        mbar_init(&bar_cb, 1);
        mbar_init(&bar_y2, 1);
        mbar_init(&bar_ds, 1);
        mbar_init(&bar_y, 1);
        mbar_init(&bar_end, 1);
        mbar_init(&bar_xh, kWarps);
        mbar_init(&bar_h, kWarps);
        mbar_init(&bar_sc, kWarps);
        mbar_init(&bar_ys, kWarps);
        mbar_init(&bar_hfree, 1);
        fence_barrier_init();
        make_plan(prm, s_plan);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const bool want_final = prm.final_state != nullptr;

    if (warp == 8) {
        // ---------------- TMA loads.  The tile-it loads wait for tile it-1 to
        // release each buffer: x of a factorized head once its X_hat is built,
        // x of a wide head once its score product is done, B / C once CB, Y2
        // and the state jump are done.
        if ((tid & 31) == 0) {
            prefetch_tmap(&tm_x);
            prefetch_tmap(&tm_b);
            prefetch_tmap(&tm_c);
            uint32_t it = 0;
            bool ok = true;
            const int n_my = s_plan.count;
            for (int j = 0; j < n_my && ok; ++j) {
                const PItem w = my_item(prm, s_plan, j);
                for (int t = w.t0; t < w.t1; ++t, ++it) {
                    const int tok = t * kTile;
                    auto load_x = [&](int k) {
                        mbar_arrive_expect_tx(&bar_x[k], kRegion);
                        tma4(smem + Lay::off_x + k * kRegion, &tm_x, &bar_x[k], 0, w.h0 + k, tok, w.b);
                    };
                    auto load_bc = [&]() {
                        mbar_arrive_expect_tx(&bar_bc, 2 * Lay::kB);
                        for (int r = 0; r < Lay::kSReg; ++r) {
                            tma4(smem + Lay::off_b + r * kRegion, &tm_b, &bar_bc, r * 64, w.grp, tok, w.b);
                            tma4(smem + Lay::off_c + r * kRegion, &tm_c, &bar_bc, r * 64, w.grp, tok, w.b);
                        }
                    };
                    if (it == 0) {
                        load_x(0);
                        load_x(1);
                        load_bc();
                        continue;
                    }
                    const uint32_t pp = (it - 1) & 1;
                    if (!mbar_wait(&bar_xh, pp, wait_ns)) {
                        ok = false;
                        break;
                    }
                    const int m0 = s_mode[pp][0], m1 = s_mode[pp][1];
                    if (m0)
                        load_x(0);
                    if (m1)
                        load_x(1);
                    if (!mbar_wait(&bar_ds, pp, wait_ns)) {
                        ok = false;
                        break;
                    }
                    load_bc();
                    if (!m0 || !m1) {
                        if (!mbar_wait(&bar_y, pp, wait_ns)) {
                            ok = false;
                            break;
                        }
                        if (!m0)
                            load_x(0);
                        if (!m1)
                            load_x(1);
                    }
                }
            }
            if (!ok)
                atomicOr(prm.status, 1u);
        }
    } else if (warp == 9) {
        // ---------------- MMA issue.  Per tile: CB; Y2 (both heads); the state
        // jump (both heads, hi + lo); then Y1 once the scores are ready.
        if ((tid & 31) == 0) {
            const uint32_t id_cb = idesc_bf16(128, 128, false, false);
            const uint32_t id_y2 = idesc_bf16(128, 128, false, true);  // H is MN-major
            const uint32_t id_ds = idesc_bf16(128, 128, true, true);   // B^T, X_hat MN-major
            const uint32_t id_y1p = idesc_bf16(128, 128, false, true);  // A (scores) from TMEM
            const uint32_t id_y1h = idesc_bf16(128, 64, false, true);
            const uint64_t d_bk = desc_k0(smem_u32(smem + Lay::off_b));
            const uint64_t d_ck = desc_k0(smem_u32(smem + Lay::off_c));
            const uint64_t d_bmn = desc_mn0(smem_u32(smem + Lay::off_b), kRegion);
            const uint64_t d_h = desc_mn0(smem_u32(smem + Lay::off_h), kRegion);
            const uint64_t d_hi = desc_mn0(smem_u32(smem + Lay::off_xh), kRegion);
            const uint64_t d_lo = desc_mn0(smem_u32(smem + Lay::off_xh + 2 * kRegion), kRegion);
            const uint64_t d_x = desc_mn0(smem_u32(smem + Lay::off_x), kRegion);
            constexpr uint32_t kStep = kRegion >> 4;  // one region in descriptor units
            uint32_t it = 0;
            bool ok = true;
            const int n_my = s_plan.count;
            for (int j = 0; j < n_my && ok; ++j) {
                const PItem w = my_item(prm, s_plan, j);
                for (int t = w.t0; t < w.t1; ++t, ++it) {
                    const bool last_seq = t + 1 == prm.n_tiles;
                    const bool do_state = !last_seq || want_final;
                    const uint32_t par = it & 1;
                    // CB overwrites the previous tile's CB, whose conversion
                    // ended before that tile's Y1 was issued
                    if (!mbar_spin(&bar_bc, par, wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < S / 16; ++ks)
                        mma_ss(tmem + Lay::t_cb, desc_k(d_ck, kRegion, ks), desc_k(d_bk, kRegion, ks),
                               id_cb, ks > 0);
                    mma_commit(&bar_cb);
                    if (!mbar_spin(&bar_xh, par, wait_ns) || !mbar_spin(&bar_h, par, wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // Y += C [H_0 | H_1]^T  (Y holds D x / r, or zero for a wide head)
#pragma unroll
                    for (int ks = 0; ks < S / 16; ++ks)
                        mma_ss(tmem + Lay::t_y, desc_k(d_ck, kRegion, ks), desc_mn(d_h, ks), id_y2, 1u);
                    mma_commit(&bar_y2);
                    // The state jump (hi, then lo) right after Y2, in one straight
                    // run of MMAs: with Y2 it is the last reader of the B / C tiles,
                    // the H buffers and the X_hat lo buffers, so their reuse for the
                    // next tile can start as soon as it completes; the compute warps
                    // build the next tile's H from its result while Y1 runs.
                    if (do_state) {
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            mma_ss(tmem + Lay::t_st, desc_mn(d_bmn, u), desc_mn(d_hi, u), id_ds, 1u);
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            mma_ss(tmem + Lay::t_st, desc_mn(d_bmn, u), desc_mn(d_lo, u), id_ds, 1u);
                    }
                    mma_commit(&bar_ds);
                    // Y1 once the scores are ready: both heads in one N = 128 MMA
                    // when both are factorized, else per head.
                    auto issue_y1 = [&]() {
                        tc_fence_after();
                        const int m0 = s_mode[par][0], m1 = s_mode[par][1];
                        if (m0 && m1) {
#pragma unroll
                            for (int ks = 0; ks < kTile / 16; ++ks)
                                mma_ts(tmem + Lay::t_y, tmem + Lay::t_sc + ks * 8, desc_mn(d_hi, ks),
                                       id_y1p, 1u);
                        } else {
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                const int mk = k ? m1 : m0;
                                // a wide head 0 uses the shared region when head 1 is wide too
                                const uint32_t a =
                                    mk ? Lay::t_sc : ((k == 0 && !m1) ? Lay::t_sc : Lay::t_wide);
                                const uint64_t bd = (mk ? d_hi : d_x) + k * kStep;
#pragma unroll
                                for (int ks = 0; ks < kTile / 16; ++ks)
                                    mma_ts(tmem + Lay::t_y + 64 * k, tmem + a + ks * 8,
                                           desc_mn(bd, ks), id_y1h, 1u);
                            }
                        }
                        mma_commit(&bar_y);
                    };
                    if (!mbar_spin(&bar_sc, par, wait_ns)) {
                        ok = false;
                        break;
                    }
                    issue_y1();
                    if (!ok)
                        break;
                }
            }
            if (!ok)
                atomicOr(prm.status, 1u);
            // every MMA this thread issued has completed before TMEM is freed
            mma_commit(&bar_end);
            if (!mbar_wait(&bar_end, 0, wait_ns))
                atomicOr(prm.status, 1u);
        }
    } else if (warp == 10) {
        // ---------------- y store from the X_hat lo buffers (its staging)
        if ((tid & 31) == 0) {
            prefetch_tmap(&tm_y);
            uint32_t it = 0;
            bool ok = true;
            const int n_my = s_plan.count;
            for (int j = 0; j < n_my && ok; ++j) {
                const PItem w = my_item(prm, s_plan, j);
                for (int t = w.t0; t < w.t1; ++t, ++it) {
                    if (!mbar_wait(&bar_ys, it & 1, wait_ns)) {
                        ok = false;
                        break;
                    }
                    tma4_store(&tm_y, smem + Lay::off_xh + 2 * kRegion, 0, w.h0, t * kTile, w.b);
                    tma4_store(&tm_y, smem + Lay::off_xh + 3 * kRegion, 0, w.h0 + 1, t * kTile, w.b);
                    bulk_commit();
                    bulk_wait_read();
                    mbar_arrive(&bar_hfree);
                }
            }
            bulk_wait_all();
            if (!ok)
                atomicOr(prm.status, 1u);
        }
    } else if (warp < kWarps) {
        // ---------------- compute: warpgroup k owns head h0 + k
        //
        // Order per tile `it` (the next tile is it + 1):
        //   scores(it) -> G of it + 1 -> [state leaving the item] -> H(it + 1)
        //   -> epilogue(it) -> X_hat(it + 1)
        // so the next tile's H is built while Y1(it) runs on the tensor cores,
        // and y(it) is staged in the X_hat lo buffers (free once the state
        // jump of `it` is done), which leaves the H buffers to H(it + 1).
        const int k = warp >> 2, q = warp & 3;
        const int i = q * 32 + (tid & 31);
        const int row_lo = q * 32, row_hi = q * 32 + 31;
        const uint32_t tl = tmem_at(tmem, (uint32_t)(q * 32), 0);
        const uint32_t ty = tl + Lay::t_y + 64 * k, tst = tl + Lay::t_st + 64 * k;
        const bool srow = q * 32 < S;  // warp-uniform: this warp's rows are state rows
        float *gtab_all = reinterpret_cast<float *>(smem + Lay::off_g);
        uint8_t *sx = smem + Lay::off_x + k * kRegion;
        uint8_t *s_hi = smem + Lay::off_xh + k * kRegion;
        uint8_t *s_lo = smem + Lay::off_xh + (2 + k) * kRegion;
        uint8_t *s_h = smem + Lay::off_h + k * kRegion;
        const int tpc_mask = (1 << prm.tpc_shift) - 1;

        // dt of a tile for both heads (adjacent in the [B, L, H] input), copied
        // two tiles ahead by cp.async: thread i of warpgroup 0 copies row i's
        // pair of words into slot [parity][i][2].  Each thread waits for its
        // copy before arriving at the X_hat barrier of the tile before it, so
        // every compute thread may read the whole tile once it has passed that
        // barrier.  G within the tile is then a prefix sum each warp computes
        // with shuffles, so no separate cumsum pass is needed.
        float *raw_all = reinterpret_cast<float *>(smem + Lay::off_raw);
        const int lane_id = tid & 31;
        auto prefetch_dt = [&](const PItem &w, int t, uint32_t buf) {
            if (k != 0)
                return;
            float *slot = raw_all + (buf * 128 + i) * 2;
            const int tau = t * kTile;
            const int n = min(kTile, (int)g.L - tau);
            if (i < n) {
                cp_async8(slot, prm.dt + ((int64_t)w.b * g.L + tau + i) * prm.H + w.h0);
            } else {  // past the sequence end: dt = 0
                slot[0] = 0.f;
                slot[1] = 0.f;
            }
            cp_async_commit();
        };
        // Within-tile G (log2 units, relative to the token before the tile):
        // this row's g and dt, the first row's g and the tile total g_L.
        struct TileG {
            float gi, dti, g0, gL;
        };
        auto tile_g = [&](uint32_t buf, float a_l2) {
            const float *slot = raw_all + buf * 128 * 2 + k;
            float incl[4], d[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                d[m] = slot[(32 * m + lane_id) * 2];
                float v = a_l2 * d[m];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float u = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane_id >= o)
                        v += u;
                }
                incl[m] = v;
            }
            float tot[4], pre = 0.f, mine_pre = 0.f, mine = 0.f, mine_d = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                tot[m] = __shfl_sync(0xffffffffu, incl[m], 31);
                if (m == q) {
                    mine_pre = pre;
                    mine = incl[m];
                    mine_d = d[m];
                }
                pre += tot[m];
            }
            TileG tg;
            tg.gi = mine_pre + mine;
            tg.dti = mine_d;
            tg.g0 = __shfl_sync(0xffffffffu, incl[0], 0);
            tg.gL = pre;  // rows past the end add nothing
            return tg;
        };

        // Position of a tile in this CTA's work: item j, tile t, and the
        // item's head's A and D.
        struct Pos {
            PItem w;
            int j, t;
            float a, d;
            bool valid;
        };
        const int n_my = s_plan.count;
        auto first_pos = [&]() {
            Pos p{};
            p.valid = n_my > 0;
            if (p.valid) {
                p.j = 0;
                p.w = my_item(prm, s_plan, 0);
                p.t = p.w.t0;
                p.a = ld_early(prm.A + p.w.h0 + k);
                p.d = ld_early(prm.D + p.w.h0 + k);
            }
            return p;
        };
        auto next_pos = [&](const Pos &p) {
            Pos n = p;
            if (!p.valid)
                return n;
            if (p.t + 1 < p.w.t1) {
                n.t = p.t + 1;
                return n;
            }
            if (p.j + 1 >= n_my) {
                n.valid = false;
                return n;
            }
            n.j = p.j + 1;
            n.w = my_item(prm, s_plan, n.j);
            n.t = n.w.t0;
            n.a = ld_early(prm.A + n.w.h0 + k);
            n.d = ld_early(prm.D + n.w.h0 + k);
            return n;
        };

        // One tile: its place, its G, and the decay reference chosen for it.
        // Reference gref of the factorized form: keep the stored state's scale
        // (gref = -lp) while every exponent gref - g_j, g_i - gref stays within
        // kRefRange; else fold the scale into the state with gref at the middle
        // of the tile's range; beyond 2 kRefRange the exact per-element form
        // for this head (gref = g_L).
        struct Tile {
            PItem w;
            int t, n;
            uint32_t it;
            bool first, last_item, last_seq, do_state, keep, narrow;
            float gi, dti, gL, gref, Dh, lp;  // lp: the stored state's scale on entry
            int64_t bh;
        };
        auto make_tile = [&](const Pos &p, uint32_t it, const TileG &tg, float lp) {
            Tile c;
            c.w = p.w;
            c.t = p.t;
            c.it = it;
            c.n = min(kTile, (int)g.L - p.t * kTile);
            c.first = p.t == p.w.t0;
            c.last_item = p.t + 1 == p.w.t1;
            c.last_seq = p.t + 1 == prm.n_tiles;
            c.do_state = !c.last_seq || want_final;
            c.gi = tg.gi;
            c.dti = tg.dti;
            c.gL = tg.gL;
            const float gmin = fminf(tg.g0, tg.gL), gmax = fmaxf(tg.g0, tg.gL);
            c.keep = !c.first && -lp - gmin <= kRefRange && gmax + lp <= kRefRange;
            c.narrow = c.keep || gmax - gmin <= 2.f * kRefRange;
            c.gref = c.keep ? -lp : (c.narrow ? 0.5f * (gmin + gmax) : tg.gL);
            c.Dh = p.d;
            c.lp = c.first ? 0.f : lp;
            c.bh = (int64_t)p.w.b * prm.H + p.w.h0 + k;
            return c;
        };

        // ---- X_hat = dt exp2(gref - g) x (hi, lo) and Y = D x / r (0 if wide).
        // Packed bf16 arithmetic with the weight w split as w_hi + w_lo:
        // hi = bf16(x w_hi); the rounding residual x w_hi - hi is exact in
        // bf16 (x and w_hi carry 8 significant bits each), so
        // lo = bf16(x w_lo + residual) leaves hi + lo within ~2^-16 of x w.
        // hi and Y go out first; lo is held in registers until the previous
        // tile's y store has read the lo buffers (its staging area).
        auto build_xhat = [&](const Tile &c) -> bool {
            const uint32_t par = c.it & 1;
            float *gtab = gtab_all + (par * 2 + k) * 256;
            gtab[i] = c.gi;
            gtab[128 + i] = c.dti;
            if (i == 0)
                s_mode[par][k] = c.narrow ? 1 : 0;
            if (!mbar_wait(&bar_x[k], par, wait_ns))
                return false;
            tc_fence_after();
            const float e = ex2_approx(c.gref - c.gi);
            const float wv = i < c.n ? c.dti * e : 0.f;
            const float dsc = c.narrow ? c.Dh * e : 0.f;
            const uint32_t whi = pack_bf16x2(wv, wv);
            const float wv_lo = wv - bf_lo(whi);
            const uint32_t wlo = pack_bf16x2(wv_lo, wv_lo);
            const uint64_t dsc2 = f2_pack(__float_as_uint(dsc), __float_as_uint(dsc));
            uint32_t lo_keep[8][4];
            // every x load before the first store (the stores go to other
            // buffers, which the compiler cannot tell)
            uint4 xv[8];
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                xv[ch] = *reinterpret_cast<const uint4 *>(sx + sw128_offset(i, ch));
#pragma unroll
            for (int c2 = 0; c2 < 4; ++c2) {
                uint32_t dx[16];
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int ch = 2 * c2 + cc;
                    const uint32_t off = sw128_offset(i, ch);
                    const uint4 v = xv[ch];
                    const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
                    uint32_t hi[4];
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {
                        hi[e2] = bf2_mul(vv[e2], whi);
                        lo_keep[ch][e2] = bf2_fma(vv[e2], wlo, bf2_fma(vv[e2], whi, hi[e2] ^ 0x80008000u));
                        f2_unpack(f2_mul(bf2_to_f2(vv[e2]), dsc2), dx[8 * cc + 2 * e2],
                                  dx[8 * cc + 2 * e2 + 1]);
                    }
                    *reinterpret_cast<uint4 *>(s_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                }
                tmem_st16(ty + 16 * c2, dx);
            }
            // the previous tile's y store has read the lo buffers
            if (c.it > 0 && !mbar_wait(&bar_hfree, par ^ 1u, wait_ns))
                return false;
            if (c.do_state) {
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    *reinterpret_cast<uint4 *>(s_lo + sw128_offset(i, ch)) =
                        make_uint4(lo_keep[ch][0], lo_keep[ch][1], lo_keep[ch][2], lo_keep[ch][3]);
            }
            fence_proxy_async_smem();
            tmem_st_wait();
            tc_fence_before();
            cp_async_wait_all();  // the dt copied for the tile after this one
            if (!(prm.fault_skip_arrive && c.it == 0 && warp == 0))
                warp_arrive(&bar_xh);
            return true;
        };

        // ---- H = bf16(exp2(gref) h) for the factorized form, bf16(h) for the
        // exact one (MN-major [s][p]).  The stored state is rewritten only
        // when its scale is folded in: S <- exp2(lp) S, times exp2(g_L) if
        // exact.  A non-first tile reads the state the previous tile's jump
        // left (the caller waited for that jump); an item's first tile loads
        // its start state (a later segment waits until its predecessor has
        // published it).
        auto build_h = [&](const Tile &c) -> bool {
            if (c.first && c.w.seg > 0 && !prm.prefilled) {
                const unsigned int *cnt = prm.seg_count + c.bh * prm.n_seg + c.w.seg - 1;
                bool ready = ld_acquire_gpu(cnt) >= 4u;
                const uint64_t t_start = globaltimer_ns();
                while (!ready) {
                    if (globaltimer_ns() - t_start > wait_ns)
                        break;
                    __nanosleep(256);
                    ready = ld_acquire_gpu(cnt) >= 4u;
                }
                if (!ready)
                    return false;
            }
            const bool fold = !c.keep;
            const bool emit = prm.states_out && (c.t & tpc_mask) == 0;
            if (srow) {
                const float *src = nullptr;
                if (c.first) {
                    if (c.w.seg > 0)
                        src = prm.seg_state + ((c.bh * prm.n_seg + c.w.seg - 1) * g.P) * g.S;
                    else if (prm.init)
                        src = prm.init + c.bh * g.P * g.S;
                }
                float *emit_dst =
                    emit ? prm.states_out + ((c.bh * g.nc + (c.t >> prm.tpc_shift)) * g.P) * g.S
                         : nullptr;
                // The pending scale and the new reference scale are applied one
                // after the other: their product can fall below the f32 range
                // even though each scaled value does not.
                const float pv = c.first ? 1.f : ex2_approx(c.lp);
                const float eref = ex2_approx(c.gref);
                const float hsc = c.narrow ? eref : 1.f;
                // the whole 64-column state row in one TMEM round trip
                uint32_t r[64];
                if (c.first) {
#pragma unroll
                    for (int jj = 0; jj < 64; ++jj)
                        r[jj] = __float_as_uint(src ? __ldcg(src + (int64_t)jj * S + i) : 0.f);
                } else {
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq)
                        tmem_ld16(tst + 16 * qq, *reinterpret_cast<uint32_t(*)[16]>(r + 16 * qq));
                    tmem_ld_wait();
                }
                if (emit_dst) {
#pragma unroll
                    for (int jj = 0; jj < 64; ++jj)
                        emit_dst[(int64_t)jj * S + i] = pv * __uint_as_float(r[jj]);
                }
                // scaling runs on f32 pairs
                auto scaled = [&](int jj, uint64_t s2, uint32_t &a, uint32_t &b) {
                    f2_unpack(f2_mul(f2_pack(r[jj], r[jj + 1]), s2), a, b);
                };
                if (fold) {  // r <- the true state h
                    const uint64_t pv2 = f2_pack(__float_as_uint(pv), __float_as_uint(pv));
#pragma unroll
                    for (int jj = 0; jj < 64; jj += 2)
                        scaled(jj, pv2, r[jj], r[jj + 1]);
                }
                // keep: H = bf16(S); fold: H = bf16(hsc h)
                const uint64_t hs2 = f2_pack(__float_as_uint(hsc), __float_as_uint(hsc));
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    uint32_t hp[4];
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {
                        const int jj = 8 * cc + 2 * e2;
                        uint32_t a = r[jj], b = r[jj + 1];
                        if (!c.keep)
                            scaled(jj, hs2, a, b);
                        hp[e2] = pack_bf16x2(__uint_as_float(a), __uint_as_float(b));
                    }
                    *reinterpret_cast<uint4 *>(s_h + sw128_offset(i, cc)) =
                        make_uint4(hp[0], hp[1], hp[2], hp[3]);
                }
                if (fold && c.do_state) {  // stored state <- exp2(gref) h
                    const uint64_t er2 = f2_pack(__float_as_uint(eref), __float_as_uint(eref));
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        uint32_t o[16];
#pragma unroll
                        for (int jj = 0; jj < 16; jj += 2)
                            scaled(16 * qq + jj, er2, o[jj], o[jj + 1]);
                        tmem_st16(tst + 16 * qq, o);
                    }
                }
                if (fold && c.do_state)
                    tmem_st_wait();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(&bar_h);
            return true;
        };

        // ---- scores.  Shared masked CB (keys [64k, 64k + 64) here) when a
        // head is factorized; the exact per-element scores of a wide head.
        auto build_scores = [&](const Tile &c, const Pos &p_after_next) -> bool {
            const uint32_t par = c.it & 1;
            if (!mbar_wait(&bar_cb, par, wait_ns) || !mbar_wait(&bar_xh, par, wait_ns))
                return false;
            tc_fence_after();
            // dt two tiles ahead, into this tile's buffer: every compute warp
            // has formed this tile's G (it arrived at this tile's X_hat
            // barrier after doing so)
            if (p_after_next.valid)
                prefetch_dt(p_after_next.w, p_after_next.t, par);
            const int m0 = s_mode[par][0], m1 = s_mode[par][1];
            if (m0 || m1) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t cbv[2][16];
#pragma unroll
                    for (int gq = 0; gq < 2; ++gq) {
                        const int j0 = 64 * k + 32 * half + 16 * gq;
                        if (j0 <= row_hi)
                            tmem_ld16(tl + Lay::t_cb + j0, cbv[gq]);
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int gq = 0; gq < 2; ++gq) {
                        const int j0 = 64 * k + 32 * half + 16 * gq;
                        uint32_t pk[8];
                        if (j0 > row_hi) {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                pk[e] = 0u;
                        } else if (j0 + 15 < row_lo) {  // whole group below the diagonal
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                pk[e] = pack_bf16x2(__uint_as_float(cbv[gq][2 * e]),
                                                    __uint_as_float(cbv[gq][2 * e + 1]));
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int jk = j0 + 2 * e;
                                pk[e] = pack_bf16x2(jk <= i ? __uint_as_float(cbv[gq][2 * e]) : 0.f,
                                                    jk + 1 <= i ? __uint_as_float(cbv[gq][2 * e + 1]) : 0.f);
                            }
                        }
                        tmem_st8(tl + Lay::t_sc + j0 / 2, pk);
                    }
                }
            }
            if (!c.narrow) {
                // exact scores CB_ij exp2(g_i - g_j) dt_j of this head, all keys
                const float *gtab = gtab_all + (par * 2 + k) * 256;
                const uint32_t region = (k == 0 && !m1) ? Lay::t_sc : Lay::t_wide;
#pragma unroll 1
                for (int j0 = 0; j0 < kTile; j0 += 16) {
                    uint32_t cbv[16], pk[8];
                    if (j0 <= row_hi) {  // warp-uniform
                        tmem_ld16(tl + Lay::t_cb + j0, cbv);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            float v2[2];
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const int jk = j0 + 2 * e + u;
                                v2[u] = jk <= i ? __uint_as_float(cbv[2 * e + u]) *
                                                      ex2_approx(c.gi - gtab[jk]) * gtab[128 + jk]
                                                : 0.f;
                            }
                            pk[e] = pack_bf16x2(v2[0], v2[1]);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            pk[e] = 0u;
                    }
                    tmem_st8(tl + region + j0 / 2, pk);
                }
                // Y = exp2(g_i) (C H^T) + D x, before the score product adds on
                if (!mbar_wait(&bar_y2, par, wait_ns))
                    return false;
                tc_fence_after();
                const float er = ex2_approx(c.gi);
#pragma unroll
                for (int c2 = 0; c2 < 4; ++c2) {
                    uint32_t yv[16];
                    tmem_ld16(ty + 16 * c2, yv);
                    tmem_ld_wait();
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(sx + sw128_offset(i, 2 * c2 + cc));
                        const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            const int o = 8 * cc + 2 * e2;
                            yv[o] = __float_as_uint(er * __uint_as_float(yv[o]) + c.Dh * bf_lo(vv[e2]));
                            yv[o + 1] =
                                __float_as_uint(er * __uint_as_float(yv[o + 1]) + c.Dh * bf_hi(vv[e2]));
                        }
                    }
                    tmem_st16(ty + 16 * c2, yv);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            warp_arrive(&bar_sc);
            return true;
        };

        // ---- the state leaving an item: the next segment's start, or the
        // final state (the caller waited for the item's last jump)
        auto leave_state = [&](const Tile &c) {
            const bool handoff = !c.last_seq && !prm.prefilled;
            float *dst = handoff ? prm.seg_state + ((c.bh * prm.n_seg + c.w.seg) * g.P) * g.S
                                 : ((c.last_seq && want_final) ? prm.final_state + c.bh * g.P * g.S
                                                               : nullptr);
            if (dst && srow) {
                const float pscale = ex2_approx(c.gL - c.gref);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t r[32];
                    tmem_ld16(tst + 32 * half, *reinterpret_cast<uint32_t(*)[16]>(r));
                    tmem_ld16(tst + 32 * half + 16, *reinterpret_cast<uint32_t(*)[16]>(r + 16));
                    tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        __stcg(dst + (int64_t)(32 * half + jj) * S + i, pscale * __uint_as_float(r[jj]));
                }
            }
            if (dst && handoff) {
                __threadfence();
                __syncwarp();
                if ((tid & 31) == 0)
                    atomicAdd(prm.seg_count + c.bh * prm.n_seg + c.w.seg, 1u);
            }
        };

        // ---- epilogue: y = r Y, staged in this head's lo buffer (free once
        // the tile's state jump is done; the caller waited for it)
        auto epilogue = [&](const Tile &c) -> bool {
            const uint32_t par = c.it & 1;
            if (!mbar_wait(&bar_y, par, wait_ns))
                return false;
            tc_fence_after();
            const float r = c.narrow ? ex2_approx(c.gi - c.gref) : 1.f;
            const uint64_t r2 = f2_pack(__float_as_uint(r), __float_as_uint(r));
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t yv[32];
                tmem_ld16(ty + 32 * half, *reinterpret_cast<uint32_t(*)[16]>(yv));
                tmem_ld16(ty + 32 * half + 16, *reinterpret_cast<uint32_t(*)[16]>(yv + 16));
                tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t o[4];
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {
                        uint32_t a, b;
                        f2_unpack(f2_mul(f2_pack(yv[8 * cc + 2 * e2], yv[8 * cc + 2 * e2 + 1]), r2), a, b);
                        o[e2] = pack_bf16x2(__uint_as_float(a), __uint_as_float(b));
                    }
                    *reinterpret_cast<uint4 *>(s_lo + sw128_offset(i, 4 * half + cc)) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(&bar_ys);
            return true;
        };

        bool ok = true;
        Pos p0 = first_pos();
        if (p0.valid) {
            Pos p1 = next_pos(p0);
            Pos p2 = next_pos(p1);
            prefetch_dt(p0.w, p0.t, 0);
            cp_async_wait_all();
            // the first tile's dt is visible to all 256 compute threads
            // (non-aligned form: the copies above leave lanes diverged)
            asm volatile("barrier.sync 1, %0;" ::"r"(kWarps * 32) : "memory");
            Tile cur = make_tile(p0, 0, tile_g(0, kLog2e * p0.a), 0.f);
            if (p1.valid)
                prefetch_dt(p1.w, p1.t, 1);
            ok = build_xhat(cur) && build_h(cur);
            for (uint32_t it = 0; ok; ++it) {
                if (!build_scores(cur, p2)) {
                    ok = false;
                    break;
                }
                TileG tg1{};
                if (p1.valid)  // the next tile's G while the jump runs on the tensor cores
                    tg1 = tile_g((it + 1) & 1, kLog2e * p1.a);

                // this tile's state jump is done: the state, the H buffers and
                // the lo buffers are free
                if (!mbar_wait(&bar_ds, it & 1, wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (cur.last_item && cur.do_state)
                    leave_state(cur);
                Tile nxt{};
                if (p1.valid) {
                    nxt = make_tile(p1, it + 1, tg1, cur.gL - cur.gref);
                    if (!build_h(nxt)) {
                        ok = false;
                        break;
                    }
                }
                if (!epilogue(cur)) {
                    ok = false;
                    break;
                }
                if (!p1.valid)
                    break;
                if (!build_xhat(nxt)) {
                    ok = false;
                    break;
                }
                cur = nxt;
                p1 = p2;
                p2 = next_pos(p2);
            }
        }
        if (!ok)
            atomicOr(prm.status, 1u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

int sm_count_pair()
{
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0)
            n = 1;
    }
    return n;
}

// Work plan.  With at least one head pair per SM: the wrap schedule (one
// contiguous piece of the pair-major tile sequence per CTA, at most one
// hand-off slot per sequence).  With at most half as many head pairs as SMs:
// prefilled segments -- one to four waves of (pair, segment) items, every
// segment's start state computed beforehand by the segmented tensor-core
// state pass, so no item waits for another.  Otherwise one item per head pair, run end to
// end by one CTA: only one segment of a sequence can run at a time, so
// cutting the sequences into segments that hand their states on adds waits
// and no parallelism (B 4, L 65536, H 64, S 128 took 1.75 ms against 1.87 ms
// with about eight hand-off segments per SM).  SSD_PAIR_PREFILL=0 turns the
// prefilled plan off (a test and measurement switch).
constexpr int kMaxPrefillSeg = 64;  // segments the state pass's combine handles
constexpr int64_t kMinWaveSeg = 96;  // tiles of a prefilled segment past the first wave

struct PairSegPlan {
    bool wrap, prefill;
    int seg_tiles, n_seg;
    size_t state_bytes, count_bytes, gd_bytes;  // gd: G and dt^T for the prefill
};

PairSegPlan pair_seg_plan(const Geom &g, bool allow_prefill = true)
{
    PairSegPlan sp;
    const int64_t n_tiles = (g.L + kTile - 1) / kTile;
    const int64_t units = g.B * (g.H / 2);
    const int64_t nbh = g.B * g.H;
    sp.wrap = units >= sm_count_pair() && n_tiles > 1;
    sp.prefill = false;
    sp.gd_bytes = 0;
    if (sp.wrap) {
        sp.seg_tiles = (int)n_tiles;
        sp.n_seg = 2;  // slot 0: the state a sequence's first part hands to its second
        sp.state_bytes = (size_t)(nbh * 2 * g.P * g.S) * sizeof(float);
        sp.count_bytes = (size_t)(nbh * 2) * sizeof(unsigned int);
        return sp;
    }
    const char *env = getenv("SSD_PAIR_PREFILL");
    const int tpc = g.T / kTile;
    // one wave of items, or two or four while the segments stay at least
    // kMinWaveSeg tiles long (B 1, L 262144, H 64: S 128 2.80 -> 2.51 ms and
    // S 64 2.68 -> 2.35 ms at four waves, eight were slower; B 4, L 16384,
    // H 8 is fastest with one)
    int64_t waves = 1;
    while (waves < 4 && n_tiles * units / (2 * waves * sm_count_pair()) >= kMinWaveSeg)
        waves *= 2;
    int64_t want1 = waves * sm_count_pair() / units;
    if (want1 > kMaxPrefillSeg)
        want1 = kMaxPrefillSeg;
    if (want1 * 2 * tpc > n_tiles)
        want1 = n_tiles / (2 * tpc);
    if (allow_prefill && want1 >= 2 && state_pass_tc_supported(g) && !(env && strcmp(env, "0") == 0)) {
        int64_t st = (n_tiles + want1 - 1) / want1;
        st = (st + tpc - 1) / tpc * tpc;
        sp.seg_tiles = (int)st;
        sp.n_seg = (int)((n_tiles + st - 1) / st);
        if (sp.n_seg >= 2) {
            sp.prefill = true;
            sp.state_bytes = (size_t)(nbh * sp.n_seg * g.P * g.S) * sizeof(float);
            sp.count_bytes = 0;
            sp.gd_bytes = 2 * (size_t)(nbh * g.L) * sizeof(float);
            return sp;
        }
    }
    sp.seg_tiles = (int)n_tiles;
    sp.n_seg = 1;
    sp.state_bytes = 0;
    sp.count_bytes = 0;
    return sp;
}

template <int S>
cudaError_t launch_pair(const CUtensorMap &tx, const CUtensorMap &tb, const CUtensorMap &tcm,
                        const CUtensorMap &ty, const PairParams &prm, cudaStream_t st)
{
    using Lay = PairLayout<S>;
    const size_t smem = Lay::bytes + 1024;
    auto k = pair_tc_kernel<S>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const int grid = prm.wrap ? sm_count_pair()
                              : (prm.n_items < sm_count_pair() ? prm.n_items : sm_count_pair());
    // CTAs wait on each other's state hand-offs, so the grid (one CTA per SM)
    // must be co-resident: a cooperative launch guarantees it or fails.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k, tx, tb, tcm, ty, prm);
    note_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool pair_tc_supported(const Geom &g)
{
    const int64_t n_tiles = (g.L + kTile - 1) / kTile;
    return g.P == 64 && (g.S == 64 || g.S == 128) && g.hpg % 2 == 0 &&
           (g.T == kTile || g.T == 2 * kTile) && g.L > 0 && g.L < (1LL << 31) && g.H <= 65535 &&
           g.G <= 65535 && g.B <= 65535 && g.B * g.H * n_tiles < (1LL << 31);
}

size_t pair_tc_scratch_bytes(const Geom &g, bool allow_prefill)
{
    const PairSegPlan sp = pair_seg_plan(g, allow_prefill);
    if (!sp.wrap && sp.n_seg <= 1)
        return 0;
    return (sp.state_bytes + 255) / 256 * 256 + (sp.count_bytes + 255) / 256 * 256 +
           (sp.gd_bytes + 511) / 512 * 512;
}

bool pair_tc_prefers_prefill(const Geom &g) { return pair_tc_supported(g) && pair_seg_plan(g).prefill; }

cudaError_t launch_fused_pair_tc(const void *x, const void *Bm, const void *Cm, const float *dt,
                                 const float *A, const float *D, const float *init, float *states,
                                 float *final_state, void *y, const Geom &g, void *scratch,
                                 size_t scratch_bytes, cudaStream_t st, bool allow_prefill)
{
    if (!pair_tc_supported(g))
        return cudaErrorNotSupported;
    PairParams prm{};
    prm.dt = dt;
    prm.A = A;
    prm.D = D;
    prm.init = init;
    prm.states_out = states;
    prm.final_state = final_state;
    prm.g = g;
    prm.n_tiles = (int)((g.L + kTile - 1) / kTile);
    prm.tpc_shift = g.T == 2 * kTile ? 1 : 0;
    prm.batch = (int)g.B;
    prm.H = (int)g.H;
    prm.npairs = (int)(g.H / 2);
    prm.hpg = g.hpg;
    // the prefilled plan when the scratch holds it, else the hand-off plan
    // (the caller checked that one of the two fits)
    PairSegPlan sp = pair_seg_plan(g, allow_prefill);
    if (sp.prefill && scratch_bytes < pair_tc_scratch_bytes(g, true))
        sp = pair_seg_plan(g, false);
    prm.seg_tiles = sp.seg_tiles;
    prm.n_seg = sp.n_seg;
    prm.wrap = sp.wrap ? 1 : 0;
    prm.prefilled = sp.prefill ? 1 : 0;
    prm.wrap_units = (long long)(g.B * (g.H / 2)) * prm.n_tiles;
    prm.n_items = (int)(g.B * (g.H / 2) * (sp.wrap ? 1 : sp.n_seg));
    if (sp.wrap || sp.n_seg > 1) {
        const size_t off = (sp.state_bytes + 255) / 256 * 256;
        const size_t off_gd = off + (sp.count_bytes + 255) / 256 * 256;
        if (!scratch || scratch_bytes < off_gd + sp.gd_bytes)
            return cudaErrorInvalidValue;
        prm.seg_state = static_cast<float *>(scratch);
        prm.seg_count = reinterpret_cast<unsigned int *>(static_cast<char *>(scratch) + off);
        cudaError_t e;
        if (sp.prefill) {
            // every segment's start state: G, then the segmented state pass
            float *Gc = reinterpret_cast<float *>(static_cast<char *>(scratch) + off_gd);
            float *dtT = Gc + g.B * g.H * g.L;
            if ((e = launch_chunk_cumsum(dt, A, Gc, dtT, g, st)) != cudaSuccess ||
                (e = launch_segment_starts_tc(x, Bm, dtT, Gc, init, prm.seg_state, sp.seg_tiles,
                                              sp.n_seg, g, st)) != cudaSuccess)
                return e;
        } else if ((e = cudaMemsetAsync(prm.seg_count, 0, sp.count_bytes, st)) != cudaSuccess) {
            return e;
        }
    }
    prm.status = device_status_word();
    if (!prm.status)
        return cudaErrorUnknown;
    // SSD_FAULT_SKIP_ARRIVE=1 (debug only) injects a lost barrier arrival on
    // every CTA's first tile and shortens every wait to 20 ms, so a test can
    // see the timeout path report SSD_ERR_TIMEOUT through ssd_stream_status.
    // What is in flight when the waits run out: the first tile's TMA loads
    // (each already waited for by its consumer) and its C B^T MMA (waited for
    // by the compute warps through its commit barrier before the wait that
    // runs out), so every role leaves with nothing outstanding.
    const char *fault = getenv("SSD_FAULT_SKIP_ARRIVE");
    prm.fault_skip_arrive = (fault && strcmp(fault, "1") == 0) ? 1 : 0;
    prm.wait_ns = prm.fault_skip_arrive ? 20000000ull : 2000000000ull;
    CUtensorMap tx, tb, tcm, ty;
    if (!make_tmap_tokens_heads(&tx, x, g) || !make_tmap_tokens_groups(&tb, Bm, g) ||
        !make_tmap_tokens_groups(&tcm, Cm, g) || !make_tmap_tokens_heads(&ty, y, g))
        return cudaErrorInvalidValue;
    return g.S == 64 ? launch_pair<64>(tx, tb, tcm, ty, prm, st)
                     : launch_pair<128>(tx, tb, tcm, ty, prm, st);
}

}  // namespace ssd
