// Stage 3 (chunk output) and the fused single-pass forward on tensor cores,
// bf16 inputs.
//
// "Accelerating Mamba-2 forward-pass kernels with CUDA Tile (cuTile)",
// section "Kernel 3: compute_out", per (batch, chunk, head):
//     Y = exp2(G) * (C h_c^T) + (exp2(G_i - G_j) * (C B^T) * M)(dt * X) + D X
// and section "Kernel 2: fwd_pass_state" for the state jump
//     h <- exp2(G_last) h + X^T (B * dt * exp2(G_last - G)).
//
// chunk_tc_kernel, dstate 64 / 128 / 256, has two modes:
//   OUT   -- a work item is (batch, chunk, head); h_c comes from chunk_states.
//   FUSED -- a work item is (batch, head, segment of the sequence); the state
//            is carried on chip from tile to tile, so chunk states never go
//            through HBM unless the caller asks for them.
// chunk_big_kernel is the FUSED mode for dstate 384 / 512, with B and C
// streamed in 128-row dstate blocks (its own description is further down).
// Tokens are processed in 128-token tiles (the tcgen05 M and K extent).  A
// chunk of 256 tokens is two tiles: the second tile's starting state is the
// first tile's state jump applied to h_c, and its G is taken relative to the
// token before it, which is the same arithmetic regrouped
// (exp2(G_i - G_j) = exp2(G_i - G_m) exp2(G_m - G_j) with both factors <= 1).
//
// Per tile (all contractions are tcgen05.mma kind::f16, f32 accumulate in TMEM):
//   CB  = C B^T                 M 128 (i) x N 128 (j), K = S     [TMEM]
//   scores_ij = CB_ij exp2(g_i - g_j) dt_j for j <= i (masked entries are set
//               to zero without evaluating the exponent), bf16 into TMEM
//   Y1  = scores X              N = P, K = 128, A operand from TMEM
//   Y2  = C H^T, H = bf16(h_c)  N = P, K = S
//   y   = Y1 + exp2(g_i) Y2 + D x      (f32 epilogue, bf16; D x is written
//                                       into Y1's accumulator before its MMAs)
//   and, when a later tile needs the state: h <- exp2(g_L) h + B^T X_hat with
//   X_hat = dt exp2(g_L - g) X split into bf16 hi + lo (two MMA passes); the
//   state h^T [S, P] is an f32 TMEM accumulator.
// When the tile's decay range is narrow the decay factorizes:
//   exp2(g_i - g_j) dt_j = exp2(g_i - g_L) * [dt_j exp2(g_L - g_j)],
// so the scores are just the masked CB and Y1 = scores X_hat with the row
// factor exp2(g_i - g_L) applied in the epilogue; no per-element exponent.
//
// Roles (one CTA per SM, persistent over work items):
//   warps 0-7  two compute warpgroups; thread (wg, q, lane) owns tile row /
//              TMEM lane i = 32 q + lane, warpgroup wg owns half of the
//              columns of every per-tile step;
//   warp 8     TMA loads of B, C and x tiles into a STAGES-deep ring
//              (128-byte swizzle); a stage's B / C are reloaded as soon as
//              the tile's state jump is done, its x once its y is stored;
//   warp 9     MMA issue;
//   warp 10    TMA store of y: the epilogue writes y over the x tile it has
//              consumed, this warp stores it and then frees the x slot.
// Every wait is bounded; a timeout sets the kernel status word and the role
// leaves its loop.
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "ssd_internal.h"
#include "tc05.cuh"

namespace ssd {
namespace {
using namespace tc;

constexpr int kTile = 128;
constexpr int kComputeWarps = 8;  // two warpgroups
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kThreads = kComputeThreads + 96;
constexpr uint32_t kRegion = 128 * 128;
// A tile takes the factorized decay when |g_first - g_last| <= kNarrow
// (log2 units): then exp2(g_i - g_L) <= 2^64 and dt exp2(g_L - g_j) >= dt 2^-64,
// both comfortably inside the normal f32 / bf16 range.
constexpr float kNarrow = 64.f;

template <int P, int S, int STAGES>
struct CoLayout {
    static constexpr int kSReg = S / 64;           // 64-wide dstate regions of B / C
    static constexpr int kPReg = P / 64;           // 64-wide headdim regions of x
    static constexpr int kSBlk = (S + 127) / 128;  // 128-row blocks of the state
    static constexpr uint32_t kB = kSReg * kRegion;
    static constexpr uint32_t kX = kPReg * kRegion;
    static constexpr uint32_t kStage = 2 * kB;  // B, C
    // x has a ring of its own, at least two slots deep: the next tile's x
    // lands while an exact tile's Y1 still reads its own x
    static constexpr int kXSt = STAGES < 2 ? 2 : STAGES;
    static constexpr uint32_t off_x = STAGES * kStage;
    static constexpr uint32_t off_xh = off_x + kXSt * kX;  // X_hat hi, then lo (then y)
    static constexpr uint32_t off_h = off_xh + 2 * kX;
    // H is stored MN-major: one 128-byte row of P bf16 per state index s
    static constexpr uint32_t kH = S * 128;
    // [g 128 | dt 128] f32 of the tile whose X_hat was built last (every
    // warp has converted the previous tile's scores by then: its epilogue
    // waited for Y1, which waited for the scores)
    static constexpr uint32_t off_g = off_h + kH;
    static constexpr uint32_t bytes = off_g + 256 * 4;
    // TMEM columns: CB (f32), the bf16 score operand (two per column), Y1, Y2,
    // and the f32 state accumulator
    static constexpr uint32_t t_cb = 0, t_sc = 128, t_y1 = 192, t_y2 = 192 + P,
                              t_st = 192 + 2 * P;
    static constexpr uint32_t cols_used = t_st + kSBlk * P;
    static constexpr uint32_t kTmemCols = cols_used <= 256 ? 256 : 512;
    static_assert(P == 64, "one 128-byte row of x / y / H per token or state index");
    static_assert(cols_used <= 512, "TMEM budget");
    // dynamic bytes + alignment pad + static barriers within the 227 KB opt-in limit
    static_assert(bytes + 1024 + 256 <= 232448, "shared memory budget");
};

enum Mode { kModeOut = 0, kModeFused = 1 };

struct Params {
    const float *dtT, *Gc, *D;
    const float *h_src;   // OUT: chunk_states; FUSED: init_state (may be null)
    float *states_out;    // FUSED: chunk_states to emit (may be null)
    float *final_state;   // FUSED: may be null
    Geom g;
    // Work geometry in 32-bit (the launcher checks that it fits): per-tile
    // index arithmetic stays in cheap 32-bit integer operations.
    int n_items;
    int n_tiles;  // tiles per sequence
    int tpc_shift;  // log2(tiles per chunk); chunk_size / 128 is 1 or 2
    int H, nc, nbh;
    // FUSED: each (batch, head) sequence is split into n_seg segments of
    // seg_tiles tiles; segment k > 0 starts from the state segment k-1 leaves
    // in seg_state, published by seg_count reaching kComputeWarps.
    int seg_tiles;
    int n_seg;
    float *seg_state;          // [B*H*n_seg][P][S]
    unsigned int *seg_count;   // [B*H*n_seg], zero at launch
    // prefilled: a state pass has already put every segment's start state in
    // seg_state, so no segment waits for another and none hands off
    int prefilled;
    unsigned int *status;
};

// A work item: tiles [t0, t1) of sequence (b, h); chunk is the chunk index
// (OUT) or the segment index (FUSED).
struct Item {
    int b, h, bh, t0, t1, chunk;
};

template <int MODE>
__device__ __forceinline__ Item decode_item(const Params &p, int item)
{
    Item it;
    const unsigned u = (unsigned)item;
    if (MODE == kModeOut) {
        // consecutive items share (b, chunk) so their B/C tiles hit in L2
        it.h = (int)(u % (unsigned)p.H);
        const unsigned bc = u / (unsigned)p.H;
        it.chunk = (int)(bc % (unsigned)p.nc);
        it.b = (int)(bc / (unsigned)p.nc);
        it.t0 = it.chunk << p.tpc_shift;
        it.t1 = min(it.t0 + (1 << p.tpc_shift), p.n_tiles);
    } else {
        // segment-major: every segment k of every sequence comes before any
        // segment k+1, so a segment's predecessor is always an earlier item
        const unsigned seg = u / (unsigned)p.nbh, bh = u % (unsigned)p.nbh;
        it.h = (int)(bh % (unsigned)p.H);
        it.b = (int)(bh / (unsigned)p.H);
        it.t0 = (int)seg * p.seg_tiles;
        it.t1 = min(it.t0 + p.seg_tiles, p.n_tiles);
        it.chunk = (int)seg;
    }
    it.bh = it.b * p.H + it.h;
    return it;
}

template <int P, int S, int STAGES, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_y,
                const Params prm)
{
    using Lay = CoLayout<P, S, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // per B / C stage: landed; free (the tile's C B^T, C H^T and state jump
    // done).  Per x slot: landed; free (X_hat built; for an exact tile, Y1 done)
    __shared__ uint64_t bar_full[STAGES], bar_empty[STAGES], bar_full_x[Lay::kXSt],
        bar_empty_x[Lay::kXSt];
    // y staged in the X_hat lo buffer (compute warps); that buffer read by
    // the y store
    __shared__ uint64_t bar_ys, bar_lofree;
    // MMA completions: cb (CB), y (Y1 and Y2), ds (state jump and all before)
    __shared__ uint64_t bar_cb, bar_y, bar_ds, bar_end;
    // compute warps done with: X_hat and the g / dt table, H and the state
    // decay, the score operand
    __shared__ uint64_t bar_xh, bar_h, bar_scores;
    __shared__ uint32_t tmem_slot;
    __shared__ int s_mode[2];  // per tile parity: 1 = factorized (narrow) decay

    const Geom &g = prm.g;
    const int tid = threadIdx.x, warp = tid >> 5;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], 1);
        }
        for (int s = 0; s < Lay::kXSt; ++s) {
            mbar_init(&bar_full_x[s], 1);
            mbar_init(&bar_empty_x[s], kComputeWarps);
        }
        mbar_init(&bar_ys, kComputeWarps);
        mbar_init(&bar_lofree, 1);
        mbar_init(&bar_cb, 1);
        mbar_init(&bar_y, 1);
        mbar_init(&bar_end, 1);
        mbar_init(&bar_ds, 1);
        mbar_init(&bar_xh, kComputeWarps);
        mbar_init(&bar_h, kComputeWarps);
        mbar_init(&bar_scores, kComputeWarps);
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
    const bool want_final = MODE == kModeFused && prm.final_state != nullptr;

    if (warp == 8) {
        // ---------------- TMA producer
        if ((tid & 31) == 0) {
            prefetch_tmap(&tm_x);
            prefetch_tmap(&tm_b);
            prefetch_tmap(&tm_c);
            uint32_t it = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < prm.n_items && ok; item += gridDim.x) {
                const Item w = decode_item<MODE>(prm, item);
                const int grp = w.h / g.hpg;
                for (int t = w.t0; t < w.t1; ++t, ++it) {
                    const int s = (int)(it % STAGES), sx = (int)(it % Lay::kXSt);
                    const int tok = t * kTile;
                    // x once its slot's previous tile no longer reads it (X_hat
                    // built, or for an exact tile Y1 done); then B / C once the
                    // stage's previous tile no longer reads them (its state
                    // jump and Y2 done).  x never waits behind B / C: its slot
                    // frees no later than the epilogue before the next X_hat,
                    // which the state jump that frees B / C waits for.
                    if (it >= Lay::kXSt &&
                        !mbar_wait(&bar_empty_x[sx], ((it / Lay::kXSt) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sxp = smem + Lay::off_x + sx * Lay::kX;
                    mbar_arrive_expect_tx(&bar_full_x[sx], Lay::kX);
                    for (int r = 0; r < Lay::kPReg; ++r)
                        tma4(sxp + r * kRegion, &tm_x, &bar_full_x[sx], r * 64, w.h, tok, w.b);
                    if (it >= STAGES &&
                        !mbar_wait(&bar_empty[s], ((it / STAGES) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = smem + s * Lay::kStage;
                    mbar_arrive_expect_tx(&bar_full[s], 2 * Lay::kB);
                    for (int r = 0; r < Lay::kSReg; ++r) {
                        tma4(st + r * kRegion, &tm_b, &bar_full[s], r * 64, grp, tok, w.b);
                        tma4(st + Lay::kB + r * kRegion, &tm_c, &bar_full[s], r * 64, grp, tok, w.b);
                    }
                }
            }
            if (!ok)
                atomicOr(prm.status, 1u);
        }
    } else if (warp == 9) {
        // ---------------- MMA issuer.  Per tile: CB; Y2 and the state jump as
        // one straight run once H and X_hat are ready; Y1 once the scores are.
        // The waits poll with test_wait (never parked).
        if ((tid & 31) == 0) {
            const uint32_t id_cb = idesc_bf16(128, 128, false, false);
            const uint32_t id_y1 = idesc_bf16(128, P, false, true);  // A (scores) from TMEM
            const uint32_t id_y2 = idesc_bf16(128, P, false, true);  // H is MN-major
            const uint32_t id_ds = idesc_bf16(128, P, true, true);
            // base descriptors: per stage B, C (K-major and, for B, MN-major
            // as the state jump's A) and x; X_hat hi / lo; H
            const uint64_t d_xh = desc_mn0(smem_u32(smem + Lay::off_xh));
            const uint64_t d_h = desc_mn0(smem_u32(smem + Lay::off_h));
            uint32_t it = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < prm.n_items && ok; item += gridDim.x) {
                const Item w = decode_item<MODE>(prm, item);
                for (int t = w.t0; t < w.t1; ++t, ++it) {
                    const bool last_seq = MODE == kModeOut ? t + 1 == w.t1 : t + 1 == prm.n_tiles;
                    const bool do_state = !last_seq || want_final;
                    const int s = (int)(it % STAGES), sx = (int)(it % Lay::kXSt);
                    const uint32_t sb = smem_u32(smem + s * Lay::kStage);
                    const uint64_t d_bk = desc_k0(sb), d_ck = desc_k0(sb + Lay::kB);
                    const uint64_t d_bmn = desc_mn0(sb);
                    const uint64_t d_x = desc_mn0(smem_u32(smem + Lay::off_x + sx * Lay::kX));
                    const uint32_t par = it & 1;
                    // CB overwrites the previous tile's CB, whose conversion
                    // ended before that tile's Y1 was issued
                    if (!mbar_wait(&bar_full[s], (it / STAGES) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < S / 16; ++ks)
                        mma_ss(tmem + Lay::t_cb, desc_k(d_ck, kRegion, ks), desc_k(d_bk, kRegion, ks),
                               id_cb, ks > 0);
                    mma_commit(&bar_cb);
                    // Y2 once H is built and X_hat too (X_hat comes after the
                    // previous tile's epilogue has read Y2).  An exact tile's Y1
                    // reads raw x: wait for it to have landed (its slot is held
                    // until that Y1 is done; a factorized tile's slot may already
                    // be reloading, and its MMAs never read raw x).
                    if (!mbar_spin(&bar_h, par) || !mbar_spin(&bar_xh, par) ||
                        (!s_mode[par] && !mbar_spin(&bar_full_x[sx], (it / Lay::kXSt) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < S / 16; ++ks)
                        mma_ss(tmem + Lay::t_y2, desc_k(d_ck, kRegion, ks), desc_mn(d_h, ks), id_y2,
                               ks > 0);
                    // the state jump right after Y2, in one straight run: with
                    // them the tile's B / C are done with, so their reload starts
                    if (do_state) {
#pragma unroll
                        for (int mb = 0; mb < Lay::kSBlk; ++mb)
#pragma unroll
                            for (int part = 0; part < 2; ++part)
#pragma unroll
                                for (int ks = 0; ks < kTile / 16; ++ks)
                                    mma_ss(tmem + Lay::t_st + mb * P,
                                           desc_mn(d_bmn + ((2 * mb * kRegion) >> 4), ks),
                                           desc_mn(d_xh + ((part * Lay::kX) >> 4), ks), id_ds, 1u);
                    }
                    mma_commit(&bar_ds);
                    mma_commit(&bar_empty[s]);
                    // Y1 (adding onto D x / r1) once the scores are converted
                    if (!mbar_spin(&bar_scores, par)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    {
                        const uint64_t d_y1b = s_mode[par] ? d_xh : d_x;  // X_hat or raw x
#pragma unroll
                        for (int ks = 0; ks < kTile / 16; ++ks)
                            mma_ts(tmem + Lay::t_y1, tmem + Lay::t_sc + ks * 8, desc_mn(d_y1b, ks),
                                   id_y1, 1u);
                        mma_commit(&bar_y);
                    }
                    if (!ok)
                        break;
                }
            }
            if (!ok)
                atomicOr(prm.status, 1u);
            // every MMA this thread issued has completed before TMEM is freed
            mma_commit(&bar_end);
            if (!mbar_wait(&bar_end, 0))
                atomicOr(prm.status, 1u);
        }
    } else if (warp == 10) {
        // ---------------- y store: the epilogue left y in the X_hat lo buffer
        if ((tid & 31) == 0) {
            prefetch_tmap(&tm_y);
            uint32_t it = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < prm.n_items && ok; item += gridDim.x) {
                const Item w = decode_item<MODE>(prm, item);
                for (int t = w.t0; t < w.t1; ++t, ++it) {
                    if (!mbar_wait(&bar_ys, it & 1)) {
                        ok = false;
                        break;
                    }
                    const uint8_t *sy = smem + Lay::off_xh + Lay::kX;  // the X_hat lo buffer
                    for (int r = 0; r < Lay::kPReg; ++r)
                        tma4_store(&tm_y, sy + r * kRegion, r * 64, w.h, t * kTile, w.b);
                    bulk_commit();
                    bulk_wait_read();
                    mbar_arrive(&bar_lofree);
                }
            }
            bulk_wait_all();
            if (!ok)
                atomicOr(prm.status, 1u);
        }
    } else if (warp < kComputeWarps) {
        // ---------------- two compute warpgroups.  Order per tile `it`:
        //   scores(it) -> [state leaving the item] -> H(it + 1) -> epilogue(it)
        //   -> X_hat(it + 1)
        // so the next tile's H is built from the state the jump of `it` left
        // while Y1(it) runs on the tensor cores.  y is staged in the X_hat lo
        // buffer (free once the jump of `it` is done) and D x goes into the Y1
        // accumulator when X_hat is built, so x is free as soon as X_hat is
        // (Y1 of a wide tile, which reads raw x, keeps it until Y1 is done).
        const int wg = warp >> 2, q = warp & 3;
        const int i = q * 32 + (tid & 31);
        const int row_lo = q * 32, row_hi = q * 32 + 31;  // this warp's rows
        const uint32_t lane = tmem_at(tmem, (uint32_t)(q * 32), 0);
        float *gtab_all = reinterpret_cast<float *>(smem + Lay::off_g);
        uint8_t *s_xh = smem + Lay::off_xh;
        uint8_t *s_lo = s_xh + Lay::kX;
        uint8_t *s_h = smem + Lay::off_h;
        constexpr int kPHalf = P / 2;
        const int c0w = wg * kPHalf;  // this warpgroup's first headdim column

        // raw G / dt words of a tile, loaded two tiles ahead.  Every load is
        // unconditional (addresses clamped into the row) and the choices
        // between a loaded word and a default are made in make_tile, a tile
        // later: a select on a load still in flight would hold the thread
        // until the load returns.
        struct Raw {
            float base, g0, gL, gi, dti;
        };
        const int tpc_mask = (1 << prm.tpc_shift) - 1;
        auto load_raw = [&](const Item &w, int t) {
            const float *grow = prm.Gc + (int64_t)w.bh * g.L;
            const int tau = t * kTile;
            const int n = min(kTile, (int)g.L - tau);
            const int ic = i < n ? i : n - 1;
            Raw r;
            r.base = ld_early(grow + (tau > 0 ? tau - 1 : 0));
            r.g0 = ld_early(grow + tau);
            r.gL = ld_early(grow + tau + n - 1);
            r.gi = ld_early(grow + tau + ic);
            r.dti = ld_early(prm.dtT + (int64_t)w.bh * g.L + tau + ic);
            return r;
        };
        // Position of a tile in this CTA's work: item, tile, the head's D.
        struct Pos {
            Item w;
            int item, t;
            float Dh;
            bool valid;
        };
        auto first_pos = [&]() {
            Pos p{};
            p.item = blockIdx.x;
            p.valid = p.item < prm.n_items;
            if (p.valid) {
                p.w = decode_item<MODE>(prm, p.item);
                p.t = p.w.t0;
                p.Dh = prm.D[p.w.h];
            }
            return p;
        };
        // next_pos past the last tile returns valid = false with the last
        // tile's place unchanged
        auto next_pos = [&](const Pos &p) {
            Pos n = p;
            if (!p.valid)
                return n;
            if (p.t + 1 < p.w.t1) {
                n.t = p.t + 1;
                return n;
            }
            n.item = p.item + (int)gridDim.x;
            n.valid = n.item < prm.n_items;
            if (n.valid) {
                n.w = decode_item<MODE>(prm, n.item);
                n.t = n.w.t0;
                n.Dh = prm.D[n.w.h];
            }
            return n;
        };
        struct Tile {
            Item w;
            int t, n, sx;  // sx: x slot
            uint32_t it;
            bool first, last_item, last_seq, do_state, narrow;
            float gi, dti, gL, Dh;
        };
        auto make_tile = [&](const Pos &p, uint32_t it, const Raw &raw) {
            Tile c;
            c.w = p.w;
            c.t = p.t;
            c.it = it;
            c.sx = (int)(it % Lay::kXSt);
            c.n = min(kTile, (int)g.L - p.t * kTile);
            c.first = p.t == p.w.t0;
            c.last_item = p.t + 1 == p.w.t1;
            c.last_seq = MODE == kModeOut ? c.last_item : p.t + 1 == prm.n_tiles;
            c.do_state = !c.last_seq || want_final;
            // G restarts at chunk starts; a tile inside a chunk is relative to
            // G just before it
            const float base = (p.t & tpc_mask) == 0 ? 0.f : raw.base;
            c.gL = raw.gL - base;
            const float range = (raw.g0 - base) - c.gL;
            c.narrow = range <= kNarrow && range >= -kNarrow;
            c.gi = i < c.n ? raw.gi - base : 0.f;
            c.dti = i < c.n ? raw.dti : 0.f;
            c.Dh = p.Dh;
            return c;
        };

        // ---- X_hat = dt exp2(g_L - g) x as bf16 hi (+ lo for the state jump),
        // and Y1 <- D x / r1 (r1 = exp2(g_i - g_L) factorized, 1 exact), which
        // Y1's MMAs add onto.  lo goes in once the previous tile's y store has
        // read the lo buffer.
        auto build_xhat = [&](const Tile &c) -> bool {
            const uint32_t par = c.it & 1;
            float *gtab = gtab_all;
            if (wg == 0)
                gtab[i] = c.gi;
            else
                gtab[128 + i] = c.dti;
            if (tid == 0)
                s_mode[par] = c.narrow ? 1 : 0;
            if (!mbar_wait(&bar_full_x[c.sx], (c.it / Lay::kXSt) & 1))
                return false;
            tc_fence_after();
            const uint8_t *sx = smem + Lay::off_x + c.sx * Lay::kX;
            const bool build = c.narrow || c.do_state;
            const float e = ex2_approx(c.gL - c.gi);
            const float w = (build && i < c.n) ? c.dti * e : 0.f;
            const float dsc = c.narrow ? c.Dh * e : c.Dh;
            uint32_t lo_keep[4][4];
            uint32_t dx[32];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int ch = wg * 4 + k;
                const uint32_t off = sw128_offset(i, ch);
                const uint4 v = *reinterpret_cast<const uint4 *>(sx + off);
                const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
                uint32_t hi[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const float x0 = bf_lo(vv[e2]), x1 = bf_hi(vv[e2]);
                    const float a = x0 * w, bb = x1 * w;
                    hi[e2] = pack_bf16x2(a, bb);
                    lo_keep[k][e2] = pack_bf16x2(a - bf_lo(hi[e2]), bb - bf_hi(hi[e2]));
                    dx[8 * k + 2 * e2] = __float_as_uint(dsc * x0);
                    dx[8 * k + 2 * e2 + 1] = __float_as_uint(dsc * x1);
                }
                if (build)
                    *reinterpret_cast<uint4 *>(s_xh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            }
            tmem_st16(lane + Lay::t_y1 + c0w, *reinterpret_cast<uint32_t(*)[16]>(dx));
            tmem_st16(lane + Lay::t_y1 + c0w + 16, *reinterpret_cast<uint32_t(*)[16]>(dx + 16));
            // a factorized tile no longer needs raw x: its slot may be reloaded
            if (c.narrow)
                warp_arrive(&bar_empty_x[c.sx]);
            // the previous tile's y store has read the lo buffer
            if (c.it > 0 && !mbar_wait(&bar_lofree, par ^ 1u))
                return false;
            if (c.do_state) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    *reinterpret_cast<uint4 *>(s_lo + sw128_offset(i, wg * 4 + k)) =
                        make_uint4(lo_keep[k][0], lo_keep[k][1], lo_keep[k][2], lo_keep[k][3]);
            }
            fence_proxy_async_smem();
            tmem_st_wait();
            tc_fence_before();
            warp_arrive(&bar_xh);
            return true;
        };

        // ---- H = bf16(hscale * h), MN-major [s][p]; emit and decay the state.
        // A non-first tile reads the state the previous tile's jump left (the
        // caller waited for it); an item's first tile loads its start state (a
        // later segment waits until its predecessor has published it).
        auto build_h = [&](const Tile &c) -> bool {
            const int64_t bh = c.w.bh;
            const int chunk = c.w.chunk;
            if (MODE == kModeFused && c.first && chunk > 0 && !prm.prefilled) {
                const unsigned int *cnt = prm.seg_count + bh * prm.n_seg + chunk - 1;
                bool ready = ld_acquire_gpu(cnt) >= (unsigned)kComputeWarps;
                const uint64_t t_start = globaltimer_ns();
                while (!ready) {
                    if (globaltimer_ns() - t_start > 2000000000ull)
                        break;
                    __nanosleep(256);
                    ready = ld_acquire_gpu(cnt) >= (unsigned)kComputeWarps;
                }
                if (!ready)
                    return false;
            }
            const float decay = ex2_approx(c.gL);
            const float hscale = c.narrow ? decay : 1.f;
            const bool emit = MODE == kModeFused && prm.states_out && (c.t & tpc_mask) == 0;
#pragma unroll
            for (int mb = 0; mb < Lay::kSBlk; ++mb) {
                const int sidx = mb * 128 + i;
                const bool s_ok = sidx < S;
                const uint32_t acc = lane + Lay::t_st + mb * P + c0w;
                uint32_t r[kPHalf];
                if (c.first) {
                    const float *src = nullptr;
                    if (MODE == kModeOut)
                        src = prm.h_src + ((bh * g.nc + chunk) * g.P) * g.S;
                    else if (chunk > 0)  // later segment: the predecessor's state
                        src = prm.seg_state + ((bh * prm.n_seg + chunk - 1) * g.P) * g.S;
                    else if (prm.h_src)
                        src = prm.h_src + bh * g.P * g.S;
#pragma unroll
                    for (int j = 0; j < kPHalf; ++j)
                        r[j] = __float_as_uint(
                            (src && s_ok) ? __ldcg(src + (int64_t)(c0w + j) * S + sidx) : 0.f);
                } else {
#pragma unroll
                    for (int cc = 0; cc < kPHalf; cc += 16)
                        tmem_ld16(acc + cc, *reinterpret_cast<uint32_t(*)[16]>(r + cc));
                    tmem_ld_wait();
                }
                float *emit_dst =
                    emit ? prm.states_out + ((bh * g.nc + (c.t >> prm.tpc_shift)) * g.P) * g.S
                         : nullptr;
                uint32_t hp[kPHalf / 2];
#pragma unroll
                for (int j = 0; j < kPHalf; j += 2) {
                    const float v0 = __uint_as_float(r[j]), v1 = __uint_as_float(r[j + 1]);
                    if (emit_dst && s_ok) {
                        emit_dst[(int64_t)(c0w + j) * S + sidx] = v0;
                        emit_dst[(int64_t)(c0w + j + 1) * S + sidx] = v1;
                    }
                    hp[j / 2] = pack_bf16x2(v0 * hscale, v1 * hscale);
                    r[j] = __float_as_uint(v0 * decay);
                    r[j + 1] = __float_as_uint(v1 * decay);
                }
                if (s_ok) {  // row sidx, columns c0w .. c0w + 31: four 16-byte chunks
#pragma unroll
                    for (int k = 0; k < kPHalf / 8; ++k)
                        *reinterpret_cast<uint4 *>(s_h + sw128_offset(sidx, c0w / 8 + k)) =
                            make_uint4(hp[4 * k], hp[4 * k + 1], hp[4 * k + 2], hp[4 * k + 3]);
                }
                if (c.do_state) {
#pragma unroll
                    for (int cc = 0; cc < kPHalf; cc += 16)
                        tmem_st16(acc + cc, *reinterpret_cast<uint32_t(*)[16]>(r + cc));
                }
            }
            if (c.do_state)
                tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(&bar_h);
            return true;
        };

        // ---- scores: CB (f32) -> masked, decayed bf16 A operand in TMEM.
        // Warpgroup wg converts keys [64 wg, 64 wg + 64): one TMEM round trip
        // for all of them.  The g / dt table is complete once every warp has
        // published X_hat.
        auto build_scores = [&](const Tile &c) -> bool {
            const uint32_t par = c.it & 1;
            if (!mbar_wait(&bar_cb, par) || !mbar_wait(&bar_xh, par))
                return false;
            tc_fence_after();
            const float *gtab = gtab_all;
            const bool full = c.n == kTile;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t cbv[2][16];
#pragma unroll
                for (int gq = 0; gq < 2; ++gq) {
                    const int j0 = wg * 64 + half * 32 + gq * 16;
                    if (j0 <= row_hi)  // warp-uniform: keys above the diagonal stay zero
                        tmem_ld16(lane + Lay::t_cb + j0, cbv[gq]);
                }
                tmem_ld_wait();
#pragma unroll
                for (int gq = 0; gq < 2; ++gq) {
                    const int j0 = wg * 64 + half * 32 + gq * 16;
                    uint32_t pk[8];
                    if (j0 > row_hi) {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            pk[e] = 0u;
                    } else if (c.narrow) {
                        if (full && j0 + 15 < row_lo) {  // whole group below the diagonal
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                pk[e] = pack_bf16x2(__uint_as_float(cbv[gq][2 * e]),
                                                    __uint_as_float(cbv[gq][2 * e + 1]));
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int j = j0 + 2 * e;
                                const float a =
                                    (j <= i && j < c.n) ? __uint_as_float(cbv[gq][2 * e]) : 0.f;
                                const float bb = (j + 1 <= i && j + 1 < c.n)
                                                     ? __uint_as_float(cbv[gq][2 * e + 1])
                                                     : 0.f;
                                pk[e] = pack_bf16x2(a, bb);
                            }
                        }
                    } else {
                        const float4 *g4 = reinterpret_cast<const float4 *>(gtab + j0);
                        const float4 *d4 = reinterpret_cast<const float4 *>(gtab + 128 + j0);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            const float4 gg = g4[v4], dd = d4[v4];
                            const float gj[4] = {gg.x, gg.y, gg.z, gg.w};
                            const float dj[4] = {dd.x, dd.y, dd.z, dd.w};
                            float val[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int j = j0 + 4 * v4 + e;
                                val[e] = (j <= i && j < c.n)
                                             ? __uint_as_float(cbv[gq][4 * v4 + e]) *
                                                   ex2_approx(c.gi - gj[e]) * dj[e]
                                             : 0.f;
                            }
                            pk[2 * v4] = pack_bf16x2(val[0], val[1]);
                            pk[2 * v4 + 1] = pack_bf16x2(val[2], val[3]);
                        }
                    }
                    tmem_st8(lane + Lay::t_sc + j0 / 2, pk);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            warp_arrive(&bar_scores);
            return true;
        };

        // ---- the state leaving an item: the next segment's start, or the
        // final state (the caller waited for the item's last jump)
        auto leave_state = [&](const Tile &c) {
            const int64_t bh = c.w.bh;
            float *dst = nullptr;
            const bool handoff = MODE == kModeFused && !c.last_seq && !prm.prefilled;
            if (handoff)
                dst = prm.seg_state + ((bh * prm.n_seg + c.w.chunk) * g.P) * g.S;
            else if (c.last_seq && want_final)
                dst = prm.final_state + bh * g.P * g.S;
            if (dst) {
#pragma unroll
                for (int mb = 0; mb < Lay::kSBlk; ++mb) {
                    const int sidx = mb * 128 + i;
                    uint32_t r[kPHalf];
#pragma unroll
                    for (int cc = 0; cc < kPHalf; cc += 16)
                        tmem_ld16(lane + Lay::t_st + mb * P + c0w + cc,
                                  *reinterpret_cast<uint32_t(*)[16]>(r + cc));
                    tmem_ld_wait();
                    if (sidx < S) {
#pragma unroll
                        for (int j = 0; j < kPHalf; ++j)
                            __stcg(dst + (int64_t)(c0w + j) * S + sidx, __uint_as_float(r[j]));
                    }
                }
            }
            if (handoff) {
                __threadfence();
                __syncwarp();
                if ((tid & 31) == 0)
                    atomicAdd(prm.seg_count + bh * prm.n_seg + c.w.chunk, 1u);
            }
        };

        // ---- epilogue: y = r1 Y1 + r2 Y2 (Y1 holds D x / r1), staged in the
        // lo buffer (free: the caller waited for this tile's jump)
        auto epilogue = [&](const Tile &c) -> bool {
            const uint32_t par = c.it & 1;
            if (!mbar_wait(&bar_y, par))
                return false;
            tc_fence_after();
            // an exact tile's Y1 read raw x: its slot may be reloaded now
            if (!c.narrow)
                warp_arrive(&bar_empty_x[c.sx]);
            const float r1 = c.narrow ? ex2_approx(c.gi - c.gL) : 1.f;
            const float r2 = c.narrow ? r1 : ex2_approx(c.gi);
#pragma unroll
            for (int c16 = 0; c16 < kPHalf; c16 += 16) {
                uint32_t ra[16], rb[16];
                tmem_ld16(lane + Lay::t_y1 + c0w + c16, ra);
                tmem_ld16(lane + Lay::t_y2 + c0w + c16, rb);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int cc = 8 * k + 2 * e;
                        o[e] = pack_bf16x2(r1 * __uint_as_float(ra[cc]) + r2 * __uint_as_float(rb[cc]),
                                           r1 * __uint_as_float(ra[cc + 1]) +
                                               r2 * __uint_as_float(rb[cc + 1]));
                    }
                    *reinterpret_cast<uint4 *>(s_lo + sw128_offset(i, (c0w + c16) / 8 + k)) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(&bar_ys);
            return true;
        };

        bool ok = true;
        Pos p1 = first_pos();
        if (p1.valid) {
            const Raw raw0 = load_raw(p1.w, p1.t);
            Tile cur = make_tile(p1, 0, raw0);
            p1 = next_pos(p1);
            // (a position past the CTA's last tile keeps that tile's place, so
            // these loads are always in bounds; selecting between a load and
            // a default would make the thread wait for the load right here)
            Raw raw1 = load_raw(p1.w, p1.t);
            ok = build_xhat(cur) && build_h(cur);
            for (uint32_t it = 0; ok; ++it) {
                // the tile after the next one, its G / dt in flight
                const Pos p2 = next_pos(p1);
                const Raw raw2 = load_raw(p2.w, p2.t);
                if (!build_scores(cur)) {
                    ok = false;
                    break;
                }
                // this tile's jump (and Y2, CB before it) is done: the state, the
                // H buffer and the lo buffer are free
                if (!mbar_wait(&bar_ds, it & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (cur.last_item && cur.do_state)
                    leave_state(cur);
                Tile nxt{};
                if (p1.valid) {
                    nxt = make_tile(p1, it + 1, raw1);
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
                raw1 = raw2;
            }
        }
        if (!ok)
            atomicOr(prm.status, 1u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, Lay::kTmemCols);
    }
}

// ---------------------------------------------------------------- dstate 384 / 512
// The fused forward for dstate 384 and 512, one head per CTA item.  One
// tile's B and C (128 KB each at S = 512) do not fit in shared memory next to
// x, X_hat and H, so they stream through a two-slot ring in 128-row dstate
// blocks and every contraction over S runs block by block: per block b,
//   [CB | Y] += C_b [B_b | H_b]^T (one N = 192 MMA per K step, so C_b is read
//   once),  state_b += B_b^T (X_hat hi + lo),
// where H_b = bf16 of the tile's start state rows of block b, written by the
// compute warps transposed (K-major, [p][s]) into the block's ring slot, in
// the 64 rows after each B region's 128 token rows, before the block's MMAs.
// CB is complete with the last block's C B^T: the score conversion overlaps
// that block's C H^T and jump, and Y1 follows the block loop.  Y holds C H^T and, for a factorized tile, Y1 on top
// (y = exp2(g_i - g_L) Y + D x); an exact tile's Y1 goes to the CB columns
// (y = exp2(g_i) Y + Y1 + D x).  D x is added in the epilogue from the x tile,
// which stays in its slot until then; y is written over it and stored.
//
// Per tile `it`, compute warps: scores(it) -> [state leaving the item] ->
// H blocks 0, 1 of it + 1 -> (Y1 done) epilogue(it) -> X_hat(it + 1) -> the
// remaining H blocks of it + 1.  MMA thread, per block: C B^T, C H^T (after
// the block's H; block 0 after the previous epilogue has read Y), the jump
// (block 0 after X_hat, which the compute warps build while that C H^T
// runs); then Y1 once the scores are converted.
//
// Shared memory (P 64, S 512): B (+ H^T) / C ring 2 x 80 KB, x ring 2 x 16 KB,
// X_hat hi / lo 32 KB, g / dt 1 KB = 225 KB.  TMEM: CB 128 columns and Y 64
// (adjacent: one accumulator of the N = 192 MMA), scores 64, state S / 128
// blocks of 64.
template <int P, int S>
struct BigLayout {
    static constexpr int kSBlk = S / 128;            // 128-row dstate blocks
    // a B region: 128 token rows of 64 s (TMA), then 64 rows of H^T (p) over
    // the same 64 s (compute warps), all K-major with the 128-byte swizzle
    static constexpr uint32_t kRegB = kRegion + 64 * 128;
    static constexpr uint32_t kBlkB = 2 * kRegB;     // one block of B and H^T
    static constexpr uint32_t kBlkC = 2 * kRegion;   // one block of C: 128 tokens x 128 s
    static constexpr uint32_t kSlot = kBlkB + kBlkC;
    static constexpr uint32_t kX = kRegion;          // x / y tile (P = 64)
    static constexpr uint32_t off_x = 2 * kSlot;     // two x slots (y is staged over x)
    static constexpr uint32_t off_xh = off_x + 2 * kX;  // X_hat hi, then lo
    static constexpr uint32_t off_g = off_xh + 2 * kX;  // [g 128 | dt 128] f32
    static constexpr uint32_t bytes = off_g + 256 * 4;
    static constexpr uint32_t t_cb = 0, t_y = 128, t_sc = 192, t_st = 256;
    static constexpr uint32_t kTmemCols = 512;
    static_assert(P == 64, "one 128-byte row of x / y / H per token or state index");
    static_assert(S % 128 == 0 && S >= 384 && t_st + kSBlk * P <= 512, "TMEM budget");
    static_assert(bytes + 1024 + 256 <= 232448, "shared memory budget");
};

template <int P, int S>
__global__ void __launch_bounds__(kThreads, 1)
chunk_big_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                 const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_y,
                 const Params prm)
{
    using Lay = BigLayout<P, S>;
    constexpr int kSBlk = Lay::kSBlk;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // B / C slots: landed, free (the block's C B^T, jump and C H^T done)
    __shared__ uint64_t bar_full[2], bar_empty[2];
    // x slots: landed, free (y stored from it); y staged in the slot
    __shared__ uint64_t bar_full_x[2], bar_empty_x[2], bar_ys[2];
    // H buffers: built (compute warps), free (the block's C H^T done)
    __shared__ uint64_t bar_hr[2], bar_hf[2];
    // X_hat built; CB complete (the last block's C B^T done); the block loop
    // done (state jumped); scores converted; Y complete (Y1 done); the
    // epilogue has read Y; teardown
    __shared__ uint64_t bar_xh, bar_cb, bar_blk, bar_sc, bar_y, bar_ep, bar_end;
    __shared__ uint32_t tmem_slot;
    __shared__ int s_mode[2];  // per tile parity: 1 = factorized (narrow) decay

    const Geom &g = prm.g;
    const int tid = threadIdx.x, warp = tid >> 5;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], 1);
            mbar_init(&bar_full_x[s], 1);
            mbar_init(&bar_empty_x[s], 1);
            mbar_init(&bar_ys[s], kComputeWarps);
            mbar_init(&bar_hr[s], kComputeWarps);
            mbar_init(&bar_hf[s], 1);
        }
        mbar_init(&bar_xh, kComputeWarps);
        mbar_init(&bar_cb, 1);
        mbar_init(&bar_blk, 1);
        mbar_init(&bar_sc, kComputeWarps);
        mbar_init(&bar_y, 1);
        mbar_init(&bar_ep, kComputeWarps);
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
    const bool want_final = prm.final_state != nullptr;

    if (warp == 8) {
        // ---------------- TMA loads: per tile, x into slot it & 1 once the
        // y stored from that slot two tiles back has been read, then B / C
        // block by block into the ring
        if ((tid & 31) == 0) {
            prefetch_tmap(&tm_x);
            prefetch_tmap(&tm_b);
            prefetch_tmap(&tm_c);
            uint32_t it = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < prm.n_items && ok; item += gridDim.x) {
                const Item w = decode_item<kModeFused>(prm, item);
                const int grp = w.h / g.hpg;
                for (int t = w.t0; t < w.t1 && ok; ++t, ++it) {
                    const int tok = t * kTile;
                    const int sx = (int)(it & 1);
                    if (it >= 2 && !mbar_wait(&bar_empty_x[sx], ((it >> 1) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar_full_x[sx], Lay::kX);
                    tma4(smem + Lay::off_x + sx * Lay::kX, &tm_x, &bar_full_x[sx], 0, w.h, tok, w.b);
                    for (int k = 0; k < kSBlk; ++k) {
                        const uint32_t gb = it * kSBlk + k;
                        const int slot = (int)(gb & 1);
                        if (gb >= 2 && !mbar_wait(&bar_empty[slot], ((gb >> 1) - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        uint8_t *sb = smem + slot * Lay::kSlot;
                        mbar_arrive_expect_tx(&bar_full[slot], 4 * kRegion);
                        for (int r = 0; r < 2; ++r) {
                            tma4(sb + r * Lay::kRegB, &tm_b, &bar_full[slot], (2 * k + r) * 64, grp, tok, w.b);
                            tma4(sb + Lay::kBlkB + r * kRegion, &tm_c, &bar_full[slot], (2 * k + r) * 64, grp,
                                 tok, w.b);
                        }
                    }
                }
            }
            if (!ok)
                atomicOr(prm.status, 1u);
        }
    } else if (warp == 9) {
        // ---------------- MMA issuer (waits poll with test_wait)
        if ((tid & 31) == 0) {
            // [CB | Y] += C [B | H]^T: N = 128 tokens + P, both operands K-major
            const uint32_t id_cby = idesc_bf16(128, 128 + P, false, false);
            const uint32_t id_y1 = idesc_bf16(128, P, false, true);  // A (scores) from TMEM
            const uint32_t id_ds = idesc_bf16(128, P, true, true);
            const uint64_t d_xh = desc_mn0(smem_u32(smem + Lay::off_xh));
            const uint64_t d_lo = desc_mn0(smem_u32(smem + Lay::off_xh + Lay::kX));
            uint32_t it = 0;
            bool ok = true, prev_exact = false;
            for (int item = blockIdx.x; item < prm.n_items && ok; item += gridDim.x) {
                const Item w = decode_item<kModeFused>(prm, item);
                for (int t = w.t0; t < w.t1; ++t, ++it) {
                    const bool do_state = t + 1 != prm.n_tiles || want_final;
                    const uint32_t par = it & 1;
                    // the previous tile's epilogue reads Y (and, for an exact
                    // tile, Y1 in the CB columns): wait for it once per tile,
                    // before the first MMA that overwrites what it reads
                    bool ep_done = it == 0;
                    if (prev_exact && !ep_done) {
                        if (!mbar_spin(&bar_ep, (it - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        ep_done = true;
                    }
                    for (int k = 0; k < kSBlk && ok; ++k) {
                        const uint32_t gb = it * kSBlk + k;
                        const int slot = (int)(gb & 1);
                        if (!mbar_spin(&bar_full[slot], (gb >> 1) & 1)) {
                            ok = false;
                            break;
                        }
                        // C [B | H]^T once the block's H^T is in its slot (block
                        // 0: once the previous epilogue has read Y), then the
                        // jump (block 0: once X_hat is built, which the compute
                        // warps do after that epilogue, while these MMAs run)
                        if (!mbar_spin(&bar_hr[slot], (gb >> 1) & 1)) {
                            ok = false;
                            break;
                        }
                        if (!ep_done) {
                            if (!mbar_spin(&bar_ep, (it - 1) & 1)) {
                                ok = false;
                                break;
                            }
                            ep_done = true;
                        }
                        tc_fence_after();
                        const uint32_t sb = smem_u32(smem + slot * Lay::kSlot);
                        const uint64_t d_bk = desc_k0(sb), d_ck = desc_k0(sb + Lay::kBlkB);
                        const uint64_t d_bmn = desc_mn0(sb, Lay::kRegB);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            mma_ss(tmem + Lay::t_cb, desc_k(d_ck, kRegion, ks), desc_k(d_bk, Lay::kRegB, ks),
                                   id_cby, (k > 0 || ks > 0) ? 1u : 0u);
                        // CB is complete with the last block's MMAs above: the
                        // score conversion may overlap that block's jump
                        if (k == kSBlk - 1)
                            mma_commit(&bar_cb);
                        if (k == 0 && !mbar_spin(&bar_xh, par)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (do_state) {
#pragma unroll
                            for (int part = 0; part < 2; ++part)
#pragma unroll
                                for (int ks = 0; ks < 8; ++ks)
                                    mma_ss(tmem + Lay::t_st + k * P, desc_mn(d_bmn, ks),
                                           desc_mn(part ? d_lo : d_xh, ks), id_ds, 1u);
                        }
                        mma_commit(&bar_hf[slot]);
                        mma_commit(&bar_empty[slot]);
                    }
                    if (!ok)
                        break;
                    mma_commit(&bar_blk);
                    if (!mbar_spin(&bar_sc, par)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const bool narrow = s_mode[par] != 0;
                    if (narrow) {
#pragma unroll
                        for (int ks = 0; ks < kTile / 16; ++ks)
                            mma_ts(tmem + Lay::t_y, tmem + Lay::t_sc + ks * 8, desc_mn(d_xh, ks), id_y1, 1u);
                    } else {
                        const uint64_t d_x = desc_mn0(smem_u32(smem + Lay::off_x + (it & 1) * Lay::kX));
#pragma unroll
                        for (int ks = 0; ks < kTile / 16; ++ks)
                            mma_ts(tmem + Lay::t_cb, tmem + Lay::t_sc + ks * 8, desc_mn(d_x, ks), id_y1,
                                   ks > 0 ? 1u : 0u);
                    }
                    mma_commit(&bar_y);
                    prev_exact = !narrow;
                }
            }
            if (!ok)
                atomicOr(prm.status, 1u);
            // every MMA this thread issued has completed before TMEM is freed
            mma_commit(&bar_end);
            if (!mbar_wait(&bar_end, 0))
                atomicOr(prm.status, 1u);
        }
    } else if (warp == 10) {
        // ---------------- y store: the epilogue wrote y over its tile's x
        if ((tid & 31) == 0) {
            prefetch_tmap(&tm_y);
            uint32_t it = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < prm.n_items && ok; item += gridDim.x) {
                const Item w = decode_item<kModeFused>(prm, item);
                for (int t = w.t0; t < w.t1; ++t, ++it) {
                    const int sx = (int)(it & 1);
                    if (!mbar_wait(&bar_ys[sx], (it >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tma4_store(&tm_y, smem + Lay::off_x + sx * Lay::kX, 0, w.h, t * kTile, w.b);
                    bulk_commit();
                    bulk_wait_read();
                    mbar_arrive(&bar_empty_x[sx]);
                }
            }
            bulk_wait_all();
            if (!ok)
                atomicOr(prm.status, 1u);
        }
    } else if (warp < kComputeWarps) {
        // ---------------- two compute warpgroups; thread (wg, q, lane) owns
        // tile row / TMEM lane i = 32 q + lane, warpgroup wg half of the
        // columns of every step
        const int wg = warp >> 2, q = warp & 3;
        const int i = q * 32 + (tid & 31);
        const int row_lo = q * 32, row_hi = q * 32 + 31;
        const uint32_t lane = tmem_at(tmem, (uint32_t)(q * 32), 0);
        float *gtab = reinterpret_cast<float *>(smem + Lay::off_g);
        uint8_t *s_xh = smem + Lay::off_xh;
        uint8_t *s_lo = s_xh + Lay::kX;
        constexpr int kPHalf = P / 2;
        const int c0w = wg * kPHalf;
        const int tpc_mask = (1 << prm.tpc_shift) - 1;

        // raw G / dt words of a tile, loaded two tiles ahead, unconditionally
        // (addresses clamped into the row; defaults chosen a tile later)
        struct Raw {
            float base, g0, gL, gi, dti;
        };
        auto load_raw = [&](const Item &w, int t) {
            const float *grow = prm.Gc + (int64_t)w.bh * g.L;
            const int tau = t * kTile;
            const int n = min(kTile, (int)g.L - tau);
            const int ic = i < n ? i : n - 1;
            Raw r;
            r.base = ld_early(grow + (tau > 0 ? tau - 1 : 0));
            r.g0 = ld_early(grow + tau);
            r.gL = ld_early(grow + tau + n - 1);
            r.gi = ld_early(grow + tau + ic);
            r.dti = ld_early(prm.dtT + (int64_t)w.bh * g.L + tau + ic);
            return r;
        };
        struct Pos {
            Item w;
            int item, t;
            float Dh;
            bool valid;
        };
        auto first_pos = [&]() {
            Pos p{};
            p.item = blockIdx.x;
            p.valid = p.item < prm.n_items;
            if (p.valid) {
                p.w = decode_item<kModeFused>(prm, p.item);
                p.t = p.w.t0;
                p.Dh = prm.D[p.w.h];
            }
            return p;
        };
        // past the last tile: valid = false, the last tile's place kept
        auto next_pos = [&](const Pos &p) {
            Pos n = p;
            if (!p.valid)
                return n;
            if (p.t + 1 < p.w.t1) {
                n.t = p.t + 1;
                return n;
            }
            n.item = p.item + (int)gridDim.x;
            n.valid = n.item < prm.n_items;
            if (n.valid) {
                n.w = decode_item<kModeFused>(prm, n.item);
                n.t = n.w.t0;
                n.Dh = prm.D[n.w.h];
            }
            return n;
        };
        // a tile of sequence bh, segment seg
        struct Tile {
            int bh, seg, t, n, sx;
            uint32_t it;
            bool first, last_item, last_seq, do_state, narrow;
            float gi, dti, gL, Dh;
        };
        auto make_tile = [&](const Pos &p, uint32_t it, const Raw &raw) {
            Tile c;
            c.bh = p.w.bh;
            c.seg = p.w.chunk;
            c.t = p.t;
            c.it = it;
            c.sx = (int)(it & 1);
            c.n = min(kTile, (int)g.L - p.t * kTile);
            c.first = p.t == p.w.t0;
            c.last_item = p.t + 1 == p.w.t1;
            c.last_seq = p.t + 1 == prm.n_tiles;
            c.do_state = !c.last_seq || want_final;
            const float base = (p.t & tpc_mask) == 0 ? 0.f : raw.base;
            c.gL = raw.gL - base;
            const float range = (raw.g0 - base) - c.gL;
            c.narrow = range <= kNarrow && range >= -kNarrow;
            c.gi = i < c.n ? raw.gi - base : 0.f;
            c.dti = i < c.n ? raw.dti : 0.f;
            c.Dh = p.Dh;
            return c;
        };

        // ---- X_hat = dt exp2(g_L - g) x, bf16 hi (+ lo for the jump).  The
        // caller waited for the previous tile's Y1 (the last reader of hi, of
        // the table and, through the jumps before it, of lo).
        auto build_xhat = [&](const Tile &c) -> bool {
            const uint32_t par = c.it & 1;
            if (wg == 0)
                gtab[i] = c.gi;
            else
                gtab[128 + i] = c.dti;
            if (tid == 0)
                s_mode[par] = c.narrow ? 1 : 0;
            if (!mbar_wait(&bar_full_x[c.sx], (c.it >> 1) & 1))
                return false;
            const uint8_t *sx = smem + Lay::off_x + c.sx * Lay::kX;
            const bool build = c.narrow || c.do_state;
            const float e = ex2_approx(c.gL - c.gi);
            const float w = (build && i < c.n) ? c.dti * e : 0.f;
            uint4 xv[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                xv[k] = *reinterpret_cast<const uint4 *>(sx + sw128_offset(i, wg * 4 + k));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t off = sw128_offset(i, wg * 4 + k);
                const uint32_t vv[4] = {xv[k].x, xv[k].y, xv[k].z, xv[k].w};
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const float a = bf_lo(vv[e2]) * w, bb = bf_hi(vv[e2]) * w;
                    hi[e2] = pack_bf16x2(a, bb);
                    lo[e2] = pack_bf16x2(a - bf_lo(hi[e2]), bb - bf_hi(hi[e2]));
                }
                if (build)
                    *reinterpret_cast<uint4 *>(s_xh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                if (c.do_state)
                    *reinterpret_cast<uint4 *>(s_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async_smem();
            warp_arrive(&bar_xh);
            return true;
        };

        // ---- H block k = bf16(hscale h) rows 128 k .. 128 k + 127, stored
        // transposed (K-major [p][s]) in the ring slot of block (it kSBlk + k)
        // once that slot's previous block is done; the chunk state emitted if
        // asked for; the decay written back.  A non-first tile reads the state the previous tile's
        // jumps left (the caller waited for them); an item's first tile loads
        // its start state (a later segment waits until its predecessor has
        // published it).
        auto build_h = [&](const Tile &c, int k) -> bool {
            const uint32_t gh = c.it * kSBlk + k;
            const int buf = (int)(gh & 1);
            if (gh >= 2 && !mbar_wait(&bar_hf[buf], ((gh >> 1) - 1) & 1))
                return false;
            const int64_t bh = c.bh;
            const int seg = c.seg;
            if (k == 0 && c.first && seg > 0 && !prm.prefilled) {
                const unsigned int *cnt = prm.seg_count + bh * prm.n_seg + seg - 1;
                bool ready = ld_acquire_gpu(cnt) >= (unsigned)kComputeWarps;
                const uint64_t t_start = globaltimer_ns();
                while (!ready) {
                    if (globaltimer_ns() - t_start > 2000000000ull)
                        break;
                    __nanosleep(256);
                    ready = ld_acquire_gpu(cnt) >= (unsigned)kComputeWarps;
                }
                if (!ready)
                    return false;
            }
            tc_fence_after();
            const float decay = ex2_approx(c.gL);
            const float hscale = c.narrow ? decay : 1.f;
            const int sidx = k * 128 + i;
            const uint32_t acc = lane + Lay::t_st + k * P + c0w;
            uint32_t r[kPHalf];
            if (c.first) {
                const float *src = nullptr;
                if (seg > 0)  // later segment: the predecessor's state
                    src = prm.seg_state + ((bh * prm.n_seg + seg - 1) * g.P) * g.S;
                else if (prm.h_src)
                    src = prm.h_src + bh * g.P * g.S;
#pragma unroll
                for (int j = 0; j < kPHalf; ++j)
                    r[j] = __float_as_uint(src ? __ldcg(src + (int64_t)(c0w + j) * S + sidx) : 0.f);
            } else {
#pragma unroll
                for (int cc = 0; cc < kPHalf; cc += 16)
                    tmem_ld16(acc + cc, *reinterpret_cast<uint32_t(*)[16]>(r + cc));
                tmem_ld_wait();
            }
            float *emit_dst = (prm.states_out && (c.t & tpc_mask) == 0)
                                  ? prm.states_out + ((bh * g.nc + (c.t >> prm.tpc_shift)) * g.P) * g.S
                                  : nullptr;
            // H^T, K-major: row 128 + p of this state row's 64-s region of the
            // slot, element s % 64, 128-byte swizzle.  The swizzle XORs the
            // 16-byte chunk index (address bits 4-6, zero in every other term
            // here) with row & 7 == j & 7, so the address of row c0w + j is
            // (h0 + 128 j) ^ ((j & 7) << 4).  Lanes of a warp cover 32
            // consecutive s, so a row's 2-byte stores fall in 16 distinct banks.
            const uint32_t h0 = smem_u32(smem + buf * Lay::kSlot + (i >> 6) * Lay::kRegB + (128 + c0w) * 128 +
                                         (i & 7) * 2) +
                                ((uint32_t)((i & 63) >> 3) << 4);
#pragma unroll
            for (int j = 0; j < kPHalf; j += 2) {
                const float v0 = __uint_as_float(r[j]), v1 = __uint_as_float(r[j + 1]);
                if (emit_dst) {
                    emit_dst[(int64_t)(c0w + j) * S + sidx] = v0;
                    emit_dst[(int64_t)(c0w + j + 1) * S + sidx] = v1;
                }
                const uint32_t hv = pack_bf16x2(v0 * hscale, v1 * hscale);
                asm volatile("st.shared.b16 [%0], %1;" ::"r"((h0 + j * 128) ^ (uint32_t)((j & 7) << 4)),
                             "h"((unsigned short)(hv & 0xffffu))
                             : "memory");
                asm volatile("st.shared.b16 [%0], %1;" ::"r"((h0 + (j + 1) * 128) ^ (uint32_t)(((j + 1) & 7) << 4)),
                             "h"((unsigned short)(hv >> 16))
                             : "memory");
                r[j] = __float_as_uint(v0 * decay);
                r[j + 1] = __float_as_uint(v1 * decay);
            }
            if (c.do_state) {
#pragma unroll
                for (int cc = 0; cc < kPHalf; cc += 16)
                    tmem_st16(acc + cc, *reinterpret_cast<uint32_t(*)[16]>(r + cc));
                tmem_st_wait();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(&bar_hr[buf]);
            return true;
        };

        // ---- scores: CB (f32, complete after the last block's C B^T) ->
        // masked, decayed bf16 A operand in TMEM; warpgroup wg converts keys
        // [64 wg, 64 wg + 64).  X_hat's barrier also publishes the g / dt table.
        auto build_scores = [&](const Tile &c) -> bool {
            const uint32_t par = c.it & 1;
            if (!mbar_wait(&bar_cb, par) || !mbar_wait(&bar_xh, par))
                return false;
            tc_fence_after();
            const bool full = c.n == kTile;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t cbv[2][16];
#pragma unroll
                for (int gq = 0; gq < 2; ++gq) {
                    const int j0 = wg * 64 + half * 32 + gq * 16;
                    if (j0 <= row_hi)  // warp-uniform: keys above the diagonal stay zero
                        tmem_ld16(lane + Lay::t_cb + j0, cbv[gq]);
                }
                tmem_ld_wait();
#pragma unroll
                for (int gq = 0; gq < 2; ++gq) {
                    const int j0 = wg * 64 + half * 32 + gq * 16;
                    uint32_t pk[8];
                    if (j0 > row_hi) {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            pk[e] = 0u;
                    } else if (c.narrow) {
                        if (full && j0 + 15 < row_lo) {  // whole group below the diagonal
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                pk[e] = pack_bf16x2(__uint_as_float(cbv[gq][2 * e]),
                                                    __uint_as_float(cbv[gq][2 * e + 1]));
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int j = j0 + 2 * e;
                                const float a = (j <= i && j < c.n) ? __uint_as_float(cbv[gq][2 * e]) : 0.f;
                                const float bb =
                                    (j + 1 <= i && j + 1 < c.n) ? __uint_as_float(cbv[gq][2 * e + 1]) : 0.f;
                                pk[e] = pack_bf16x2(a, bb);
                            }
                        }
                    } else {
                        const float4 *g4 = reinterpret_cast<const float4 *>(gtab + j0);
                        const float4 *d4 = reinterpret_cast<const float4 *>(gtab + 128 + j0);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            const float4 gg = g4[v4], dd = d4[v4];
                            const float gj[4] = {gg.x, gg.y, gg.z, gg.w};
                            const float dj[4] = {dd.x, dd.y, dd.z, dd.w};
                            float val[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int j = j0 + 4 * v4 + e;
                                val[e] = (j <= i && j < c.n) ? __uint_as_float(cbv[gq][4 * v4 + e]) *
                                                                   ex2_approx(c.gi - gj[e]) * dj[e]
                                                             : 0.f;
                            }
                            pk[2 * v4] = pack_bf16x2(val[0], val[1]);
                            pk[2 * v4 + 1] = pack_bf16x2(val[2], val[3]);
                        }
                    }
                    tmem_st8(lane + Lay::t_sc + j0 / 2, pk);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            warp_arrive(&bar_sc);
            return true;
        };

        // ---- the state leaving an item: the next segment's start, or the
        // final state (the caller waited for the item's last jumps)
        auto leave_state = [&](const Tile &c) {
            const int64_t bh = c.bh;
            float *dst = nullptr;
            const bool handoff = !c.last_seq && !prm.prefilled;
            if (handoff)
                dst = prm.seg_state + ((bh * prm.n_seg + c.seg) * g.P) * g.S;
            else if (c.last_seq && want_final)
                dst = prm.final_state + bh * g.P * g.S;
            if (dst) {
#pragma unroll 1
                for (int k = 0; k < kSBlk; ++k) {
                    const int sidx = k * 128 + i;
                    uint32_t r[kPHalf];
#pragma unroll
                    for (int cc = 0; cc < kPHalf; cc += 16)
                        tmem_ld16(lane + Lay::t_st + k * P + c0w + cc, *reinterpret_cast<uint32_t(*)[16]>(r + cc));
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < kPHalf; ++j)
                        __stcg(dst + (int64_t)(c0w + j) * S + sidx, __uint_as_float(r[j]));
                }
            }
            if (handoff) {
                __threadfence();
                __syncwarp();
                if ((tid & 31) == 0)
                    atomicAdd(prm.seg_count + bh * prm.n_seg + c.seg, 1u);
            }
        };

        // ---- epilogue (the caller waited for Y): factorized y = r1 Y + D x
        // with r1 = exp2(g_i - g_L); exact y = exp2(g_i) Y + Y1 + D x with Y1
        // in the CB columns.  y goes over the tile's x in its slot.
        auto epilogue = [&](const Tile &c) -> bool {
            tc_fence_after();
            const float r = c.narrow ? ex2_approx(c.gi - c.gL) : ex2_approx(c.gi);
            uint8_t *sx = smem + Lay::off_x + c.sx * Lay::kX;
#pragma unroll
            for (int c16 = 0; c16 < kPHalf; c16 += 16) {
                uint32_t ya[16], yb[16];
                tmem_ld16(lane + Lay::t_y + c0w + c16, ya);
                if (!c.narrow)
                    tmem_ld16(lane + Lay::t_cb + c0w + c16, yb);
                tmem_ld_wait();
#pragma unroll
                for (int k2 = 0; k2 < 2; ++k2) {
                    const uint32_t off = sw128_offset(i, (c0w + c16) / 8 + k2);
                    const uint4 xv = *reinterpret_cast<const uint4 *>(sx + off);
                    const uint32_t vv[4] = {xv.x, xv.y, xv.z, xv.w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int cc = 8 * k2 + 2 * e;
                        float y0 = fmaf(r, __uint_as_float(ya[cc]), c.Dh * bf_lo(vv[e]));
                        float y1 = fmaf(r, __uint_as_float(ya[cc + 1]), c.Dh * bf_hi(vv[e]));
                        if (!c.narrow) {
                            y0 += __uint_as_float(yb[cc]);
                            y1 += __uint_as_float(yb[cc + 1]);
                        }
                        o[e] = pack_bf16x2(y0, y1);
                    }
                    *reinterpret_cast<uint4 *>(sx + off) = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            // Y (and the CB columns) read: the next tile's MMAs may overwrite them
            tc_fence_before();
            warp_arrive(&bar_ep);
            fence_proxy_async_smem();
            warp_arrive(&bar_ys[c.sx]);
            return true;
        };

        bool ok = true;
        Pos p1 = first_pos();
        if (p1.valid) {
            const Raw raw0 = load_raw(p1.w, p1.t);
            Tile cur = make_tile(p1, 0, raw0);
            p1 = next_pos(p1);
            Raw raw1 = load_raw(p1.w, p1.t);
            ok = build_xhat(cur);
            for (int k = 0; k < kSBlk && ok; ++k)
                ok = build_h(cur, k);
            for (uint32_t it = 0; ok; ++it) {
                if (!build_scores(cur)) {
                    ok = false;
                    break;
                }
                // the block loop of `it` done: its jumps have left the state
                if (!mbar_wait(&bar_blk, it & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (cur.last_item && cur.do_state)
                    leave_state(cur);
                Tile nxt{};
                if (p1.valid) {
                    nxt = make_tile(p1, it + 1, raw1);
                    for (int k = 0; k < 2 && ok; ++k)
                        ok = build_h(nxt, k);
                    if (!ok)
                        break;
                }
                // Y1 done: X_hat hi, lo and the table are free, Y is complete
                if (!mbar_wait(&bar_y, it & 1)) {
                    ok = false;
                    break;
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
                // the tile after the next one: its G / dt words are in flight
                // for a whole tile before make_tile reads them
                const Pos p2 = next_pos(p1);
                const Raw raw2 = load_raw(p2.w, p2.t);
                for (int k = 2; k < kSBlk && ok; ++k)
                    ok = build_h(nxt, k);
                cur = nxt;
                p1 = p2;
                raw1 = raw2;
            }
        }
        if (!ok)
            atomicOr(prm.status, 1u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, Lay::kTmemCols);
    }
}

int sm_count()
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

template <int P, int S, int STAGES, int MODE>
cudaError_t launch_cfg(const CUtensorMap &tx, const CUtensorMap &tb, const CUtensorMap &tcm,
                       const CUtensorMap &ty, const Params &prm, cudaStream_t st)
{
    using Lay = CoLayout<P, S, STAGES>;
    const size_t smem = Lay::bytes + 1024;
    auto k = chunk_tc_kernel<P, S, STAGES, MODE>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const int grid = prm.n_items < sm_count() ? prm.n_items : sm_count();
    k<<<(unsigned)grid, kThreads, smem, st>>>(tx, tb, tcm, ty, prm);
    note_launch();
    return cudaGetLastError();
}

template <int P, int S>
cudaError_t launch_big(const CUtensorMap &tx, const CUtensorMap &tb, const CUtensorMap &tcm,
                       const CUtensorMap &ty, const Params &prm, cudaStream_t st)
{
    using Lay = BigLayout<P, S>;
    const size_t smem = Lay::bytes + 1024;
    auto k = chunk_big_kernel<P, S>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const int grid = prm.n_items < sm_count() ? prm.n_items : sm_count();
    k<<<(unsigned)grid, kThreads, smem, st>>>(tx, tb, tcm, ty, prm);
    note_launch();
    return cudaGetLastError();
}

template <int MODE>
cudaError_t dispatch(const CUtensorMap &tx, const CUtensorMap &tb, const CUtensorMap &tcm,
                     const CUtensorMap &ty, const Params &prm, cudaStream_t st)
{
    const Geom &g = prm.g;
    if (g.P == 64 && g.S == 64)
        return launch_cfg<64, 64, 3, MODE>(tx, tb, tcm, ty, prm, st);
    if (g.P == 64 && g.S == 128)
        return launch_cfg<64, 128, 2, MODE>(tx, tb, tcm, ty, prm, st);
    if (g.P == 64 && g.S == 256)
        return launch_cfg<64, 256, 1, MODE>(tx, tb, tcm, ty, prm, st);
    return cudaErrorNotSupported;
}

struct SegPlan {
    int seg_tiles;
    int n_seg;
    bool prefill;
    size_t state_bytes, count_bytes;
};

// Segments of the fused pass.  With at most half as many (batch, head)
// sequences as SMs, segments that hand their states to one another run as a
// wavefront (at most one segment of each sequence makes progress at a time),
// so the sequences are cut into up to kMaxPrefillSeg segments of whole chunks
// -- about eight items per SM, at least two chunks each -- whose start states
// a segmented state pass computes first (the prefilled plan): every item is
// then independent.  (With more sequences the extra state pass costs more
// than the wavefront: B 2, L 32768, H 64, S 256 took 1.74 ms prefilled
// against 1.39 ms with hand-offs; B 1, L 262144, H 64, S 256 took 6.17 ms
// against 10.66 ms.)  With at most one sequence per SM: one segment each, a
// CTA runs its sequence end to end (only one segment of a sequence can run at
// a time, so cutting it adds hand-offs and lets one late segment hold up the
// others queued behind it on the same CTA: B 2, L 32768, H 64, S 256 took
// 1.22 ms against 1.32 ms with ten segments each).  With more sequences than
// SMs: enough hand-off segments for about sixteen items per SM, none shorter
// than two tiles, so that CTAs whose tiles run slower (their share of L2
// bandwidth differs) end near the others (B 4, L 65536, H 64, S 256: 3.94 ms
// against 4.05 ms with about eight).
constexpr int kMaxPrefillSeg = 64;  // segments the state pass's combine handles

SegPlan seg_plan(const Geom &g)
{
    SegPlan sp;
    sp.prefill = false;
    const int64_t n_tiles = (g.L + kTile - 1) / kTile;
    const int64_t nbh = g.B * g.H;
    const int tpc = g.T / kTile;
    if (2 * nbh <= sm_count() && state_pass_tc_supported(g)) {
        int64_t want = (8LL * sm_count() + nbh - 1) / nbh;
        if (want > kMaxPrefillSeg)
            want = kMaxPrefillSeg;
        if (want * 2 * tpc > n_tiles)
            want = n_tiles / (2 * tpc);
        if (want >= 2) {
            int64_t st = (n_tiles + want - 1) / want;
            st = (st + tpc - 1) / tpc * tpc;
            sp.seg_tiles = (int)st;
            sp.n_seg = (int)((n_tiles + st - 1) / st);
            if (sp.n_seg >= 2) {
                sp.prefill = true;
                sp.state_bytes = (size_t)(nbh * sp.n_seg * g.P * g.S) * sizeof(float);
                sp.count_bytes = 0;
                return sp;
            }
        }
    }
    // one segment per sequence while every sequence has an SM of its own
    int64_t want = nbh <= sm_count() ? 1 : (16LL * sm_count() + nbh - 1) / nbh;
    want = want < 1 ? 1 : want;
    if (want > (n_tiles + 1) / 2)
        want = (n_tiles + 1) / 2 < 1 ? 1 : (n_tiles + 1) / 2;
    sp.seg_tiles = (int)((n_tiles + want - 1) / want);
    sp.n_seg = (int)((n_tiles + sp.seg_tiles - 1) / sp.seg_tiles);
    sp.state_bytes = sp.n_seg > 1 ? (size_t)(nbh * sp.n_seg * g.P * g.S) * sizeof(float) : 0;
    sp.count_bytes = sp.n_seg > 1 ? (size_t)(nbh * sp.n_seg) * sizeof(unsigned int) : 0;
    return sp;
}

cudaError_t run(int mode, const void *x, const void *Bm, const void *Cm, const float *dtT,
                const float *Gc, const float *D, const float *h_src, float *states_out,
                float *final_state, void *y, const Geom &g, void *scratch, size_t scratch_bytes,
                cudaStream_t st)
{
    if (mode == kModeOut ? !chunk_tc_supported(g) : !fused_tc_supported(g))
        return cudaErrorNotSupported;
    Params prm{};
    prm.dtT = dtT;
    prm.Gc = Gc;
    prm.D = D;
    prm.h_src = h_src;
    prm.states_out = states_out;
    prm.final_state = final_state;
    prm.g = g;
    prm.n_tiles = (int)((g.L + kTile - 1) / kTile);
    prm.tpc_shift = g.T == 2 * kTile ? 1 : 0;
    prm.H = (int)g.H;
    prm.nc = (int)g.nc;
    prm.nbh = (int)(g.B * g.H);
    prm.n_items = (int)(g.B * g.nc * g.H);
    prm.seg_tiles = prm.n_tiles;
    prm.n_seg = 1;
    if (mode == kModeFused) {
        const SegPlan sp = seg_plan(g);
        prm.seg_tiles = sp.seg_tiles;
        prm.n_seg = sp.n_seg;
        prm.n_items = (int)(g.B * g.H * sp.n_seg);
        prm.prefilled = sp.prefill ? 1 : 0;
        if (sp.n_seg > 1) {
            const size_t off = (sp.state_bytes + 255) / 256 * 256;
            if (!scratch || scratch_bytes < off + sp.count_bytes)
                return cudaErrorInvalidValue;
            prm.seg_state = static_cast<float *>(scratch);
            cudaError_t e;
            if (sp.prefill) {
                // every segment's start state (segment 0's is the initial state)
                e = launch_segment_starts_tc(x, Bm, dtT, Gc, h_src, prm.seg_state, sp.seg_tiles,
                                             sp.n_seg, g, st);
            } else {
                prm.seg_count = reinterpret_cast<unsigned int *>(static_cast<char *>(scratch) + off);
                e = cudaMemsetAsync(prm.seg_count, 0, sp.count_bytes, st);
            }
            if (e != cudaSuccess)
                return e;
        }
    }
    prm.status = device_status_word();
    if (!prm.status)
        return cudaErrorUnknown;
    CUtensorMap tx, tb, tcm, ty;
    if (!make_tmap_tokens_heads(&tx, x, g) || !make_tmap_tokens_groups(&tb, Bm, g) ||
        !make_tmap_tokens_groups(&tcm, Cm, g) || !make_tmap_tokens_heads(&ty, y, g))
        return cudaErrorInvalidValue;
    if (mode == kModeFused && g.P == 64 && g.S == 384)
        return launch_big<64, 384>(tx, tb, tcm, ty, prm, st);
    if (mode == kModeFused && g.P == 64 && g.S == 512)
        return launch_big<64, 512>(tx, tb, tcm, ty, prm, st);
    return mode == kModeOut ? dispatch<kModeOut>(tx, tb, tcm, ty, prm, st)
                            : dispatch<kModeFused>(tx, tb, tcm, ty, prm, st);
}

}  // namespace

namespace {
// work items and tile indices are 32-bit in the kernels
bool tile_geometry_ok(const Geom &g)
{
    const int64_t n_tiles = (g.L + kTile - 1) / kTile;
    return (g.T == kTile || g.T == 2 * kTile) && g.L > 0 && g.L < (1LL << 31) && g.H <= 65535 &&
           g.G <= 65535 && g.B <= 65535 && g.B * g.H * n_tiles < (1LL << 31);
}
}  // namespace

bool chunk_tc_supported(const Geom &g)
{
    return g.P == 64 && (g.S == 64 || g.S == 128 || g.S == 256) && tile_geometry_ok(g);
}

bool fused_tc_supported(const Geom &g)
{
    return chunk_tc_supported(g) || (g.P == 64 && (g.S == 384 || g.S == 512) && tile_geometry_ok(g));
}

cudaError_t launch_chunk_out_tc(const void *x, const void *Bm, const void *Cm, const float *dtT,
                                const float *Gc, const float *states, const float *D, void *y,
                                const Geom &g, cudaStream_t st)
{
    return run(kModeOut, x, Bm, Cm, dtT, Gc, D, states, nullptr, nullptr, y, g, nullptr, 0, st);
}

bool fused_pair_enabled(const Geom &g)
{
    const char *env = getenv("SSD_FUSED_KERNEL");
    return pair_tc_supported(g) && !(env && strcmp(env, "single") == 0);
}

size_t fused_tc_scratch_bytes(const Geom &g)
{
    const SegPlan sp = seg_plan(g);
    if (sp.n_seg <= 1)
        return 0;
    return (sp.state_bytes + 255) / 256 * 256 + (sp.count_bytes + 255) / 256 * 256;
}

cudaError_t launch_fused_tc(const void *x, const void *Bm, const void *Cm, const float *dtT,
                            const float *Gc, const float *D, const float *init, float *states,
                            float *final_state, void *y, const Geom &g, void *scratch,
                            size_t scratch_bytes, cudaStream_t st)
{
    return run(kModeFused, x, Bm, Cm, dtT, Gc, D, init, states, final_state, y, g, scratch,
               scratch_bytes, st);
}

}  // namespace ssd
