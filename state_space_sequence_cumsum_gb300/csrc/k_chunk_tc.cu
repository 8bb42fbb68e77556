// Stage 3 (chunk output) and the fused single-pass forward on tensor cores,
// bf16 inputs.
//
// "Accelerating Mamba-2 forward-pass kernels with CUDA Tile (cuTile)",
// section "Kernel 3: compute_out", per (batch, chunk, head):
//     Y = exp2(G) * (C h_c^T) + (exp2(G_i - G_j) * (C B^T) * M)(dt * X) + D X
// and section "Kernel 2: fwd_pass_state" for the state jump
//     h <- exp2(G_last) h + X^T (B * dt * exp2(G_last - G)).
//
// One kernel, two modes:
//   OUT   -- a work item is (batch, chunk, head); h_c comes from chunk_states.
//   FUSED -- a work item is (batch, head) over the whole sequence; the state
//            is carried on chip from tile to tile, so chunk states never go
//            through HBM unless the caller asks for them.
// Tokens are processed in 128-token tiles (the tcgen05 M and K extent).  A
// chunk of 256 tokens is two tiles: the second tile's starting state is the
// first tile's state jump applied to h_c, and its G is taken relative to the
// token before it, which is the same arithmetic regrouped
// (exp2(G_i - G_j) = exp2(G_i - G_m) exp2(G_m - G_j) with both factors <= 1).
//
// Per tile (all contractions are tcgen05.mma kind::f16, f32 accumulate in TMEM):
//   CB  = C B^T                 M 128 (i) x N 128 (j), K = S     [TMEM cols 0..127]
//   scores_ij = CB_ij exp2(g_i - g_j) dt_j for j <= i (masked entries are set
//               to zero without evaluating the exponent), bf16 into shared memory
//   Y1  = scores X              N = P, K = 128                   [TMEM]
//   Y2  = C H^T, H = bf16(h_c)  N = P, K = S                     [TMEM]
//   y   = Y1 + exp2(g_i) Y2 + D x      (f32 epilogue, bf16 store)
//   and, when a later tile needs the state: h <- exp2(g_L) h + B^T X_hat with
//   X_hat = dt exp2(g_L - g) X split into bf16 hi + lo (two MMA passes); the
//   state h^T [S, P] is an f32 TMEM accumulator.
//
// Roles: warps 0-3 are the compute warpgroup (thread i owns tile row i, i.e.
// TMEM lane i); warp 4 lane 0 issues TMA loads into a STAGES-deep ring
// (B, C and x tiles, 128-byte swizzle); warp 5 lane 0 issues the MMAs.  The
// CTA is persistent over work items.  Every wait is bounded; a timeout sets
// the kernel status word and the role leaves its loop.
#include "common.cuh"
#include "ssd_internal.h"
#include "tc05.cuh"

namespace ssd {
namespace {
using namespace tc;

constexpr int kTile = 128;
constexpr int kComputeThreads = 256;  // two warpgroups
constexpr int kThreads = kComputeThreads + 64;
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
    static constexpr uint32_t kStage = 2 * kB + kX;  // B, C, x
    static constexpr uint32_t off_xh = STAGES * kStage;  // X_hat hi, then lo
    static constexpr uint32_t off_h = off_xh + 2 * kX;
    static constexpr uint32_t kHRegion = P * 128;  // P rows x 128 bytes
    static constexpr uint32_t kH = kSReg * kHRegion;
    static constexpr uint32_t off_g = off_h + kH;  // [2 tiles][g 128 | dt 128] f32
    static constexpr uint32_t bytes = off_g + 2 * 256 * 4;
    // TMEM columns: CB (f32), the bf16 score operand (two per column), Y1, Y2,
    // and the f32 state accumulator
    static constexpr uint32_t t_cb = 0, t_sc = 128, t_y1 = 192, t_y2 = 192 + P,
                              t_st = 192 + 2 * P;
    static constexpr uint32_t cols_used = t_st + kSBlk * P;
    static constexpr uint32_t kTmemCols = cols_used <= 256 ? 256 : 512;
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
    __nv_bfloat16 *y;
    Geom g;
    int64_t n_items;
    int64_t n_tiles;  // tiles per sequence
    int tiles_per_chunk;
    // FUSED: each (batch, head) sequence is split into n_seg segments of
    // seg_tiles tiles; segment k > 0 starts from the state segment k-1 leaves
    // in seg_state, published by seg_count reaching kComputeThreads.
    int64_t seg_tiles;
    int n_seg;
    float *seg_state;          // [B*H*n_seg][P][S]
    unsigned int *seg_count;   // [B*H*n_seg], zero at launch
    unsigned int *status;
};

template <int MODE>
__device__ __forceinline__ void decode_item(const Params &p, int64_t item, int64_t &b, int64_t &h,
                                            int64_t &t0, int64_t &t1, int64_t &chunk)
{
    if (MODE == kModeOut) {
        // consecutive items share (b, chunk) so their B/C tiles hit in L2
        h = item % p.g.H;
        const int64_t bc = item / p.g.H;
        chunk = bc % p.g.nc;
        b = bc / p.g.nc;
        t0 = chunk * p.tiles_per_chunk;
        t1 = min64(t0 + p.tiles_per_chunk, p.n_tiles);
    } else {
        // segment-major: every segment k of every sequence comes before any
        // segment k+1, so a segment's predecessor is always an earlier item
        const int64_t nbh = p.g.B * p.g.H;
        const int64_t seg = item / nbh, bh = item % nbh;
        h = bh % p.g.H;
        b = bh / p.g.H;
        t0 = seg * p.seg_tiles;
        t1 = min64(t0 + p.seg_tiles, p.n_tiles);
        chunk = seg;
    }
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int *p)
{
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void tma4(void *dst, const void *tmap, uint64_t *bar, int c0, int c1,
                                     int c2, int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// K-major operand (rows x K, 64 K-elements per 128-byte row, one region per
// 64 K): descriptor for the 16-wide K step ks.
__device__ __forceinline__ uint64_t desc_k(uint32_t base, uint32_t region_bytes, int ks)
{
    return smem_desc(base + (ks >> 2) * region_bytes + (ks & 3) * 32, 16, 1024);
}
// MN-major operand (128 K-rows of 64 M/N elements per region): K step ks.
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, int ks)
{
    return smem_desc(base + ks * 2048, kRegion, 1024);
}

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

template <int P, int S, int STAGES, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ CUtensorMap tm_c, const Params prm)
{
    using Lay = CoLayout<P, S, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_full[STAGES], bar_empty[STAGES];
    __shared__ uint64_t bar_cb, bar_scores, bar_xh, bar_h, bar_done, bar_g;
    __shared__ uint32_t tmem_slot;
    __shared__ int s_mode[2];  // per tile parity: 1 = factorized (narrow) decay

    const Geom &g = prm.g;
    const int tid = threadIdx.x, warp = tid >> 5;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], 1 + kComputeThreads);
        }
        mbar_init(&bar_cb, 1);
        mbar_init(&bar_scores, kComputeThreads);
        mbar_init(&bar_xh, kComputeThreads);
        mbar_init(&bar_h, kComputeThreads);
        mbar_init(&bar_done, 1);
        mbar_init(&bar_g, kComputeThreads);
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
            int64_t it = 0;
            bool ok = true;
            for (int64_t item = blockIdx.x; item < prm.n_items && ok; item += gridDim.x) {
                int64_t b, h, t0, t1, chunk;
                decode_item<MODE>(prm, item, b, h, t0, t1, chunk);
                const int64_t grp = h / g.hpg;
                for (int64_t t = t0; t < t1; ++t, ++it) {
                    const int s = (int)(it % STAGES);
                    if (it >= STAGES &&
                        !mbar_wait(&bar_empty[s], (uint32_t)(((it / STAGES) - 1) & 1))) {
                        atomicOr(prm.status, 1u);
                        ok = false;
                        break;
                    }
                    uint8_t *st = smem + s * Lay::kStage;
                    mbar_arrive_expect_tx(&bar_full[s], Lay::kStage);
                    const int tok = (int)(t * kTile);
                    for (int r = 0; r < Lay::kSReg; ++r) {
                        tma4(st + r * kRegion, &tm_b, &bar_full[s], r * 64, (int)grp, tok, (int)b);
                        tma4(st + Lay::kB + r * kRegion, &tm_c, &bar_full[s], r * 64, (int)grp,
                             tok, (int)b);
                    }
                    for (int r = 0; r < Lay::kPReg; ++r)
                        tma4(st + 2 * Lay::kB + r * kRegion, &tm_x, &bar_full[s], r * 64, (int)h,
                             tok, (int)b);
                }
            }
        }
    } else if (warp == 9) {
        // ---------------- MMA issuer.  Per tile: CB; then (X_hat and H ready)
        // Y2 and the state jump; then (scores ready) Y1; one commit covers all.
        if ((tid & 31) == 0) {
            const uint32_t id_cb = idesc_bf16(128, 128, false, false);
            const uint32_t id_y1 = idesc_bf16(128, P, false, true);  // A (scores) from TMEM
            const uint32_t id_y2 = idesc_bf16(128, P, false, false);
            const uint32_t id_ds = idesc_bf16(128, P, true, true);
            const uint32_t s_xh = smem_u32(smem + Lay::off_xh);
            const uint32_t s_h = smem_u32(smem + Lay::off_h);
            int64_t it = 0;
            bool ok = true;
            for (int64_t item = blockIdx.x; item < prm.n_items && ok; item += gridDim.x) {
                int64_t b, h, t0, t1, chunk;
                decode_item<MODE>(prm, item, b, h, t0, t1, chunk);
                for (int64_t t = t0; t < t1; ++t, ++it) {
                    const bool last_seq = MODE == kModeOut ? t + 1 == t1 : t + 1 == prm.n_tiles;
                    const bool do_state = !last_seq || want_final;
                    const int s = (int)(it % STAGES);
                    const uint32_t sb = smem_u32(smem + s * Lay::kStage);
                    const uint32_t sc = sb + Lay::kB;
                    const uint32_t sx = sb + 2 * Lay::kB;
                    const uint32_t par = (uint32_t)(it & 1);
                    if (!mbar_wait(&bar_full[s], (uint32_t)((it / STAGES) & 1))) {
                        ok = false;
                        break;
                    }
                    // CB overwrites the previous tile's score columns
                    if (it > 0 && !mbar_wait(&bar_done, (uint32_t)((it - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < S / 16; ++ks)
                        mma_ss(tmem + Lay::t_cb, desc_k(sc, kRegion, ks), desc_k(sb, kRegion, ks),
                               id_cb, ks > 0);
                    mma_commit(&bar_cb);
                    if (!mbar_wait(&bar_xh, par) || !mbar_wait(&bar_h, par)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < S / 16; ++ks)
                        mma_ss(tmem + Lay::t_y2, desc_k(sc, kRegion, ks),
                               desc_k(s_h, Lay::kHRegion, ks), id_y2, ks > 0);
                    if (do_state) {
#pragma unroll
                        for (int mb = 0; mb < Lay::kSBlk; ++mb)
#pragma unroll
                            for (int part = 0; part < 2; ++part)
#pragma unroll
                                for (int ks = 0; ks < kTile / 16; ++ks)
                                    mma_ss(tmem + Lay::t_st + mb * P,
                                           desc_mn(sb + 2 * mb * kRegion, ks),
                                           desc_mn(s_xh + part * Lay::kX, ks), id_ds, 1u);
                    }
                    if (!mbar_wait(&bar_scores, par)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t y1b = s_mode[it & 1] ? s_xh : sx;  // X_hat or raw x
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks)
                        mma_ts(tmem + Lay::t_y1, tmem + Lay::t_sc + ks * 8, desc_mn(y1b, ks), id_y1,
                               ks > 0);
                    mma_commit(&bar_done);
                    mma_commit(&bar_empty[s]);
                }
            }
            if (!ok)
                atomicOr(prm.status, 1u);
        }
    } else {
        // ---------------- two compute warpgroups.  Thread (wg, q, lane) owns
        // tile row / TMEM lane i = 32 q + lane; warpgroup wg owns half of the
        // columns of every per-tile step.  Order per tile: X_hat, H (so the
        // MMA can start the state jump early), scores, epilogue.
        const int wg = warp >> 2, q = warp & 3;
        const int i = q * 32 + (tid & 31);
        const uint32_t lane = tmem_at(tmem, (uint32_t)(q * 32), 0);
        float *gtab_all = reinterpret_cast<float *>(smem + Lay::off_g);
        uint8_t *s_xh = smem + Lay::off_xh;
        uint8_t *s_h = smem + Lay::off_h;
        constexpr int kPHalf = P / 2;

        // raw G / dt values of a tile, loaded one tile ahead
        struct Raw {
            float base, g0, gL, gi, dti;
        };
        auto load_raw = [&](int64_t item, int64_t t) {
            int64_t b, h, t0, t1, chunk;
            decode_item<MODE>(prm, item, b, h, t0, t1, chunk);
            const int64_t bh = b * g.H + h;
            const float *grow = prm.Gc + bh * g.L;
            const int64_t tau = t * kTile;
            const int n = (int)min64(kTile, g.L - tau);
            Raw r;
            r.base = (tau % g.T == 0) ? 0.f : grow[tau - 1];
            r.g0 = grow[tau];
            r.gL = grow[tau + n - 1];
            r.gi = i < n ? grow[tau + i] : 0.f;
            r.dti = i < n ? prm.dtT[bh * g.L + tau + i] : 0.f;
            return r;
        };
        Raw nxt{};
        if ((int64_t)blockIdx.x < prm.n_items) {
            int64_t b, h, t0, t1, chunk;
            decode_item<MODE>(prm, blockIdx.x, b, h, t0, t1, chunk);
            nxt = load_raw(blockIdx.x, t0);
        }
        int64_t it = 0;
        bool ok = true;
        for (int64_t item = blockIdx.x; item < prm.n_items && ok; item += gridDim.x) {
            int64_t b, h, t0, t1, chunk;
            decode_item<MODE>(prm, item, b, h, t0, t1, chunk);
            const int64_t bh = b * g.H + h;
            const float Dh = prm.D[h];
            for (int64_t t = t0; t < t1; ++t, ++it) {
                const int64_t tau = t * kTile;
                const int n = (int)min64(kTile, g.L - tau);
                const bool first = t == t0, last_item = t + 1 == t1;
                const bool last_seq = MODE == kModeOut ? last_item : t + 1 == prm.n_tiles;
                const bool do_state = !last_seq || want_final;
                const Raw cur = nxt;
                // prefetch the next tile's G / dt while this one is processed
                if (!last_item)
                    nxt = load_raw(item, t + 1);
                else if (item + gridDim.x < prm.n_items) {
                    int64_t b2, h2, u0, u1, c2;
                    decode_item<MODE>(prm, item + gridDim.x, b2, h2, u0, u1, c2);
                    nxt = load_raw(item + gridDim.x, u0);
                }
                const float gL = cur.gL - cur.base;
                const float range = (cur.g0 - cur.base) - gL;
                const bool narrow = range <= kNarrow && range >= -kNarrow;
                const float gi = cur.gi - cur.base;
                const float dti = cur.dti;
                const int s = (int)(it % STAGES);
                const uint8_t *sx = smem + s * Lay::kStage + 2 * Lay::kB;
                const uint32_t par = (uint32_t)(it & 1);

                // ---- per-tile g / dt table (double-buffered by tile parity)
                float *gtab = gtab_all + (it & 1) * 256;
                if (wg == 0)
                    gtab[i] = gi;
                else
                    gtab[128 + i] = dti;
                if (tid == 0)
                    s_mode[it & 1] = narrow ? 1 : 0;
                mbar_arrive(&bar_g);
                if (!mbar_wait(&bar_g, par) ||
                    !mbar_wait(&bar_full[s], (uint32_t)((it / STAGES) & 1))) {
                    ok = false;
                    break;
                }
                // the previous tile's MMAs (state jump, Y1 reading X_hat) are done
                if (it > 0 && !mbar_wait(&bar_done, (uint32_t)((it - 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();

                // ---- X_hat = dt exp2(g_L - g) x as bf16 hi (+ lo for the state jump)
                if (narrow || do_state) {
                    const float w = i < n ? dti * ex2_approx(gL - gi) : 0.f;
#pragma unroll
                    for (int r = 0; r < Lay::kPReg; ++r) {
#pragma unroll
                        for (int c = wg * 4; c < wg * 4 + 4; ++c) {
                            const uint32_t off = r * kRegion + sw128_offset(i, c);
                            const uint4 v = *reinterpret_cast<const uint4 *>(sx + off);
                            const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
                            uint32_t hi[4], lo[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float a = bf_lo(vv[e]) * w, bb = bf_hi(vv[e]) * w;
                                hi[e] = pack_bf16x2(a, bb);
                                lo[e] = pack_bf16x2(a - bf_lo(hi[e]), bb - bf_hi(hi[e]));
                            }
                            *reinterpret_cast<uint4 *>(s_xh + off) =
                                make_uint4(hi[0], hi[1], hi[2], hi[3]);
                            if (do_state)
                                *reinterpret_cast<uint4 *>(s_xh + Lay::kX + off) =
                                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
                        }
                    }
                    fence_proxy_async_smem();
                }
                mbar_arrive(&bar_xh);

                // ---- a later segment waits until its predecessor published its state
                if (MODE == kModeFused && first && chunk > 0) {
                    const unsigned int *cnt = prm.seg_count + bh * prm.n_seg + chunk - 1;
                    bool ready = ld_acquire_gpu(cnt) >= (unsigned)kComputeThreads;
                    const uint64_t t_start = globaltimer_ns();
                    while (!ready) {
                        if (globaltimer_ns() - t_start > 2000000000ull)
                            break;
                        __nanosleep(256);
                        ready = ld_acquire_gpu(cnt) >= (unsigned)kComputeThreads;
                    }
                    if (!ready) {
                        ok = false;
                        break;
                    }
                }

                // ---- H = bf16(hscale * h) into K-major [p][s]; emit and decay the state
                const float decay = ex2_approx(gL);
                const float hscale = narrow ? decay : 1.f;
                const bool emit = MODE == kModeFused && prm.states_out && (tau % g.T == 0);
#pragma unroll
                for (int mb = 0; mb < Lay::kSBlk; ++mb) {
                    const int sidx = mb * 128 + i;
                    const bool s_ok = sidx < S;
                    const uint32_t acc = lane + Lay::t_st + mb * P;
                    const float *src = nullptr;
                    if (first) {
                        if (MODE == kModeOut)
                            src = prm.h_src + ((bh * g.nc + chunk) * g.P) * g.S;
                        else if (chunk > 0)  // later segment: the predecessor's state
                            src = prm.seg_state + ((bh * prm.n_seg + chunk - 1) * g.P) * g.S;
                        else if (prm.h_src)
                            src = prm.h_src + bh * g.P * g.S;
                    }
                    float *emit_dst =
                        emit ? prm.states_out + ((bh * g.nc + tau / g.T) * g.P) * g.S : nullptr;
                    uint8_t *hb = s_h + (sidx >> 6) * Lay::kHRegion;
                    const int cs = sidx & 63;
#pragma unroll
                    for (int c0 = wg * kPHalf; c0 < (wg + 1) * kPHalf; c0 += 16) {
                        uint32_t r[16];
                        if (first) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                r[j] = __float_as_uint(
                                    (src && s_ok) ? __ldcg(src + (int64_t)(c0 + j) * S + sidx) : 0.f);
                        } else {
                            tmem_ld16(acc + c0, r);
                            tmem_ld_wait();
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float v = __uint_as_float(r[j]);
                            if (s_ok) {
                                if (emit_dst)
                                    emit_dst[(int64_t)(c0 + j) * S + sidx] = v;
                                *reinterpret_cast<__nv_bfloat16 *>(
                                    hb + sw128_offset(c0 + j, cs >> 3) + (cs & 7) * 2) =
                                    __float2bfloat16_rn(v * hscale);
                            }
                            r[j] = __float_as_uint(v * decay);
                        }
                        if (do_state)
                            tmem_st16(acc + c0, r);
                    }
                }
                if (do_state)
                    tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bar_h);

                // ---- scores: CB (f32) -> masked, decayed bf16 A operand in TMEM.
                // Warpgroup wg converts keys [64 wg, 64 wg + 64), 16 at a time.
                if (!mbar_wait(&bar_cb, par)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int row_max = q * 32 + 31;  // warp-uniform bound for the collective ld/st
#pragma unroll
                for (int gq = 0; gq < 4; ++gq) {
                    const int j0 = wg * 64 + gq * 16;
                    uint32_t pk[8];
                    if (j0 <= row_max) {
                        uint32_t cbv[16];
                        tmem_ld16(lane + Lay::t_cb + j0, cbv);
                        tmem_ld_wait();
                        if (narrow) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int j = j0 + 2 * e;
                                const float a = (j <= i && j < n) ? __uint_as_float(cbv[2 * e]) : 0.f;
                                const float bb =
                                    (j + 1 <= i && j + 1 < n) ? __uint_as_float(cbv[2 * e + 1]) : 0.f;
                                pk[e] = pack_bf16x2(a, bb);
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
                                    val[e] = (j <= i && j < n) ? __uint_as_float(cbv[4 * v4 + e]) *
                                                                     ex2_approx(gi - gj[e]) * dj[e]
                                                               : 0.f;
                                }
                                pk[2 * v4] = pack_bf16x2(val[0], val[1]);
                                pk[2 * v4 + 1] = pack_bf16x2(val[2], val[3]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            pk[e] = 0u;
                    }
                    tmem_st8(lane + Lay::t_sc + j0 / 2, pk);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bar_scores);

                // ---- epilogue: y = r1 Y1 + r2 Y2 + D x
                if (!mbar_wait(&bar_done, par)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float r1 = narrow ? ex2_approx(gi - gL) : 1.f;
                const float r2 = narrow ? r1 : ex2_approx(gi);
                __nv_bfloat16 *yrow = prm.y + ((b * g.L + tau + i) * g.H + h) * g.P;
#pragma unroll
                for (int c0 = wg * kPHalf; c0 < (wg + 1) * kPHalf; c0 += 16) {
                    uint32_t ra[16], rb[16];
                    tmem_ld16(lane + Lay::t_y1 + c0, ra);
                    tmem_ld16(lane + Lay::t_y2 + c0, rb);
                    tmem_ld_wait();
                    const uint8_t *xr = sx + (c0 >> 6) * kRegion;
                    const int cc = (c0 & 63) >> 3;
                    const uint4 xa = *reinterpret_cast<const uint4 *>(xr + sw128_offset(i, cc));
                    const uint4 xb = *reinterpret_cast<const uint4 *>(xr + sw128_offset(i, cc + 1));
                    const uint32_t xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
                    uint32_t o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float a = r1 * __uint_as_float(ra[2 * e]) +
                                        r2 * __uint_as_float(rb[2 * e]) + Dh * bf_lo(xv[e]);
                        const float bb = r1 * __uint_as_float(ra[2 * e + 1]) +
                                         r2 * __uint_as_float(rb[2 * e + 1]) + Dh * bf_hi(xv[e]);
                        o[e] = pack_bf16x2(a, bb);
                    }
                    if (i < n) {
                        uint4 *dst = reinterpret_cast<uint4 *>(yrow + c0);
                        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
                    }
                }
                tc_fence_before();
                mbar_arrive(&bar_empty[s]);

                // ---- state leaving the item: the next segment's start, or the final state
                if (do_state && last_item) {
                    float *dst = nullptr;
                    const bool handoff = MODE == kModeFused && !last_seq;
                    if (handoff)
                        dst = prm.seg_state + ((bh * prm.n_seg + chunk) * g.P) * g.S;
                    else if (last_seq && want_final)
                        dst = prm.final_state + bh * g.P * g.S;
                    if (dst) {
#pragma unroll
                        for (int mb = 0; mb < Lay::kSBlk; ++mb) {
                            const int sidx = mb * 128 + i;
#pragma unroll
                            for (int c0 = wg * kPHalf; c0 < (wg + 1) * kPHalf; c0 += 16) {
                                uint32_t r[16];
                                tmem_ld16(lane + Lay::t_st + mb * P + c0, r);
                                tmem_ld_wait();
                                if (sidx < S) {
#pragma unroll
                                    for (int j = 0; j < 16; ++j)
                                        __stcg(dst + (int64_t)(c0 + j) * S + sidx,
                                               __uint_as_float(r[j]));
                                }
                            }
                        }
                    }
                    if (handoff) {
                        __threadfence();
                        atomicAdd(prm.seg_count + bh * prm.n_seg + chunk, 1u);
                    }
                }
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
                       const Params &prm, cudaStream_t st)
{
    using Lay = CoLayout<P, S, STAGES>;
    const size_t smem = Lay::bytes + 1024;
    auto k = chunk_tc_kernel<P, S, STAGES, MODE>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const int64_t grid = min64(prm.n_items, (int64_t)sm_count());
    k<<<(unsigned)grid, kThreads, smem, st>>>(tx, tb, tcm, prm);
    note_launch();
    return cudaGetLastError();
}

template <int MODE>
cudaError_t dispatch(const CUtensorMap &tx, const CUtensorMap &tb, const CUtensorMap &tcm,
                     const Params &prm, cudaStream_t st)
{
    const Geom &g = prm.g;
    if (g.P == 64 && g.S == 64)
        return launch_cfg<64, 64, 3, MODE>(tx, tb, tcm, prm, st);
    if (g.P == 64 && g.S == 128)
        return launch_cfg<64, 128, 2, MODE>(tx, tb, tcm, prm, st);
    if (g.P == 64 && g.S == 256)
        return launch_cfg<64, 256, 1, MODE>(tx, tb, tcm, prm, st);
    return cudaErrorNotSupported;
}

// Segmentation of the fused pass: enough (batch, head, segment) items for
// about eight per SM, so the persistent CTAs end within one item of each
// other; no segment shorter than two tiles.
struct SegPlan {
    int64_t seg_tiles;
    int n_seg;
    size_t state_bytes, count_bytes;
};

SegPlan seg_plan(const Geom &g)
{
    SegPlan sp;
    const int64_t n_tiles = (g.L + kTile - 1) / kTile;
    const int64_t nbh = g.B * g.H;
    int64_t want = (8LL * sm_count() + nbh - 1) / nbh;
    want = want < 1 ? 1 : want;
    if (want > (n_tiles + 1) / 2)
        want = (n_tiles + 1) / 2 < 1 ? 1 : (n_tiles + 1) / 2;
    sp.seg_tiles = (n_tiles + want - 1) / want;
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
    if (!chunk_tc_supported(g))
        return cudaErrorNotSupported;
    Params prm{};
    prm.dtT = dtT;
    prm.Gc = Gc;
    prm.D = D;
    prm.h_src = h_src;
    prm.states_out = states_out;
    prm.final_state = final_state;
    prm.y = static_cast<__nv_bfloat16 *>(y);
    prm.g = g;
    prm.n_tiles = (g.L + kTile - 1) / kTile;
    prm.tiles_per_chunk = g.T / kTile;
    prm.n_items = g.B * g.nc * g.H;
    prm.seg_tiles = prm.n_tiles;
    prm.n_seg = 1;
    if (mode == kModeFused) {
        const SegPlan sp = seg_plan(g);
        prm.seg_tiles = sp.seg_tiles;
        prm.n_seg = sp.n_seg;
        prm.n_items = g.B * g.H * sp.n_seg;
        if (sp.n_seg > 1) {
            const size_t off = (sp.state_bytes + 255) / 256 * 256;
            if (!scratch || scratch_bytes < off + sp.count_bytes)
                return cudaErrorInvalidValue;
            prm.seg_state = static_cast<float *>(scratch);
            prm.seg_count = reinterpret_cast<unsigned int *>(static_cast<char *>(scratch) + off);
            cudaError_t e = cudaMemsetAsync(prm.seg_count, 0, sp.count_bytes, st);
            if (e != cudaSuccess)
                return e;
        }
    }
    prm.status = device_status_word();
    if (!prm.status)
        return cudaErrorUnknown;
    CUtensorMap tx, tb, tcm;
    if (!make_tmap_tokens_heads(&tx, x, g) || !make_tmap_tokens_groups(&tb, Bm, g) ||
        !make_tmap_tokens_groups(&tcm, Cm, g))
        return cudaErrorInvalidValue;
    return mode == kModeOut ? dispatch<kModeOut>(tx, tb, tcm, prm, st)
                            : dispatch<kModeFused>(tx, tb, tcm, prm, st);
}

}  // namespace

bool chunk_tc_supported(const Geom &g)
{
    const bool shape = g.P == 64 && (g.S == 64 || g.S == 128 || g.S == 256);
    return shape && g.T % kTile == 0 && g.L > 0 && g.L < (1LL << 31) && g.H <= 65535 &&
           g.G <= 65535 && g.B <= 65535;
}

cudaError_t launch_chunk_out_tc(const void *x, const void *Bm, const void *Cm, const float *dtT,
                                const float *Gc, const float *states, const float *D, void *y,
                                const Geom &g, cudaStream_t st)
{
    return run(kModeOut, x, Bm, Cm, dtT, Gc, D, states, nullptr, nullptr, y, g, nullptr, 0, st);
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
