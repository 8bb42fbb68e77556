// Chunk gradients of the backward pass on tensor cores (bf16, headdim 64,
// dstate 64 or 128, 128-token chunks).
//
// The chunked adjoint of the forward of "Accelerating Mamba-2 forward-pass
// kernels with CUDA Tile (cuTile)" (sections "Kernel 2" and "Kernel 3"; the
// pages name the backward pass without giving it).  Per (batch, chunk, head),
// with W_ij = exp2(G_i - G_j) for j <= i < n (else 0), e_T(j) = exp2(G_last -
// G_j), e(i) = exp2(G_i), h_in the chunk's start state and dS the gradient of
// its end state:
//
//   phase A (tcgen05):  dyx  = dY X^T      CB   = C B^T
//                       Chin = C h_in^T    BdS  = B dS^T
//   compute:            Q1   = W * CB                         (bf16, [i][j])
//                       Q2   = W * dyx * dt_j                 (bf16, [i][j])
//                       Xs   = dt e_T X,   Ys = e dY          (bf16 row scalings)
//   phase B (tcgen05):  dX1  = Q1^T dY
//                       dB   = Q2^T C + Xs dS                 (the group's dB share)
//                       dC   = Q2 B   + Ys h_in               (the group's dC share)
//   epilogue:           dx_j = D dy_j + dt_j (dX1_j + e_T(j) BdS_j)
//                       ddt_j = x_j . dX1_j + e_T(j) x_j . BdS_j + A da_j
//   with the decay gradient dL_i = sum_j Q1_ij dyx_ij dt_j - dt_i x_i . dX1_i
//                                  + e(i) dy_i . Chin_i - R_i,
//        R_j = e_T(j) dt_j x_j . BdS_j,  dL_last += sum_j R_j + exp2(G_last) (dS . h_in),
//        da = suffix sums of dL,  dA += sum dt da,  dD += sum dy . x.
//
// Every operand is a bf16 tile in shared memory in the 128-byte-swizzled
// layout (x, dy, B, C by TMA; h_in, dS, Q1, Q2, Xs, Ys written by the compute
// warps), so each contraction is one tcgen05.mma chain with f32 accumulators
// in TMEM: dyx cols [0,128), CB [128,256), Chin [256,320), BdS [384,448); in
// phase B dX1 [0,64), dB [128,128+S), dC [256,256+S).  h_in, dS, Xs and Ys
// enter the contractions as bf16 hi + lo pairs (h_in, dS in phase A; all four
// in a second phase-B step that adds Xs dS_lo + Xs_lo dS to dB and Ys h_lo +
// Ys_lo h_in to dC, once the lo tiles are over Q1 / Q2): with single bf16
// roundings the state terms cancel badly at long sequences (dC 6e-2 of its
// rms beyond 2^-5 of each element at 4000 tokens; 1e-3 with the split).
// The lo halves of h_in and dS wait in TMEM [448, 448 + S/2) between the
// two uses.  dB and dC are summed
// over the heads of a group in f32 by TMA bulk reductions (the rows staged in
// shared memory as swizzled [128 x 32] f32 boxes); dx goes out through a
// TMA store.  Roles: warps 0-3 compute (thread i = row / TMEM lane i), one
// thread of warp 4 issues TMA and MMA.  Every wait is bounded; a timeout sets
// the status word and the CTA leaves after freeing TMEM.
#include <type_traits>

#include "common.cuh"
#include "ssd_internal.h"
#include "tc05.cuh"

namespace ssd {
namespace {
using namespace tc;

constexpr int kT = 128;
constexpr int kThreads = 160;
constexpr uint32_t kRegion = 128 * 128;  // 128 rows x 128 bytes

template <int S>
struct BtLayout {
    static constexpr uint32_t kSR = S / 64;                   // 64-wide dstate regions
    static constexpr uint32_t kStateRegion = 64 * 128;        // 64 rows (p) x 128 bytes
    static constexpr uint32_t off_x = 0;                      // x [t][p] (then dx staging)
    static constexpr uint32_t off_dy = off_x + kRegion;       // dy [t][p]
    static constexpr uint32_t off_b = off_dy + kRegion;       // B [t][s], kSR regions
    static constexpr uint32_t off_c = off_b + kSR * kRegion;  // C [t][s]
    static constexpr uint32_t off_hin = off_c + kSR * kRegion;       // h_in [p][s] bf16
    static constexpr uint32_t off_ds = off_hin + kSR * kStateRegion;  // dS [p][s] bf16
    static constexpr uint32_t off_q1 = off_ds + kSR * kStateRegion;   // Q1 [i][j], 2 regions
    static constexpr uint32_t off_q2 = off_q1 + 2 * kRegion;          // Q2 [i][j], 2 regions
    static constexpr uint32_t off_xs = off_q2 + 2 * kRegion;          // h_in lo (phase A), then Xs [t][p]
    static constexpr uint32_t off_ys = off_xs + kRegion;              // dS lo (phase A), then Ys [t][p]
    static constexpr uint32_t off_vec = off_ys + kRegion;             // g, dt, dl: 3 x 128 f32
    static constexpr uint32_t bytes = off_vec + 3 * 128 * 4;
    static_assert(bytes + 1024 + 256 <= 232448, "shared memory budget");
    static constexpr uint32_t t_dyx = 0, t_cb = 128, t_chin = 256, t_bds = 384;
    static constexpr uint32_t t_dx = 0, t_db = 128, t_dc = 256;
    // the lo halves of h_in and dS (bf16 pairs), kept from the conversion
    // at the item's start until the second phase-B step
    static constexpr uint32_t t_lo = 448;
    static_assert(t_lo + S / 2 <= 512, "TMEM budget");
};

struct BtParams {
    const float *Gc, *dtT, *A, *D, *states, *dstates;
    float *ddt, *dA, *dD, *dBacc, *dCacc;
    Geom g;
    unsigned int *status;
};

// Named barrier 1 over the four compute warps.  The non-aligned form counts
// threads, so lanes may arrive while their warp is diverged (after a
// lane-0-only block); the aligned bar.sync would be undefined there.
__device__ __forceinline__ void compute_sync() { asm volatile("barrier.sync 1, 128;" ::: "memory"); }

// TMA reduce-add of a [128 rows][32 f32] swizzled shared-memory box into
// global f32 (rows past the tensor's end are not touched).
__device__ __forceinline__ void tma4_reduce_add(const void *tmap, const void *src, int c0, int c1,
                                                int c2, int c3)
{
    asm volatile("cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.bulk_group"
                 " [%0, {%2, %3, %4, %5}], [%1];" ::"l"(tmap),
                 "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

// L2 prefetch of one TMA tile (no shared memory written, no barrier)
__device__ __forceinline__ void tma4_prefetch_l2(const void *tmap, int c0, int c1, int c2, int c3)
{
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(tmap),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

// A work item: chunk c of (batch b, head h); items run heads fastest, so the
// CTAs working at the same time share their chunk's B / C tiles through L2.
struct BtItem {
    int64_t b, h, bh, grp, tau;
    int c, n;
};

__device__ __forceinline__ BtItem bt_item(const Geom &g, int u)
{
    BtItem w;
    w.h = u % g.H;
    const int64_t bc = u / g.H;
    w.c = (int)(bc % g.nc);
    w.b = bc / g.nc;
    w.bh = w.b * g.H + w.h;
    w.grp = w.h / g.hpg;
    w.tau = (int64_t)w.c * kT;
    w.n = (int)min64(kT, g.L - w.tau);
    return w;
}

// Persistent: one CTA per SM walks the items blockIdx.x, + gridDim.x, ...
// Every barrier completes once per item (phase = item count & 1).  The
// issuing thread also sends each item's staged dx, dB and dC rows out (TMA
// store and bulk reductions), so the compute warps go on to the next item
// while those copies read shared memory; once they have, it brings the next
// item's chunk states (f32, contiguous) into the Q1 / Q2 regions with bulk
// copies and its x, dy, B, C tiles by TMA.  The item after that is
// prefetched into L2 meanwhile.
template <int S>
__global__ void __launch_bounds__(kThreads, 1)
bwd_chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
                    const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_c,
                    const __grid_constant__ CUtensorMap tm_dx, const __grid_constant__ CUtensorMap tm_db,
                    const __grid_constant__ CUtensorMap tm_dc, BtParams prm)
{
    using Lay = BtLayout<S>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_in, bar_sld, bar_st, bar_a, bar_q, bar_b1, bar_q2, bar_b, bar_stg, bar_end;
    __shared__ uint32_t tmem_slot;
    __shared__ float red[4][4];
    __shared__ int s_fail;

    const Geom &g = prm.g;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_items = (int)(g.B * g.nc * g.H);

    if (tid == 0) {
        mbar_init(&bar_in, 1);
        mbar_init(&bar_st, 4);
        mbar_init(&bar_a, 1);
        mbar_init(&bar_q, 4);
        mbar_init(&bar_b1, 1);
        mbar_init(&bar_q2, 4);
        mbar_init(&bar_b, 1);
        mbar_init(&bar_sld, 1);
        mbar_init(&bar_stg, 4);
        mbar_init(&bar_end, 1);
        fence_barrier_init();
        s_fail = 0;
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    float *sg = reinterpret_cast<float *>(smem + Lay::off_vec);
    float *sdt = sg + 128, *sdl = sdt + 128;
    const int64_t state_floats = 64 * S;  // one chunk's [P][S] state
    const uint32_t state_bytes = (uint32_t)(state_floats * 4);
    static_assert(64 * S * 4 <= 2 * kRegion, "an f32 chunk state fits the Q1 (or Q2) region");

    if (warp == 4) {
        if (lane == 0) {
            // ---------------- TMA loads, then the two MMA phases, per item
            prefetch_tmap(&tm_x);
            prefetch_tmap(&tm_dy);
            prefetch_tmap(&tm_b);
            prefetch_tmap(&tm_c);
            const uint32_t base = smem_u32(smem);
            const uint32_t id_tt = idesc_bf16(128, 128, false, false);
            const uint32_t id_tp = idesc_bf16(128, 64, false, false);
            const uint32_t id_dx = idesc_bf16(128, 64, true, true);
            const uint32_t id_ms = idesc_bf16(128, S, true, true);
            const uint32_t id_ks = idesc_bf16(128, S, false, true);
            const uint64_t d_dy = desc_k0(base + Lay::off_dy), d_x = desc_k0(base + Lay::off_x);
            const uint64_t d_c = desc_k0(base + Lay::off_c), d_b = desc_k0(base + Lay::off_b);
            const uint64_t d_hk = desc_k0(base + Lay::off_hin), d_sk = desc_k0(base + Lay::off_ds);
            const uint64_t d_q1 = desc_mn0(base + Lay::off_q1, kRegion);
            const uint64_t d_q2m = desc_mn0(base + Lay::off_q2, kRegion);
            const uint64_t d_dym = desc_mn0(base + Lay::off_dy, kRegion);
            const uint64_t d_cm = desc_mn0(base + Lay::off_c, kRegion);
            const uint64_t d_bm = desc_mn0(base + Lay::off_b, kRegion);
            const uint64_t d_dsm = desc_mn0(base + Lay::off_ds, Lay::kStateRegion);
            const uint64_t d_hm = desc_mn0(base + Lay::off_hin, Lay::kStateRegion);
            const uint64_t d_xs = desc_k0(base + Lay::off_xs), d_ys = desc_k0(base + Lay::off_ys);
            const uint64_t d_q2k = desc_k0(base + Lay::off_q2);
            // the lo halves: of h_in and dS over Xs / Ys for phase A, over Q1
            // for phase B; of Xs and Ys over Q2
            const uint64_t d_hlo_a = desc_k0(base + Lay::off_xs), d_slo_a = desc_k0(base + Lay::off_ys);
            const uint64_t d_hlo_b = desc_mn0(base + Lay::off_q1, Lay::kStateRegion);
            const uint64_t d_slo_b = desc_mn0(base + Lay::off_q1 + Lay::kSR * Lay::kStateRegion, Lay::kStateRegion);
            const uint64_t d_xslo = desc_k0(base + Lay::off_q2), d_yslo = desc_k0(base + Lay::off_q2 + kRegion);
            // an item's staged rows out: dB (over Q1) and dC (over B / C) added
            // into the f32 accumulators, dx (over x) stored; rows past the
            // sequence end are clipped by the tensor maps
            auto send_out = [&](const BtItem &w) {
                for (int r = 0; r < S / 32; ++r) {
                    tma4_reduce_add(&tm_db, smem + Lay::off_q1 + r * kRegion, 32 * r, (int)w.grp, (int)w.tau,
                                    (int)w.b);
                    tma4_reduce_add(&tm_dc, smem + Lay::off_b + r * kRegion, 32 * r, (int)w.grp, (int)w.tau,
                                    (int)w.b);
                }
                tma4_store(&tm_dx, smem + Lay::off_x, 0, (int)w.h, (int)w.tau, (int)w.b);
                bulk_commit();
            };
            prefetch_tmap(&tm_dx);
            bool ok = true;
            uint32_t k = 0;
            BtItem prev{};
            for (int u = blockIdx.x; u < n_items && ok; u += gridDim.x, ++k) {
                const uint32_t par = k & 1u;
                const BtItem w = bt_item(g, u);
                if (k > 0) {
                    // the previous item's rows are staged: out they go, and
                    // once read, their boxes take this item's loads
                    if (!mbar_wait(&bar_stg, par ^ 1u)) {
                        ok = false;
                        break;
                    }
                    send_out(prev);
                    bulk_wait_read();
                }
                const int64_t so = (w.bh * g.nc + w.c) * state_floats;
                mbar_arrive_expect_tx(&bar_sld, 2 * state_bytes);
                bulk_load(smem + Lay::off_q1, prm.states + so, state_bytes, &bar_sld);
                bulk_load(smem + Lay::off_q2, prm.dstates + so, state_bytes, &bar_sld);
                mbar_arrive_expect_tx(&bar_in, (2 + 2 * Lay::kSR) * kRegion);
                tma4(smem + Lay::off_x, &tm_x, &bar_in, 0, (int)w.h, (int)w.tau, (int)w.b);
                tma4(smem + Lay::off_dy, &tm_dy, &bar_in, 0, (int)w.h, (int)w.tau, (int)w.b);
                for (uint32_t r = 0; r < Lay::kSR; ++r) {
                    tma4(smem + Lay::off_b + r * kRegion, &tm_b, &bar_in, (int)(r * 64), (int)w.grp,
                         (int)w.tau, (int)w.b);
                    tma4(smem + Lay::off_c + r * kRegion, &tm_c, &bar_in, (int)(r * 64), (int)w.grp,
                         (int)w.tau, (int)w.b);
                }
                // the next item's tiles and chunk states into L2
                if (u + (int)gridDim.x < n_items) {
                    const BtItem nx = bt_item(g, u + (int)gridDim.x);
                    tma4_prefetch_l2(&tm_x, 0, (int)nx.h, (int)nx.tau, (int)nx.b);
                    tma4_prefetch_l2(&tm_dy, 0, (int)nx.h, (int)nx.tau, (int)nx.b);
                    for (uint32_t r = 0; r < Lay::kSR; ++r) {
                        tma4_prefetch_l2(&tm_b, (int)(r * 64), (int)nx.grp, (int)nx.tau, (int)nx.b);
                        tma4_prefetch_l2(&tm_c, (int)(r * 64), (int)nx.grp, (int)nx.tau, (int)nx.b);
                    }
                    const int64_t sn = (nx.bh * g.nc + nx.c) * state_floats;
                    bulk_prefetch_l2(prm.states + sn, state_bytes);
                    bulk_prefetch_l2(prm.dstates + sn, state_bytes);
                }
                if (!mbar_wait(&bar_in, par)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // dyx = dY X^T: M i, N j, K p (one region)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(tmem + Lay::t_dyx, desc_k(d_dy, kRegion, ks), desc_k(d_x, kRegion, ks), id_tt, ks > 0);
                // CB = C B^T: K = s over the dstate regions
#pragma unroll
                for (int ks = 0; ks < S / 16; ++ks)
                    mma_ss(tmem + Lay::t_cb, desc_k(d_c, kRegion, ks), desc_k(d_b, kRegion, ks), id_tt, ks > 0);
                if (!mbar_wait(&bar_st, par)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // Chin = C h_in^T and BdS = B dS^T: N = p (64 rows of the state
                // tiles), K = s; h_in and dS as hi + lo (the lo halves over the
                // Xs / Ys regions until the compute warps build Xs and Ys)
#pragma unroll
                for (int ks = 0; ks < S / 16; ++ks) {
                    mma_ss(tmem + Lay::t_chin, desc_k(d_c, kRegion, ks), desc_k(d_hk, Lay::kStateRegion, ks),
                           id_tp, ks > 0);
                    mma_ss(tmem + Lay::t_bds, desc_k(d_b, kRegion, ks), desc_k(d_sk, Lay::kStateRegion, ks),
                           id_tp, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < S / 16; ++ks) {
                    mma_ss(tmem + Lay::t_chin, desc_k(d_c, kRegion, ks), desc_k(d_hlo_a, Lay::kStateRegion, ks),
                           id_tp, 1u);
                    mma_ss(tmem + Lay::t_bds, desc_k(d_b, kRegion, ks), desc_k(d_slo_a, Lay::kStateRegion, ks),
                           id_tp, 1u);
                }
                mma_commit(&bar_a);
                if (!mbar_wait(&bar_q, par)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // dX1 = Q1^T dY: A = Q1 viewed M (j) -major, B = dY viewed N (p) -major, K = i
#pragma unroll
                for (int ks = 0; ks < kT / 16; ++ks)
                    mma_ss(tmem + Lay::t_dx, desc_mn(d_q1, ks), desc_mn(d_dym, ks), id_dx, ks > 0);
                // dB = Q2^T C + Xs dS
#pragma unroll
                for (int ks = 0; ks < kT / 16; ++ks)
                    mma_ss(tmem + Lay::t_db, desc_mn(d_q2m, ks), desc_mn(d_cm, ks), id_ms, ks > 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(tmem + Lay::t_db, desc_k(d_xs, kRegion, ks), desc_mn(d_dsm, ks), id_ks, 1u);
                // dC = Q2 B + Ys h_in
#pragma unroll
                for (int ks = 0; ks < kT / 16; ++ks)
                    mma_ss(tmem + Lay::t_dc, desc_k(d_q2k, kRegion, ks), desc_mn(d_bm, ks), id_ks, ks > 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(tmem + Lay::t_dc, desc_k(d_ys, kRegion, ks), desc_mn(d_hm, ks), id_ks, 1u);
                mma_commit(&bar_b1);
                // the state terms' lo parts, once the compute warps have put
                // h_in lo, dS lo (over Q1) and Xs lo, Ys lo (over Q2) in place:
                // dB += Xs dS_lo + Xs_lo dS, dC += Ys h_lo + Ys_lo h_in
                if (!mbar_wait(&bar_q2, par)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    mma_ss(tmem + Lay::t_db, desc_k(d_xs, kRegion, ks), desc_mn(d_slo_b, ks), id_ks, 1u);
                    mma_ss(tmem + Lay::t_db, desc_k(d_xslo, kRegion, ks), desc_mn(d_dsm, ks), id_ks, 1u);
                    mma_ss(tmem + Lay::t_dc, desc_k(d_ys, kRegion, ks), desc_mn(d_hlo_b, ks), id_ks, 1u);
                    mma_ss(tmem + Lay::t_dc, desc_k(d_yslo, kRegion, ks), desc_mn(d_hm, ks), id_ks, 1u);
                }
                mma_commit(&bar_b);
                prev = w;
            }
            // the last item's rows
            if (ok && k > 0) {
                if (mbar_wait(&bar_stg, (k - 1) & 1u))
                    send_out(prev);
                else
                    ok = false;
            }
            bulk_wait_all();
            if (!ok)
                atomicOr(prm.status, 1u);
            // every MMA this thread issued has completed before TMEM is freed
            mma_commit(&bar_end);
            if (!mbar_wait(&bar_end, 0))
                atomicOr(prm.status, 1u);
        }
    } else {
        // ---------------- compute: thread i owns row / TMEM lane i
        const int i = tid;
        const uint32_t tl = tmem_at(tmem, (uint32_t)(warp * 32), 0);
        uint32_t k = 0;
        for (int u = blockIdx.x; u < n_items; u += gridDim.x, ++k) {
            const uint32_t par = k & 1u;
            const BtItem w = bt_item(g, u);
            const int64_t b = w.b, h = w.h, bh = w.bh, tau = w.tau;
            const int n = w.n;
            const bool valid = i < n;
            const float *grow = prm.Gc + bh * g.L + tau;
            sg[i] = valid ? grow[i] : 0.f;
            sdt[i] = valid ? prm.dtT[bh * g.L + tau + i] : 0.f;
            // h_in and dS: f32 [P][S], brought into the Q1 / Q2 regions by the
            // issuing thread's bulk copies -> bf16 hi + lo [p][s], swizzled rows
            // of 64 s: hi into the h_in / dS tiles, lo over the Xs / Ys regions
            // (for phase A) and into TMEM (for the second phase-B step), as
            // the contractions with the states cancel strongly at long
            // sequences and a single bf16 rounding of the state showed there.
            // Warp w takes rows p = w, w + 4, ...; lane l four consecutive s.
            constexpr int kLanesPerRow = S / 4;           // 32 (S 128) or 16 (S 64)
            constexpr int kRowsPerPass = 32 / kLanesPerRow;
            constexpr int kIters = 64 / (4 * kRowsPerPass);  // rows per lane: 16 or 8
            const int st_sub = lane % kLanesPerRow, st_rsub = lane / kLanesPerRow;
            const int st_s = 4 * st_sub;
            const uint32_t st_reg = (uint32_t)(st_s / 64), st_col = (uint32_t)(st_s % 64);
            auto st_off = [&](int r, int &p) {
                p = warp * kRowsPerPass + st_rsub + r * 4 * kRowsPerPass;
                return st_reg * Lay::kStateRegion + sw128_offset((uint32_t)p, st_col / 8) + (st_col % 8) * 2;
            };
            float dshin = 0.f;
            bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_sld, par));
            if (ok) {
                const float *hin_s = reinterpret_cast<const float *>(smem + Lay::off_q1);
                const float *ds_s = reinterpret_cast<const float *>(smem + Lay::off_q2);
#pragma unroll 1
                for (int r0 = 0; r0 < kIters; r0 += 4) {
                    uint32_t lw[16];  // lo words of four rows: h (2), dS (2) each
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        int p;
                        const uint32_t off = st_off(r0 + q, p);
                        const float4 hv = *reinterpret_cast<const float4 *>(hin_s + p * S + st_s);
                        const float4 dv = *reinterpret_cast<const float4 *>(ds_s + p * S + st_s);
                        dshin += hv.x * dv.x + hv.y * dv.y + hv.z * dv.z + hv.w * dv.w;
                        const uint32_t h0 = pack_bf16x2(hv.x, hv.y), h1 = pack_bf16x2(hv.z, hv.w);
                        const uint32_t d0 = pack_bf16x2(dv.x, dv.y), d1 = pack_bf16x2(dv.z, dv.w);
                        lw[4 * q] = pack_bf16x2(hv.x - bf_lo(h0), hv.y - bf_hi(h0));
                        lw[4 * q + 1] = pack_bf16x2(hv.z - bf_lo(h1), hv.w - bf_hi(h1));
                        lw[4 * q + 2] = pack_bf16x2(dv.x - bf_lo(d0), dv.y - bf_hi(d0));
                        lw[4 * q + 3] = pack_bf16x2(dv.z - bf_lo(d1), dv.w - bf_hi(d1));
                        *reinterpret_cast<uint2 *>(smem + Lay::off_hin + off) = make_uint2(h0, h1);
                        *reinterpret_cast<uint2 *>(smem + Lay::off_ds + off) = make_uint2(d0, d1);
                        *reinterpret_cast<uint2 *>(smem + Lay::off_xs + off) = make_uint2(lw[4 * q], lw[4 * q + 1]);
                        *reinterpret_cast<uint2 *>(smem + Lay::off_ys + off) =
                            make_uint2(lw[4 * q + 2], lw[4 * q + 3]);
                    }
                    tmem_st16(tl + Lay::t_lo + 4 * r0, lw);
                }
                tmem_st_wait();
            }
            fence_proxy_async_smem();
            warp_arrive(&bar_st);
            compute_sync();  // G and dt of every row are visible
            const float glast = sg[n - 1];
            const float gi = sg[i], dti = sdt[i];
            const float eT = valid ? exp2f(glast - gi) : 0.f, ei = valid ? exp2f(gi) : 0.f;
            // Score weights exp2(g_i - g_j) = r_i c_j with a reference g_m in the
            // middle of the chunk's range, while that range stays within 200
            // (both factors within 2^100): c_j goes to shared memory (over dl),
            // and the Q loop needs no exponent.  Wider ranges take exp2 per
            // element.
            const float g0 = sg[0];
            const bool fact = fabsf(g0 - glast) <= 200.f;  // the same for the whole CTA
            const float gm = 0.5f * (g0 + glast);
            const float ri = (fact && valid) ? exp2f(gi - gm) : 0.f;
            if (fact) {
                const float cj = valid ? exp2f(gm - gi) : 0.f;
                sdl[i] = cj;
            }
            compute_sync();  // the column factors are visible

            // ok is made warp-uniform: the TMEM loads below are warp-collective
            ok = __all_sync(0xffffffffu, ok && mbar_wait(&bar_in, par) && mbar_wait(&bar_a, par));
            float rowq = 0.f, yst = 0.f, xb = 0.f, dyx_ii = 0.f;
            if (ok) {
                tc_fence_after();
                const uint8_t *sxr = smem + Lay::off_x, *sdyr = smem + Lay::off_dy;
                // e(i) dy_i . Chin_i and x_i . BdS_i; Xs and Ys rows
#pragma unroll
                for (int c2 = 0; c2 < 4; ++c2) {
                    uint32_t ch[16], bd[16];
                    tmem_ld16(tl + Lay::t_chin + 16 * c2, ch);
                    tmem_ld16(tl + Lay::t_bds + 16 * c2, bd);
                    tmem_ld_wait();
                    uint32_t xs_pk[8], ys_pk[8];
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const uint32_t off = sw128_offset((uint32_t)i, (uint32_t)(2 * c2 + cc));
                        const uint4 xv = *reinterpret_cast<const uint4 *>(sxr + off);
                        const uint4 dv = *reinterpret_cast<const uint4 *>(sdyr + off);
                        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            const int o = 8 * cc + 2 * e2;
                            const float x0 = bf_lo(xw[e2]), x1 = bf_hi(xw[e2]);
                            const float d0 = bf_lo(dw[e2]), d1 = bf_hi(dw[e2]);
                            yst = fmaf(d0, __uint_as_float(ch[o]), fmaf(d1, __uint_as_float(ch[o + 1]), yst));
                            xb = fmaf(x0, __uint_as_float(bd[o]), fmaf(x1, __uint_as_float(bd[o + 1]), xb));
                            xs_pk[4 * cc + e2] = pack_bf16x2(dti * eT * x0, dti * eT * x1);
                            ys_pk[4 * cc + e2] = pack_bf16x2(ei * d0, ei * d1);
                        }
                    }
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const uint32_t off = sw128_offset((uint32_t)i, (uint32_t)(2 * c2 + cc));
                        *reinterpret_cast<uint4 *>(smem + Lay::off_xs + off) =
                            make_uint4(xs_pk[4 * cc], xs_pk[4 * cc + 1], xs_pk[4 * cc + 2], xs_pk[4 * cc + 3]);
                        *reinterpret_cast<uint4 *>(smem + Lay::off_ys + off) =
                            make_uint4(ys_pk[4 * cc], ys_pk[4 * cc + 1], ys_pk[4 * cc + 2], ys_pk[4 * cc + 3]);
                    }
                }
                // Q1 = W * CB and Q2 = W * dyx * dt_j, row i, 16 keys at a time
                // one loop per weight form (the CTA-uniform branch stays out of
                // the unrolled body)
                auto q_block = [&](auto fact_c, int j0, uint32_t (&q1)[8], uint32_t (&q2)[8]) {
                    constexpr bool kFact = decltype(fact_c)::value;
                    uint32_t cb[16], dx[16];
                    tmem_ld16(tl + Lay::t_cb + j0, cb);
                    tmem_ld16(tl + Lay::t_dyx + j0, dx);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float a[2], bq[2], dxt[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int j = j0 + 2 * e + u;
                            const float cbv = __uint_as_float(cb[2 * e + u]);
                            const float dyxv = __uint_as_float(dx[2 * e + u]);
                            float w;
                            if (kFact)
                                w = (valid && j <= i) ? ri * sdl[j] : 0.f;
                            else
                                w = (valid && j <= i) ? exp2f(gi - sg[j]) : 0.f;
                            a[u] = w * cbv;              // Q1 = W CB
                            dxt[u] = dyxv * sdt[j];
                            bq[u] = w * dxt[u];          // Q2 = W dyx dt_j
                            if (j == i)
                                dyx_ii = dyxv;
                        }
                        q1[e] = pack_bf16x2(a[0], a[1]);
                        q2[e] = pack_bf16x2(bq[0], bq[1]);
                        // the row sum of Q1 dyx dt from the bf16 Q1 that dX1 (and
                        // with it the column sums x . dX1) is formed from: the two
                        // enter dL with opposite signs and their chunk totals are
                        // equal, so they must carry the same rounding
                        rowq = fmaf(bf_lo(q1[e]), dxt[0], fmaf(bf_hi(q1[e]), dxt[1], rowq));
                    }
                };
#pragma unroll 1
                for (int j0 = 0; j0 < kT; j0 += 16) {
                    // keys past every row of this warp: zero weights, nothing to load
                    const bool none = j0 > warp * 32 + 31;  // warp-uniform
                    uint32_t q1[8], q2[8];
                    if (none) {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            q1[e] = q2[e] = 0u;
                    } else if (fact) {
                        q_block(std::true_type{}, j0, q1, q2);
                    } else {
                        q_block(std::false_type{}, j0, q1, q2);
                    }
                    const int reg = j0 / 64, ch0 = (j0 % 64) / 8;
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const uint32_t off = reg * kRegion + sw128_offset((uint32_t)i, (uint32_t)(ch0 + cc));
                        *reinterpret_cast<uint4 *>(smem + Lay::off_q1 + off) =
                            make_uint4(q1[4 * cc], q1[4 * cc + 1], q1[4 * cc + 2], q1[4 * cc + 3]);
                        *reinterpret_cast<uint4 *>(smem + Lay::off_q2 + off) =
                            make_uint4(q2[4 * cc], q2[4 * cc + 1], q2[4 * cc + 2], q2[4 * cc + 3]);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(&bar_q);

            // ---------------- the lo halves for the second phase-B step, over
            // Q1 (h_in lo, dS lo) and Q2 (Xs lo, Ys lo).  They are read from
            // TMEM and formed in registers while phase B runs, and stored once
            // phase B has read Q1 and Q2.
            {
                constexpr int kLoWords = kIters * 4;  // 64 (S 128) or 32 (S 64)
                uint32_t lw[kLoWords];
#pragma unroll
                for (int c16 = 0; c16 < kLoWords; c16 += 16)
                    tmem_ld16(tl + Lay::t_lo + c16, *reinterpret_cast<uint32_t(*)[16]>(lw + c16));
                uint32_t xl[32], yl[32];
                {
                    const uint8_t *sxr = smem + Lay::off_x, *sdyr = smem + Lay::off_dy;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint32_t off = sw128_offset((uint32_t)i, (uint32_t)ch);
                        const uint4 xv = *reinterpret_cast<const uint4 *>(sxr + off);
                        const uint4 dv = *reinterpret_cast<const uint4 *>(sdyr + off);
                        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            const float a0 = dti * eT * bf_lo(xw[e2]), a1 = dti * eT * bf_hi(xw[e2]);
                            const float b0 = ei * bf_lo(dw[e2]), b1 = ei * bf_hi(dw[e2]);
                            const uint32_t ah = pack_bf16x2(a0, a1), bh = pack_bf16x2(b0, b1);
                            xl[4 * ch + e2] = pack_bf16x2(a0 - bf_lo(ah), a1 - bf_hi(ah));
                            yl[4 * ch + e2] = pack_bf16x2(b0 - bf_lo(bh), b1 - bf_hi(bh));
                        }
                    }
                }
                tmem_ld_wait();
                ok = __all_sync(0xffffffffu, ok && mbar_wait(&bar_b1, par));
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int r = 0; r < kIters; ++r) {
                        int p;
                        const uint32_t off = st_off(r, p);
                        *reinterpret_cast<uint2 *>(smem + Lay::off_q1 + off) = make_uint2(lw[4 * r], lw[4 * r + 1]);
                        *reinterpret_cast<uint2 *>(smem + Lay::off_q1 + Lay::kSR * Lay::kStateRegion + off) =
                            make_uint2(lw[4 * r + 2], lw[4 * r + 3]);
                    }
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint32_t off = sw128_offset((uint32_t)i, (uint32_t)ch);
                        *reinterpret_cast<uint4 *>(smem + Lay::off_q2 + off) =
                            make_uint4(xl[4 * ch], xl[4 * ch + 1], xl[4 * ch + 2], xl[4 * ch + 3]);
                        *reinterpret_cast<uint4 *>(smem + Lay::off_q2 + kRegion + off) =
                            make_uint4(yl[4 * ch], yl[4 * ch + 1], yl[4 * ch + 2], yl[4 * ch + 3]);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(&bar_q2);

            // ---------------- epilogue.  dx first: its inputs (dX1, BdS, x, dy)
            // are complete after phase B's first step, so it runs while the
            // second step is in flight, and its rows go over the x tile (each
            // thread reads its row of x before writing dx there; no MMA reads
            // x any more)
            float colq = 0.f, ddt_direct = 0.f, rj = 0.f;
            if (ok) {
                const float Dh = prm.D[h];
                const uint8_t *sxr = smem + Lay::off_x, *sdyr = smem + Lay::off_dy;
                uint8_t *stage = smem + Lay::off_x;
#pragma unroll
                for (int c2 = 0; c2 < 4; ++c2) {
                    uint32_t d1[16], bd[16];
                    tmem_ld16(tl + Lay::t_dx + 16 * c2, d1);
                    tmem_ld16(tl + Lay::t_bds + 16 * c2, bd);
                    tmem_ld_wait();
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const uint32_t off = sw128_offset((uint32_t)i, (uint32_t)(2 * c2 + cc));
                        const uint4 xv = *reinterpret_cast<const uint4 *>(sxr + off);
                        const uint4 dv = *reinterpret_cast<const uint4 *>(sdyr + off);
                        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
                        uint32_t o4[4];
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            const int o = 8 * cc + 2 * e2;
                            const float x0 = bf_lo(xw[e2]), x1 = bf_hi(xw[e2]);
                            const float a0 = __uint_as_float(d1[o]), a1 = __uint_as_float(d1[o + 1]);
                            colq = fmaf(x0, a0, fmaf(x1, a1, colq));
                            const float g0 = a0 + eT * __uint_as_float(bd[o]);
                            const float g1 = a1 + eT * __uint_as_float(bd[o + 1]);
                            o4[e2] = pack_bf16x2(Dh * bf_lo(dw[e2]) + dti * g0, Dh * bf_hi(dw[e2]) + dti * g1);
                        }
                        *reinterpret_cast<uint4 *>(stage + off) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
                    }
                }
                ddt_direct = colq + eT * xb;
                rj = eT * dti * xb;
            }
            ok = __all_sync(0xffffffffu, ok && mbar_wait(&bar_b, par));
            if (ok) {
                tc_fence_after();
                // dB and dC rows of this chunk's tokens, added into the f32
                // accumulators by TMA reductions: each row goes to shared memory in
                // [128 rows][32 f32] swizzled boxes (dB over Q1 / Q2, dC over B / C:
                // phase B has read them all), then one thread issues the bulk adds.
                // The TMEM loads are warp-collective, so every lane runs them; rows
                // past the sequence end are clipped by the tensor map.
                {
                    uint8_t *stg_db = smem + Lay::off_q1, *stg_dc = smem + Lay::off_b;
#pragma unroll
                    for (int s0 = 0; s0 < S; s0 += 16) {
                        uint32_t vb[16], vc[16];
                        tmem_ld16(tl + Lay::t_db + s0, vb);
                        tmem_ld16(tl + Lay::t_dc + s0, vc);
                        tmem_ld_wait();
                        const uint32_t box = (uint32_t)(s0 / 32) * kRegion;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t off = box + sw128_offset((uint32_t)i, (uint32_t)((s0 % 32) / 4 + q));
                            *reinterpret_cast<uint4 *>(stg_db + off) =
                                make_uint4(vb[4 * q], vb[4 * q + 1], vb[4 * q + 2], vb[4 * q + 3]);
                            *reinterpret_cast<uint4 *>(stg_dc + off) =
                                make_uint4(vc[4 * q], vc[4 * q + 1], vc[4 * q + 2], vc[4 * q + 3]);
                        }
                    }
                }
            }
            // this warp's rows of the dx tile and of the dB / dC boxes are in
            // shared memory: the issuing thread sends them out
            fence_proxy_async_smem();
            if (ok)
                warp_arrive(&bar_stg);
            // dL_i (the column part and the end-state part come from the other rows)
            sdl[i] = valid ? rowq - colq * dti + ei * yst - rj : 0.f;
            // CTA sums: R_j, dS . h_in, dy . x
            float v0 = valid ? rj : 0.f, v1 = dshin, v2 = valid ? dyx_ii : 0.f;
            for (int o = 16; o > 0; o >>= 1) {
                v0 += __shfl_xor_sync(0xffffffffu, v0, o);
                v1 += __shfl_xor_sync(0xffffffffu, v1, o);
                v2 += __shfl_xor_sync(0xffffffffu, v2, o);
            }
            if (lane == 0) {
                red[0][warp] = v0;
                red[1][warp] = v1;
                red[2][warp] = v2;
            }
            compute_sync();
            // suffix sums of dL, da_i = sum_{k >= i} dL_k, as a scan over the 128
            // rows (shuffles within a warp, then the later warps' totals); the
            // last valid row also takes the end-state terms
            float da = valid ? sdl[i] : 0.f;
            if (i == n - 1) {
                const float rsum = red[0][0] + red[0][1] + red[0][2] + red[0][3];
                const float dsh = red[1][0] + red[1][1] + red[1][2] + red[1][3];
                da += rsum + exp2f(glast) * dsh;
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_down_sync(0xffffffffu, da, o);
                if (lane + o < 32)
                    da += u;
            }
            const float dd = red[2][0] + red[2][1] + red[2][2] + red[2][3];
            compute_sync();  // every thread has read red[][]
            if (lane == 0)
                red[3][warp] = da;  // warp total (lane 0 holds the whole warp's suffix)
            compute_sync();
            for (int w2 = warp + 1; w2 < 4; ++w2)
                da += red[3][w2];
            // dA gets sum dt_k da_k
            float dasum = valid ? dti * da : 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                dasum += __shfl_xor_sync(0xffffffffu, dasum, o);
            compute_sync();  // every thread has read red[3][]
            if (lane == 0)
                red[0][warp] = dasum;
            compute_sync();
            if (ok && i == 0) {
                atomicAdd(prm.dA + h, red[0][0] + red[0][1] + red[0][2] + red[0][3]);
                atomicAdd(prm.dD + h, dd);
            }
            if (ok && valid)
                prm.ddt[(b * g.L + tau + i) * g.H + h] = ddt_direct + prm.A[h] * da;
            // dx rows out by TMA (rows past the sequence end are not written)
            if (!ok)
                s_fail = 1;
            compute_sync();
            if (s_fail)
                break;  // every compute thread leaves at the same item
        }
        if (s_fail && lane == 0)
            atomicOr(prm.status, 1u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int S>
cudaError_t launch_bt(const CUtensorMap &tx, const CUtensorMap &tdy, const CUtensorMap &tb,
                      const CUtensorMap &tc_, const CUtensorMap &tdx, const CUtensorMap &tdb,
                      const CUtensorMap &tdc, const BtParams &p, cudaStream_t st)
{
    const size_t smem = BtLayout<S>::bytes + 1024;
    auto k = bwd_chunk_tc_kernel<S>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    const int64_t items = p.g.B * p.g.nc * p.g.H;
    const unsigned grid = (unsigned)(items < sms ? items : sms);
    k<<<grid, kThreads, smem, st>>>(tx, tdy, tb, tc_, tdx, tdb, tdc, p);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

bool bwd_tc_supported(const Geom &g)
{
    return g.P == 64 && (g.S == 64 || g.S == 128) && g.T == kT && g.L > 0 && g.nc <= 2147483647LL &&
           g.B * g.H <= 65535 && g.L < (1LL << 31);
}

cudaError_t launch_bwd_chunk_tc(const void *x, const void *Bm, const void *Cm, const void *dy,
                                const float *dtT, const float *Gc, const float *A, const float *D,
                                const float *states, const float *dstates, void *dx, float *ddt,
                                float *dA, float *dD, float *dBacc, float *dCacc, const Geom &g,
                                cudaStream_t st)
{
    if (!bwd_tc_supported(g))
        return cudaErrorNotSupported;
    unsigned int *status = device_status_word();
    if (!status)
        return cudaErrorUnknown;
    CUtensorMap tx, tdy, tb, tc_, tdx, tdb, tdc;
    if (!make_tmap_tokens_heads(&tx, x, g) || !make_tmap_tokens_heads(&tdy, dy, g) ||
        !make_tmap_tokens_groups(&tb, Bm, g) || !make_tmap_tokens_groups(&tc_, Cm, g) ||
        !make_tmap_tokens_heads(&tdx, dx, g) || !make_tmap_f32_tokens_groups(&tdb, dBacc, g) ||
        !make_tmap_f32_tokens_groups(&tdc, dCacc, g))
        return cudaErrorInvalidValue;
    BtParams p{Gc, dtT, A, D, states, dstates, ddt, dA, dD, dBacc, dCacc, g, status};
    if (g.S == 64)
        return launch_bt<64>(tx, tdy, tb, tc_, tdx, tdb, tdc, p, st);
    return launch_bt<128>(tx, tdy, tb, tc_, tdx, tdb, tdc, p, st);
}

}  // namespace ssd
