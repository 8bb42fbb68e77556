// Stage 3 (chunk output) on tensor cores for large state sizes: bf16, headdim
// 64, dstate 384 or 512, 128-token chunks.
//
// "Accelerating Mamba-2 forward-pass kernels with CUDA Tile (cuTile)",
// section "Kernel 3: compute_out", per (batch, chunk, head):
//     Y = exp2(G) * (C h_c^T) + (exp2(G_i - G_j) * (C B^T) * M)(dt * X) + D X.
//
// At dstate 512 the B and C tiles of one chunk are 128 KB each, too large to
// hold with everything else in shared memory, so they are streamed in
// 128-wide dstate blocks through a two-deep TMA ring, and both contractions
// over dstate accumulate block by block in TMEM:
//     CB += C_s B_s^T    (M 128 tokens, N 128 tokens, K 128 per block)
//     Y2 += C_s H_s^T    (M 128, N = P, K 128 per block), H = bf16(h_c)
// then the exact scores CB_ij exp2(g_i - g_j) dt_j (j <= i) go to TMEM as the
// A operand of Y1 = scores X, and the epilogue forms
//     y = Y1 + exp2(g_i) Y2 + D x
// over the consumed x tile, which a TMA store writes out.  The chunk state
// (f32 [P][S], the largest stream) is read by the compute warps with
// coalesced loads and written to shared memory as bf16 H in the MN-major
// layout the MMA takes.
//
// A work item is (batch, chunk, head) with heads fastest, so consecutive
// items share their B / C tiles in L2.  Roles: warps 0-7 compute (thread i
// owns tile row / TMEM lane i; warpgroup w takes half of the columns and of
// the state rows), warp 8 TMA loads, warp 9 MMA issue, warp 10 TMA store of
// y.  Every wait is bounded; a timeout sets the kernel status word and the
// role leaves its loop.
#include "common.cuh"
#include "ssd_internal.h"
#include "tc05.cuh"

namespace ssd {
namespace {
using namespace tc;

constexpr int kTile = 128;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32 + 96;
constexpr uint32_t kRegion = 128 * 128;  // 128 rows of 128 bytes (64 bf16)

template <int S>
struct BigLayout {
    static constexpr int kSB = S / 128;           // 128-wide dstate blocks
    static constexpr uint32_t kSub = 4 * kRegion;  // B (2 regions) and C (2 regions) of a block
    static constexpr uint32_t off_sub = 0;         // two sub-stages
    static constexpr uint32_t off_x = 2 * kSub;    // x (then y) of two items
    static constexpr uint32_t off_h = off_x + 2 * kRegion;  // H [S][P] bf16, MN-major
    static constexpr uint32_t off_g = off_h + S * 128;       // g 128 | dt 128, f32
    static constexpr uint32_t bytes = off_g + 256 * 4;
    // TMEM columns: CB (f32), bf16 scores (two per column), Y1, Y2 (two
    // buffers by item parity: the next item's C H^T may start before this
    // item's epilogue has read its Y2)
    static constexpr uint32_t t_cb = 0, t_sc = 128, t_y1 = 192, t_y2 = 256;
    static_assert(S % 128 == 0 && S >= 256 && S <= 512, "dstate blocks");
    static_assert(bytes + 1024 + 512 <= 232448, "shared memory budget");
};

struct BigParams {
    const float *Gc, *dtT, *states, *D;
    Geom g;
    int n_items, H, nc;
    unsigned int *status;
};

struct BItem {
    int b, h, c, tau, n;
    int64_t bh;
};

__device__ __forceinline__ BItem big_item(const BigParams &p, int item)
{
    BItem w;
    const unsigned u = (unsigned)item;
    w.h = (int)(u % (unsigned)p.H);
    const unsigned bc = u / (unsigned)p.H;
    w.c = (int)(bc % (unsigned)p.nc);
    w.b = (int)(bc / (unsigned)p.nc);
    w.tau = w.c * kTile;
    w.n = min(kTile, (int)p.g.L - w.tau);
    w.bh = (int64_t)w.b * p.H + w.h;
    return w;
}

template <int S>
__global__ void __launch_bounds__(kThreads, 1)
out_big_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_y,
               const BigParams prm)
{
    using Lay = BigLayout<S>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // TMA: sub-stage landed / free (its MMAs done); x of an item landed / free
    // (the y written over it has been stored)
    __shared__ uint64_t bar_full[2], bar_empty[2], bar_x[2], bar_xfree[2];
    // MMA completions: CB complete; Y1 (and everything before) complete
    __shared__ uint64_t bar_cb, bar_y, bar_end;
    // compute warps (8 arrivals): H's rows of dstate block k written (block 0
    // also the g / dt table); scores written; y staged (per x buffer)
    __shared__ uint64_t bar_h[Lay::kSB], bar_sc, bar_ys[2];
    __shared__ uint32_t tmem_slot;

    const Geom &g = prm.g;
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        for (int k = 0; k < 2; ++k) {
            mbar_init(&bar_full[k], 1);
            mbar_init(&bar_empty[k], 1);
            mbar_init(&bar_x[k], 1);
            mbar_init(&bar_xfree[k], 1);
            mbar_init(&bar_ys[k], kWarps);
        }
        mbar_init(&bar_cb, 1);
        mbar_init(&bar_y, 1);
        mbar_init(&bar_end, 1);
        for (int k = 0; k < Lay::kSB; ++k)
            mbar_init(&bar_h[k], kWarps);
        mbar_init(&bar_sc, kWarps);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 8) {
        // ---------------- TMA loads: x of each item, then its dstate blocks of B, C
        if ((tid & 31) == 0) {
            prefetch_tmap(&tm_x);
            prefetch_tmap(&tm_b);
            prefetch_tmap(&tm_c);
            uint32_t it = 0, u = 0;
            bool ok = true;
            // the f32 chunk state of an item (P x S, contiguous) into L2 ahead
            // of the compute warps' loads of it: the first item's now, then
            // each next item's as the current one starts
            const uint32_t st_bytes = (uint32_t)(g.P * S) * 4u;
            auto prefetch_state = [&](int item) {
                if (item < prm.n_items) {
                    const BItem v = big_item(prm, item);
                    bulk_prefetch_l2(prm.states + ((v.bh * prm.nc + v.c) * g.P) * g.S, st_bytes);
                }
            };
            prefetch_state(blockIdx.x);
            for (int item = blockIdx.x; item < prm.n_items && ok; item += gridDim.x, ++it) {
                const BItem w = big_item(prm, item);
                const int grp = w.h / g.hpg;
                const uint32_t xs = it & 1;
                prefetch_state(item + gridDim.x);
                if (it >= 2 && !mbar_wait(&bar_xfree[xs], ((it >> 1) - 1) & 1)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&bar_x[xs], kRegion);
                tma4(smem + Lay::off_x + xs * kRegion, &tm_x, &bar_x[xs], 0, w.h, w.tau, w.b);
                for (int sb = 0; sb < Lay::kSB; ++sb, ++u) {
                    const uint32_t s = u & 1;
                    if (u >= 2 && !mbar_wait(&bar_empty[s], ((u >> 1) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sub = smem + Lay::off_sub + s * Lay::kSub;
                    mbar_arrive_expect_tx(&bar_full[s], Lay::kSub);
                    for (int r = 0; r < 2; ++r) {
                        tma4(sub + r * kRegion, &tm_b, &bar_full[s], (2 * sb + r) * 64, grp, w.tau, w.b);
                        tma4(sub + (2 + r) * kRegion, &tm_c, &bar_full[s], (2 * sb + r) * 64, grp,
                             w.tau, w.b);
                    }
                }
            }
            if (!ok)
                atomicOr(prm.status, 1u);
        }
    } else if (warp == 9) {
        // ---------------- MMA issue.  Per item: CB and Y2 block by block, then
        // Y1 once the scores are written.
        if ((tid & 31) == 0) {
            const uint32_t id_cb = idesc_bf16(128, 128, false, false);
            const uint32_t id_y2 = idesc_bf16(128, 64, false, true);  // H is MN-major
            const uint32_t id_y1 = idesc_bf16(128, 64, false, true);  // x is MN-major
            const uint64_t d_h = desc_mn0(smem_u32(smem + Lay::off_h));
            uint32_t it = 0, u = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < prm.n_items && ok; item += gridDim.x, ++it) {
                const uint32_t par = it & 1, xs = it & 1;
                for (int sb = 0; sb < Lay::kSB; ++sb, ++u) {
                    const uint32_t s = u & 1;
                    if (!mbar_wait(&bar_full[s], (u >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sub = smem_u32(smem + Lay::off_sub + s * Lay::kSub);
                    const uint64_t d_b = desc_k0(sub), d_c = desc_k0(sub + 2 * kRegion);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ss(tmem + Lay::t_cb, desc_k(d_c, kRegion, ks), desc_k(d_b, kRegion, ks),
                               id_cb, (sb | ks) != 0);
                    // this block's rows of H written (and Y2 of the last item read H)
                    if (!mbar_wait(&bar_h[sb], par)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t d_hb = d_h + ((uint32_t)(sb * 128 * 128) >> 4);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ss(tmem + Lay::t_y2 + 64 * par, desc_k(d_c, kRegion, ks), desc_mn(d_hb, ks), id_y2,
                               (sb | ks) != 0);
                    mma_commit(&bar_empty[s]);
                }
                if (!ok)
                    break;
                mma_commit(&bar_cb);
                if (!mbar_wait(&bar_sc, par) || !mbar_wait(&bar_x[xs], (it >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t d_x = desc_mn0(smem_u32(smem + Lay::off_x + xs * kRegion));
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks)
                    mma_ts(tmem + Lay::t_y1, tmem + Lay::t_sc + ks * 8, desc_mn(d_x, ks), id_y1, ks > 0);
                mma_commit(&bar_y);
            }
            if (!ok)
                atomicOr(prm.status, 1u);
            // every MMA this thread issued has completed before TMEM is freed
            mma_commit(&bar_end);
            if (!mbar_wait(&bar_end, 0))
                atomicOr(prm.status, 1u);
        }
    } else if (warp == 10) {
        // ---------------- y store (written over the item's x tile)
        if ((tid & 31) == 0) {
            prefetch_tmap(&tm_y);
            uint32_t it = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < prm.n_items && ok; item += gridDim.x, ++it) {
                const BItem w = big_item(prm, item);
                const uint32_t xs = it & 1;
                if (!mbar_wait(&bar_ys[xs], (it >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tma4_store(&tm_y, smem + Lay::off_x + xs * kRegion, 0, w.h, w.tau, w.b);
                bulk_commit();
                bulk_wait_read();
                mbar_arrive(&bar_xfree[xs]);
            }
            bulk_wait_all();
            if (!ok)
                atomicOr(prm.status, 1u);
        }
    } else if (warp < kWarps) {
        // ---------------- compute
        const int wg = warp >> 2, q = warp & 3;
        const int i = q * 32 + (tid & 31);
        const int row_hi = q * 32 + 31;
        const uint32_t tl = tmem_at(tmem, (uint32_t)(q * 32), 0);
        float *gtab = reinterpret_cast<float *>(smem + Lay::off_g);
        uint8_t *s_h = smem + Lay::off_h;
        // this row's G and dt of the next item, loaded one item ahead
        float g_nx = 0.f, d_nx = 0.f;
        auto load_gd = [&](const BItem &w) {
            const int64_t o = w.bh * g.L + w.tau + i;
            g_nx = i < w.n ? ld_early(prm.Gc + o) : 0.f;
            d_nx = i < w.n ? ld_early(prm.dtT + o) : 0.f;
        };
        // ---- g / dt table; H = bf16(h_c), MN-major [s][p], one 128-row dstate
        // block at a time, published per block so that block k's C H^T starts
        // while the next rows are written: both warpgroups take every block,
        // thread i its row 128 k + i and warpgroup wg the headdim columns
        // [32 wg, 32 wg + 32).  The caller has seen the previous item's C B^T
        // and C H^T complete (bar_cb) and every warp's scores of it done.
        auto build_h = [&](const BItem &w, float gi, float dti) {
            if (wg == 0)
                gtab[i] = gi;
            else
                gtab[128 + i] = dti;
            const float *src = prm.states + ((w.bh * prm.nc + w.c) * g.P) * g.S;
#pragma unroll 1
            for (int sb = 0; sb < Lay::kSB; ++sb) {
                const int s_row = sb * 128 + i;
                float v[32];
#pragma unroll
                for (int p = 0; p < 32; ++p)
                    v[p] = __ldcs(src + (int64_t)(32 * wg + p) * S + s_row);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 o = make_uint4(pack_bf16x2(v[8 * c], v[8 * c + 1]),
                                               pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                                               pack_bf16x2(v[8 * c + 4], v[8 * c + 5]),
                                               pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
                    *reinterpret_cast<uint4 *>(s_h + sw128_offset(s_row, 4 * wg + c)) = o;
                }
                fence_proxy_async_smem();
                warp_arrive(&bar_h[sb]);
            }
        };
        // Order per item k: scores(k), then the next item's table and H (they
        // overlap Y1(k) and the next item's C B^T), then the epilogue of k.
        float gi_cur = 0.f, dti_cur = 0.f;
        if ((int)blockIdx.x < prm.n_items) {
            load_gd(big_item(prm, blockIdx.x));
            gi_cur = g_nx;
            dti_cur = d_nx;
            if ((int)(blockIdx.x + gridDim.x) < prm.n_items)
                load_gd(big_item(prm, blockIdx.x + gridDim.x));
            build_h(big_item(prm, blockIdx.x), gi_cur, dti_cur);
        }
        uint32_t it = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < prm.n_items && ok; item += gridDim.x, ++it) {
            const BItem w = big_item(prm, item);
            const uint32_t par = it & 1, xs = it & 1;
            const float gi = gi_cur;
            const bool more = item + (int)gridDim.x < prm.n_items;

            // ---- exact scores CB_ij exp2(g_i - g_j) dt_j (j <= i); warpgroup wg
            // converts keys [64 wg, 64 wg + 64).  The table is complete once all
            // eight warps have arrived at bar_h[0].
            if (!mbar_wait(&bar_cb, par) || !mbar_wait(&bar_h[0], par)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t cbv[2][16];
#pragma unroll
                for (int gq = 0; gq < 2; ++gq) {
                    const int j0 = 64 * wg + 32 * half + 16 * gq;
                    if (j0 <= row_hi)
                        tmem_ld16(tl + Lay::t_cb + j0, cbv[gq]);
                }
                tmem_ld_wait();
#pragma unroll
                for (int gq = 0; gq < 2; ++gq) {
                    const int j0 = 64 * wg + 32 * half + 16 * gq;
                    uint32_t pk[8];
                    if (j0 > row_hi) {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            pk[e] = 0u;
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            float v2[2];
#pragma unroll
                            for (int uu = 0; uu < 2; ++uu) {
                                const int j = j0 + 2 * e + uu;
                                v2[uu] = j <= i ? __uint_as_float(cbv[gq][2 * e + uu]) *
                                                      ex2_approx(gi - gtab[j]) * gtab[128 + j]
                                                : 0.f;
                            }
                            pk[e] = pack_bf16x2(v2[0], v2[1]);
                        }
                    }
                    tmem_st8(tl + Lay::t_sc + j0 / 2, pk);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            warp_arrive(&bar_sc);

            // ---- the next item's table and H: every warp is done with this
            // item's table once bar_sc completes, and bar_cb covered this
            // item's C H^T (the last reader of H)
            if (more) {
                if (!mbar_wait(&bar_sc, par)) {
                    ok = false;
                    break;
                }
                gi_cur = g_nx;
                dti_cur = d_nx;
                if (item + 2 * (int)gridDim.x < prm.n_items)
                    load_gd(big_item(prm, item + 2 * gridDim.x));
                build_h(big_item(prm, item + gridDim.x), gi_cur, dti_cur);
            }

            // ---- epilogue: y = Y1 + exp2(g_i) Y2 + D x, written over x
            if (!mbar_wait(&bar_y, par) || !mbar_wait(&bar_x[xs], (it >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            {
                const float er = ex2_approx(gi), Dh = prm.D[w.h];
                uint8_t *sx = smem + Lay::off_x + xs * kRegion;
                const int c0w = 32 * wg;
#pragma unroll
                for (int c16 = 0; c16 < 32; c16 += 16) {
                    uint32_t ra[16], rb[16];
                    tmem_ld16(tl + Lay::t_y1 + c0w + c16, ra);
                    tmem_ld16(tl + Lay::t_y2 + 64 * par + c0w + c16, rb);
                    tmem_ld_wait();
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        uint8_t *xp = sx + sw128_offset(i, (c0w + c16) / 8 + kk);
                        const uint4 xv4 = *reinterpret_cast<const uint4 *>(xp);
                        const uint32_t xv[4] = {xv4.x, xv4.y, xv4.z, xv4.w};
                        uint32_t o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = 8 * kk + 2 * e;
                            const float a = __uint_as_float(ra[c]) + er * __uint_as_float(rb[c]) +
                                            Dh * bf_lo(xv[e]);
                            const float bb = __uint_as_float(ra[c + 1]) +
                                             er * __uint_as_float(rb[c + 1]) + Dh * bf_hi(xv[e]);
                            o[e] = pack_bf16x2(a, bb);
                        }
                        *reinterpret_cast<uint4 *>(xp) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(&bar_ys[xs]);
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

int sm_count_big()
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

template <int S>
cudaError_t launch_big(const CUtensorMap &tx, const CUtensorMap &tb, const CUtensorMap &tcm,
                       const CUtensorMap &ty, const BigParams &prm, cudaStream_t st)
{
    using Lay = BigLayout<S>;
    const size_t smem = Lay::bytes + 1024;
    auto k = out_big_kernel<S>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const int grid = prm.n_items < sm_count_big() ? prm.n_items : sm_count_big();
    k<<<(unsigned)grid, kThreads, smem, st>>>(tx, tb, tcm, ty, prm);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

bool chunk_out_big_supported(const Geom &g)
{
    const int64_t nc = (g.L + kTile - 1) / kTile;
    return g.P == 64 && (g.S == 384 || g.S == 512) && g.T == kTile && g.L > 0 &&
           g.L < (1LL << 31) && g.H <= 65535 && g.G <= 65535 && g.B <= 65535 &&
           g.B * g.H * nc < (1LL << 31);
}

cudaError_t launch_chunk_out_big(const void *x, const void *Bm, const void *Cm, const float *dtT,
                                 const float *Gc, const float *states, const float *D, void *y,
                                 const Geom &g, cudaStream_t st)
{
    if (!chunk_out_big_supported(g))
        return cudaErrorNotSupported;
    BigParams prm{};
    prm.Gc = Gc;
    prm.dtT = dtT;
    prm.states = states;
    prm.D = D;
    prm.g = g;
    prm.H = (int)g.H;
    prm.nc = (int)g.nc;
    prm.n_items = (int)(g.B * g.nc * g.H);
    prm.status = device_status_word();
    if (!prm.status)
        return cudaErrorUnknown;
    CUtensorMap tx, tb, tcm, ty;
    if (!make_tmap_tokens_heads(&tx, x, g) || !make_tmap_tokens_groups(&tb, Bm, g) ||
        !make_tmap_tokens_groups(&tcm, Cm, g) || !make_tmap_tokens_heads(&ty, y, g))
        return cudaErrorInvalidValue;
    return g.S == 384 ? launch_big<384>(tx, tb, tcm, ty, prm, st)
                      : launch_big<512>(tx, tb, tcm, ty, prm, st);
}

}  // namespace ssd
