// Single-token decode step on the carried state.
//
// "Accelerating Mamba-2 forward-pass kernels with CUDA Tile (cuTile)",
// section "Mamba-2 架构": the recurrence the chunked forward computes in
// blocks, taken one token at a time -- the inference use of the final state
// that section "Kernel 2: fwd_pass_state" hands on.  Per (b, h), g = h / hpg:
//     h[p,s] <- exp(A[h] dt) h[p,s] + dt x[p] B[s]
//     y[p]    = sum_s C[s] h[p,s] + D[h] x[p]
//
// The step is bound by streaming the f32 state through HBM once in each
// direction (4PS bytes read and written per head); everything else is small.
// A "row" is one (b, h, p): S contiguous floats of the state.  In the main
// kernel lpr lanes of a warp share a row (lpr = the largest power of two
// dividing the row's count of 4-float vectors, at most 32), each lane taking
// every lpr-th vector, at most four per row; C . h is reduced over those
// lanes with shuffles.  Work items are blocks of rows of one (b, h), so the
// index arithmetic, the decay and the B / C vectors are set up once per
// block.  Other dstates (S % 4 != 0, more than four vectors per lane, or
// unaligned state / B / C) take a plain kernel with one warp per row.  With
// L = 1 the row index is also the index of x and y, and row / P that of dt.
#include "common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kDecThreads = 256;

struct DecGeom {
    int64_t rows;  // B * H * P
    int P, H, G, hpg, S;
    int lpr;       // lanes per row (power of two, divides 32)
    int vpl;       // vectors per lane per row
    int passes;    // warp passes per work item (main kernel)
};

// four inputs of B or C as f32: one 8-byte load for bf16, 16 bytes for f32
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float (&v)[4])
{
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xffff0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xffff0000u);
}
__device__ __forceinline__ void load4(const float *p, float (&v)[4])
{
    const float4 u = *reinterpret_cast<const float4 *>(p);
    v[0] = u.x;
    v[1] = u.y;
    v[2] = u.z;
    v[3] = u.w;
}

// Where row r's inputs live, and its decay and input weight (plain kernel).
struct RowIn {
    int64_t bg;  // b * G + group: B / C vector
    float decay, dtx, xp, dh;
};
template <typename TI>
__device__ __forceinline__ RowIn row_inputs(int64_t r, const TI *x, const float *dt, const float *A,
                                            const float *D, const DecGeom &g)
{
    RowIn o;
    const int64_t bh = r / g.P;
    const int h = (int)(bh % g.H);
    const float dtv = dt[bh];
    o.bg = (bh / g.H) * g.G + h / g.hpg;
    o.xp = to_f32(x[r]);
    o.dh = D[h];
    o.decay = expf(A[h] * dtv);
    o.dtx = dtv * o.xp;
    return o;
}

// Main kernel.  A work item is a block of rows of one (b, h): its index
// arithmetic, decay and B / C vectors are set up once and reused by every
// row of the block.  A warp pass covers NSET row sets of 32 / lpr rows; the
// state loads of all of them are issued before any is used (NSET * MAXV
// 16-byte loads in flight per lane).
template <typename TI, int MAXV>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(const TI *__restrict__ x,
                                                             const float *__restrict__ dt,
                                                             const float *__restrict__ A,
                                                             const TI *__restrict__ Bm,
                                                             const TI *__restrict__ Cm,
                                                             const float *__restrict__ D,
                                                             const float *state_in, float *state_out,
                                                             TI *__restrict__ y, DecGeom g)
{
    constexpr int NSET = 8 / MAXV;
    const int lane = threadIdx.x & 31;
    const int sub = lane & (g.lpr - 1), rw = lane / g.lpr;
    const int rpw = 32 / g.lpr;                 // rows of one row set
    const int rows_per_item = NSET * rpw * g.passes;
    const unsigned npb = ((unsigned)g.P + rows_per_item - 1) / rows_per_item;
    const unsigned n_items = (unsigned)(g.rows / g.P) * npb;
    const unsigned warp0 = blockIdx.x * (kDecThreads / 32) + (threadIdx.x >> 5);
    const unsigned nwarps = gridDim.x * (kDecThreads / 32);

    for (unsigned item = warp0; item < n_items; item += nwarps) {
        const unsigned bh = item / npb, pb = item - bh * npb;
        const unsigned h = bh % (unsigned)g.H, b = bh / (unsigned)g.H;
        const unsigned bg = b * (unsigned)g.G + h / (unsigned)g.hpg;
        const float dtv = dt[bh];
        const float decay = expf(A[h] * dtv);
        const float dh = D[h];
        float bv[MAXV][4], cv[MAXV][4];
#pragma unroll
        for (int k = 0; k < MAXV; ++k)
            if (k < g.vpl) {
                load4(Bm + (size_t)bg * g.S + 4 * (sub + k * g.lpr), bv[k]);
                load4(Cm + (size_t)bg * g.S + 4 * (sub + k * g.lpr), cv[k]);
            }
        // this head's state, x and y (offsets within a head fit 32 bits)
        const size_t head0 = (size_t)bh * g.P;
        const float4 *sin4 = reinterpret_cast<const float4 *>(state_in + head0 * g.S) + sub;
        float4 *sout4 = reinterpret_cast<float4 *>(state_out + head0 * g.S) + sub;
        const TI *xh = x + head0;
        TI *yh = y + head0;
        const int vrow = g.S >> 2;  // 16-byte vectors per row
        for (int pass = 0; pass < g.passes; ++pass) {
            const int pbase = (int)pb * rows_per_item + pass * NSET * rpw + rw;
            float4 hv[NSET][MAXV];
#pragma unroll
            for (int u = 0; u < NSET; ++u) {
                const int p = pbase + u * rpw;
                if (p < g.P) {
#pragma unroll
                    for (int k = 0; k < MAXV; ++k)
                        if (k < g.vpl)
                            hv[u][k] = sin4[p * vrow + k * g.lpr];
                }
            }
#pragma unroll
            for (int u = 0; u < NSET; ++u) {
                const int p = pbase + u * rpw;
                float acc = 0.f, xp = 0.f;
                if (p < g.P) {
                    xp = to_f32(xh[p]);
                    const float dtx = dtv * xp;
                    float4 *dst = sout4 + p * vrow;
#pragma unroll
                    for (int k = 0; k < MAXV; ++k) {
                        if (k < g.vpl) {
                            float4 h4 = hv[u][k];
                            h4.x = fmaf(decay, h4.x, dtx * bv[k][0]);
                            h4.y = fmaf(decay, h4.y, dtx * bv[k][1]);
                            h4.z = fmaf(decay, h4.z, dtx * bv[k][2]);
                            h4.w = fmaf(decay, h4.w, dtx * bv[k][3]);
                            acc = fmaf(cv[k][0], h4.x, acc);
                            acc = fmaf(cv[k][1], h4.y, acc);
                            acc = fmaf(cv[k][2], h4.z, acc);
                            acc = fmaf(cv[k][3], h4.w, acc);
                            dst[k * g.lpr] = h4;
                        }
                    }
                }
                // C . h over the row's lanes (every lane takes part in the shuffles)
                for (int o = g.lpr >> 1; o > 0; o >>= 1)
                    acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (p < g.P && sub == 0)
                    yh[p] = from_f32<TI>(acc + dh * xp);
            }
        }
    }
}

// Any dstate: one warp per row, lanes striding over s.
template <typename TI>
__global__ void __launch_bounds__(kDecThreads) decode_plain_kernel(const TI *__restrict__ x,
                                                                   const float *__restrict__ dt,
                                                                   const float *__restrict__ A,
                                                                   const TI *__restrict__ Bm,
                                                                   const TI *__restrict__ Cm,
                                                                   const float *__restrict__ D,
                                                                   const float *state_in,
                                                                   float *state_out,
                                                                   TI *__restrict__ y, DecGeom g)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (int64_t)blockIdx.x * (kDecThreads / 32) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (kDecThreads / 32);
    for (int64_t r = warp0; r < g.rows; r += nwarps) {
        const RowIn in = row_inputs(r, x, dt, A, D, g);
        const TI *bp = Bm + in.bg * g.S;
        const TI *cp = Cm + in.bg * g.S;
        float acc = 0.f;
        for (int s = lane; s < g.S; s += 32) {
            const float hv = fmaf(in.decay, state_in[r * g.S + s], in.dtx * to_f32(bp[s]));
            state_out[r * g.S + s] = hv;
            acc = fmaf(to_f32(cp[s]), hv, acc);
        }
        for (int o = 16; o > 0; o >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0)
            y[r] = from_f32<TI>(acc + in.dh * in.xp);
    }
}

int sm_count_decode()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

template <typename TI>
cudaError_t launch_dec(const void *x, const float *dt, const float *A, const void *Bm, const void *Cm,
                       const float *D, const float *state_in, float *state_out, void *y, DecGeom dg,
                       cudaStream_t st)
{
    const int64_t cap = (int64_t)sm_count_decode() * (2048 / kDecThreads);
    // 16-byte state vectors when a row is a whole number of them, every
    // state row and B / C vector is then aligned for them, and a lane holds
    // at most four of a row
    const auto al = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
    const uintptr_t bc_al = 4 * sizeof(TI);
    if (dg.S % 4 == 0 && al(state_in, 16) && al(state_out, 16) && al(Bm, bc_al) && al(Cm, bc_al)) {
        const int vpr = dg.S / 4;
        dg.lpr = 1;
        while (dg.lpr < 32 && vpr % (dg.lpr * 2) == 0)
            dg.lpr *= 2;
        dg.vpl = vpr / dg.lpr;
        if (dg.vpl <= 4) {
            const int maxv = dg.vpl == 1 ? 1 : (dg.vpl == 2 ? 2 : 4);
            // two passes per item unless that leaves fewer than 16 warps per SM
            const int rows_per_pass = (8 / maxv) * (32 / dg.lpr);
            const int64_t heads = dg.rows / dg.P;
            const int64_t items2 = heads * ((dg.P + 2 * rows_per_pass - 1) / (2 * rows_per_pass));
            dg.passes = items2 >= (int64_t)sm_count_decode() * 16 ? 2 : 1;
            const int rows_per_item = rows_per_pass * dg.passes;
            const int64_t items = heads * ((dg.P + rows_per_item - 1) / rows_per_item);
            int64_t blocks = (items + kDecThreads / 32 - 1) / (kDecThreads / 32);
            if (blocks > cap)
                blocks = cap;
            const TI *xt = static_cast<const TI *>(x), *bt = static_cast<const TI *>(Bm),
                     *ct = static_cast<const TI *>(Cm);
            TI *yt = static_cast<TI *>(y);
            if (maxv == 1)
                decode_kernel<TI, 1><<<(unsigned)blocks, kDecThreads, 0, st>>>(
                    xt, dt, A, bt, ct, D, state_in, state_out, yt, dg);
            else if (maxv == 2)
                decode_kernel<TI, 2><<<(unsigned)blocks, kDecThreads, 0, st>>>(
                    xt, dt, A, bt, ct, D, state_in, state_out, yt, dg);
            else
                decode_kernel<TI, 4><<<(unsigned)blocks, kDecThreads, 0, st>>>(
                    xt, dt, A, bt, ct, D, state_in, state_out, yt, dg);
            note_launch(1);
            return cudaGetLastError();
        }
    }
    int64_t blocks = (dg.rows + kDecThreads / 32 - 1) / (kDecThreads / 32);
    if (blocks > cap)
        blocks = cap;
    decode_plain_kernel<TI><<<(unsigned)blocks, kDecThreads, 0, st>>>(
        static_cast<const TI *>(x), dt, A, static_cast<const TI *>(Bm), static_cast<const TI *>(Cm), D,
        state_in, state_out, static_cast<TI *>(y), dg);
    note_launch(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_step(const void *x, const float *dt, const float *A, const void *Bm,
                               const void *Cm, const float *D, const float *state_in, float *state_out,
                               void *y, const Geom &g, bool bf16, cudaStream_t st)
{
    DecGeom dg{};
    dg.rows = (int64_t)g.B * g.H * g.P;
    dg.P = (int)g.P;
    dg.H = (int)g.H;
    dg.G = (int)g.G;
    dg.hpg = g.hpg;
    dg.S = (int)g.S;
    if (dg.rows == 0)
        return cudaSuccess;
    return bf16 ? launch_dec<__nv_bfloat16>(x, dt, A, Bm, Cm, D, state_in, state_out, y, dg, st)
                : launch_dec<float>(x, dt, A, Bm, Cm, D, state_in, state_out, y, dg, st);
}

}  // namespace ssd
