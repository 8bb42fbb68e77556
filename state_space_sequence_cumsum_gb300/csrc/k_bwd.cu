// Backward pass of the chunked SSD forward (f32 arithmetic on CUDA cores).
//
// The pages ("Accelerating Mamba-2 forward-pass kernels with CUDA Tile
// (cuTile)") name the backward pass without giving it; it is derived here
// from the chunked forward of sections "Kernel 2" and "Kernel 3".  Within a
// chunk (tokens i, j; L_i the inclusive within-chunk sum of a = A dt, in
// natural units; G = log2(e) L as stage 1 stores it; W_ij = exp(L_i - L_j)
// for i >= j, else 0; h_in the chunk's start state, dS the gradient of its
// end state):
//
//   forward   y_i   = sum_j W_ij (C_i . B_j) dt_j x_j + e^{L_i} h_in C_i + D x_i
//             h_out = e^{L_T} h_in + sum_j e^{L_T - L_j} dt_j x_j B_j^T
//   backward  dh_in = e^{L_T} dS + sum_i e^{L_i} dy_i C_i^T     (reverse state pass)
//             dx_j  = D dy_j + dt_j [ sum_i W_ij (C_i . B_j) dy_i + e^{L_T - L_j} dS B_j ]
//             dB_j  = dt_j [ sum_i W_ij (dy_i . x_j) C_i + e^{L_T - L_j} dS^T x_j ]
//             dC_i  = sum_j W_ij (dy_i . x_j) dt_j B_j + e^{L_i} h_in^T dy_i
//             dD    = sum_i dy_i . x_i
// and, through the decays, with dL_i = d loss / d L_i:
//             dL_i += sum_j Q_ij dt_j - sum_k Q_ki dt_i,   Q_ij = W_ij (C_i . B_j)(dy_i . x_j)
//             dL_i += e^{L_i} dy_i . (h_in C_i)
//             dL_j -= R_j,  dL_last += sum_j R_j + e^{L_T} (dS . h_in),
//                                        R_j = e^{L_T - L_j} dt_j x_j . (dS B_j)
//             da_k = sum_{i >= k} dL_i,  ddt_k = x_k . [dx_k - D dy_k] / dt_k + A da_k,
//             dA  += sum_k dt_k da_k
// where x_k . [dx_k - D dy_k] / dt_k is formed directly (no division).
// dB and dC sum over the heads of a group (f32 atomics into a workspace,
// converted to the input dtype at the end).
//
// Kernels: the reverse state pass (the forward state pass's structure run
// from the last chunk to the first), the per-(batch, chunk, head) gradient
// kernel (64-token chunks, dstate streamed in 64-wide tiles), and a final
// conversion.  The chunk start states come from the forward state pass.
#include "common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kBT = 64;        // tokens per chunk of the backward
constexpr int kBThreads = 256;
constexpr int kLd = kBT + 1;   // padded row stride of the 64-wide tiles

// ---------------------------------------------------------------- reverse state pass
// CTA = (32-wide dstate tile, 64-row headdim tile, batch*head); warp w owns
// headdim rows p0 + w + 8k, lane l dstate column s0 + l.  dstates[c] receives
// the gradient of chunk c's END state before chunk c is folded in.
constexpr int kRsTok = 32;

template <typename TI>
__global__ void __launch_bounds__(kBThreads)
bwd_state_kernel(const TI *__restrict__ dy, const TI *__restrict__ Cm, const float *__restrict__ Gc,
                 const float *__restrict__ dfinal, float *__restrict__ dstates,
                 float *__restrict__ dinit, Geom g)
{
    __shared__ float sdy[kRsTok][64];  // exp2(G_i) dy_i for the CTA's headdim rows
    __shared__ float sc[kRsTok][33];   // C for the CTA's dstate columns
    __shared__ float sw[kRsTok];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t s0 = (int64_t)blockIdx.x * 32, p0 = (int64_t)blockIdx.y * 64;
    const int64_t bh = blockIdx.z, b = bh / g.H, h = bh % g.H, grp = h / g.hpg;
    const int64_t s = s0 + lane;
    const bool s_ok = s < g.S;

    float ds[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int64_t p = p0 + warp + 8 * k;
        ds[k] = (dfinal && s_ok && p < g.P) ? dfinal[(bh * g.P + p) * g.S + s] : 0.f;
    }
    const float *grow = Gc + bh * g.L;
    for (int64_t c = g.nc - 1; c >= 0; --c) {
        const int64_t t0 = c * g.T;
        const int n = (int)min64(g.T, g.L - t0);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t p = p0 + warp + 8 * k;
            if (s_ok && p < g.P)
                dstates[((bh * g.nc + c) * g.P + p) * g.S + s] = ds[k];
        }
        const float glast = grow[t0 + n - 1];
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int i0 = 0; i0 < n; i0 += kRsTok) {
            const int m = min(kRsTok, n - i0);
            __syncthreads();
            if (threadIdx.x < kRsTok) {
                const int i = threadIdx.x;
                sw[i] = i < m ? exp2f(grow[t0 + i0 + i]) : 0.f;
            }
            __syncthreads();
            for (int e = threadIdx.x; e < kRsTok * 64; e += kBThreads) {
                const int i = e / 64, pp = e % 64;
                const int64_t p = p0 + pp;
                float v = 0.f;
                if (i < m && p < g.P)
                    v = to_f32(dy[((b * g.L + t0 + i0 + i) * g.H + h) * g.P + p]) * sw[i];
                sdy[i][pp] = v;
            }
            for (int e = threadIdx.x; e < kRsTok * 32; e += kBThreads) {
                const int i = e / 32, ss = e % 32;
                float v = 0.f;
                if (i < m && s0 + ss < g.S)
                    v = to_f32(Cm[((b * g.L + t0 + i0 + i) * g.G + grp) * g.S + s0 + ss]);
                sc[i][ss] = v;
            }
            __syncthreads();
            for (int i = 0; i < m; ++i) {
                const float cv = sc[i][lane];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    acc[k] = fmaf(sdy[i][warp + 8 * k], cv, acc[k]);
            }
        }
        const float decay = exp2f(glast);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            ds[k] = fmaf(decay, ds[k], acc[k]);
    }
    if (dinit) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t p = p0 + warp + 8 * k;
            if (s_ok && p < g.P)
                dinit[(bh * g.P + p) * g.S + s] = ds[k];
        }
    }
}

// ---------------------------------------------------------------- chunk gradients
// acc[r][c] += sum_k Aop[4 ty + r][k] Bop[k][4 tx + c] over a 64 x 64 tile,
// Aop[m][k] = TA ? A[k lda + m] : A[m lda + k], Bop[k][n] = TB ? B[n ldb + k] : B[k ldb + n].
template <bool TA, bool TB>
__device__ __forceinline__ void mm64(float (&acc)[4][4], const float *A, int lda, const float *B,
                                     int ldb, int K, int ty, int tx)
{
    for (int k = 0; k < K; ++k) {
        float a[4], bv[4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
            a[r] = TA ? A[k * lda + 4 * ty + r] : A[(4 * ty + r) * lda + k];
#pragma unroll
        for (int c = 0; c < 4; ++c)
            bv[c] = TB ? B[(4 * tx + c) * ldb + k] : B[k * ldb + 4 * tx + c];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                acc[r][c] = fmaf(a[r], bv[c], acc[r][c]);
    }
}

__device__ __forceinline__ void zero44(float (&a)[4][4])
{
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c)
            a[r][c] = 0.f;
}

struct BwdSmem {
    // 64 x 65 f32 tiles
    static constexpr int kTile = kBT * kLd;
    static constexpr int x = 0, dy = x + kTile, dyx = dy + kTile, cb = dyx + kTile,
                         bds = cb + kTile, chin = bds + kTile, bt = chin + kTile, ct = bt + kTile,
                         hin = ct + kTile, dst = hin + kTile, wd = dst + kTile;
    static constexpr int vec = wd + kTile;  // g[64], dt[64], w[64], dl[64], red[64]
    static constexpr int floats = vec + 5 * kBT;
};

template <typename TI>
__global__ void __launch_bounds__(kBThreads)
bwd_chunk_kernel(const TI *__restrict__ x, const TI *__restrict__ Bm, const TI *__restrict__ Cm,
                 const TI *__restrict__ dy, const float *__restrict__ dtT,
                 const float *__restrict__ Gc, const float *__restrict__ A,
                 const float *__restrict__ D, const float *__restrict__ states,
                 const float *__restrict__ dstates, TI *__restrict__ dx, float *__restrict__ ddt,
                 float *__restrict__ dA, float *__restrict__ dD, float *__restrict__ dBacc,
                 float *__restrict__ dCacc, Geom g)
{
    extern __shared__ float sm[];
    using L = BwdSmem;
    float *sx = sm + L::x, *sdy = sm + L::dy, *sdyx = sm + L::dyx, *scb = sm + L::cb,
          *sbds = sm + L::bds, *schin = sm + L::chin, *sbt = sm + L::bt, *sct = sm + L::ct,
          *shin = sm + L::hin, *sdst = sm + L::dst, *swd = sm + L::wd;
    float *sg = sm + L::vec, *sdt = sg + kBT, *sw2 = sdt + kBT, *sdl = sw2 + kBT, *sred = sdl + kBT;

    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int64_t c = blockIdx.x, bh = blockIdx.y;
    const int64_t b = bh / g.H, h = bh % g.H, grp = h / g.hpg;
    const int64_t t0 = c * kBT;
    const int n = (int)min64(kBT, g.L - t0);
    const int P = (int)g.P;

    // ---- chunk inputs: x, dy (rows past n are zero), G, dt
    for (int e = tid; e < kBT * kBT; e += kBThreads) {
        const int i = e / kBT, p = e % kBT;
        float xv = 0.f, dv = 0.f;
        if (i < n && p < P) {
            const int64_t o = ((b * g.L + t0 + i) * g.H + h) * g.P + p;
            xv = to_f32(x[o]);
            dv = to_f32(dy[o]);
        }
        sx[i * kLd + p] = xv;
        sdy[i * kLd + p] = dv;
    }
    if (tid < kBT) {
        const bool ok = tid < n;
        sg[tid] = ok ? Gc[bh * g.L + t0 + tid] : 0.f;
        sdt[tid] = ok ? dtT[bh * g.L + t0 + tid] : 0.f;
        sdl[tid] = 0.f;
    }
    __syncthreads();
    const float glast = sg[n - 1];
    if (tid < kBT)
        sw2[tid] = tid < n ? exp2f(glast - sg[tid]) : 0.f;  // e^{L_T - L_j}

    // ---- dyx[i][j] = dy_i . x_j, then wd = W * dyx (masked)
    {
        float acc[4][4];
        zero44(acc);
        mm64<false, true>(acc, sdy, kLd, sx, kLd, P, ty, tx);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int i = 4 * ty + r, j = 4 * tx + cc;
                sdyx[i * kLd + j] = acc[r][cc];
                swd[i * kLd + j] = (j <= i && i < n) ? exp2f(sg[i] - sg[j]) * acc[r][cc] : 0.f;
                scb[i * kLd + j] = 0.f;
            }
    }
    for (int e = tid; e < kBT * kBT; e += kBThreads) {
        const int j = e / kBT, p = e % kBT;
        sbds[j * kLd + p] = 0.f;
        schin[j * kLd + p] = 0.f;
    }
    float dshin = 0.f;  // this thread's part of sum dS * h_in
    __syncthreads();

    // ---- dstate tiles
    const float *hin_g = states + (bh * g.nc + c) * g.P * g.S;
    const float *dst_g = dstates + (bh * g.nc + c) * g.P * g.S;
    for (int s0 = 0; s0 < (int)g.S; s0 += kBT) {
        const int sw = min(kBT, (int)g.S - s0);
        for (int e = tid; e < kBT * kBT; e += kBThreads) {
            const int r = e / kBT, s = e % kBT;
            float bv = 0.f, cv = 0.f, hv = 0.f, dv = 0.f;
            if (s < sw) {
                if (r < n) {
                    const int64_t o = ((b * g.L + t0 + r) * g.G + grp) * g.S + s0 + s;
                    bv = to_f32(Bm[o]);
                    cv = to_f32(Cm[o]);
                }
                if (r < P) {
                    hv = hin_g[(int64_t)r * g.S + s0 + s];
                    dv = dst_g[(int64_t)r * g.S + s0 + s];
                }
            }
            sbt[r * kLd + s] = bv;
            sct[r * kLd + s] = cv;
            shin[r * kLd + s] = hv;
            sdst[r * kLd + s] = dv;
            dshin = fmaf(hv, dv, dshin);
        }
        __syncthreads();
        {
            float acc[4][4];
            // CB += C_t B_t^T ; BdS += B_t dS_t^T ; Chin += C_t h_in_t^T
            zero44(acc);
            mm64<false, true>(acc, sct, kLd, sbt, kLd, sw, ty, tx);
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    scb[(4 * ty + r) * kLd + 4 * tx + cc] += acc[r][cc];
            zero44(acc);
            mm64<false, true>(acc, sbt, kLd, sdst, kLd, sw, ty, tx);
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    sbds[(4 * ty + r) * kLd + 4 * tx + cc] += acc[r][cc];
            zero44(acc);
            mm64<false, true>(acc, sct, kLd, shin, kLd, sw, ty, tx);
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    schin[(4 * ty + r) * kLd + 4 * tx + cc] += acc[r][cc];

            // dB_t[j][s] = dt_j [ sum_i wd[i][j] C_t[i][s] + e^{L_T - L_j} sum_p x_j[p] dS_t[p][s] ]
            float a1[4][4], a2[4][4];
            zero44(a1);
            zero44(a2);
            mm64<true, false>(a1, swd, kLd, sct, kLd, kBT, ty, tx);
            mm64<false, false>(a2, sx, kLd, sdst, kLd, P, ty, tx);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int j = 4 * ty + r;
                if (j >= n)
                    continue;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int s = 4 * tx + cc;
                    if (s < sw)
                        atomicAdd(dBacc + ((b * g.L + t0 + j) * g.G + grp) * g.S + s0 + s,
                                  sdt[j] * (a1[r][cc] + sw2[j] * a2[r][cc]));
                }
            }
            // dC_t[i][s] = sum_j wd[i][j] dt_j B_t[j][s] + e^{L_i} sum_p dy_i[p] h_in_t[p][s]
            zero44(a1);
            zero44(a2);
            for (int k = 0; k < kBT; ++k) {
                float av[4], bv4[4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    av[r] = swd[(4 * ty + r) * kLd + k] * sdt[k];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    bv4[cc] = sbt[k * kLd + 4 * tx + cc];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        a1[r][cc] = fmaf(av[r], bv4[cc], a1[r][cc]);
            }
            mm64<false, false>(a2, sdy, kLd, shin, kLd, P, ty, tx);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = 4 * ty + r;
                if (i >= n)
                    continue;
                const float el = exp2f(sg[i]);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int s = 4 * tx + cc;
                    if (s < sw)
                        atomicAdd(dCacc + ((b * g.L + t0 + i) * g.G + grp) * g.S + s0 + s,
                                  a1[r][cc] + el * a2[r][cc]);
                }
            }
        }
        __syncthreads();
    }

    // ---- dx, ddt (direct part), dL
    const float Ah = A[h], Dh = D[h];
    {
        // m1 = W * CB (masked), overwriting cb; q = m1 * dyx * dt_j for dL
        for (int e = tid; e < kBT * kBT; e += kBThreads) {
            const int i = e / kBT, j = e % kBT;
            scb[i * kLd + j] = (j <= i && i < n) ? exp2f(sg[i] - sg[j]) * scb[i * kLd + j] : 0.f;
        }
        __syncthreads();
        // dx_j[p] = D dy_j[p] + dt_j [ sum_i m1[i][j] dy_i[p] + e^{L_T - L_j} BdS[j][p] ]
        float acc[4][4];
        zero44(acc);
        mm64<true, false>(acc, scb, kLd, sdy, kLd, kBT, ty, tx);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int j = 4 * ty + r;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int p = 4 * tx + cc;
                if (j < n && p < P) {
                    const float gpart = acc[r][cc] + sw2[j] * sbds[j * kLd + p];
                    dx[((b * g.L + t0 + j) * g.H + h) * g.P + p] =
                        from_f32<TI>(Dh * sdy[j * kLd + p] + sdt[j] * gpart);
                }
            }
        }
    }
    __syncthreads();  // every thread is done reading e^{L_T - L_j} (sw2)
    // per-token reductions: thread j < 64 walks its row / column
    if (tid < kBT) {
        const int j = tid;
        float direct = 0.f, dl = 0.f, rj = 0.f;
        if (j < n) {
            // x_j . (sum_p dS B_j) and the state read through y_j
            float xb = 0.f, yst = 0.f;
            for (int p = 0; p < P; ++p) {
                xb = fmaf(sx[j * kLd + p], sbds[j * kLd + p], xb);
                yst = fmaf(sdy[j * kLd + p], schin[j * kLd + p], yst);
            }
            // column j of m1 * dyx, and row j of m1 * dyx * dt
            float colq = 0.f, rowq = 0.f;
            for (int i = j; i < n; ++i)
                colq = fmaf(scb[i * kLd + j], sdyx[i * kLd + j], colq);
            for (int k = 0; k <= j; ++k)
                rowq = fmaf(scb[j * kLd + k] * sdyx[j * kLd + k], sdt[k], rowq);
            direct = colq + sw2[j] * xb;  // x_j . g_j: the dt-free part of ddt_j
            rj = sw2[j] * sdt[j] * xb;
            dl = rowq - colq * sdt[j] + exp2f(sg[j]) * yst - rj;
        }
        sred[j] = rj;
        sdl[j] = dl;
        sw2[j] = direct;
    }
    // sum of dS * h_in over the CTA, then the serial per-chunk tail
    __shared__ float wsum[kBThreads / 32];
    {
        float v = dshin;
        for (int o = 16; o > 0; o >>= 1)
            v += __shfl_xor_sync(0xffffffffu, v, o);
        if ((tid & 31) == 0)
            wsum[tid >> 5] = v;
    }
    __syncthreads();
    if (tid == 0) {
        float tot = 0.f, rsum = 0.f;
        for (int w = 0; w < kBThreads / 32; ++w)
            tot += wsum[w];
        for (int j = 0; j < n; ++j)
            rsum += sred[j];
        sdl[n - 1] += rsum + exp2f(glast) * tot;
        // da_k = suffix sums of dL; ddt_k = direct_k + A da_k; dA gets sum dt_k da_k
        float da = 0.f, dasum = 0.f, dd = 0.f;
        for (int k = n - 1; k >= 0; --k) {
            da += sdl[k];
            ddt[(b * g.L + t0 + k) * g.H + h] = sw2[k] + Ah * da;
            dasum = fmaf(sdt[k], da, dasum);
        }
        for (int i = 0; i < n; ++i)
            dd += sdyx[i * kLd + i];
        atomicAdd(dA + h, dasum);
        atomicAdd(dD + h, dd);
    }
}

template <typename TO>
__global__ void convert_kernel(const float *__restrict__ src, TO *__restrict__ dst, int64_t n)
{
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n;
         k += (int64_t)gridDim.x * blockDim.x)
        dst[k] = from_f32<TO>(src[k]);
}

}  // namespace

cudaError_t launch_convert_f32(const float *src, void *dst, int64_t n, bool bf16, cudaStream_t st)
{
    if (n <= 0)
        return cudaSuccess;
    const int blocks = (int)min64((n + 255) / 256, 4096);
    if (bf16)
        convert_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(src, static_cast<__nv_bfloat16 *>(dst), n);
    else
        convert_kernel<float><<<blocks, 256, 0, st>>>(src, static_cast<float *>(dst), n);
    note_launch(1);
    return cudaGetLastError();
}

bool bwd_supported(const Geom &g) { return g.P <= kBT && g.S <= 512 && g.L >= 1; }

int bwd_chunk_size() { return kBT; }

size_t bwd_chunk_smem_bytes() { return BwdSmem::floats * sizeof(float); }

cudaError_t launch_bwd(const void *x, const void *Bm, const void *Cm, const void *dy,
                       const float *dtT, const float *Gc, const float *A, const float *D,
                       const float *states, const float *dfinal, float *dstates, void *dx,
                       float *ddt, float *dA, float *dD, float *dBacc, float *dCacc, void *dB,
                       void *dC, float *dinit, const Geom &g, bool bf16, cudaStream_t st)
{
    // g.T must be kBT: states / dstates / G are per 64-token chunk
    const dim3 rs_grid((unsigned)((g.S + 31) / 32), (unsigned)((g.P + 63) / 64), (unsigned)(g.B * g.H));
    const dim3 ck_grid((unsigned)g.nc, (unsigned)(g.B * g.H));
    const size_t smem = bwd_chunk_smem_bytes();
    const int64_t nbc = g.B * g.L * g.G * g.S;
    const int cv_blocks = (int)min64((nbc + 255) / 256, 4096);
    cudaError_t e;
    if (bf16) {
        using T = __nv_bfloat16;
        bwd_state_kernel<T><<<rs_grid, kBThreads, 0, st>>>(static_cast<const T *>(dy),
                                                          static_cast<const T *>(Cm), Gc, dfinal,
                                                          dstates, dinit, g);
        e = cudaFuncSetAttribute(bwd_chunk_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess)
            return e;
        bwd_chunk_kernel<T><<<ck_grid, kBThreads, smem, st>>>(
            static_cast<const T *>(x), static_cast<const T *>(Bm), static_cast<const T *>(Cm),
            static_cast<const T *>(dy), dtT, Gc, A, D, states, dstates, static_cast<T *>(dx), ddt,
            dA, dD, dBacc, dCacc, g);
        convert_kernel<T><<<cv_blocks, 256, 0, st>>>(dBacc, static_cast<T *>(dB), nbc);
        convert_kernel<T><<<cv_blocks, 256, 0, st>>>(dCacc, static_cast<T *>(dC), nbc);
    } else {
        using T = float;
        bwd_state_kernel<T><<<rs_grid, kBThreads, 0, st>>>(static_cast<const T *>(dy),
                                                          static_cast<const T *>(Cm), Gc, dfinal,
                                                          dstates, dinit, g);
        e = cudaFuncSetAttribute(bwd_chunk_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess)
            return e;
        bwd_chunk_kernel<T><<<ck_grid, kBThreads, smem, st>>>(
            static_cast<const T *>(x), static_cast<const T *>(Bm), static_cast<const T *>(Cm),
            static_cast<const T *>(dy), dtT, Gc, A, D, states, dstates, static_cast<T *>(dx), ddt,
            dA, dD, dBacc, dCacc, g);
        convert_kernel<T><<<cv_blocks, 256, 0, st>>>(dBacc, static_cast<T *>(dB), nbc);
        convert_kernel<T><<<cv_blocks, 256, 0, st>>>(dCacc, static_cast<T *>(dC), nbc);
    }
    note_launch(4);
    return cudaGetLastError();
}

}  // namespace ssd
