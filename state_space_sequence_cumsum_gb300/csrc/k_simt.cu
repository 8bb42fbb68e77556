// Stages 2 and 3 on CUDA cores with f32 arithmetic.
//
// These kernels serve the f32-input path (whose tolerance, 1e-4 of the
// output's rms, rules out bf16/tf32 tensor-core operands) and every shape the
// tensor-core path does not cover.  They follow "Accelerating Mamba-2
// forward-pass kernels with CUDA Tile (cuTile)":
//   * state pass, section "Kernel 2: fwd_pass_state" -- per chunk
//       chunk_states[c] = h;  h <- exp2(G_last) h + X^T (B * dt * exp2(G_last - G))
//   * chunk output, section "Kernel 3: compute_out" --
//       Y = exp2(G) (C h_c^T) + (exp2(G_i - G_j) (C B^T) M)(dt X) + D X
// G_last is G at the chunk's last valid token (a ragged last chunk does not
// use zero padding as its last element).  Masked score entries (j > i) are
// set to zero without evaluating their (possibly overflowing) exponent.
#include "common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

// ---------------------------------------------------------------- state pass
// CTA = (32-wide dstate tile, 64-row headdim tile, batch*head).  Warp w owns
// headdim rows p0 + w + 8k (k < 8); lane l owns dstate column s0 + l.  The
// running state stays in registers across the serial chunk loop.
constexpr int kSpThreads = 256;
constexpr int kSpTok = 32;  // tokens staged per step

template <typename TI>
__global__ void __launch_bounds__(kSpThreads)
state_pass_simt_kernel(const TI *__restrict__ x, const TI *__restrict__ Bm,
                       const float *__restrict__ dtT, const float *__restrict__ Gc,
                       const float *__restrict__ init, float *__restrict__ states,
                       float *__restrict__ final_state, Geom g)
{
    __shared__ float sxw[kSpTok][64];  // x * w for the CTA's headdim rows
    __shared__ float sb[kSpTok][33];   // B for the CTA's dstate columns
    __shared__ float sw[kSpTok];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t s0 = (int64_t)blockIdx.x * 32, p0 = (int64_t)blockIdx.y * 64;
    const int64_t bh = blockIdx.z, b = bh / g.H, h = bh % g.H, grp = h / g.hpg;
    const int64_t s = s0 + lane;
    const bool s_ok = s < g.S;

    float hs[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int64_t p = p0 + warp + 8 * k;
        hs[k] = (init && s_ok && p < g.P) ? init[(bh * g.P + p) * g.S + s] : 0.f;
    }

    const float *grow = Gc + bh * g.L;
    const float *drow = dtT + bh * g.L;
    for (int64_t c = 0; c < g.nc; ++c) {
        const int64_t t0 = c * g.T;
        const int n = (int)min64(g.T, g.L - t0);
        if (states) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int64_t p = p0 + warp + 8 * k;
                if (s_ok && p < g.P)
                    states[((bh * g.nc + c) * g.P + p) * g.S + s] = hs[k];
            }
        }
        const float glast = grow[t0 + n - 1];
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j0 = 0; j0 < n; j0 += kSpTok) {
            const int m = min(kSpTok, n - j0);
            __syncthreads();
            if (threadIdx.x < kSpTok) {
                const int j = threadIdx.x;
                sw[j] = j < m ? drow[t0 + j0 + j] * exp2f(glast - grow[t0 + j0 + j]) : 0.f;
            }
            __syncthreads();
            for (int e = threadIdx.x; e < kSpTok * 64; e += kSpThreads) {
                const int j = e / 64, pp = e % 64;
                const int64_t p = p0 + pp;
                float v = 0.f;
                if (j < m && p < g.P)
                    v = to_f32(x[((b * g.L + t0 + j0 + j) * g.H + h) * g.P + p]) * sw[j];
                sxw[j][pp] = v;
            }
            for (int e = threadIdx.x; e < kSpTok * 32; e += kSpThreads) {
                const int j = e / 32, ss = e % 32;
                float v = 0.f;
                if (j < m && s0 + ss < g.S)
                    v = to_f32(Bm[((b * g.L + t0 + j0 + j) * g.G + grp) * g.S + s0 + ss]);
                sb[j][ss] = v;
            }
            __syncthreads();
            for (int j = 0; j < m; ++j) {
                const float bv = sb[j][lane];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    acc[k] = fmaf(sxw[j][warp + 8 * k], bv, acc[k]);
            }
        }
        const float decay = exp2f(glast);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            hs[k] = fmaf(decay, hs[k], acc[k]);
    }
    if (final_state) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t p = p0 + warp + 8 * k;
            if (s_ok && p < g.P)
                final_state[(bh * g.P + p) * g.S + s] = hs[k];
        }
    }
}

// ---------------------------------------------------------------- chunk output
// CTA = (chunk, 32-row query tile, batch*head), 256 threads.  The CB row
// block, the C h^T term and the output tile live in shared memory; dstate,
// keys and headdim are streamed in 64-wide tiles.
constexpr int kCoThreads = 256;
constexpr int kCoRows = 32;
constexpr int kCoTile = 64;

template <typename TI>
__global__ void __launch_bounds__(kCoThreads)
chunk_out_simt_kernel(const TI *__restrict__ x, const TI *__restrict__ Bm,
                      const TI *__restrict__ Cm, const float *__restrict__ dtT,
                      const float *__restrict__ Gc, const float *__restrict__ states,
                      const float *__restrict__ D, TI *__restrict__ y, Geom g)
{
    extern __shared__ float smem[];
    const int T = g.T;
    const int P = (int)g.P;
    float *scb = smem;                       // [kCoRows][T]   CB, then scores
    float *sy = scb + kCoRows * T;           // [kCoRows][P]   C h^T, then output
    float *sc = sy + kCoRows * P;            // [kCoRows][kCoTile]   C tile
    float *st = sc + kCoRows * kCoTile;      // [kCoTile][kCoTile+1] B / h / x tile
    float *sg = st + kCoTile * (kCoTile + 1);  // [T] G of the chunk
    float *sdt = sg + T;                     // [T] dt of the chunk
    constexpr int ldt = kCoTile + 1;

    const int64_t c = blockIdx.x, i0 = (int64_t)blockIdx.y * kCoRows;
    const int64_t bh = blockIdx.z, b = bh / g.H, h = bh % g.H, grp = h / g.hpg;
    const int64_t t0 = c * T;
    const int n = (int)min64(T, g.L - t0);
    if (i0 >= n)
        return;
    const int rows = (int)min64(kCoRows, n - i0);
    const int keys = (int)min64(n, i0 + rows);  // causal: keys < i0 + rows
    const int tid = threadIdx.x;

    for (int j = tid; j < T; j += kCoThreads) {
        sg[j] = j < n ? Gc[bh * g.L + t0 + j] : 0.f;
        sdt[j] = j < n ? dtT[bh * g.L + t0 + j] : 0.f;
    }
    for (int e = tid; e < kCoRows * T; e += kCoThreads)
        scb[e] = 0.f;
    for (int e = tid; e < kCoRows * P; e += kCoThreads)
        sy[e] = 0.f;
    __syncthreads();

    const float *hc = states + (bh * g.nc + c) * g.P * g.S;
    for (int64_t s0 = 0; s0 < g.S; s0 += kCoTile) {
        const int sw = (int)min64(kCoTile, g.S - s0);
        for (int e = tid; e < kCoRows * kCoTile; e += kCoThreads) {
            const int r = e / kCoTile, ss = e % kCoTile;
            float v = 0.f;
            if (r < rows && ss < sw)
                v = to_f32(Cm[((b * g.L + t0 + i0 + r) * g.G + grp) * g.S + s0 + ss]);
            sc[e] = v;
        }
        // CB[r][j] += sum_s C[r][s] B[j][s]
        for (int j0 = 0; j0 < keys; j0 += kCoTile) {
            const int kw = min(kCoTile, keys - j0);
            __syncthreads();
            for (int e = tid; e < kCoTile * kCoTile; e += kCoThreads) {
                const int j = e / kCoTile, ss = e % kCoTile;
                float v = 0.f;
                if (j < kw && ss < sw)
                    v = to_f32(Bm[((b * g.L + t0 + j0 + j) * g.G + grp) * g.S + s0 + ss]);
                st[j * ldt + ss] = v;
            }
            __syncthreads();
            for (int e = tid; e < kCoRows * kCoTile; e += kCoThreads) {
                const int r = e / kCoTile, j = e % kCoTile;
                if (r < rows && j < kw) {
                    float a = 0.f;
                    for (int ss = 0; ss < sw; ++ss)
                        a = fmaf(sc[r * kCoTile + ss], st[j * ldt + ss], a);
                    scb[r * T + j0 + j] += a;
                }
            }
        }
        // Ch[r][p] += sum_s C[r][s] h[p][s]
        for (int pb = 0; pb < P; pb += kCoTile) {
            const int pw = min(kCoTile, P - pb);
            __syncthreads();
            for (int e = tid; e < kCoTile * kCoTile; e += kCoThreads) {
                const int p = e / kCoTile, ss = e % kCoTile;
                float v = 0.f;
                if (p < pw && ss < sw)
                    v = hc[(int64_t)(pb + p) * g.S + s0 + ss];
                st[p * ldt + ss] = v;
            }
            __syncthreads();
            for (int e = tid; e < kCoRows * kCoTile; e += kCoThreads) {
                const int r = e / kCoTile, p = e % kCoTile;
                if (r < rows && p < pw) {
                    float a = 0.f;
                    for (int ss = 0; ss < sw; ++ss)
                        a = fmaf(sc[r * kCoTile + ss], st[p * ldt + ss], a);
                    sy[r * P + pb + p] += a;
                }
            }
        }
        __syncthreads();
    }

    // scores[r][j] = CB * exp2(G_i - G_j) * dt_j for j <= i, else 0; the
    // carried-state term is scaled by exp2(G_i).
    for (int e = tid; e < kCoRows * T; e += kCoThreads) {
        const int r = e / T, j = e % T;
        const int i = (int)i0 + r;
        float v = 0.f;
        if (r < rows && j <= i && j < n)
            v = scb[e] * exp2f(sg[i] - sg[j]) * sdt[j];
        scb[e] = v;
    }
    __syncthreads();
    for (int e = tid; e < kCoRows * P; e += kCoThreads) {
        const int r = e / P;
        if (r < rows)
            sy[e] *= exp2f(sg[i0 + r]);
    }
    // Y += scores X
    for (int j0 = 0; j0 < keys; j0 += kCoTile) {
        const int kw = min(kCoTile, keys - j0);
        for (int pb = 0; pb < P; pb += kCoTile) {
            const int pw = min(kCoTile, P - pb);
            __syncthreads();
            for (int e = tid; e < kCoTile * kCoTile; e += kCoThreads) {
                const int j = e / kCoTile, p = e % kCoTile;
                float v = 0.f;
                if (j < kw && p < pw)
                    v = to_f32(x[((b * g.L + t0 + j0 + j) * g.H + h) * g.P + pb + p]);
                st[j * ldt + p] = v;
            }
            __syncthreads();
            for (int e = tid; e < kCoRows * kCoTile; e += kCoThreads) {
                const int r = e / kCoTile, p = e % kCoTile;
                if (r < rows && p < pw) {
                    float a = 0.f;
                    for (int j = 0; j < kw; ++j)
                        a = fmaf(scb[r * T + j0 + j], st[j * ldt + p], a);
                    sy[r * P + pb + p] += a;
                }
            }
        }
    }
    __syncthreads();
    const float dh = D[h];
    for (int e = tid; e < kCoRows * P; e += kCoThreads) {
        const int r = e / P, p = e % P;
        if (r < rows) {
            const int64_t idx = ((b * g.L + t0 + i0 + r) * g.H + h) * g.P + p;
            y[idx] = from_f32<TI>(sy[e] + dh * to_f32(x[idx]));
        }
    }
}

}  // namespace

cudaError_t launch_state_pass_simt(const void *x, const void *Bm, const float *dtT,
                                   const float *Gc, const float *init, float *states,
                                   float *final_state, const Geom &g, bool bf16,
                                   cudaStream_t st)
{
    if (g.B == 0 || g.L == 0)
        return cudaSuccess;
    dim3 grid((unsigned)((g.S + 31) / 32), (unsigned)((g.P + 63) / 64), (unsigned)(g.B * g.H));
    if (bf16)
        state_pass_simt_kernel<__nv_bfloat16><<<grid, kSpThreads, 0, st>>>(
            (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)Bm, dtT, Gc, init, states,
            final_state, g);
    else
        state_pass_simt_kernel<float><<<grid, kSpThreads, 0, st>>>(
            (const float *)x, (const float *)Bm, dtT, Gc, init, states, final_state, g);
    note_launch();
    return cudaGetLastError();
}

static size_t chunk_out_simt_smem(const Geom &g)
{
    return sizeof(float) * ((size_t)kCoRows * g.T + (size_t)kCoRows * g.P +
                            (size_t)kCoRows * kCoTile + (size_t)kCoTile * (kCoTile + 1) +
                            2 * (size_t)g.T);
}

cudaError_t launch_chunk_out_simt(const void *x, const void *Bm, const void *Cm,
                                  const float *dtT, const float *Gc, const float *states,
                                  const float *D, void *y, const Geom &g, bool bf16,
                                  cudaStream_t st)
{
    if (g.B == 0 || g.L == 0)
        return cudaSuccess;
    const size_t smem = chunk_out_simt_smem(g);
    dim3 grid((unsigned)g.nc, (unsigned)((g.T + kCoRows - 1) / kCoRows), (unsigned)(g.B * g.H));
    cudaError_t e;
    if (bf16) {
        auto k = chunk_out_simt_kernel<__nv_bfloat16>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem)) != cudaSuccess)
            return e;
        k<<<grid, kCoThreads, smem, st>>>((const __nv_bfloat16 *)x, (const __nv_bfloat16 *)Bm,
                                          (const __nv_bfloat16 *)Cm, dtT, Gc, states, D,
                                          (__nv_bfloat16 *)y, g);
    } else {
        auto k = chunk_out_simt_kernel<float>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem)) != cudaSuccess)
            return e;
        k<<<grid, kCoThreads, smem, st>>>((const float *)x, (const float *)Bm,
                                          (const float *)Cm, dtT, Gc, states, D, (float *)y, g);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace ssd
