// Stage 1: within-chunk cumulative decay in log2 units.
//
// "Accelerating Mamba-2 forward-pass kernels with CUDA Tile (cuTile)",
// section "Kernel 1": G[b,h,t] = log2(e) * cumsum_{t' in chunk, t' <= t} A[h] dt[b,t',h];
// the scan restarts at every chunk boundary.  Section "Mamba-2 性能优化" moves
// decay_cumsum and dt to a token-contiguous [batch, head, token] layout; this
// kernel writes both G and dt in that layout so the later stages read them
// with contiguous (TMA-able) loads.
//
// One CTA per (chunk, 32-head tile, batch row).  The [T x 32] slice of dt is
// read row by row (128-byte coalesced rows along heads) into shared memory,
// transposed through it, and each warp scans one head at a time: every lane
// sums ceil(T/32) consecutive tokens serially, the lane totals are combined
// with a warp-shuffle inclusive scan, and each lane writes its run of tokens
// contiguously.
#include "common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kHeadsPerCta = 32;
constexpr int kThreads = 256;
constexpr int kMaxPerLane = 8;  // T <= 256

__global__ void __launch_bounds__(kThreads)
chunk_cumsum_kernel(const float *__restrict__ dt, const float *__restrict__ A,
                    float *__restrict__ Gc, float *__restrict__ dtT, int64_t L, int H, int T)
{
    extern __shared__ float tile[];  // [T][kHeadsPerCta + 1]
    constexpr int ld = kHeadsPerCta + 1;
    const int c = blockIdx.x, h0 = blockIdx.y * kHeadsPerCta, b = blockIdx.z;
    const int64_t t0 = (int64_t)c * T;
    const int n = (int)min64(T, L - t0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int h = h0 + lane;

    // [T x 32] slice of dt, one 128-byte row per warp instruction; the loads
    // of a thread are independent, so they are all in flight together
    const float *src = dt + ((int64_t)b * L + t0) * H + h;
#pragma unroll 8
    for (int r = warp; r < T; r += kThreads / 32)
        tile[r * ld + lane] = (r < n && h < H) ? src[(int64_t)r * H] : 0.f;  // zero padding
    __syncthreads();

    const int per = (T + 31) / 32;
    for (int hl = warp; hl < kHeadsPerCta; hl += kThreads / 32) {
        const int hh = h0 + hl;
        if (hh >= H)
            break;
        float *drow = dtT ? dtT + ((int64_t)b * H + hh) * L + t0 : nullptr;
        float *grow = Gc + ((int64_t)b * H + hh) * L + t0;
        // dt transposed: consecutive lanes write consecutive tokens
        if (drow)
            for (int t = lane; t < n; t += 32)
                drow[t] = tile[t * ld + hl];
        // lane-serial partial sums over `per` consecutive tokens, then a
        // warp-shuffle scan of the lane totals
        const float a = A[hh];
        float run = 0.f, vals[kMaxPerLane];
#pragma unroll
        for (int k = 0; k < kMaxPerLane; ++k) {
            const int t = lane * per + k;
            float v = 0.f;
            if (k < per && t < T)
                v = a * tile[t * ld + hl];
            run += v;
            vals[k] = run;
        }
        float incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off)
                incl += o;
        }
        const float excl = incl - run;
        __syncwarp();
#pragma unroll
        for (int k = 0; k < kMaxPerLane; ++k) {
            const int t = lane * per + k;
            if (k < per && t < T)
                tile[t * ld + hl] = (excl + vals[k]) * kLog2e;  // this warp's column only
        }
        __syncwarp();
        for (int t = lane; t < n; t += 32)
            grow[t] = tile[t * ld + hl];
    }
}

}  // namespace

cudaError_t launch_chunk_cumsum(const float *dt, const float *A, float *Gc, float *dtT,
                                const Geom &g, cudaStream_t st)
{
    if (g.L == 0 || g.B == 0)
        return cudaSuccess;
    const size_t smem = sizeof(float) * (size_t)g.T * (kHeadsPerCta + 1);
    dim3 grid((unsigned)g.nc, (unsigned)((g.H + kHeadsPerCta - 1) / kHeadsPerCta),
              (unsigned)g.B);
    chunk_cumsum_kernel<<<grid, kThreads, smem, st>>>(dt, A, Gc, dtT, g.L, (int)g.H, g.T);
    note_launch();
    return cudaGetLastError();
}

}  // namespace ssd
