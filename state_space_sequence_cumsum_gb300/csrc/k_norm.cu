// Gated RMS norm: the gating and normalisation that follow the scan.
//
// "Accelerating Mamba-2 forward-pass kernels with CUDA Tile (cuTile)",
// operator-fusion section: after the scan come gating, normalisation and the
// output projection; fusing the element-wise / light steps keeps the
// intermediates on chip.  Here the gate and the norm are one pass (the
// projection is a plain GEMM):
//     g   = y * silu(z),   silu(z) = z / (1 + e^{-z})
//     out = g / sqrt(mean(g^2 over each group of gs channels) + eps) * w
// Rows of up to 32 x 4 16-byte vectors go to one warp each, which reads the
// row once, keeps g in registers and reduces sum g^2 with shuffles.  Rows of
// up to 24 KB (the 2.7B layer's 5120 bf16 channels: 10 KB) are streamed
// through shared memory by bulk copies, two rows in flight per CTA, so the
// HBM reads never wait for the arithmetic.  Other rows take a 256-thread
// register team, or a warp that sweeps the row twice.  HBM traffic is y and
// z read once and out written once (except in the last case).
#include "common.cuh"
#include "ssd_internal.h"
#include "tc05.cuh"

namespace ssd {
namespace {

constexpr int kNormThreads = 256;

template <typename TI, int VEC> struct Vec;
template <> struct Vec<__nv_bfloat16, 8> {
    using T = uint4;
    __device__ static void unpack(const uint4 &u, float (&v)[8])
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    }
    __device__ static uint4 pack(const float (&v)[8])
    {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
            w[k] = *reinterpret_cast<const uint32_t *>(&p);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct Vec<float, 4> {
    using T = float4;
    __device__ static void unpack(const float4 &u, float (&v)[4])
    {
        v[0] = u.x;
        v[1] = u.y;
        v[2] = u.z;
        v[3] = u.w;
    }
    __device__ static float4 pack(const float (&v)[4]) { return make_float4(v[0], v[1], v[2], v[3]); }
};
template <typename TI> struct Vec<TI, 1> {
    using T = TI;
    __device__ static void unpack(const TI &u, float (&v)[1]) { v[0] = to_f32(u); }
    __device__ static TI pack(const float (&v)[1]) { return from_f32<TI>(v[0]); }
};

// z / (1 + e^-z) with the fast exponential and division intrinsics (a few
// ulp each); for z < -88 e^-z overflows to inf and the quotient is -0.
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.f + __expf(-z)); }

template <typename TI, int VEC>
__global__ void __launch_bounds__(kNormThreads)
gated_rmsnorm_kernel(const TI *y, const TI *z, const float *__restrict__ w, TI *out, int64_t rows, int gs, int ngroups, float eps)
{
    using V = typename Vec<TI, VEC>::T;
    const int lane = threadIdx.x & 31;
    const int nv = gs / VEC;
    const int64_t warp0 = (int64_t)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (kNormThreads / 32);
    for (int64_t r = warp0; r < rows; r += nwarps) {
        const V *yr = reinterpret_cast<const V *>(y + r * gs);
        const V *zr = reinterpret_cast<const V *>(z + r * gs);
        float ss = 0.f;
        for (int v = lane; v < nv; v += 32) {
            float a[VEC], b[VEC];
            Vec<TI, VEC>::unpack(yr[v], a);
            Vec<TI, VEC>::unpack(zr[v], b);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float g = a[e] * silu(b[e]);
                ss = fmaf(g, g, ss);
            }
        }
        for (int o = 16; o > 0; o >>= 1)
            ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float scale = rsqrtf(ss / (float)gs + eps);
        const float *wr = w + (int)(r % ngroups) * gs;
        V *orow = reinterpret_cast<V *>(out + r * gs);
        for (int v = lane; v < nv; v += 32) {
            float a[VEC], b[VEC];
            Vec<TI, VEC>::unpack(yr[v], a);
            Vec<TI, VEC>::unpack(zr[v], b);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                a[e] = a[e] * silu(b[e]) * scale * wr[v * VEC + e];
            orow[v] = Vec<TI, VEC>::pack(a);
        }
    }
}

// TEAM threads per row, each holding at most 4 vectors of g.
template <typename TI, int VEC, int TEAM>
__global__ void __launch_bounds__(kNormThreads)
gated_rmsnorm_reg_kernel(const TI *y, const TI *z, const float *__restrict__ w, TI *out, int64_t rows, int gs, int ngroups, float eps)
{
    using V = typename Vec<TI, VEC>::T;
    constexpr int kMaxV = 4;
    constexpr int kTeams = kNormThreads / TEAM;
    __shared__ float part[kTeams][TEAM / 32 > 0 ? TEAM / 32 : 1];
    const int lane = threadIdx.x % TEAM, team = threadIdx.x / TEAM;
    const int nv = gs / VEC;
    for (int64_t r = (int64_t)blockIdx.x * kTeams + team; r - team < rows;
         r += (int64_t)gridDim.x * kTeams) {
        const bool live = r < rows;  // the whole CTA stays in the loop for the barriers
        float g[kMaxV][VEC];
        float ss = 0.f;
        if (live) {
            const V *yr = reinterpret_cast<const V *>(y + r * gs);
            const V *zr = reinterpret_cast<const V *>(z + r * gs);
#pragma unroll
            for (int k = 0; k < kMaxV; ++k) {
                const int v = lane + k * TEAM;
                if (v < nv) {
                    float a[VEC], b[VEC];
                    Vec<TI, VEC>::unpack(yr[v], a);
                    Vec<TI, VEC>::unpack(zr[v], b);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        g[k][e] = a[e] * silu(b[e]);
                        ss = fmaf(g[k][e], g[k][e], ss);
                    }
                }
            }
        }
        for (int o = 16; o > 0; o >>= 1)
            ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (TEAM > 32) {
            if ((threadIdx.x & 31) == 0)
                part[team][lane / 32] = ss;
            __syncthreads();
            ss = 0.f;
#pragma unroll
            for (int k = 0; k < TEAM / 32; ++k)
                ss += part[team][k];
            __syncthreads();
        }
        if (live) {
            const float scale = rsqrtf(ss / (float)gs + eps);
            const float *wr = w + (int)(r % ngroups) * gs;
            V *orow = reinterpret_cast<V *>(out + r * gs);
#pragma unroll
            for (int k = 0; k < kMaxV; ++k) {
                const int v = lane + k * TEAM;
                if (v < nv) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        g[k][e] *= scale * wr[v * VEC + e];
                    orow[v] = Vec<TI, VEC>::pack(g[k]);
                }
            }
        }
    }
}

// Rows streamed through shared memory: one CTA per row at a time, the next
// row's y and z in flight (bulk copies into a two-stage buffer) while the
// current row is reduced and written.  Thread 0 alone waits on the copy
// barrier (bounded) and the outcome is shared, so every thread leaves the
// loop together.
template <typename TI, int VEC>
__global__ void __launch_bounds__(kNormThreads)
gated_rmsnorm_stream_kernel(const TI *y, const TI *z, const float *__restrict__ w, TI *out,
                            int64_t rows, int gs, int ngroups, float eps, unsigned int *status)
{
    using V = typename Vec<TI, VEC>::T;
    extern __shared__ __align__(16) uint8_t sbuf[];
    __shared__ uint64_t full[2];
    __shared__ float part[kNormThreads / 32];
    __shared__ int s_ok;
    const int tid = threadIdx.x;
    const uint32_t rb = (uint32_t)gs * sizeof(TI);  // bytes of one row of y (or z)
    const int nv = gs / VEC;
    if (tid == 0) {
        tc::mbar_init(&full[0], 1);
        tc::mbar_init(&full[1], 1);
        tc::fence_barrier_init();
        s_ok = 1;
    }
    __syncthreads();
    auto issue = [&](int64_t k) {
        const int64_t r = blockIdx.x + k * gridDim.x;
        if (r >= rows)
            return;
        uint8_t *st = sbuf + (k & 1) * 2 * rb;
        tc::mbar_arrive_expect_tx(&full[k & 1], 2 * rb);
        tc::bulk_load(st, y + r * gs, rb, &full[k & 1]);
        tc::bulk_load(st + rb, z + r * gs, rb, &full[k & 1]);
    };
    if (tid == 0) {
        issue(0);
        issue(1);
    }
    for (int64_t k = 0;; ++k) {
        const int64_t r = blockIdx.x + k * gridDim.x;
        if (r >= rows)
            break;
        if (tid == 0 && !tc::mbar_wait(&full[k & 1], (uint32_t)((k >> 1) & 1))) {
            atomicOr(status, 1u);
            s_ok = 0;
        }
        __syncthreads();
        if (!s_ok)
            break;
        const V *ys = reinterpret_cast<const V *>(sbuf + (k & 1) * 2 * rb);
        const V *zs = reinterpret_cast<const V *>(sbuf + (k & 1) * 2 * rb + rb);
        // g of this thread's (at most four) vectors stays in registers
        float g[4][VEC];
        float ss = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int v = tid + q * kNormThreads;
            if (v < nv) {
                float a[VEC], b[VEC];
                Vec<TI, VEC>::unpack(ys[v], a);
                Vec<TI, VEC>::unpack(zs[v], b);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    g[q][e] = a[e] * silu(b[e]);
                    ss = fmaf(g[q][e], g[q][e], ss);
                }
            }
        }
        for (int o = 16; o > 0; o >>= 1)
            ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if ((tid & 31) == 0)
            part[tid >> 5] = ss;
        __syncthreads();
        ss = 0.f;
#pragma unroll
        for (int q = 0; q < kNormThreads / 32; ++q)
            ss += part[q];
        const float scale = rsqrtf(ss / (float)gs + eps);
        const float *wr = w + (int)(r % ngroups) * gs;
        V *orow = reinterpret_cast<V *>(out + r * gs);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int v = tid + q * kNormThreads;
            if (v < nv) {
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    g[q][e] *= scale * wr[v * VEC + e];
                orow[v] = Vec<TI, VEC>::pack(g[q]);
            }
        }
        __syncthreads();  // the stage and part[] are free again
        if (tid == 0)
            issue(k + 2);
    }
}

int sm_count_norm()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

template <typename TI, int VEC>
cudaError_t launch_norm_v(const void *y, const void *z, const float *w, void *out, int64_t rows, int gs,
                          int ngroups, float eps, cudaStream_t st)
{
    const int64_t cap = (int64_t)sm_count_norm() * (2048 / kNormThreads) * 4;
    const TI *yt = static_cast<const TI *>(y), *zt = static_cast<const TI *>(z);
    TI *ot = static_cast<TI *>(out);
    const int nv = gs / VEC;
    auto grid = [&](int teams_per_cta) {
        int64_t b = (rows + teams_per_cta - 1) / teams_per_cta;
        return (unsigned)(b > cap ? cap : b);
    };
    const size_t row_bytes = (size_t)gs * sizeof(TI);
    if (nv <= 32 * 4) {
        gated_rmsnorm_reg_kernel<TI, VEC, 32><<<grid(kNormThreads / 32), kNormThreads, 0, st>>>(
            yt, zt, w, ot, rows, gs, ngroups, eps);
    } else if (VEC > 1 && row_bytes % 16 == 0 && row_bytes <= 24 * 1024 && nv <= 4 * kNormThreads) {
        // y and z rows streamed through a two-stage shared buffer
        unsigned int *status = device_status_word();
        if (!status)
            return cudaErrorUnknown;
        const size_t smem = 4 * row_bytes;
        auto k = gated_rmsnorm_stream_kernel<TI, VEC>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        int per_sm = (int)((200 * 1024) / (smem + 1024));
        per_sm = per_sm < 1 ? 1 : (per_sm > 8 ? 8 : per_sm);
        int64_t b = (int64_t)sm_count_norm() * per_sm;
        if (b > rows)
            b = rows;
        k<<<(unsigned)b, kNormThreads, smem, st>>>(yt, zt, w, ot, rows, gs, ngroups, eps, status);
    } else if (nv <= kNormThreads * 4) {
        gated_rmsnorm_reg_kernel<TI, VEC, kNormThreads><<<grid(1), kNormThreads, 0, st>>>(
            yt, zt, w, ot, rows, gs, ngroups, eps);
    } else
        gated_rmsnorm_kernel<TI, VEC><<<grid(kNormThreads / 32), kNormThreads, 0, st>>>(
            yt, zt, w, ot, rows, gs, ngroups, eps);
    note_launch(1);
    return cudaGetLastError();
}

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_gated_rmsnorm(const void *y, const void *z, const float *w, void *out,
                                 int64_t ntokens, int64_t dim, int64_t gs, float eps, bool bf16,
                                 cudaStream_t st)
{
    const int64_t rows = ntokens * (dim / gs);
    if (rows == 0)
        return cudaSuccess;
    const int ng = (int)(dim / gs);
    const bool vec_ok = al16(y) && al16(z) && al16(out);
    if (bf16) {
        if (vec_ok && gs % 8 == 0)
            return launch_norm_v<__nv_bfloat16, 8>(y, z, w, out, rows, (int)gs, ng, eps, st);
        return launch_norm_v<__nv_bfloat16, 1>(y, z, w, out, rows, (int)gs, ng, eps, st);
    }
    if (vec_ok && gs % 4 == 0)
        return launch_norm_v<float, 4>(y, z, w, out, rows, (int)gs, ng, eps, st);
    return launch_norm_v<float, 1>(y, z, w, out, rows, (int)gs, ng, eps, st);
}

}  // namespace ssd
