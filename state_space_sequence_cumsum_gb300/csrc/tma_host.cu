// Host-side TMA tensor-map encoding.  cuTensorMapEncodeTiled is a driver
// entry point; it is fetched through the runtime so the library does not
// link libcuda (loading it needs no GPU).
#include <cudaTypedefs.h>
#include <mutex>

#include "ssd_internal.h"

namespace ssd {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
}  // namespace

namespace {
bool encode(CUtensorMap *map, CUtensorMapDataType type, const void *base, int rank,
            const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
            CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo)
{
    std::call_once(g_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode)
        return false;
    cuuint64_t gdim[5];
    cuuint64_t gstride[4];
    cuuint32_t bdim[5], estride[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estride[i] = 1;
        if (i + 1 < rank)
            gstride[i] = strides_bytes[i];
    }
    CUresult r = g_encode(map, type, (cuuint32_t)rank, const_cast<void *>(base), gdim, gstride,
                          bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
}  // namespace

bool make_tmap_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                    const uint64_t *strides_bytes, const uint32_t *box)
{
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides_bytes, box,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// f32 matrix [rows, cols] with a row pitch of cols * 4 bytes; box {box_cols,
// box_rows}, unswizzled (shared memory holds the box row-major).
bool make_tmap_f32_rows(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
                        uint32_t box_cols, uint32_t box_rows)
{
    const uint64_t dims[2] = {cols, rows};
    const uint64_t st[1] = {cols * 4};
    const uint32_t box[2] = {box_cols, box_rows};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, 2, dims, st, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

// x, y [B, L, H, P] viewed as 4-D {P, H, L, B}; box {64, 1, 128, 1}.
bool make_tmap_tokens_heads(CUtensorMap *map, const void *base, const Geom &g)
{
    const uint64_t dims[4] = {(uint64_t)g.P, (uint64_t)g.H, (uint64_t)g.L, (uint64_t)g.B};
    const uint64_t st[3] = {(uint64_t)g.P * 2, (uint64_t)(g.H * g.P) * 2,
                            (uint64_t)(g.L * g.H * g.P) * 2};
    const uint32_t box[4] = {64, 1, 128, 1};
    return make_tmap_bf16(map, base, 4, dims, st, box);
}

// B, C [B, L, G, S] viewed as 4-D {S, G, L, B}; box {64, 1, 128, 1}.
bool make_tmap_tokens_groups(CUtensorMap *map, const void *base, const Geom &g)
{
    const uint64_t dims[4] = {(uint64_t)g.S, (uint64_t)g.G, (uint64_t)g.L, (uint64_t)g.B};
    const uint64_t st[3] = {(uint64_t)g.S * 2, (uint64_t)(g.G * g.S) * 2,
                            (uint64_t)(g.L * g.G * g.S) * 2};
    const uint32_t box[4] = {64, 1, 128, 1};
    return make_tmap_bf16(map, base, 4, dims, st, box);
}

// f32 [B, L, G, S] (the dB / dC accumulators) viewed as 4-D {S, G, L, B};
// box {32, 1, 128, 1}: 128 token rows of 32 f32 (128 bytes), 128-byte swizzle.
bool make_tmap_f32_tokens_groups(CUtensorMap *map, const void *base, const Geom &g)
{
    const uint64_t dims[4] = {(uint64_t)g.S, (uint64_t)g.G, (uint64_t)g.L, (uint64_t)g.B};
    const uint64_t st[3] = {(uint64_t)g.S * 4, (uint64_t)(g.G * g.S) * 4,
                            (uint64_t)(g.L * g.G * g.S) * 4};
    const uint32_t box[4] = {32, 1, 128, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, 4, dims, st, box,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

}  // namespace ssd
