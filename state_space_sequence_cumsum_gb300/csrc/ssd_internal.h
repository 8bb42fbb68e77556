// Host-side declarations shared by the library's translation units.
// Not part of the public ABI (include/ssd.h is).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/ssd.h"

namespace ssd {

// Problem geometry after validation.  hpg = heads per B/C group.
struct Geom {
    int64_t B, L, H, P, S, G;
    int T;
    int64_t nc;
    int hpg;
};

// Kernel-side error word (bit 0: a bounded wait ran out).  Returns its
// device address for the current device, or nullptr on failure.
unsigned int *device_status_word();

// Counts kernel launches (ssd_launch_count); every launcher calls it once per
// kernel it enqueues.
void note_launch(unsigned n = 1);

// Stage launchers (one translation unit each).
cudaError_t launch_chunk_cumsum(const float *dt, const float *A, float *Gc, float *dtT,
                                const Geom &g, cudaStream_t st);

// CUDA-core kernels with f32 arithmetic; serve every shape and both dtypes.
cudaError_t launch_state_pass_simt(const void *x, const void *Bm, const float *dtT,
                                   const float *Gc, const float *init, float *states,
                                   float *final_state, const Geom &g, bool bf16,
                                   cudaStream_t st);
cudaError_t launch_chunk_out_simt(const void *x, const void *Bm, const void *Cm,
                                  const float *dtT, const float *Gc, const float *states,
                                  const float *D, void *y, const Geom &g, bool bf16,
                                  cudaStream_t st);

// TMA tensor maps (bf16, 128-byte swizzle, zero fill out of bounds).
bool make_tmap_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                    const uint64_t *strides_bytes, const uint32_t *box);
bool make_tmap_f32_rows(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
                        uint32_t box_cols, uint32_t box_rows);
bool make_tmap_tokens_heads(CUtensorMap *map, const void *base, const Geom &g);
bool make_tmap_f32_tokens_groups(CUtensorMap *map, const void *base, const Geom &g);
bool make_tmap_tokens_groups(CUtensorMap *map, const void *base, const Geom &g);

// Tensor-core (tcgen05) state pass; bf16 inputs.  Returns cudaErrorNotSupported
// for shapes it does not serve (the caller then uses the CUDA-core kernel).
bool state_pass_tc_supported(const Geom &g);
cudaError_t launch_state_pass_tc(const void *x, const void *Bm, const float *dtT,
                                 const float *Gc, const float *init, float *states,
                                 float *final_state, const Geom &g, cudaStream_t st);
// The same pass split into segments of the sequence run in parallel (end
// states from zero, a serial combine, then the segments again from their true
// start states), for long sequences with few (batch, head) units; needs the
// chunk-state array.  cudaErrorNotSupported: too few tiles to split.
void state_pass_seg_plan(const Geom &g, int sms, int *seg_tiles, int *n_seg);
cudaError_t launch_segment_starts_tc(const void *x, const void *Bm, const float *dtT,
                                     const float *Gc, const float *init, float *slots,
                                     int seg_tiles, int n_seg, const Geom &g, cudaStream_t st);
cudaError_t launch_state_pass_tc_segmented(const void *x, const void *Bm, const float *dtT,
                                           const float *Gc, const float *init, float *states,
                                           float *final_state, const Geom &g, cudaStream_t st);

// Tensor-core chunk output (stage 3) and fused single-pass forward (bf16).
bool chunk_tc_supported(const Geom &g);
// the fused one-head forward: chunk_tc_supported shapes, and dstate 384 / 512
// (B / C streamed in 128-row dstate blocks)
bool fused_tc_supported(const Geom &g);
cudaError_t launch_chunk_out_tc(const void *x, const void *Bm, const void *Cm, const float *dtT,
                                const float *Gc, const float *states, const float *D, void *y,
                                const Geom &g, cudaStream_t st);
// Tensor-core chunk output for dstate 384 / 512 (bf16, P = 64, chunk 128),
// streaming B / C in 128-wide dstate blocks.
bool chunk_out_big_supported(const Geom &g);
// Reverse state pass of the backward on tensor cores (k_state_pass_tc.cu):
// bf16, P in {64, 128}, S % 64 == 0, 128-token chunks.
bool reverse_state_pass_tc_supported(const Geom &g);
cudaError_t launch_reverse_state_pass_tc(const void *dy, const void *Cm, const float *Gc,
                                         const float *dfinal, float *dstates, float *dinit,
                                         const Geom &g, cudaStream_t st);
// Chunk gradients of the backward on tensor cores (k_bwd_tc.cu): bf16,
// P == 64, S in {64, 128}, 128-token chunks; states / dstates / Gc / dtT per
// 128-token chunk; dBacc / dCacc / dA / dD zeroed f32 accumulators.
bool bwd_tc_supported(const Geom &g);
cudaError_t launch_bwd_chunk_tc(const void *x, const void *Bm, const void *Cm, const void *dy,
                                const float *dtT, const float *Gc, const float *A, const float *D,
                                const float *states, const float *dstates, void *dx, float *ddt,
                                float *dA, float *dD, float *dBacc, float *dCacc, const Geom &g,
                                cudaStream_t st);
cudaError_t launch_convert_f32(const float *src, void *dst, int64_t n, bool bf16, cudaStream_t st);
// Backward pass (k_bwd.cu): 64-token chunks, P <= 64.  states / dstates /
// Gc / dtT are per 64-token chunk; dBacc / dCacc are zeroed f32 [B,L,G,S]
// accumulators; dA / dD are zeroed f32 [H] accumulators.
bool bwd_supported(const Geom &g);
int bwd_chunk_size();
cudaError_t launch_bwd(const void *x, const void *Bm, const void *Cm, const void *dy,
                       const float *dtT, const float *Gc, const float *A, const float *D,
                       const float *states, const float *dfinal, float *dstates, void *dx,
                       float *ddt, float *dA, float *dD, float *dBacc, float *dCacc, void *dB,
                       void *dC, float *dinit, const Geom &g, bool bf16, cudaStream_t st);
// Gated RMS norm (k_norm.cu): rows of group_size channels, ntokens * dim / gs rows.
cudaError_t launch_gated_rmsnorm(const void *y, const void *z, const float *w, void *out,
                                 int64_t ntokens, int64_t dim, int64_t gs, float eps, bool bf16,
                                 cudaStream_t st);
// Single-token decode step (k_decode.cu); state_in may equal state_out.
cudaError_t launch_decode_step(const void *x, const float *dt, const float *A, const void *Bm,
                               const void *Cm, const float *D, const float *state_in, float *state_out,
                               void *y, const Geom &g, bool bf16, cudaStream_t st);
cudaError_t launch_chunk_out_big(const void *x, const void *Bm, const void *Cm, const float *dtT,
                                 const float *Gc, const float *states, const float *D, void *y,
                                 const Geom &g, cudaStream_t st);

// Scratch the one-head fused pass needs (segment hand-off states and
// counters), 0 if none.
size_t fused_tc_scratch_bytes(const Geom &g);
cudaError_t launch_fused_tc(const void *x, const void *Bm, const void *Cm, const float *dtT,
                            const float *Gc, const float *D, const float *init, float *states,
                            float *final_state, void *y, const Geom &g, void *scratch,
                            size_t scratch_bytes, cudaStream_t st);

// Fused forward for two heads of one B/C group per CTA (bf16, P = 64,
// S in {64, 128}, an even number of heads per group), straight from dt and A
// (it forms G itself).  ssd_fwd uses it where it applies unless
// SSD_FUSED_KERNEL=single asks for the cumsum + one-head fused pair.
bool pair_tc_supported(const Geom &g);
bool fused_pair_enabled(const Geom &g);
// The least workspace ssd_fwd runs with for these arguments (its own
// ssd_fwd_workspace_size reports the preferred size; the head-pair kernel
// also runs with the smaller hand-off plan's).  0: invalid arguments.
size_t fwd_workspace_min_size(ssd_dims_t dims, ssd_dtype_t dtype, int chunk_size,
                              int want_chunk_states);
// The chunk size ssd_fwd(chunk_size = 0) would use now, without fixing the
// choice (the cached one, else the static rule); 0 for invalid arguments.
int chunk_size_peek(ssd_dims_t dims, ssd_dtype_t dtype);
// Scratch of the head-pair kernel: with allow_prefill, that of the plan it
// prefers (the prefilled segments where they apply, which also hold G and
// dt^T); without, that of the hand-off plan, the least it runs with.
size_t pair_tc_scratch_bytes(const Geom &g, bool allow_prefill = true);
// True when the head-pair kernel would run the prefilled-segment plan for g.
bool pair_tc_prefers_prefill(const Geom &g);
// allow_prefill = false keeps the hand-off plan even where the prefilled one
// applies and fits (the chunk-size tuner times both).
cudaError_t launch_fused_pair_tc(const void *x, const void *Bm, const void *Cm, const float *dt,
                                 const float *A, const float *D, const float *init, float *states,
                                 float *final_state, void *y, const Geom &g, void *scratch,
                                 size_t scratch_bytes, cudaStream_t st, bool allow_prefill = true);

}  // namespace ssd
