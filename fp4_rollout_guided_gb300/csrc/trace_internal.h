// trace_internal.h - launch interface between the C ABI (trace_api.cu) and
// the sm_103a kernels (trace_kernels.cu, trace_fakequant.cu).  Not part of the
// public ABI.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "trace_fp4.h"

namespace tfp4 {

// Segment table as a kernel parameter: row offsets narrowed to int32 (rows
// are validated to fit), passed by value in the parameter bank so that calls
// need no device copy of the table and stay stream-ordered by construction.
struct SegParam {
  int32_t n;
  int32_t off[TRACE_MAX_SEGMENTS + 1];
};

// Waves of the fused amax + quantisation kernel: wave w holds the whole
// segments [seg0[w], seg0[w+1]); seg0[n] is the segment count.
struct WaveParam {
  int32_t n;
  uint16_t seg0[TRACE_MAX_SEGMENTS + 1];
};
static_assert(TRACE_MAX_SEGMENTS < 65536, "wave table holds 16-bit segment indices");

// Unsigned division by a runtime constant (chunk index -> row) without a
// hardware divide: q = (mulhi(n, mul) + n) >> shift with shift = ceil(log2 d)
// and mul = floor(2^32 * (2^shift - d) / d) + 1, exact for every 32-bit n.
struct FastDivU {
  uint32_t mul, shift, d;
  explicit FastDivU(uint32_t d_) : d(d_) {
    uint32_t l = 0;
    const uint32_t d = d_;
    while ((1ull << l) < d) ++l;
    shift = l;
    mul = (uint32_t)((((1ull << 32) * ((1ull << l) - d)) / d) + 1);
  }
  __host__ __device__ __forceinline__ uint32_t div(uint32_t n) const {
#ifdef __CUDA_ARCH__
    const uint32_t t = __umulhi(n, mul);
#else
    const uint32_t t = (uint32_t)(((uint64_t)n * mul) >> 32);
#endif
    return (uint32_t)(((uint64_t)t + n) >> shift);
  }
};

// Debug builds (TRACE_DEBUG_BOUNDS): the byte ranges of global memory the
// next launches on a stream may touch.  Each API call registers its buffers
// and its scratch before it launches (stream-ordered); the kernels' memory
// helpers check every access against the table, count one that falls
// outside, and skip it.  Release builds register nothing and check nothing.
constexpr int kDbgRanges = 24;
struct DbgRanges {
  uint32_t n;
  uint64_t lo[kDbgRanges];
  uint64_t hi[kDbgRanges];
};
// Register the ranges in every translation unit's table (on st); read and
// clear the accesses counted outside the ranges since the last call.
cudaError_t dbg_set_ranges(const DbgRanges& r, cudaStream_t st);
unsigned long long dbg_take_violations();
// per translation unit
cudaError_t dbg_set_ranges_kernels(const DbgRanges& r, cudaStream_t st);
unsigned long long dbg_take_kernels();
cudaError_t dbg_set_ranges_fakequant(const DbgRanges& r, cudaStream_t st);
unsigned long long dbg_take_fakequant();

// Device scratch owned by a handle.  amax_bits holds per-segment maxima as
// binary32 bit patterns (non-negative floats order like unsigned integers);
// the amax kernel's last CTA converts them to global scales and re-zeroes
// them, so the array is all-zero between calls.
struct Scratch {
  uint32_t* amax_bits;  // [TRACE_MAX_SEGMENTS]
  uint32_t* done;       // completion ticket of the amax kernel
  float* gs_train;      // [TRACE_MAX_SEGMENTS] training-side global scales
  uint32_t* wave_cnt;   // [TRACE_MAX_SEGMENTS] fused kernel: CTAs done with a wave's amax
  uint32_t* err;        // fused kernel: nonzero once an in-kernel wait ran out
};

// a1: per-segment amax of x, then gs[s] = amax/2688 written to gs_out.
cudaError_t launch_amax(const void* x, int64_t nchunks, int32_t cpr, const SegParam& seg,
                        const Scratch& s, float* gs_out, int sm_count, cudaStream_t st);

// Block scales in the tensor-core tile layout, written by the rollout
// quantiser next to (or instead of) the row-major ones: 512-byte tiles of
// 128 rows x 4 scale columns, tiles_per_row tiles along a row band.
struct MmaOut {
  uint8_t* p;  // null: not written
  uint32_t tiles_per_row;
};

// a2: RTN codes, block scales (row-major and/or tile layout; either may be
// null), compact words (guide may be null).
cudaError_t launch_rollout_quant(const void* x, int64_t nchunks, int32_t cpr,
                                 const SegParam& seg, const float* gs, void* codes, void* bs,
                                 MmaOut mma, uint32_t* guide, int sm_count, cudaStream_t st);

// gs[s] = amax[s] / 2688 from given maxima (delayed scaling).
cudaError_t launch_scales_from_amax(const float* amax, int32_t n, float* gs, cudaStream_t st);

// a2 with the global scales from given maxima (gs = amax_in / 2688, written
// to gs) instead of this tensor's; amax_out (zeroed by the caller, may be
// null) receives this tensor's segment maxima for a later call.
cudaError_t launch_rollout_quant_delayed(const void* x, int64_t nchunks, int32_t cpr,
                                         const SegParam& seg, const float* amax_in, float* gs,
                                         void* codes, void* bs, MmaOut mma, uint32_t* guide,
                                         float* amax_out, int sm_count, cudaStream_t st);

// a1 + a2 in one cooperative launch (see k_rollout_fused).  plan_waves
// groups whole segments into waves of about wave_bytes of x; it returns
// false when a segment is too large to stay in L2 between the two phases.
bool plan_waves(const SegParam& seg, int32_t cols, int64_t wave_bytes, WaveParam* wv);
cudaError_t launch_rollout_fused(const void* x, int64_t nchunks, int32_t cpr, const SegParam& seg,
                                 const WaveParam& wv, const Scratch& s, float* gs_out,
                                 void* codes, void* bs, MmaOut mma, uint32_t* guide, int sm_count,
                                 uint32_t wait_extra, uint64_t wait_ns, cudaStream_t st);

// a3: codes -> compact words.
cudaError_t launch_guide_pack(const void* codes, int64_t nchunks, uint32_t* guide,
                              int sm_count, cudaStream_t st);

// a4: compact words + reference values -> codes.
cudaError_t launch_guide_unpack(const void* x_ref, const uint32_t* guide, const void* bs_r,
                                const float* gs_r, int64_t nchunks, int32_t cpr,
                                const SegParam& seg_r, void* codes, int sm_count,
                                cudaStream_t st);

// backward: straight-through gradient through the fake quantiser.
cudaError_t launch_ste_backward(const void* g, const uint32_t* mask, int64_t nchunks, void* out,
                                int sm_count, cudaStream_t st);

// a5 + a6: training-side guided fake quantisation.
struct FakequantArgs {
  const void* x;
  int64_t nchunks;
  int32_t cpr;
  const float* gs_t;  // per training segment
  int kind;
  const void* guide;
  const void* bs_r;
  const float* gs_r;
  void* y;
  uint32_t* mask;
  void* codes_t;
  trace_stats_t* stats;
  uint32_t* amax_out = nullptr;  // delayed scaling: the training maxima (y and mask only)
};
cudaError_t launch_fakequant(const FakequantArgs& a, const SegParam& seg_t,
                             const SegParam& seg_r, int sm_count, cudaStream_t st);

// f4: block scales in the tensor-core tile layout, and the NVFP4 GEMM
// through cuBLASLt (trace_gemm.cu).
int64_t mma_scales_bytes(int64_t rows, int64_t cols);
cudaError_t launch_mma_scales(const void* bs, int64_t rows, int64_t cols, void* out, int sm_count,
                              cudaStream_t st);
cudaError_t launch_gemm_scalars(const float* gs_a, const float* gs_b, float* out,
                                cudaStream_t st);
// The hand-written tcgen05 form (trace_gemm_tc.cu): output tiles of
// 128 x 256, 128 x 128, or 256 x 256 on an SM pair; a wait that runs out
// sets *err.
enum { kGemmTile256 = 0, kGemmTile128 = 1, kGemmTilePair = 2 };
cudaError_t launch_nvfp4_gemm_tc(const void* a_codes, const void* a_sf, const float* a_gs,
                                 const void* b_codes, const void* b_sf, const float* b_gs,
                                 int64_t m, int64_t n, int64_t k, void* d, int d_bf16,
                                 int tile, uint32_t* err, uint64_t wait_ns, int sm_count,
                                 cudaStream_t st);
// The driver's tensor-map encoder (null if the driver lacks it).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
bool lt_available();
void lt_destroy(void* lt);
// 0 on success, -1 if cuBLASLt cannot be loaded, else a cublasStatus_t.
int lt_nvfp4_gemm(void** lt, void* workspace, size_t ws_bytes, const void* a_codes,
                  const void* a_scales, const void* b_codes, const void* b_scales,
                  const float* alpha_beta, int64_t m, int64_t n, int64_t k, void* d, int d_bf16,
                  cudaStream_t st);

}  // namespace tfp4
