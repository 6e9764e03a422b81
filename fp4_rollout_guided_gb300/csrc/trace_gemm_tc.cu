// trace_gemm_tc.cu - the NVFP4 GEMM over rollout codes on the fifth-
// generation tensor cores: block-scaled E2M1 x E2M1 products with UE4M3 block
// scales (one per 16 elements along k), FP32 accumulation in tensor memory.
//
// Source: "Alibaba Qwen Proposes TRACE for 5.4x Faster FP4 RL Rollouts",
// section "TRACE Core Concept": rollout runs weights and activations in
// NVFP4, so the rollout codes and their block scales are the operands of its
// GEMMs.  The operand, scale and descriptor formats are NVIDIA's documented
// interfaces (PTX ISA, tcgen05 shared-memory and instruction descriptors and
// block scaling; cuBLAS, "1D block scaling factors layout").
//
// d [m, n] = fl32(gs_a * gs_b) * sum_k A[i, k] B[j, k], A and B as codes
// [rows, k/2] (element 2i in the low nibble: the packed E2M1 operand format)
// and block scales in the 512-byte tile layout the rollout quantiser writes.
//
// One CTA per output tile of 128 x BN, one CTA per SM (its shared memory
// allows no second), 192 threads in three roles:
//   - warp 0 (one lane): producer.  Per k-block of 256 elements it loads the
//     A tile (128 rows x 128 bytes) and the B tile (BN rows x 128 bytes) with
//     2-D tensor-map copies in 128-byte swizzle, and the block-scale tiles
//     (512 bytes per 128 rows and 64 elements of k) with bulk copies, into a
//     ring of stages completing on mbarriers;
//   - warp 1: allocates the tensor memory; one lane copies each stage's scale
//     tiles into tensor memory (tcgen05.cp, 32 lines x 128 bits to all four
//     lane quarters) and issues the block-scaled MMAs (128 x BN x 64 each),
//     then commits the stage back to the producer;
//   - warps 2-5: epilogue.  Once the last MMA has completed each thread reads
//     its accumulator row from tensor memory (its warp's lane quarter),
//     multiplies by fl32(gs_a * gs_b) and stores fp32 or bf16.
// Rows and columns past m, n and k are zero-filled by the tensor-map copies
// (zero codes contribute nothing whatever their scales); scale tiles past the
// end of a scale tensor are not read, and only the output rows and columns
// inside d are stored.
//
// Tensor memory (512 columns of 32-bit lanes): the accumulator in columns
// [0, BN); per stage, the A scales of its four k-steps (four columns each) and
// the B scales (BN / 32 columns per k-step).  In a 512-byte scale tile, line
// L holds rows L, L + 32, L + 64, L + 96; copied to lane L of every quarter,
// column c of lane L holds the four scales of row L + 32 c for the k-step.
//
// Every wait is bounded (wait_ns): one that runs out sets *err, the role
// stops issuing, the producer still waits (bounded) for its own copies in
// flight, and the tensor memory is freed before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "trace_async.cuh"
#include "trace_internal.h"

namespace tfp4 {
namespace {

constexpr int kGemmThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBK = 256;            // k elements per stage (128 bytes of codes a row)
constexpr uint32_t kSfTile = 512;        // bytes of one scale tile: 128 rows x 64 k
constexpr uint32_t kStepsPerStage = 4;   // 64-element MMA k-steps per stage

template <int BN>
struct GemmShape {
  static constexpr uint32_t kABytes = 128u * kBK / 2;
  static constexpr uint32_t kBBytes = (uint32_t)BN * kBK / 2;
  static constexpr uint32_t kBands = (uint32_t)BN / 128;  // 128-row scale bands of a B tile
  static constexpr uint32_t kSfaBytes = kStepsPerStage * kSfTile;
  static constexpr uint32_t kSfbBytes = kBands * kStepsPerStage * kSfTile;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr uint32_t kStages = BN == 256 ? 4 : 6;
  static constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024;  // + alignment slack
  // tensor-memory columns
  static constexpr uint32_t kSfaCols = 4;                 // per k-step
  static constexpr uint32_t kSfbCols = (uint32_t)BN / 32; // per k-step
  static constexpr uint32_t kSfaBase = BN;
  static constexpr uint32_t kSfbBase = kSfaBase + kStages * kStepsPerStage * kSfaCols;
  static constexpr uint32_t kColsUsed = kSfbBase + kStages * kStepsPerStage * kSfbCols;
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned (128-byte swizzle)");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory of one CTA");
  static_assert(kColsUsed <= kTmemCols, "tensor-memory columns");
};

// ---- tcgen05 ----------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_addr(dst_smem)), "r"(cols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: start address, leading- and stride-
// dimension byte offsets (all in 16-byte units), the fixed version field
// (bits 46-48 = 0b001) and the swizzle mode (bits 61-63).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}

// K-major operand tile staged by a 128-byte-swizzled tensor-map copy: rows
// of 128 bytes, 8-row swizzle atoms 1024 bytes apart (mode 2 = 128-byte
// swizzle; the leading offset is unused for this layout).
__device__ __forceinline__ uint64_t operand_desc(uint32_t saddr) {
  return smem_desc(saddr, 16, 1024, 2);
}

// One 512-byte scale tile: 32 lines of 16 bytes, no swizzle, 8-line groups
// 128 bytes apart (a single 16-byte column, so no leading offset).
__device__ __forceinline__ uint64_t scale_desc(uint32_t saddr) {
  return smem_desc(saddr, 0, 128, 0);
}

// Instruction descriptor of the block-scaled MMA: A and B E2M1 (format 1 of
// the FP4 kinds, bits 7-9 and 10-11), both K-major, no negation, dense,
// UE4M3 scales (bit 23 = 0), scale-factor ids 0, N / 8 at bits 17-22,
// M / 16 at bits 24-28.
__host__ __device__ constexpr uint32_t mma_idesc(uint32_t m, uint32_t n) {
  return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// 32 lines x 128 bits of shared memory into four columns of tensor memory,
// the same lines in each of the four lane quarters.
__device__ __forceinline__ void tmem_copy_scales(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// d (tensor memory) (+)= A B^T over one 64-element k-step, A and B scaled
// per 16-element block by the UE4M3 scales in tensor memory at sfa / sfb.
__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
      "r"(accumulate)
      : "memory");
}

// Arrive on bar once every tcgen05 operation this thread issued so far has
// completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_addr(bar))
               : "memory");
}

// 32 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
      " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
      " [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
        "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
        "=r"(v[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- the kernel ---------------------------------------------------------------

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_nvfp4_gemm(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                 const uint8_t* __restrict__ sfa, const uint8_t* __restrict__ sfb,
                 const float* __restrict__ gs_a, const float* __restrict__ gs_b, uint32_t m,
                 uint32_t n, uint32_t k, void* __restrict__ d, uint32_t d_bf16,
                 uint32_t* __restrict__ err, uint64_t wait_ns) {
  using S = GemmShape<BN>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[S::kStages], empty[S::kStages], acc_full;
  __shared__ uint32_t tmem_base;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~uintptr_t(1023));

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  const uint32_t m0 = blockIdx.y * 128u, n0 = blockIdx.x * (uint32_t)BN;
  const uint32_t nkb = (k + kBK - 1) / kBK;
  const uint32_t tiles_per_row = (k + 63) / 64;  // scale tiles along k (64 elements each)

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < S::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&acc_full, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0 && lane == 0) {
    // ---- producer ----
    const uint32_t band_a = m0 / 128u, band_b0 = n0 / 128u;
    const uint32_t bands_b = (n + 127u) / 128u;
    uint32_t kb = 0;
    for (; kb < nkb; ++kb) {
      const uint32_t s = kb % S::kStages, ph = (kb / S::kStages) & 1u;
      if (!mbar_wait(&empty[s], ph ^ 1u, wait_ns, err)) break;
      uint8_t* st = smem + s * S::kStageBytes;
      const uint32_t steps = min(kStepsPerStage, tiles_per_row - kStepsPerStage * kb);
      uint32_t nb = 0;
      for (uint32_t b = 0; b < S::kBands; ++b) nb += band_b0 + b < bands_b ? 1u : 0u;
      mbar_expect_tx(&full[s], S::kABytes + S::kBBytes + (1u + nb) * steps * kSfTile);
      tensor_load_2d(st, &map_a, kb * (kBK / 2), m0, &full[s]);
      tensor_load_2d(st + S::kABytes, &map_b, kb * (kBK / 2), n0, &full[s]);
      const uint64_t tile0 = kStepsPerStage * kb;
      bulk_load(st + S::kABytes + S::kBBytes,
                sfa + ((uint64_t)band_a * tiles_per_row + tile0) * kSfTile, steps * kSfTile,
                &full[s]);
      for (uint32_t b = 0; b < nb; ++b)
        bulk_load(st + S::kABytes + S::kBBytes + S::kSfaBytes + b * kStepsPerStage * kSfTile,
                  sfb + ((uint64_t)(band_b0 + b) * tiles_per_row + tile0) * kSfTile,
                  steps * kSfTile, &full[s]);
    }
    // the copies still in flight complete before the CTA may exit
    const uint32_t first = kb > S::kStages ? kb - S::kStages : 0u;
    for (uint32_t j = first; j < kb; ++j)
      mbar_wait(&full[j % S::kStages], (j / S::kStages) & 1u, wait_ns, err);
  } else if (warp == 1 && lane == 0) {
    // ---- scale copies and MMAs ----
    constexpr uint32_t idesc = mma_idesc(128, BN);
    const uint32_t bands_b = (n + 127u) / 128u, band_b0 = n0 / 128u;
    bool ok = true;
    for (uint32_t kb = 0; kb < nkb; ++kb) {
      const uint32_t s = kb % S::kStages, ph = (kb / S::kStages) & 1u;
      if (!mbar_wait(&full[s], ph, wait_ns, err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t st = smem_addr(smem + s * S::kStageBytes);
      const uint32_t sf_a = st + S::kABytes + S::kBBytes, sf_b = sf_a + S::kSfaBytes;
      const uint32_t steps = min(kStepsPerStage, tiles_per_row - kStepsPerStage * kb);
      for (uint32_t j = 0; j < steps; ++j) {
        const uint32_t ta = tmem + S::kSfaBase + (s * kStepsPerStage + j) * S::kSfaCols;
        const uint32_t tb = tmem + S::kSfbBase + (s * kStepsPerStage + j) * S::kSfbCols;
        tmem_copy_scales(ta, scale_desc(sf_a + j * kSfTile));
        for (uint32_t b = 0; b < S::kBands; ++b)
          if (band_b0 + b < bands_b)
            tmem_copy_scales(tb + 4u * b, scale_desc(sf_b + (b * kStepsPerStage + j) * kSfTile));
        // k-step j sits 32 bytes further along each 128-byte row
        mma_nvf4(tmem, operand_desc(st + 32u * j), operand_desc(st + S::kABytes + 32u * j), idesc,
                 ta, tb, (kb | j) != 0u ? 1u : 0u);
      }
      tc_commit(&empty[s]);
    }
    if (ok) tc_commit(&acc_full);
  } else if (warp >= 2) {
    // ---- epilogue: warp w reads lane quarter w mod 4 ----
    const uint32_t q = warp & 3u;
    const bool ok = mbar_wait(&acc_full, 0, wait_ns, err);
    tc_fence_after();
    if (ok) {
      const float alpha = __fmul_rn(gs_a[0], gs_b[0]);
      const uint32_t row = m0 + 32u * q + lane;
      const bool row_in = row < m;
      for (uint32_t c = 0; c < (uint32_t)BN; c += 32) {
        uint32_t v[32];
        tmem_load32(tmem + ((32u * q) << 16) + c, v);
        const uint32_t col = n0 + c;
        if (!row_in || col >= n) continue;
        const uint32_t cnt = min(32u, n - col);
        if (d_bf16) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(d) + (uint64_t)row * n + col;
          if (cnt == 32 && (n & 7u) == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t w[4];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const __nv_bfloat162 pr = __floats2bfloat162_rn(
                    __fmul_rn(alpha, __uint_as_float(v[8 * i + 2 * t])),
                    __fmul_rn(alpha, __uint_as_float(v[8 * i + 2 * t + 1])));
                w[t] = *reinterpret_cast<const uint32_t*>(&pr);
              }
              reinterpret_cast<uint4*>(out)[i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            for (uint32_t i = 0; i < cnt; ++i)
              out[i] = __float2bfloat16_rn(__fmul_rn(alpha, __uint_as_float(v[i])));
          }
        } else {
          float* out = static_cast<float*>(d) + (uint64_t)row * n + col;
          if (cnt == 32 && (n & 3u) == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              reinterpret_cast<float4*>(out)[i] =
                  make_float4(__fmul_rn(alpha, __uint_as_float(v[4 * i])),
                              __fmul_rn(alpha, __uint_as_float(v[4 * i + 1])),
                              __fmul_rn(alpha, __uint_as_float(v[4 * i + 2])),
                              __fmul_rn(alpha, __uint_as_float(v[4 * i + 3])));
          } else {
            for (uint32_t i = 0; i < cnt; ++i) out[i] = __fmul_rn(alpha, __uint_as_float(v[i]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Codes [rows, k/2] as a 2-D byte tensor, boxes of box_rows rows x 128 bytes
// in 128-byte swizzle; out-of-range rows and bytes read as zero.
bool encode_operand_map(const void* codes, int64_t rows, int64_t k, uint32_t box_rows,
                        CUtensorMap* map) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dim[2] = {(cuuint64_t)(k / 2), (cuuint64_t)rows};
  const cuuint64_t stride[1] = {(cuuint64_t)(k / 2)};
  const cuuint32_t box[2] = {kBK / 2, box_rows};
  const cuuint32_t estride[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(codes), dim, stride, box,
             estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
cudaError_t launch_tc(const void* a_codes, const void* a_sf, const float* a_gs,
                      const void* b_codes, const void* b_sf, const float* b_gs, int64_t m,
                      int64_t n, int64_t k, void* d, int d_bf16, uint32_t* err, uint64_t wait_ns,
                      cudaStream_t st) {
  using S = GemmShape<BN>;
  static std::mutex mu;
  static bool set_for[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!set_for[dev]) {
      e = cudaFuncSetAttribute(k_nvfp4_gemm<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)S::kSmemBytes);
      if (e != cudaSuccess) return e;
      set_for[dev] = true;
    }
  }
  CUtensorMap ma, mb;
  if (!encode_operand_map(a_codes, m, k, 128, &ma) || !encode_operand_map(b_codes, n, k, BN, &mb))
    return cudaErrorInvalidValue;
  const dim3 grid((unsigned)((n + BN - 1) / BN), (unsigned)((m + 127) / 128));
  k_nvfp4_gemm<BN><<<grid, kGemmThreads, S::kSmemBytes, st>>>(
      ma, mb, (const uint8_t*)a_sf, (const uint8_t*)b_sf, a_gs, b_gs, (uint32_t)m, (uint32_t)n,
      (uint32_t)k, d, d_bf16 ? 1u : 0u, err, wait_ns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_nvfp4_gemm_tc(const void* a_codes, const void* a_sf, const float* a_gs,
                                 const void* b_codes, const void* b_sf, const float* b_gs,
                                 int64_t m, int64_t n, int64_t k, void* d, int d_bf16,
                                 int tile_n, uint32_t* err, uint64_t wait_ns, cudaStream_t st) {
  if (m <= 0 || n <= 0 || k <= 0 || k % 32 || m > 65535LL * 128 || m > UINT32_MAX ||
      n > UINT32_MAX || k > UINT32_MAX)
    return cudaErrorInvalidValue;
  return tile_n == 128
             ? launch_tc<128>(a_codes, a_sf, a_gs, b_codes, b_sf, b_gs, m, n, k, d, d_bf16, err,
                              wait_ns, st)
             : launch_tc<256>(a_codes, a_sf, a_gs, b_codes, b_sf, b_gs, m, n, k, d, d_bf16, err,
                              wait_ns, st);
}

}  // namespace tfp4
