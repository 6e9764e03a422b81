// trace_gemm_tc.cu - the NVFP4 GEMM over rollout codes on the fifth-
// generation tensor cores: block-scaled E2M1 x E2M1 products with UE4M3 block
// scales (one per 16 elements along k), FP32 accumulation in tensor memory.
//
// Source: "Alibaba Qwen Proposes TRACE for 5.4x Faster FP4 RL Rollouts",
// section "TRACE Core Concept": rollout runs weights and activations in
// NVFP4, so the rollout codes and their block scales are the operands of its
// GEMMs.  The operand, scale and descriptor formats are NVIDIA's documented
// interfaces (PTX ISA, tcgen05 shared-memory and instruction descriptors,
// tensor-memory operands and block scaling; cuBLAS, "1D block scaling factors
// layout").
//
// d [m, n] = fl32(gs_a * gs_b) * sum_k A[i, k] B[j, k], A and B as codes
// [rows, k/2] (element 2i in the low nibble: the packed E2M1 operand format)
// and block scales in the 512-byte tile layout the rollout quantiser writes.
//
// A persistent grid, one CTA per SM (its shared memory allows no second),
// each CTA taking output tiles of 128 x BN in turn; 320 threads in roles:
//   - warp 0 (one lane): producer.  Per k-block of 256 elements it loads the
//     A tile (128 rows x 128 bytes) and the B tile (BN rows x 128 bytes) with
//     2-D tensor-map copies in 128-byte swizzle, and the block-scale tiles
//     (512 bytes per 128 rows and 64 elements of k) with bulk copies, into a
//     ring of stages completing on mbarriers;
//   - warps 2-5: stagers.  Per stage each warp moves the stage's scale lines
//     from shared into tensor memory (tcgen05.st, warp w owning lane quarter
//     w mod 4), so that no scale copy occupies the tensor pipe;
//   - warp 1: allocates the tensor memory; one lane issues the block-scaled
//     MMAs (128 x BN x 64 each, A and B in shared memory, the scales in
//     tensor memory), commits each stage back to the producer and each tile
//     to the epilogue;
//   - warps 6-9: epilogue.  Each thread reads its accumulator row (its
//     warp's lane quarter), releases the accumulator to the next tile's
//     MMAs, multiplies by fl32(gs_a * gs_b) and stores fp32 or bf16, while
//     the next tile's loads and staging already run.
// On an SM pair (two-CTA cluster, tcgen05 cta_group::2) the tile is 256 x 256:
// each CTA holds 128 rows of A and of the accumulator and 128 rows of B; the
// even CTA issues the MMAs and the scale copies for both (paired tcgen05.cp,
// each CTA's scales from its own shared memory), the MMAs read A and B from
// both CTAs' shared memory, commits arrive in both CTAs, and a thread of the
// odd CTA relays its stages' arrival to the even one.
// Rows and columns past m, n and k are zero-filled by the tensor-map copies
// (zero codes contribute nothing whatever their scales); scale tiles past the
// end of a scale tensor are not read (their lanes hold stale scales that
// only reach output columns past n, never stored), and only rows and
// columns inside d are stored.
//
// Tensor memory (512 columns of 32-bit lanes, lane = tile row): the
// accumulator in columns [0, BN), then a slot per shared-memory stage
// holding the stage's A scales (four columns per k-step) and B scales
// (BN / 32 columns per k-step).  (A staged in tensor memory instead, read
// by the MMAs from there, left room for fewer slots than stages, and the
// stagers then waited for slots: slower.)  Scales follow the tile layout: line L of a
// 512-byte tile holds rows L, L + 32, L + 64, L + 96, and lane L of every
// quarter holds line L, so column c of lane L holds the four scales of row
// L + 32 c for the k-step.
//
// Every wait is bounded (wait_ns): one that runs out sets *err, the role
// stops, the producer still waits (bounded) for its own copies in flight,
// and the tensor memory is freed before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "trace_async.cuh"
#include "trace_internal.h"

namespace tfp4 {
namespace {

constexpr int kGemmThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBK = 256;            // k elements per stage (128 bytes of codes a row)
constexpr uint32_t kSfTile = 512;        // bytes of one scale tile: 128 rows x 64 k
constexpr uint32_t kStepsPerStage = 4;   // 64-element MMA k-steps per stage

// PAIR: one tile of 256 x BN on an SM pair (tcgen05 cta_group::2): each CTA
// holds 128 rows of A and of the accumulator and BN / 2 rows of B.
template <int BN, bool PAIR>
struct GemmShape {
  static_assert(!PAIR || BN == 256, "pair tiles are 256 x 256");
  static constexpr uint32_t kBRows = PAIR ? (uint32_t)BN / 2 : (uint32_t)BN;  // B rows per CTA
  static constexpr uint32_t kABytes = 128u * kBK / 2;
  static constexpr uint32_t kBBytes = kBRows * kBK / 2;
  static constexpr uint32_t kBands = (uint32_t)BN / 128;  // 128-row scale bands of a B tile
  static constexpr uint32_t kSfaBytes = kStepsPerStage * kSfTile;
  static constexpr uint32_t kSfbBytes = kBands * kStepsPerStage * kSfTile;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr uint32_t kStages = PAIR ? 5 : BN == 256 ? 4 : 6;  // shared-memory ring
  static constexpr uint32_t kSlots = kStages;  // tensor-memory scale slots, one per stage
  static constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024;  // + alignment slack
  // tensor-memory columns per k-step and their regions
  static constexpr uint32_t kSfaCols = 4;
  static constexpr uint32_t kSfbCols = 4 * kBands;
  static constexpr uint32_t kSfaBase = BN;
  static constexpr uint32_t kSfbBase = kSfaBase + kSlots * kStepsPerStage * kSfaCols;
  static constexpr uint32_t kColsUsed = kSfbBase + kSlots * kStepsPerStage * kSfbCols;
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned (128-byte swizzle)");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory of one CTA");
  static_assert(kColsUsed + 8 <= kTmemCols, "tensor-memory columns");
  static_assert(kSlots <= kStages, "a slot is refilled only after its stage's MMAs");
};

// ---- tcgen05 ----------------------------------------------------------------

// Allocation, MMAs and commits name the CTA group: 1 (this CTA) or 2 (the
// SM pair of a two-CTA cluster, where both CTAs allocate the same columns
// together and the even CTA issues the MMAs for both).
template <bool PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t cols) {
  if constexpr (PAIR)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_addr(dst_smem)), "r"(cols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_addr(dst_smem)), "r"(cols)
                 : "memory");
}

template <bool PAIR>
__device__ __forceinline__ void tmem_relinquish() {
  if constexpr (PAIR)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  if constexpr (PAIR)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
                 : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
                 : "memory");
}

// ---- clusters -----------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(rank));
  return a;
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Bounded wait that also acquires what other CTAs of the cluster released.
__device__ __forceinline__ bool mbar_try_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __noinline__ bool mbar_wait_cluster_slow(uint64_t* bar, uint32_t parity,
                                                    uint64_t limit_ns, uint32_t* err) {
  for (uint32_t it = 0; it < 16; ++it)
    if (mbar_try_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 22); ++it) {
    if (mbar_try_cluster(bar, parity)) return true;
    if ((it & 15u) == 15u && global_ns() - t0 > limit_ns) break;
  }
  atomicOr(err, 2u);
  return false;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns, uint32_t* err) {
  return mbar_try_cluster(bar, parity) || mbar_wait_cluster_slow(bar, parity, limit_ns, err);
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

// Instruction descriptor of the block-scaled MMA: A and B E2M1 (format 1 of
// the FP4 kinds, bits 7-9 and 10-11), both K-major, no negation, dense,
// UE4M3 scales (bit 23 = 0), scale-factor ids 0, N / 8 at bits 17-22,
// M / 16 at bits 24-28.
__host__ __device__ constexpr uint32_t mma_idesc(uint32_t m, uint32_t n) {
  return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// d (tensor memory) (+)= A B^T over one 64-element k-step, A and B in shared
// memory (descriptors adesc, bdesc), both scaled per 16-element block by the
// UE4M3 scales in tensor memory at sfa / sfb.  For a pair, the same addresses
// name both CTAs' tensor and shared memory.
template <bool PAIR>
__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  if constexpr (PAIR)
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
        "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
        "r"(accumulate)
        : "memory");
}

// 32 lines x 128 bits of shared memory into four columns of tensor memory,
// the same lines in each of the four lane quarters; for a pair, each CTA's
// lines at this address into its own tensor memory.
template <bool PAIR>
__device__ __forceinline__ void tmem_copy_scales(uint32_t taddr, uint32_t saddr) {
  const uint64_t desc = smem_desc(saddr, 0, 128, 0);  // 8-line groups 128 bytes apart
  if constexpr (PAIR)
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
                 : "memory");
  else
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
                 : "memory");
}

// Arrive on bar (in this CTA, or for a pair in both CTAs) once every tcgen05
// operation this thread issued so far has completed.
template <bool PAIR>
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  if constexpr (PAIR)
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_addr(bar)), "h"((uint16_t)3)
        : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_addr(bar))
                 : "memory");
}

// Arrive on bar in this CTA only once this thread's tcgen05 operations completed.
template <bool PAIR>
__device__ __forceinline__ void tc_commit_local(uint64_t* bar) {
  if constexpr (PAIR)
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_addr(bar))
                 : "memory");
  else
    tc_commit<false>(bar);
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

// 16 / 32 consecutive 32-bit columns of this thread's lane from registers.
__device__ __forceinline__ void tmem_store16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0],"
      " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
      ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
      "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
      "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_store32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
      " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16,"
      " %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
      ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
      "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
      "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]),
      "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
      "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_store_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t saddr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(saddr)
               : "memory");
  return v;
}


__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// ---- the kernel ---------------------------------------------------------------

// Bounded wait on a barrier that CTAs of the cluster may also release.
template <bool PAIR>
__device__ __forceinline__ bool wait_any(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                         uint32_t* err) {
  if constexpr (PAIR)
    return mbar_wait_cluster(bar, parity, limit_ns, err);
  else
    return mbar_wait(bar, parity, limit_ns, err);
}

// Arrive on `bar` of the even CTA (this CTA unless it is a pair's odd CTA).
template <bool PAIR>
__device__ __forceinline__ void arrive_even(uint64_t* bar, uint32_t rank) {
  if (PAIR && rank != 0)
    mbar_arrive_remote(peer_addr(bar, 0));
  else
    mbar_arrive(bar);
}

// Persistent: each CTA (each pair) takes output tiles u, u + units, ... with
// u its index; tile t covers rows (t / tiles_n) * TM and columns
// (t % tiles_n) * BN.  The rings of stages and slots run on across tiles
// (g counts k-blocks over all of the CTA's tiles).
template <int BN, bool PAIR>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_nvfp4_gemm(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                 const uint8_t* __restrict__ sfa, const uint8_t* __restrict__ sfb,
                 const float* __restrict__ gs_a, const float* __restrict__ gs_b, uint32_t m,
                 uint32_t n, uint32_t k, void* __restrict__ d, uint32_t d_bf16,
                 uint32_t* __restrict__ err, uint64_t wait_ns) {
  using S = GemmShape<BN, PAIR>;
  constexpr uint32_t TM = PAIR ? 256u : 128u;
  extern __shared__ uint8_t smem_raw[];
  // full: a stage's copies landed; empty: its MMAs completed (its shared
  // memory and its tensor-memory slot are free again); staged: a slot holds
  // its stage's scales (pair: the odd CTA's stage landed); acc_full:
  // a tile's last MMA completed; acc_free: the epilogue read the
  // accumulator (pair: in both CTAs); drain: this CTA's MMAs retired
  __shared__ __align__(8) uint64_t full[S::kStages], empty[S::kStages], staged[S::kSlots],
      acc_full, acc_free, drain;
  __shared__ uint32_t tmem_base;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~uintptr_t(1023));

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  const uint32_t unit = PAIR ? blockIdx.x >> 1 : blockIdx.x;
  const uint32_t units = PAIR ? gridDim.x >> 1 : gridDim.x;
  const uint32_t tiles_n = (n + BN - 1) / BN;
  const uint32_t ntiles = ((m + TM - 1) / TM) * tiles_n;
  const uint32_t nkb = (k + kBK - 1) / kBK;
  const uint32_t tiles_per_row = (k + 63) / 64;  // scale tiles along k (64 elements each)

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < S::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (uint32_t t = 0; t < S::kSlots; ++t) mbar_init(&staged[t], PAIR ? 1 : 4);
    mbar_init(&acc_full, 1);
    mbar_init(&acc_free, PAIR ? 8 : 4);
    mbar_init(&drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc<PAIR>(&tmem_base, kTmemCols);
    tmem_relinquish<PAIR>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // both CTAs' barriers and columns exist
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0 && lane == 0) {
    // ---- producer ----
    const uint32_t bands_a = (m + 127u) / 128u, bands_b = (n + 127u) / 128u;
    uint32_t g = 0;
    bool ok = true;
    for (uint32_t tile = unit; tile < ntiles && ok; tile += units) {
      // this CTA's A rows, the tile's columns, this CTA's B rows
      const uint32_t m0 = (tile / tiles_n) * TM + 128u * rank, n0 = (tile % tiles_n) * BN;
      const uint32_t nb0 = n0 + S::kBRows * rank;
      const uint32_t band_a = m0 / 128u, band_b0 = n0 / 128u;
      const uint32_t na = band_a < bands_a ? 1u : 0u;  // (a pair's odd CTA may lie past m)
      uint32_t nb = 0;
      for (uint32_t b = 0; b < S::kBands; ++b) nb += band_b0 + b < bands_b ? 1u : 0u;
      for (uint32_t kb = 0; kb < nkb; ++kb, ++g) {
        const uint32_t s = g % S::kStages, ph = (g / S::kStages) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u, wait_ns, err)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + s * S::kStageBytes;
        const uint32_t steps = min(kStepsPerStage, tiles_per_row - kStepsPerStage * kb);
        mbar_expect_tx(&full[s], S::kABytes + S::kBBytes + (na + nb) * steps * kSfTile);
        tensor_load_2d(st, &map_a, kb * (kBK / 2), m0, &full[s]);
        tensor_load_2d(st + S::kABytes, &map_b, kb * (kBK / 2), nb0, &full[s]);
        const uint64_t tile0 = kStepsPerStage * kb;
        if (na)
          bulk_load(st + S::kABytes + S::kBBytes,
                    sfa + ((uint64_t)band_a * tiles_per_row + tile0) * kSfTile, steps * kSfTile,
                    &full[s]);
        for (uint32_t b = 0; b < nb; ++b)
          bulk_load(st + S::kABytes + S::kBBytes + S::kSfaBytes + b * kStepsPerStage * kSfTile,
                    sfb + ((uint64_t)(band_b0 + b) * tiles_per_row + tile0) * kSfTile,
                    steps * kSfTile, &full[s]);
      }
    }
    // the copies still in flight complete before the CTA may exit
    for (uint32_t j = g > S::kStages ? g - S::kStages : 0u; j < g; ++j)
      mbar_wait(&full[j % S::kStages], (j / S::kStages) & 1u, wait_ns, err);
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---- MMAs (for a pair: the even CTA, for both) ----
    constexpr uint32_t idesc = mma_idesc(TM, BN);
    uint32_t g = 0, it = 0;
    bool ok = true;
    for (uint32_t tile = unit; tile < ntiles && ok; tile += units, ++it) {
      // the epilogue has read the previous tile's accumulator
      if (it > 0 && !wait_any<PAIR>(&acc_free, (it - 1) & 1u, wait_ns, err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (uint32_t kb = 0; kb < nkb; ++kb, ++g) {
        const uint32_t s = g % S::kStages, ph = (g / S::kStages) & 1u;
        const uint32_t t = g % S::kSlots, pt = (g / S::kSlots) & 1u;
        if (!wait_any<PAIR>(&staged[t], pt, wait_ns, err) ||
            !mbar_wait(&full[s], ph, wait_ns, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_smem = smem_addr(smem + s * S::kStageBytes);
        const uint32_t b_smem = a_smem + S::kABytes;
        const uint32_t steps = min(kStepsPerStage, tiles_per_row - kStepsPerStage * kb);
        const uint32_t step0 = t * kStepsPerStage;
        if constexpr (PAIR) {
          // scales of both CTAs, each from its own shared memory (paired copies)
          const uint32_t sf_a = b_smem + S::kBBytes, sf_b = sf_a + S::kSfaBytes;
          for (uint32_t j = 0; j < steps; ++j) {
            tmem_copy_scales<true>(tmem + S::kSfaBase + (step0 + j) * S::kSfaCols,
                                   sf_a + j * kSfTile);
            for (uint32_t b = 0; b < S::kBands; ++b)
              tmem_copy_scales<true>(tmem + S::kSfbBase + (step0 + j) * S::kSfbCols + 4u * b,
                                     sf_b + (b * kStepsPerStage + j) * kSfTile);
          }
        }
        for (uint32_t j = 0; j < steps; ++j) {
          // k-step j sits 32 bytes further along each 128-byte row of A and B
          const uint32_t sfa_t = tmem + S::kSfaBase + (step0 + j) * S::kSfaCols;
          const uint32_t sfb_t = tmem + S::kSfbBase + (step0 + j) * S::kSfbCols;
          const uint32_t acc = (kb | j) != 0u ? 1u : 0u;
          mma_nvf4<PAIR>(tmem, operand_desc(a_smem + 32u * j), operand_desc(b_smem + 32u * j),
                         idesc, sfa_t, sfb_t, acc);
        }
        tc_commit<PAIR>(&empty[s]);
      }
      if (ok) tc_commit<PAIR>(&acc_full);
    }
    // every MMA issued here has retired before the columns are freed
    tc_commit_local<PAIR>(&drain);
    mbar_wait(&drain, 0, wait_ns, err);
  } else if (PAIR && warp == 1 && lane == 0) {
    // ---- the odd CTA's relay: its stage landed -> the even CTA's staged ----
    const uint32_t remote = peer_addr(&staged[0], 0);
    uint32_t g = 0;
    bool ok = true;
    for (uint32_t tile = unit; tile < ntiles && ok; tile += units)
      for (uint32_t kb = 0; kb < nkb; ++kb, ++g) {
        if (!mbar_wait(&full[g % S::kStages], (g / S::kStages) & 1u, wait_ns, err)) {
          ok = false;
          break;
        }
        mbar_arrive_remote(remote + (g % S::kSlots) * (uint32_t)sizeof(uint64_t));
      }
  } else if (!PAIR && warp >= 2 && warp < 6) {
    // ---- stagers: warp w owns lane quarter q = w mod 4 (tile rows 32 q ..) ----
    const uint32_t q = warp & 3u;
    const uint32_t lane_base = tmem + ((32u * q) << 16);
    uint32_t g = 0;
    bool ok = true;
    for (uint32_t tile = unit; tile < ntiles && ok; tile += units)
      for (uint32_t kb = 0; kb < nkb; ++kb, ++g) {
        // slot t = stage s: the stage's copies land only after the MMAs of
        // its previous use (which read the slot) completed
        const uint32_t s = g % S::kStages, ph = (g / S::kStages) & 1u;
        const uint32_t t = g % S::kSlots;
        if (!mbar_wait(&full[s], ph, wait_ns, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t st = smem_addr(smem + s * S::kStageBytes);
        const uint32_t sf_a = st + S::kABytes + S::kBBytes, sf_b = sf_a + S::kSfaBytes;
        const uint32_t step0 = t * kStepsPerStage;
        {
          // A scales: line `lane` of each k-step's tile
          uint32_t w[16];
#pragma unroll
          for (uint32_t j = 0; j < 4; ++j) {
            const uint4 v = lds128(sf_a + j * kSfTile + lane * 16u);
            w[4 * j] = v.x;
            w[4 * j + 1] = v.y;
            w[4 * j + 2] = v.z;
            w[4 * j + 3] = v.w;
          }
          tmem_store16(lane_base + S::kSfaBase + step0 * S::kSfaCols, w);
        }
        if constexpr (S::kBands == 2) {
          // B scales, k-step j: band 0 then band 1
          uint32_t w[32];
#pragma unroll
          for (uint32_t j = 0; j < 4; ++j)
#pragma unroll
            for (uint32_t b = 0; b < 2; ++b) {
              const uint4 v = lds128(sf_b + (b * kStepsPerStage + j) * kSfTile + lane * 16u);
              w[8 * j + 4 * b] = v.x;
              w[8 * j + 4 * b + 1] = v.y;
              w[8 * j + 4 * b + 2] = v.z;
              w[8 * j + 4 * b + 3] = v.w;
            }
          tmem_store32(lane_base + S::kSfbBase + step0 * S::kSfbCols, w);
        } else {
          uint32_t w[16];
#pragma unroll
          for (uint32_t j = 0; j < 4; ++j) {
            const uint4 v = lds128(sf_b + j * kSfTile + lane * 16u);
            w[4 * j] = v.x;
            w[4 * j + 1] = v.y;
            w[4 * j + 2] = v.z;
            w[4 * j + 3] = v.w;
          }
          tmem_store16(lane_base + S::kSfbBase + step0 * S::kSfbCols, w);
        }
        tmem_store_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&staged[t]);
      }
  } else if (warp >= 6) {
    // ---- epilogue: warp w reads lane quarter q = w mod 4 ----
    const uint32_t q = warp & 3u;
    const uint32_t lane_base = tmem + ((32u * q) << 16);
    const float alpha = __fmul_rn(gs_a[0], gs_b[0]);
    const bool vec = d_bf16 ? (n & 7u) == 0 : (n & 3u) == 0;  // 16-byte row pieces aligned
    uint32_t it = 0;
    for (uint32_t tile = unit; tile < ntiles; tile += units, ++it) {
      if (!mbar_wait(&acc_full, it & 1u, wait_ns, err)) break;
      tc_fence_after();
      const uint32_t grow = (tile / tiles_n) * TM + 128u * rank + 32u * q + lane;
      const uint32_t n0 = (tile % tiles_n) * BN;
      if (d_bf16 && vec && n0 + BN <= n) {
        // A whole bf16 tile: the accumulator row, scaled and rounded to bf16
        // pairs, is held in registers before the accumulator is released, so
        // the next tile's MMAs run while this tile's rows are stored (a
        // lane's row pieces make 32 separate pieces per store instruction,
        // slow enough to hold the tensor pipe idle if they came first).
        uint32_t p[BN / 2];
#pragma unroll
        for (uint32_t c = 0; c < (uint32_t)BN; c += 32) {
          uint32_t v[32];
          tmem_load32(lane_base + c, v);
#pragma unroll
          for (uint32_t i = 0; i < 16; ++i)
            p[c / 2 + i] = bf16x2(__fmul_rn(alpha, __uint_as_float(v[2 * i])),
                                  __fmul_rn(alpha, __uint_as_float(v[2 * i + 1])));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_even<PAIR>(&acc_free, rank);
        if (grow < m) {
          uint4* out = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(d) +
                                                (uint64_t)grow * n + n0);
#pragma unroll
          for (uint32_t j = 0; j < (uint32_t)BN / 8; ++j)
            out[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
        }
        continue;
      }
      // fp32 output, or a tile cut by n: chunk by chunk, the accumulator
      // released after its last chunk is read
      for (uint32_t c = 0; c < (uint32_t)BN; c += 32) {
        uint32_t v[32];
        tmem_load32(lane_base + c, v);
        if (c + 32 == (uint32_t)BN) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_even<PAIR>(&acc_free, rank);
        }
        const uint32_t col = n0 + c;
        if (grow >= m || col >= n) continue;
        const uint32_t cnt = min(32u, n - col);
        if (d_bf16) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(d) + (uint64_t)grow * n + col;
          if (vec && cnt == 32) {
#pragma unroll
            for (uint32_t i = 0; i < 4; ++i) {
              const uint32_t* u = v + 8 * i;
              reinterpret_cast<uint4*>(out)[i] =
                  make_uint4(bf16x2(__fmul_rn(alpha, __uint_as_float(u[0])),
                                    __fmul_rn(alpha, __uint_as_float(u[1]))),
                             bf16x2(__fmul_rn(alpha, __uint_as_float(u[2])),
                                    __fmul_rn(alpha, __uint_as_float(u[3]))),
                             bf16x2(__fmul_rn(alpha, __uint_as_float(u[4])),
                                    __fmul_rn(alpha, __uint_as_float(u[5]))),
                             bf16x2(__fmul_rn(alpha, __uint_as_float(u[6])),
                                    __fmul_rn(alpha, __uint_as_float(u[7]))));
            }
          } else {
#pragma unroll
            for (uint32_t i = 0; i < 32; ++i)
              if (i < cnt) out[i] = __float2bfloat16_rn(__fmul_rn(alpha, __uint_as_float(v[i])));
          }
        } else {
          float* out = static_cast<float*>(d) + (uint64_t)grow * n + col;
          if (vec && cnt == 32) {
#pragma unroll
            for (uint32_t i = 0; i < 8; ++i)
              reinterpret_cast<float4*>(out)[i] =
                  make_float4(__fmul_rn(alpha, __uint_as_float(v[4 * i])),
                              __fmul_rn(alpha, __uint_as_float(v[4 * i + 1])),
                              __fmul_rn(alpha, __uint_as_float(v[4 * i + 2])),
                              __fmul_rn(alpha, __uint_as_float(v[4 * i + 3])));
          } else {
#pragma unroll
            for (uint32_t i = 0; i < 32; ++i)
              if (i < cnt) out[i] = __fmul_rn(alpha, __uint_as_float(v[i]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // the pair's MMAs and reads are done in both CTAs
  if (warp == 1) tmem_dealloc<PAIR>(tmem, kTmemCols);
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

template <int BN, bool PAIR>
cudaError_t launch_tc(const void* a_codes, const void* a_sf, const float* a_gs,
                      const void* b_codes, const void* b_sf, const float* b_gs, int64_t m,
                      int64_t n, int64_t k, void* d, int d_bf16, uint32_t* err, uint64_t wait_ns,
                      int sm_count, cudaStream_t st) {
  using S = GemmShape<BN, PAIR>;
  static std::mutex mu;
  static bool set_for[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!set_for[dev]) {
      e = cudaFuncSetAttribute(k_nvfp4_gemm<BN, PAIR>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::kSmemBytes);
      if (e != cudaSuccess) return e;
      set_for[dev] = true;
    }
  }
  CUtensorMap ma, mb;
  if (!encode_operand_map(a_codes, m, k, 128, &ma) ||
      !encode_operand_map(b_codes, n, k, S::kBRows, &mb))
    return cudaErrorInvalidValue;
  // one CTA per SM (pair: per two SMs), each taking tiles in turn
  const int64_t tm = PAIR ? 256 : 128;
  const int64_t ntiles = (m + tm - 1) / tm * ((n + BN - 1) / BN);
  int64_t units = PAIR ? sm_count / 2 : sm_count;
  if (units > ntiles) units = ntiles;
  if (units < 1) units = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units * (PAIR ? 2 : 1)));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = S::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_nvfp4_gemm<BN, PAIR>, ma, mb, (const uint8_t*)a_sf,
                            (const uint8_t*)b_sf, a_gs, b_gs, (uint32_t)m, (uint32_t)n,
                            (uint32_t)k, d, d_bf16 ? 1u : 0u, err, wait_ns);
}

}  // namespace

cudaError_t launch_nvfp4_gemm_tc(const void* a_codes, const void* a_sf, const float* a_gs,
                                 const void* b_codes, const void* b_sf, const float* b_gs,
                                 int64_t m, int64_t n, int64_t k, void* d, int d_bf16,
                                 int tile, uint32_t* err, uint64_t wait_ns, int sm_count,
                                 cudaStream_t st) {
  if (m <= 0 || n <= 0 || k <= 0 || k % 32 || m > UINT32_MAX || n > UINT32_MAX ||
      k > UINT32_MAX)
    return cudaErrorInvalidValue;
  if (tile == kGemmTilePair)
    return launch_tc<256, true>(a_codes, a_sf, a_gs, b_codes, b_sf, b_gs, m, n, k, d, d_bf16,
                                err, wait_ns, sm_count, st);
  return tile == kGemmTile128
             ? launch_tc<128, false>(a_codes, a_sf, a_gs, b_codes, b_sf, b_gs, m, n, k, d,
                                     d_bf16, err, wait_ns, sm_count, st)
             : launch_tc<256, false>(a_codes, a_sf, a_gs, b_codes, b_sf, b_gs, m, n, k, d,
                                     d_bf16, err, wait_ns, sm_count, st);
}

}  // namespace tfp4
