// trace_kernels.cu - sm_103a kernels of the guided-NVFP4 hot path of TRACE
// except the training-side fake quantiser (trace_fakequant.cu): segment
// amax, rollout quantisation (two-kernel and fused forms), guide pack and
// unpack, and the straight-through backward.  The work decomposition and
// arithmetic conventions are described in trace_device.cuh.
//
// Sources: "Alibaba Qwen Proposes TRACE for 5.4x Faster FP4 RL Rollouts",
// section "TRACE Core Concept", and the worked example of section "Why
// Does FP4 Rollout 'Break' RL Training?".
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "trace_async.cuh"
#include "trace_device.cuh"

namespace tfp4 {
namespace {

// ---------------------------------------------------------------------------
// a1: segment amax + global scales
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t chunk_amax_bits(const Chunk& c) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = max_u16x2(m, c.w[i] & kAbs2);
  const uint32_t hi = m >> 16, lo = m & 0xFFFFu;
  return (hi > lo ? hi : lo) << 16;  // binary32 bits of the largest |x|
}

// CTA-wide max of v, folded into *dst with one atomic (called uniformly).
__device__ __forceinline__ void cta_flush_max(uint32_t v, uint32_t* dst, uint32_t* red) {
  v = __reduce_max_sync(0xFFFFFFFFu, v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) m = red[i] > m ? red[i] : m;
    if (m && TFP4_OK(dst, 4)) atomicMax(dst, m);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads)
    k_amax(const uint8_t* __restrict__ x, uint32_t nchunks, FastDivU cpr,
           uint32_t steps_per_cta, const __grid_constant__ SegParam seg,
           uint32_t* __restrict__ amax_bits, uint32_t* __restrict__ done,
           float* __restrict__ gs_out) {
  __shared__ uint32_t red[kThreads / 32];
  __shared__ int is_last;
  const uint32_t nsteps = (nchunks + kThreads - 1) / kThreads;
  uint32_t step = blockIdx.x * steps_per_cta;
  const uint32_t step_end = min(step + steps_per_cta, nsteps);

  StepSeg ss;
  ss.cur = step < step_end ? seg_search(seg, cpr.div(step * kThreads)) : 0;
  int open = -1;  // segment whose running max this CTA holds
  uint32_t run = 0;

  Chunk cur, nxt;
  if (step < step_end) {
    const uint32_t c = step * kThreads + threadIdx.x;
    if (c < nchunks) load_chunk(cur, x, c);
  }
  for (; step < step_end; ++step) {
    const uint32_t c0 = step * kThreads;
    const uint32_t c = c0 + threadIdx.x;
    if (step + 1 < step_end) {
      const uint32_t cn = c + kThreads;
      if (cn < nchunks) load_chunk(nxt, x, cn);
    }
    const uint32_t last = min(c0 + kThreads, nchunks) - 1;
    const bool uniform = ss.update(seg, cpr.div(c0), cpr.div(last));
    const uint32_t m = c < nchunks ? chunk_amax_bits(cur) : 0u;
    if (uniform) {
      if (ss.cur != open) {
        if (open >= 0) cta_flush_max(run, amax_bits + open, red);
        open = ss.cur;
        run = 0;
      }
      run = m > run ? m : run;
    } else {
      if (open >= 0) cta_flush_max(run, amax_bits + open, red);
      open = -1;
      run = 0;
      if (c < nchunks && m) {
        uint32_t* dst = amax_bits + seg_advance(seg, ss.cur, cpr.div(c));
        if (TFP4_OK(dst, 4)) atomicMax(dst, m);
      }
    }
    cur = nxt;
  }
  if (open >= 0) cta_flush_max(run, amax_bits + open, red);

  // The last CTA to finish turns maxima into global scales and re-zeroes the
  // maxima for the next call.  No CTA ever waits for another.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t ticket = TFP4_OK(done, 4) ? atomicAdd(done, 1u) : 0u;
    is_last = (ticket == gridDim.x - 1);
  }
  __syncthreads();
  if (is_last) {
    __threadfence();
    for (int s = threadIdx.x; s < seg.n; s += kThreads) {
      const uint32_t a = TFP4_OK(amax_bits + s, 4) ? atomicExch(amax_bits + s, 0u) : 0u;
      if (TFP4_OK(gs_out + s, 4)) gs_out[s] = global_scale_of(a);
    }
    if (threadIdx.x == 0 && TFP4_OK(done, 4)) atomicExch(done, 0u);
  }
}

// ---------------------------------------------------------------------------
// compact word helpers
// ---------------------------------------------------------------------------

// Bits b (0: index LSB, 3: sign) of the eight nibbles of w, nibble i at bit
// 24 + i (bits 0..23 hold junk).  After the mask and fold, nibbles 2j and
// 2j + 1 sit in bits s, s + 1 of byte j (s = 0 for the LSB, 3 for the sign);
// the multiply adds byte j shifted by 24 - s - 6j, which lands the pair at
// bits 24 + 2j.  The other partial products fall in disjoint bit pairs below
// bit 24 or above bit 31, so no carry reaches the result.
__device__ __forceinline__ uint32_t nibble_lsb_hi(uint32_t w) {
  const uint32_t v = w & 0x11111111u;
  return ((v | (v >> 3)) & 0x03030303u) * 0x01041040u;  // 2^24 + 2^18 + 2^12 + 2^6
}
__device__ __forceinline__ uint32_t nibble_sign_hi(uint32_t w) {
  const uint32_t v = w & 0x88888888u;
  return ((v | (v >> 3)) & 0x18181818u) * 0x00208208u;  // 2^21 + 2^15 + 2^9 + 2^3
}

// Sixteen nibbles (one block, two words) -> compact word.
__device__ __forceinline__ uint32_t compact_word(uint32_t c0, uint32_t c1) {
  const uint32_t sgn = __byte_perm(nibble_sign_hi(c0), nibble_sign_hi(c1), 0x0073u);
  const uint32_t lsb = __byte_perm(nibble_lsb_hi(c0), nibble_lsb_hi(c1), 0x0073u);
  return __byte_perm(sgn, lsb, 0x5410u);
}

// ---------------------------------------------------------------------------
// a2: rollout quantisation
// ---------------------------------------------------------------------------

// Per-segment table of 1/S for every E4M3 code (S = dec(code) * gs), built
// by the n threads tid = 0..n-1 of a CTA or warp group.
__device__ __forceinline__ void build_inv_tab(float* inv, float gs, int tid, int n) {
  for (int c = tid; c < 128; c += n) {
    float S, r;
    real_scale((uint32_t)c, gs, S, r);
    inv[c] = r;
  }
}

// Block-scale codes of a chunk and their reciprocal scales, with the
// segment's constants (den = gs * 6, rden = 1 / den) and 1/S table, from the
// chunk's two block maxima.
__device__ __forceinline__ PairScale bamax_scale_tab(float b0, float b1, float gs, float den,
                                                     float rden, const float* inv_tab) {
  PairScale ps;
  ps.codes = pair_codes(b0, b1, gs, den, rden);
  ps.inv[0] = inv_tab[ps.codes & 0x7Fu];
  ps.inv[1] = inv_tab[(ps.codes >> 8) & 0x7Fu];
  return ps;
}

// Block-scale codes and reciprocal scales of a chunk from the global scale
// alone (a step that straddles segments).
__device__ __forceinline__ PairScale chunk_scale(const Chunk& cur, float gs) {
  float b0, b1;
  chunk_bamax(cur, b0, b1);
  return pair_scale(b0, b1, gs);
}


// Per-segment constants of the rollout scale (den, rden, 1/S table).
struct SegScale {
  float gs, den, rden;
  __device__ __forceinline__ void set(float g) {
    gs = g;
    den = __fmul_rn(g, 6.0f);
    rden = g > 0.0f ? __frcp_rn(den) : 0.0f;
  }
};

// One chunk (two blocks) -> 16 code bytes, two block-scale codes and two
// compact words, given its block-scale codes and reciprocal scales.
__device__ __forceinline__ void quant_chunk(const Chunk& cur, const PairScale& ps, uint32_t c,
                                            uint8_t* __restrict__ codes, uint8_t* __restrict__ bs,
                                            const MmaOut& mma, const FastDivU& cpr,
                                            uint8_t* __restrict__ guide) {
  uint32_t out[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    // signed x * inv keeps the input's sign in the nibble
    const F2 inv = splat(ps.inv[q >> 1]);
    F2 t[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t w = cur.w[4 * q + k];
      t[k] = mul2_rn(F2{__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)}, inv);
    }
    out[q] = e2m1x8(t[0], t[1], t[2], t[3]);
  }
  st_stream(codes + (uint64_t)c * 16u, out[0], out[1], out[2], out[3]);
  if (bs) st_stream_u16(bs + (uint64_t)c * 2u, ps.codes);
  if (mma.p) {
    // chunk q of row r holds scale columns 2q, 2q + 1: adjacent bytes of the
    // tile (r / 128, q / 2) at 16 (r mod 32) + 4 ((r / 32) mod 4) + 2 (q mod 2)
    const uint32_t r = cpr.div(c), q = c - r * cpr.d;
    const uint64_t off = ((uint64_t)(r >> 7) * mma.tiles_per_row + (q >> 1)) * 512u +
                         ((r & 31u) << 4) + (((r >> 5) & 3u) << 2) + ((q & 1u) << 1);
    st_stream_u16(mma.p + off, ps.codes);
  }
  if (guide)
    st_stream2(guide + (uint64_t)c * 8u, compact_word(out[0], out[1]), compact_word(out[2], out[3]));
}

// AMAX_OUT: also the segment maxima of x into amax_out (zeroed by the
// caller), for a later call that quantises with them (delayed scaling).
template <bool AMAX_OUT>
__global__ void __launch_bounds__(kThreads)
    k_rollout_quant(const uint8_t* __restrict__ x, uint32_t nchunks, FastDivU cpr,
                    uint32_t steps_per_cta, const __grid_constant__ SegParam seg,
                    const float* __restrict__ gs, uint8_t* __restrict__ codes,
                    uint8_t* __restrict__ bs, MmaOut mma, uint8_t* __restrict__ guide,
                    uint32_t* __restrict__ amax_out) {
  const uint32_t nsteps = (nchunks + kThreads - 1) / kThreads;
  uint32_t step = blockIdx.x * steps_per_cta;
  const uint32_t step_end = min(step + steps_per_cta, nsteps);
  StepSeg ss;
  ss.cur = step < step_end ? seg_search(seg, cpr.div(step * kThreads)) : 0;
  __shared__ float inv_tab[128];
  int tseg = -1;
  SegScale sc = {0.f, 0.f, 0.f};
  uint32_t mseg = 0u;  // AMAX_OUT: this thread's maximum in segment fseg
  int fseg = -1;

  Chunk cur, nxt;
  if (step < step_end) {
    const uint32_t c = step * kThreads + threadIdx.x;
    if (c < nchunks) load_chunk(cur, x, c);
  }
  for (; step < step_end; ++step) {
    const uint32_t c0 = step * kThreads;
    const uint32_t c = c0 + threadIdx.x;
    if (step + 1 < step_end) {
      const uint32_t cn = c + kThreads;
      if (cn < nchunks) load_chunk(nxt, x, cn);
    }
    const uint32_t last = min(c0 + kThreads, nchunks) - 1;
    const bool uniform = ss.update(seg, cpr.div(c0), cpr.div(last));
    if (AMAX_OUT && uniform && ss.cur != fseg) {
      if (fseg >= 0) flush_seg_max(mseg, amax_out + fseg);
      fseg = ss.cur;
    }
    if (uniform && ss.cur != tseg) {
      __syncthreads();
      tseg = ss.cur;
      sc.set(ldf(gs + tseg));
      build_inv_tab(inv_tab, sc.gs, threadIdx.x, kThreads);
      __syncthreads();
    }
    if (c < nchunks) {
      float b0, b1;
      chunk_bamax(cur, b0, b1);
      PairScale ps;
      if (uniform) {
        ps = bamax_scale_tab(b0, b1, sc.gs, sc.den, sc.rden, inv_tab);
        if (AMAX_OUT) mseg = max(mseg, max(__float_as_uint(b0), __float_as_uint(b1)));
      } else {
        // a step across segments: each chunk (part of one row) is in one
        const int cs = seg_advance(seg, ss.cur, cpr.div(c));
        ps = pair_scale(b0, b1, ldf(gs + cs));
        const uint32_t mb = max(__float_as_uint(b0), __float_as_uint(b1));
        if (AMAX_OUT && mb && TFP4_OK(amax_out + cs, 4)) atomicMax(amax_out + cs, mb);
      }
      quant_chunk(cur, ps, c, codes, bs, mma, cpr, guide);
    }
    cur = nxt;
  }
  if (AMAX_OUT && fseg >= 0) flush_seg_max(mseg, amax_out + fseg);
}

// Delayed scaling: gs[s] = amax[s] / 2688 from given maxima (binary32; a
// maximum that is not positive gives 0), as the amax kernel computes it.
__global__ void k_scales_from_amax(const float* __restrict__ amax, int32_t n,
                                   float* __restrict__ gs) {
  for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    if (!TFP4_OK(amax + i, 4) || !TFP4_OK(gs + i, 4)) continue;
    gs[i] = global_scale_of(__float_as_uint(amax[i]));
  }
}

// ---------------------------------------------------------------------------
// a1 + a2 fused: segment amax and quantisation in one cooperative launch
// ---------------------------------------------------------------------------
//
// The segments are grouped into waves of whole segments small enough to stay
// in L2 (host-planned, WaveParam, at most kWaveSegs segments each).  The
// 256-chunk steps of each wave are dealt to the CTAs, one CTA per SM, in
// contiguous ranges or round-robin (WaveCursor).  In each CTA two producer
// threads stage steps into shared memory with TMA copies (a 2-D tensor map
// with 128-byte swizzle when rows hold an even number of chunks, else
// cp.async.bulk; completion on mbarriers) on two rings:
//   - the amax producer streams this CTA's steps from HBM; four amax warps
//     fold per-segment maxima into shared memory and, at the end of each
//     wave, into amax_bits, then count the CTA done with that wave
//     (wave_cnt);
//   - the quantiser producer waits until every CTA has counted a wave, then
//     re-reads the same steps, from L2; two groups of eight quantiser warps
//     turn each staged chunk into codes, block scales and compact words with
//     gs = amax/2688.
// The amax stream leads the quantiser by a bounded number of steps, which
// bounds what L2 must hold, and otherwise never waits, so HBM streaming and
// quantisation overlap.
//
// The launch is cooperative (all CTAs co-resident).  Every wait is bounded
// by the same time limit: a wait that runs out sets *err (the outputs are
// then undefined) and gives up the cross-CTA waits that follow, and each
// producer waits for its own copies in flight before the CTA exits.


__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_l2(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}


// One thread: true once *p >= target; false after limit_ns (or a fixed
// number of polls, whichever comes first).
// Bounded waits read the global timer only once a wait has lasted a while:
// a timer read costs far more than a poll, and on a producer's path it would
// be paid on every step.
__device__ __noinline__ bool wait_at_least(const uint32_t* p, uint32_t target, uint64_t limit_ns) {
  for (uint32_t it = 0; it < 64; ++it) {
    if (ld_acquire(p) >= target) return true;
    __nanosleep(32);
  }
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 22); ++it) {
    if (ld_acquire(p) >= target) return true;
    __nanosleep(32);
    if ((it & 31u) == 31u && global_ns() - t0 > limit_ns) return false;
  }
  return false;
}

__device__ __forceinline__ void st_release_cta(int* p, int v) {
  asm volatile("st.release.cta.shared.s32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire_cta(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared.s32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}


// ---- TMA copies with an L2 policy -------------------------------------------

__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Chunk i of a staged step (64 B at 64 i).
__device__ __forceinline__ void smem_chunk(Chunk& c, const uint8_t* step, uint32_t i) {
  const uint4* p = reinterpret_cast<const uint4*>(step + 64u * i);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = p[q];
    c.w[4 * q + 0] = v.x;
    c.w[4 * q + 1] = v.y;
    c.w[4 * q + 2] = v.z;
    c.w[4 * q + 3] = v.w;
  }
}

// Packed |bf16| maximum of a 16-byte word (eight elements).
// Lane-wise |max| of a 16-byte word (lane signs junk: see absmax_bf16x2).
__device__ __forceinline__ uint32_t quad_max2(uint4 v) {
  return absmax_bf16x2(absmax_bf16x2(v.x, v.y), absmax_bf16x2(v.z, v.w));
}

__device__ __forceinline__ uint32_t max2_bits(uint32_t m) { return absmax_lanes_bits(m); }

// Number of CTAs c < bb in the cyclic range [o, o + R) of 0..G-1 (R < G).
__device__ __forceinline__ uint32_t extras_before(uint32_t bb, uint32_t o, uint32_t R,
                                                  uint32_t G) {
  if (o + R <= G) return min(max(bb, o), o + R) - o;
  return (bb > o ? bb - o : 0u) + min(bb, o + R - G);
}

// Step cursor over the waves.  Contiguous dealing: CTA b owns one
// contiguous range of each wave's nst steps, floor(nst / G) or one more, so
// consecutive steps of a CTA mostly stay in one segment (better when a wave
// holds many small segments: fewer global-scale lookups); which CTAs take
// the remainder rotates from wave to wave, since a wave completes only when
// its last CTA does.  Round-robin dealing: global step base + k goes to CTA
// (base + k) mod G (better when a wave holds few large segments: all CTAs
// stream neighbouring steps).  The host picks.
struct WaveCursor {
  int w;
  uint32_t kend, k, nst, c0, c1, base, contig;
  __device__ __forceinline__ void enter(const SegParam& seg, const WaveParam& wv, uint32_t cpr_u,
                                        uint32_t b, uint32_t G) {
    // skip waves in which this CTA owns no step
    while (w < wv.n) {
      c0 = (uint32_t)seg.off[wv.seg0[w]] * cpr_u;
      c1 = (uint32_t)seg.off[wv.seg0[w + 1]] * cpr_u;
      nst = (c1 - c0 + kThreads - 1) / kThreads;
      if (contig) {
        // q steps each, and one more for the R CTAs of the cyclic range
        // [o, o + R) with o = w R mod G: the CTAs that take the extra step
        // change from wave to wave, so none falls a step behind per wave
        const uint32_t q = nst / G, R = nst - q * G;
        const uint32_t o = (uint32_t)(((uint64_t)w * R) % G);
        k = b * q + extras_before(b, o, R, G);
        kend = (b + 1) * q + extras_before(b + 1, o, R, G);
      } else {
        const uint32_t r = base % G;
        k = b >= r ? b - r : b + G - r;
        kend = nst;
        base += nst;
      }
      if (k < kend) return;
      ++w;
    }
  }
  // advances to the next owned step, entering the next wave at a wave's end
  __device__ __forceinline__ void next(const SegParam& seg, const WaveParam& wv, uint32_t cpr_u,
                                       uint32_t b, uint32_t G) {
    k += contig ? 1u : G;
    if (k >= kend) {
      ++w;
      enter(seg, wv, cpr_u, b, G);
    }
  }
  __device__ __forceinline__ uint32_t step_chunk() const { return c0 + k * kThreads; }
  __device__ __forceinline__ uint32_t step_chunks() const {
    return min((uint32_t)kThreads, c1 - step_chunk());
  }
};

#ifndef TFP4_FUSED_SLOTS_A
#define TFP4_FUSED_SLOTS_A 5
#endif
#ifndef TFP4_FUSED_SLOTS_Q
#define TFP4_FUSED_SLOTS_Q 8
#endif
#ifndef TFP4_FUSED_AMAX_WARPS
#define TFP4_FUSED_AMAX_WARPS 4
#endif
#ifndef TFP4_FUSED_QUANT_GROUPS
#define TFP4_FUSED_QUANT_GROUPS 2
#endif
constexpr int kSlotsA = TFP4_FUSED_SLOTS_A;  // staged steps of the amax stream
constexpr int kSlotsQ = TFP4_FUSED_SLOTS_Q;  // staged steps of the quantiser
constexpr int kStepBytes = kThreads * 64;    // 256 chunks
constexpr int kAmaxWarps = TFP4_FUSED_AMAX_WARPS;
// Quantiser warps come in groups of eight (one chunk per thread of a step);
// group g takes the staged steps n with n mod kQuantGroups == g.
constexpr int kQuantGroups = TFP4_FUSED_QUANT_GROUPS, kQuantWarps = 8;
// warp 0: the amax stream's copies; warp 1: watches the wave counters and
// issues the quantiser stream's copies; then the amax warps and the
// quantiser groups
constexpr int kFirstAmaxWarp = 2;
constexpr int kFusedThreads = 32 * (kFirstAmaxWarp + kAmaxWarps + kQuantGroups * kQuantWarps);
static_assert(kSlotsQ % kQuantGroups == 0, "each quantiser group owns whole slots");
// The amax stream may always run through the wave the quantiser waits for;
// beyond it, it leads the quantiser by at most kLeadSteps staged steps (a
// bound on what L2 must hold: kLeadSteps x 16 KB per CTA).
#ifndef TFP4_FUSED_LEAD_STEPS
#define TFP4_FUSED_LEAD_STEPS 24
#endif
constexpr uint32_t kLeadSteps = TFP4_FUSED_LEAD_STEPS;

// Barrier of the amax warps only (id 1; 0 is __syncthreads).
__device__ __forceinline__ void amax_warps_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(32 * kAmaxWarps) : "memory");
}


// Slots are 1024-byte aligned: a 128-byte-swizzled TMA tile repeats its
// pattern every eight 128-byte rows.
struct FusedSmem {
  alignas(1024) uint8_t a[kSlotsA][kStepBytes];
  alignas(1024) uint8_t q[kSlotsQ][kStepBytes];
  uint64_t full_a[kSlotsA], empty_a[kSlotsA], full_q[kSlotsQ], empty_q[kSlotsQ];
  uint32_t smax[kWaveSegs];
};
constexpr size_t kFusedSmemBytes = sizeof(FusedSmem) + 1024;
static_assert(kFusedSmemBytes <= 227 * 1024, "one CTA per SM within the shared-memory opt-in");

// Swizzled staging (cols % 64 == 0): x is a 2-D tensor of 128-byte rows (two
// chunks each) and a step is one box of 128 rows, copied with 128-byte
// swizzle: 16-byte unit u of row r lands at unit u ^ (r mod 8).  Chunk i of
// the step is half i % 2 of row i / 2, so a quarter-warp reading one unit of
// eight consecutive chunks touches eight different bank groups.
__device__ __forceinline__ void smem_chunk_swz(Chunk& c, const uint8_t* step, uint32_t i) {
  const uint32_t row = i >> 1, h = (i & 1u) << 2, sw = row & 7u;
  const uint8_t* base = step + row * 128u;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = *reinterpret_cast<const uint4*>(base + (((h + q) ^ sw) << 4));
    c.w[4 * q + 0] = v.x;
    c.w[4 * q + 1] = v.y;
    c.w[4 * q + 2] = v.z;
    c.w[4 * q + 3] = v.w;
  }
}

// Step-local chunk held by physical 16-byte unit u of a swizzled step.
__device__ __forceinline__ uint32_t swz_unit_chunk(uint32_t u) {
  const uint32_t row = u >> 3;
  return 2u * row + ((((u & 7u) ^ (row & 7u))) >> 2);
}


__device__ __forceinline__ void tensor_load_2d_hint(void* dst, const CUtensorMap* map,
                                                    uint32_t c0, uint32_t c1, uint64_t* bar,
                                                    uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1),
      "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__global__ void __launch_bounds__(kFusedThreads, 1)
    k_rollout_fused(const uint8_t* __restrict__ x, uint32_t cpr_u, FastDivU cpr,
                    const __grid_constant__ SegParam seg, const __grid_constant__ WaveParam wv,
                    float* __restrict__ gs_out, uint8_t* __restrict__ codes,
                    uint8_t* __restrict__ bs, MmaOut mma, uint8_t* __restrict__ guide,
                    uint32_t* __restrict__ amax_bits, uint32_t* __restrict__ wave_cnt,
                    uint32_t* __restrict__ done, uint32_t* __restrict__ err,
                    uint32_t wait_extra, uint64_t wait_ns, uint32_t contig,
                    const __grid_constant__ CUtensorMap xmap, uint32_t swz) {
  extern __shared__ uint8_t smem_raw[];
  FusedSmem& sm = *reinterpret_cast<FusedSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ int is_last;
  // the quantiser producer's position: the wave it waits for or streams, and
  // its copies issued (the amax producer's lead bound)
  __shared__ int q_wave, q_issued;
  const uint32_t G = gridDim.x, b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    q_wave = 0;
    q_issued = 0;
    for (int i = 0; i < kSlotsA; ++i) {
      mbar_init(&sm.full_a[i], 1);
      mbar_init(&sm.empty_a[i], kAmaxWarps);
    }
    for (int i = 0; i < kSlotsQ; ++i) {
      mbar_init(&sm.full_q[i], 1);
      mbar_init(&sm.empty_q[i], kQuantWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = threadIdx.x; i < kWaveSegs; i += kFusedThreads) sm.smax[i] = 0u;
  __syncthreads();

  if (warp == 0) {
    // ---- amax producer: streams the CTA's steps from HBM into ring A ----
    if (lane == 0) {
      WaveCursor ca = {0, 0, 0, 0, 0, 0, 0, contig};
      ca.enter(seg, wv, cpr_u, b, G);
      uint32_t na = 0;  // copies issued
      bool broken = false;
      while (ca.w < wv.n) {
        // through the quantiser producer's wave, then at most kLeadSteps
        // steps ahead of its issued copies
        if (!broken) {
          uint64_t t0 = 0;
          uint32_t nap = 32;
          for (uint32_t it = 1;; ++it) {
            if (ca.w <= ld_acquire_cta(&q_wave) ||
                na - (uint32_t)ld_acquire_cta(&q_issued) < kLeadSteps)
              break;
            __nanosleep(nap);
            nap = nap < 1024u ? 2u * nap : nap;
            if ((it & 7u) == 0u) {
              const uint64_t t = global_ns();
              if (t0 == 0) {
                t0 = t;
              } else if (t - t0 > wait_ns || it > (1u << 22)) {
                atomicOr(err, 1u);
                broken = true;
                break;
              }
            }
          }
        }
        const uint32_t slot = na % kSlotsA, use = na / kSlotsA;
        if (use > 0 && !mbar_wait(&sm.empty_a[slot], (use - 1) & 1u, wait_ns, err)) break;
        // the consumers' generic-proxy reads of the slot come before the
        // copy's async-proxy writes
        fence_proxy_async();
        if (swz) {
          mbar_expect_tx(&sm.full_a[slot], kStepBytes);
          if (TFP4_OK(x + (uint64_t)(ca.step_chunk() >> 1) * 128u, 128))
            tensor_load_2d(sm.a[slot], &xmap, 0u, ca.step_chunk() >> 1, &sm.full_a[slot]);
        } else {
          const uint32_t bytes = ca.step_chunks() * 64u;
          mbar_expect_tx(&sm.full_a[slot], bytes);
          if (TFP4_OK(x + (uint64_t)ca.step_chunk() * 64u, bytes))
            bulk_load(sm.a[slot], x + (uint64_t)ca.step_chunk() * 64u, bytes, &sm.full_a[slot]);
        }
        ++na;
        ca.next(seg, wv, cpr_u, b, G);
      }
      // no copy may still be in flight when the CTA exits
      for (uint32_t i = 0; i < kSlotsA && i < na; ++i) {
        const uint32_t n = na - 1 - i, slot = n % kSlotsA;
        mbar_wait(&sm.full_a[slot], (n / kSlotsA) & 1u, wait_ns, err);
      }
    }
  } else if (warp == 1) {
    // ---- quantiser producer: wave by wave, waits until every CTA has
    // counted the wave's maxima, then re-reads the CTA's steps of the wave
    // (now from L2) into ring Q ----
    if (lane == 0) {
      uint64_t evict_first;
      asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(evict_first));
      WaveCursor cq = {0, 0, 0, 0, 0, 0, 0, contig};
      cq.enter(seg, wv, cpr_u, b, G);
      uint32_t nq = 0;  // copies issued
      bool broken = false, dead = false;
      for (int w = 0; w < wv.n && !dead; ++w) {
        st_release_cta(&q_wave, w);
        if (!broken && !wait_at_least(wave_cnt + w, G + wait_extra, wait_ns)) {
          atomicOr(err, 1u);
          broken = true;
        }
        for (; cq.w == w; cq.next(seg, wv, cpr_u, b, G)) {
          const uint32_t slot = nq % kSlotsQ, use = nq / kSlotsQ;
          if (use > 0 && !mbar_wait(&sm.empty_q[slot], (use - 1) & 1u, wait_ns, err)) {
            dead = true;
            break;
          }
          fence_proxy_async();
          if (swz) {
            mbar_expect_tx(&sm.full_q[slot], kStepBytes);
            if (TFP4_OK(x + (uint64_t)(cq.step_chunk() >> 1) * 128u, 128))
            tensor_load_2d_hint(sm.q[slot], &xmap, 0u, cq.step_chunk() >> 1, &sm.full_q[slot],
                                evict_first);
          } else {
            const uint32_t bytes = cq.step_chunks() * 64u;
            mbar_expect_tx(&sm.full_q[slot], bytes);
            if (TFP4_OK(x + (uint64_t)cq.step_chunk() * 64u, bytes))
            bulk_load_hint(sm.q[slot], x + (uint64_t)cq.step_chunk() * 64u, bytes,
                           &sm.full_q[slot], evict_first);
          }
          ++nq;
          st_release_cta(&q_issued, (int)nq);
        }
      }
      // lift the amax producer's lead bound before leaving
      st_release_cta(&q_wave, wv.n);
      for (uint32_t i = 0; i < kSlotsQ && i < nq; ++i) {
        const uint32_t n = nq - 1 - i, slot = n % kSlotsQ;
        mbar_wait(&sm.full_q[slot], (n / kSlotsQ) & 1u, wait_ns, err);
      }
    }
  } else if (warp < kFirstAmaxWarp + kAmaxWarps) {
    // ---- amax warps: per-segment maxima of each staged step ----
    const int t = threadIdx.x - 32 * kFirstAmaxWarp;  // 0..127
    WaveCursor c = {0, 0, 0, 0, 0, 0, 0, contig};
    c.enter(seg, wv, cpr_u, b, G);
    StepSeg ss;
    ss.cur = 0;
    uint32_t n = 0;
    bool broken = false;
    // every CTA counts itself done with every wave; waves in which it owns
    // no step are counted as soon as the cursor passes them
    int counted = 0;
    if (t == 0)
      for (; counted < c.w; ++counted)
        if (TFP4_OK(wave_cnt + counted, 4)) red_release_add(wave_cnt + counted, 1u);
    while (c.w < wv.n) {
      const int w = c.w;
      const int s0 = wv.seg0[w];
      const uint32_t slot = n % kSlotsA;
      if (!broken) broken = !mbar_wait(&sm.full_a[slot], (n / kSlotsA) & 1u, wait_ns, err);
      const uint32_t cs = c.step_chunk(), cnt = c.step_chunks();
      const bool uniform = ss.update(seg, cpr.div(cs), cpr.div(cs + cnt - 1));
      // 16-byte words dealt contiguously (a warp reads 512 B: no bank
      // conflicts); word u belongs to chunk cs + u/4
      const uint4* st4 = reinterpret_cast<const uint4*>(sm.a[slot]);
      const uint32_t nu = cnt * 4;
      if (uniform) {
        uint32_t m = 0;
        if (cnt == (uint32_t)kThreads) {
          // a full step: every unit holds data
#pragma unroll
          for (int j = 0; j < kStepBytes / 16 / (32 * kAmaxWarps); ++j)
            m = absmax_bf16x2(m, quad_max2(st4[t + 32 * kAmaxWarps * j]));
        } else if (swz) {
          // a swizzled step holds whole rows; skip units of chunks past cnt
#pragma unroll
          for (int j = 0; j < kStepBytes / 16 / (32 * kAmaxWarps); ++j) {
            const uint32_t u = t + 32 * kAmaxWarps * j;
            if (swz_unit_chunk(u) < cnt) m = absmax_bf16x2(m, quad_max2(st4[u]));
          }
        } else {
#pragma unroll
          for (int j = 0; j < kStepBytes / 16 / (32 * kAmaxWarps); ++j) {
            const uint32_t u = t + 32 * kAmaxWarps * j;
            if (u < nu) m = absmax_bf16x2(m, quad_max2(st4[u]));
          }
        }
        const uint32_t mw = __reduce_max_sync(0xFFFFFFFFu, max2_bits(m));
        if (lane == 0) {
          mbar_arrive(&sm.empty_a[slot]);
          if (mw) atomicMax(&sm.smax[ss.cur - s0], mw);
        }
      } else {
        for (int j = 0; j < kStepBytes / 16 / (32 * kAmaxWarps); ++j) {
          const uint32_t u = t + 32 * kAmaxWarps * j;
          const uint32_t lc = swz ? swz_unit_chunk(u) : u / 4;  // step-local chunk
          if (lc < cnt) {
            const uint32_t m = max2_bits(quad_max2(st4[u]));
            if (m) atomicMax(&sm.smax[seg_advance(seg, ss.cur, cpr.div(cs + lc)) - s0], m);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty_a[slot]);
      }
      ++n;
      c.next(seg, wv, cpr_u, b, G);
      if (c.w != w) {
        // wave w done here: publish its maxima, count this CTA for it and
        // for the skipped waves before the next one
        amax_warps_sync();
        for (int i = t; i < wv.seg0[w + 1] - s0; i += 32 * kAmaxWarps) {
          const uint32_t m = sm.smax[i];
          if (m) {
            if (TFP4_OK(amax_bits + s0 + i, 4)) atomicMax(amax_bits + s0 + i, m);
            sm.smax[i] = 0u;
          }
        }
        amax_warps_sync();
        if (t == 0)
          for (; counted < c.w; ++counted)
        if (TFP4_OK(wave_cnt + counted, 4)) red_release_add(wave_cnt + counted, 1u);
      }
    }
  } else {
    // ---- quantiser warps: one chunk of each staged step per thread ----
    const int qt = threadIdx.x - 32 * (kFirstAmaxWarp + kAmaxWarps);
    const int group = qt / (32 * kQuantWarps), t = qt % (32 * kQuantWarps);  // t: 0..255
    WaveCursor c = {0, 0, 0, 0, 0, 0, 0, contig};
    c.enter(seg, wv, cpr_u, b, G);
    StepSeg ss;
    ss.cur = 0;
    uint32_t n = 0;
    for (; n < (uint32_t)group && c.w < wv.n; ++n) c.next(seg, wv, cpr_u, b, G);
    bool broken = false;
    int gseg = -1;
    float g = 0.f;
    while (c.w < wv.n) {
      const uint32_t slot = n % kSlotsQ;
      if (!broken) broken = !mbar_wait(&sm.full_q[slot], (n / kSlotsQ) & 1u, wait_ns, err);
      const uint32_t cs = c.step_chunk(), cnt = c.step_chunks();
      const bool uniform = ss.update(seg, cpr.div(cs), cpr.div(cs + cnt - 1));
      if ((uint32_t)t < cnt) {
        Chunk ch;
        if (swz)
          smem_chunk_swz(ch, sm.q[slot], t);
        else
          smem_chunk(ch, sm.q[slot], t);
        const uint32_t cidx = cs + t;
        const int s = uniform ? ss.cur : seg_advance(seg, ss.cur, cpr.div(cidx));
        if (s != gseg) {
          gseg = s;
          g = TFP4_OK(amax_bits + s, 4) ? global_scale_of(ld_acquire(amax_bits + s)) : 0.0f;
        }
        quant_chunk(ch, chunk_scale(ch, g), cidx, codes, bs, mma, cpr, guide);
      }
      // release the slot only once every lane's values are in use
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty_q[slot]);
      for (int i = 0; i < kQuantGroups && c.w < wv.n; ++i) {
        ++n;
        c.next(seg, wv, cpr_u, b, G);
      }
    }
  }

  // The last CTA to finish writes the global scales and re-zeroes the
  // maxima and the wave counters for the next call (every CTA has finished
  // reading them by then).
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t ticket = TFP4_OK(done, 4) ? atomicAdd(done, 1u) : 0u;
    is_last = (ticket == G - 1);
  }
  __syncthreads();
  if (is_last) {
    __threadfence();
    // the global scales are written here, all at once: a producer that
    // wrote a wave's scales before streaming the wave would start it late
    for (int s = threadIdx.x; s < seg.n; s += kFusedThreads) {
      if (TFP4_OK(gs_out + s, 4) && TFP4_OK(amax_bits + s, 4)) {
        gs_out[s] = global_scale_of(ld_l2(amax_bits + s));
        amax_bits[s] = 0u;
      }
    }
    for (int w = threadIdx.x; w < wv.n; w += kFusedThreads)
      if (TFP4_OK(wave_cnt + w, 4)) wave_cnt[w] = 0u;
    if (threadIdx.x == 0 && TFP4_OK(done, 4)) *done = 0u;
  }
}

// ---------------------------------------------------------------------------
// a3: guide pack
// ---------------------------------------------------------------------------

constexpr int kPackPerThread = 4;  // 4 x 16 B of codes in flight per thread

__global__ void __launch_bounds__(kThreads)
    k_guide_pack(const uint8_t* __restrict__ codes, uint32_t nchunks, uint32_t steps_per_cta,
                 uint8_t* __restrict__ guide) {
  constexpr uint32_t kStep = kThreads * kPackPerThread;
  const uint32_t nsteps = (nchunks + kStep - 1) / kStep;
  uint32_t step = blockIdx.x * steps_per_cta;
  const uint32_t step_end = min(step + steps_per_cta, nsteps);
  for (; step < step_end; ++step) {
    uint4 v[kPackPerThread];
#pragma unroll
    for (int k = 0; k < kPackPerThread; ++k) {
      const uint32_t c = step * kStep + k * kThreads + threadIdx.x;
      if (c < nchunks) v[k] = ld_stream(codes + (uint64_t)c * 16u);
    }
#pragma unroll
    for (int k = 0; k < kPackPerThread; ++k) {
      const uint32_t c = step * kStep + k * kThreads + threadIdx.x;
      if (c < nchunks)
        st_stream2(guide + (uint64_t)c * 8u, compact_word(v[k].x, v[k].y),
                   compact_word(v[k].z, v[k].w));
    }
  }
}

// ---------------------------------------------------------------------------
// a4: guide unpack
// ---------------------------------------------------------------------------

// Eight bits (bit k = sign of element k) -> bit 3 of nibble k of a word.
__device__ __forceinline__ uint32_t signs_to_nibbles(uint32_t s8) {
  uint32_t t = (s8 | (s8 << 12)) & 0x000F000Fu;
  t = (t | (t << 6)) & 0x03030303u;
  t = (t | (t << 3)) & 0x11111111u;
  return t << 3;
}

// Two elements of one bf16x2 word -> their E2M1 magnitudes in the rollout
// frame (the signs are added per eight elements).
__device__ __forceinline__ F2 unpack_pair_mag(uint32_t w, float inv, uint32_t gw, int j0) {
  const uint32_t a = w & kAbs2;
  const F2 ax = {__uint_as_float(a << 16), __uint_as_float(a & 0xFFFF0000u)};
  return decode_pair(mul2_rn(ax, splat(inv)), gw, j0);
}

#ifndef TFP4_UNPACK_MIN_CTAS
#define TFP4_UNPACK_MIN_CTAS 4
#endif

__global__ void __launch_bounds__(kThreads, TFP4_UNPACK_MIN_CTAS)
    k_guide_unpack(const uint8_t* __restrict__ x, const uint8_t* __restrict__ guide,
                   const uint8_t* __restrict__ bs_r, const float* __restrict__ gs_r,
                   uint32_t nchunks, FastDivU cpr, uint32_t steps_per_cta,
                   const __grid_constant__ SegParam seg, uint8_t* __restrict__ codes) {
  const uint32_t nsteps = (nchunks + kThreads - 1) / kThreads;
  uint32_t step = blockIdx.x * steps_per_cta;
  const uint32_t step_end = min(step + steps_per_cta, nsteps);
  StepSeg ss;
  ss.cur = step < step_end ? seg_search(seg, cpr.div(step * kThreads)) : 0;
  __shared__ ScaleTab tab;
  int tseg = -1;

  Chunk cur, nxt;
  uint2 gcur = make_uint2(0, 0), gnxt = make_uint2(0, 0);
  uint32_t bcur = 0, bnxt = 0;
  if (step < step_end) {
    const uint32_t c = step * kThreads + threadIdx.x;
    if (c < nchunks) {
      load_chunk(cur, x, c);
      gcur = ld_stream2(guide + (uint64_t)c * 8u);
      bcur = ld_stream_u16(bs_r + (uint64_t)c * 2u);
    }
  }
  for (; step < step_end; ++step) {
    const uint32_t c0 = step * kThreads;
    const uint32_t c = c0 + threadIdx.x;
    if (step + 1 < step_end) {
      const uint32_t cn = c + kThreads;
      if (cn < nchunks) {
        load_chunk(nxt, x, cn);
        gnxt = ld_stream2(guide + (uint64_t)cn * 8u);
        bnxt = ld_stream_u16(bs_r + (uint64_t)cn * 2u);
      }
    }
    const uint32_t last = min(c0 + kThreads, nchunks) - 1;
    const bool uniform = ss.update(seg, cpr.div(c0), cpr.div(last));
    // per-segment table of S and 1/S for every code (rebuilt when a uniform
    // step enters a new segment)
    if (uniform && ss.cur != tseg) {
      __syncthreads();
      tseg = ss.cur;
      build_tab(tab, ldf(gs_r + tseg));
      __syncthreads();
    }
    if (c < nchunks) {
      const int s = uniform ? ss.cur : seg_advance(seg, ss.cur, cpr.div(c));
      float inv[2];
      if (uniform) {
        inv[0] = tab.sinv[bcur & 0x7Fu].y;
        inv[1] = tab.sinv[(bcur >> 8) & 0x7Fu].y;
      } else {
        const PairScale ps = pair_scale_stored(bcur, ldf(gs_r + s));
        inv[0] = ps.inv[0];
        inv[1] = ps.inv[1];
      }
      uint32_t out[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int b = q >> 1;
        const uint32_t gw = b ? gcur.y : gcur.x;
        F2 g[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          g[k] = unpack_pair_mag(cur.w[4 * q + k], inv[b], gw, (q & 1) * 8 + 2 * k);
        // the record's signs of these eight elements onto the nibbles
        out[q] = e2m1x8(g[0], g[1], g[2], g[3]) | signs_to_nibbles((gw >> ((q & 1) * 8)) & 0xFFu);
      }
      st_stream(codes + (uint64_t)c * 16u, out[0], out[1], out[2], out[3]);
    }
    cur = nxt;
    gcur = gnxt;
    bcur = bnxt;
  }
}

// ---------------------------------------------------------------------------
// straight-through backward: grad_in = grad_out where the mask bit is 1, +0
// elsewhere.  One chunk (32 elements, one mask word) per thread per step;
// each mask bit pair becomes a 0xFFFF / 0x0000 lane mask for a bf16x2 word
// (a mask byte's even and odd bits are first compacted into one word).
// ---------------------------------------------------------------------------

constexpr int kSteChunks = 2;  // chunks per thread per step (bytes in flight)

// Bits 0, 2, ..., 30 of x -> bits 0..15.
__device__ __forceinline__ uint32_t compact_even16(uint32_t x) {
  x &= 0x55555555u;
  x = (x | (x >> 1)) & 0x33333333u;
  x = (x | (x >> 2)) & 0x0F0F0F0Fu;
  x = (x | (x >> 4)) & 0x00FF00FFu;
  return (x | (x >> 8)) & 0x0000FFFFu;
}

__global__ void __launch_bounds__(kThreads)
    k_ste_backward(const uint8_t* __restrict__ g, const uint8_t* __restrict__ mask,
                   uint32_t nchunks, uint32_t steps_per_cta, uint8_t* __restrict__ out) {
  // a step is kSteChunks x 256 chunks; each warp instruction moves 512
  // contiguous bytes: thread t takes 16-byte words t + 256 j of the step
  // (eight elements, one byte of the mask)
  constexpr uint32_t kStep = kThreads * kSteChunks;
  constexpr int kWords = 4 * kSteChunks;  // 16-byte words per thread per step
  const uint32_t nsteps = (nchunks + kStep - 1) / kStep;
  const uint32_t nwords = nchunks * 4u;
  uint32_t step = blockIdx.x * steps_per_cta;
  const uint32_t step_end = min(step + steps_per_cta, nsteps);
  for (; step < step_end; ++step) {
    uint4 v[kWords];
    uint32_t mb[kWords];
#pragma unroll
    for (int j = 0; j < kWords; ++j) {
      const uint32_t u = step * kStep * 4u + j * kThreads + threadIdx.x;
      if (u < nwords) {
        v[j] = ld_stream(g + (uint64_t)u * 16u);
        unsigned short b;
        asm("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(b) : "l"(mask + u));
        mb[j] = b;
      }
    }
#pragma unroll
    for (int j = 0; j < kWords; ++j) {
      const uint32_t u = step * kStep * 4u + j * kThreads + threadIdx.x;
      if (u < nwords) {
        // mask byte: bit 2i / 2i+1 keeps the low / high element of bf16x2 word i
        const uint32_t P = compact_even16(mb[j]) | (compact_even16(mb[j] >> 1) << 16);
        const uint4 w = v[j];
        st_stream(out + (uint64_t)u * 16u, w.x & imad(P & 0x00010001u, 0xFFFFu, 0u),
                  w.y & imad((P >> 1) & 0x00010001u, 0xFFFFu, 0u),
                  w.z & imad((P >> 2) & 0x00010001u, 0xFFFFu, 0u),
                  w.w & imad((P >> 3) & 0x00010001u, 0xFFFFu, 0u));
      }
    }
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

cudaError_t launch_amax(const void* x, int64_t nchunks, int32_t cpr, const SegParam& seg,
                        const Scratch& s, float* gs_out, int sm_count, cudaStream_t st) {
  const Plan p = plan_for((const void*)k_amax, steps_of(nchunks, kThreads), sm_count);
  k_amax<<<p.grid, kThreads, 0, st>>>((const uint8_t*)x, (uint32_t)nchunks,
                                      FastDivU((uint32_t)cpr), p.steps_per_cta, seg,
                                      s.amax_bits, s.done, gs_out);
  return cudaGetLastError();
}

cudaError_t launch_rollout_quant(const void* x, int64_t nchunks, int32_t cpr,
                                 const SegParam& seg, const float* gs, void* codes, void* bs,
                                 MmaOut mma, uint32_t* guide, int sm_count, cudaStream_t st) {
  const Plan p =
      plan_for((const void*)k_rollout_quant<false>, steps_of(nchunks, kThreads), sm_count);
  k_rollout_quant<false><<<p.grid, kThreads, 0, st>>>(
      (const uint8_t*)x, (uint32_t)nchunks, FastDivU((uint32_t)cpr), p.steps_per_cta, seg, gs,
      (uint8_t*)codes, (uint8_t*)bs, mma, (uint8_t*)guide, nullptr);
  return cudaGetLastError();
}

cudaError_t launch_scales_from_amax(const float* amax, int32_t n, float* gs, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  k_scales_from_amax<<<(n + 255) / 256, 256, 0, st>>>(amax, n, gs);
  return cudaGetLastError();
}

cudaError_t launch_rollout_quant_delayed(const void* x, int64_t nchunks, int32_t cpr,
                                         const SegParam& seg, const float* amax_in, float* gs,
                                         void* codes, void* bs, MmaOut mma, uint32_t* guide,
                                         float* amax_out, int sm_count, cudaStream_t st) {
  cudaError_t e = launch_scales_from_amax(amax_in, seg.n, gs, st);
  if (e != cudaSuccess || nchunks == 0) return e;
  if (amax_out) {
    const Plan p =
        plan_for((const void*)k_rollout_quant<true>, steps_of(nchunks, kThreads), sm_count);
    k_rollout_quant<true><<<p.grid, kThreads, 0, st>>>(
        (const uint8_t*)x, (uint32_t)nchunks, FastDivU((uint32_t)cpr), p.steps_per_cta, seg, gs,
        (uint8_t*)codes, (uint8_t*)bs, mma, (uint8_t*)guide, reinterpret_cast<uint32_t*>(amax_out));
    return cudaGetLastError();
  }
  return launch_rollout_quant(x, nchunks, cpr, seg, gs, codes, bs, mma, guide, sm_count, st);
}

// Largest x bytes a single segment may hold on the fused path: two waves of
// reads plus the writes in between stay well inside the 126 MB of L2.
constexpr int64_t kWaveMaxBytes = int64_t(40) << 20;

bool plan_waves(const SegParam& seg, int32_t cols, int64_t wave_bytes, WaveParam* wv) {
  const int64_t row_bytes = int64_t(cols) * 2;
  wv->n = 0;
  int s = 0;
  while (s < seg.n) {
    const int start = s;
    int64_t bytes = int64_t(seg.off[s + 1] - seg.off[s]) * row_bytes;
    if (bytes > kWaveMaxBytes) return false;
    ++s;
    while (s < seg.n && s - start < kWaveSegs) {
      const int64_t b = int64_t(seg.off[s + 1] - seg.off[s]) * row_bytes;
      if (bytes + b > wave_bytes) break;
      bytes += b;
      ++s;
    }
    wv->seg0[wv->n++] = (uint16_t)start;
  }
  wv->seg0[wv->n] = (uint16_t)seg.n;
  return true;
}

#ifndef TFP4_FUSED_SWIZZLE
#define TFP4_FUSED_SWIZZLE 1
#endif

// The driver's tensor-map encoder, looked up once through the runtime (no
// link against the driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      (void)cudaGetLastError();
  });
  return fn;
}

// x viewed as rows of 128 bytes (two chunks), one box = one step of 128 rows,
// copied with 128-byte swizzle.  Returns false (bulk copies are used) when the
// rows of x hold an odd number of chunks or the encoder is unavailable.
bool encode_step_map(const void* x, int64_t nchunks, int32_t cpr, CUtensorMap* map) {
  if (!TFP4_FUSED_SWIZZLE || (cpr & 1) || (nchunks & 1) || nchunks < 2 ||
      (reinterpret_cast<uintptr_t>(x) & 15u))
    return false;
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dim[2] = {64, (cuuint64_t)(nchunks / 2)};
  const cuuint64_t stride[1] = {128};
  const cuuint32_t box[2] = {64, kStepBytes / 128};
  const cuuint32_t estride[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(x), dim, stride, box,
             estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_rollout_fused(const void* x, int64_t nchunks, int32_t cpr, const SegParam& seg,
                                 const WaveParam& wv, const Scratch& s, float* gs_out,
                                 void* codes, void* bs, MmaOut mma, uint32_t* guide, int sm_count,
                                 uint32_t wait_extra, uint64_t wait_ns, cudaStream_t st) {
  // the shared-memory opt-in and the occupancy, once per device
  static std::mutex mu;
  static int occ_of[64];
  static bool set_for[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int occ;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!set_for[dev]) {
      e = cudaFuncSetAttribute(k_rollout_fused, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kFusedSmemBytes);
      if (e != cudaSuccess) return e;
      int n = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_rollout_fused, kFusedThreads,
                                                        kFusedSmemBytes);
      if (e != cudaSuccess) return e;
      occ_of[dev] = n;
      set_for[dev] = true;
    }
    occ = occ_of[dev];
  }
  if (occ < 1) return cudaErrorCooperativeLaunchTooLarge;
  // contiguous step ranges when a wave averages three or more segments
  const uint32_t contig = seg.n >= 3 * wv.n ? 1u : 0u;
  int64_t g = (int64_t)sm_count * occ;
  const int64_t nsteps = steps_of(nchunks, kThreads);
  if (nsteps < g) g = nsteps;
  if (g < 1) g = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)g);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = kFusedSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  CUtensorMap xmap;
  memset(&xmap, 0, sizeof(xmap));
  const uint32_t swz = encode_step_map(x, nchunks, cpr, &xmap) ? 1u : 0u;
  return cudaLaunchKernelEx(&cfg, k_rollout_fused, (const uint8_t*)x, (uint32_t)cpr,
                            FastDivU((uint32_t)cpr), seg, wv, gs_out, (uint8_t*)codes,
                            (uint8_t*)bs, mma, (uint8_t*)guide, s.amax_bits, s.wave_cnt, s.done,
                            s.err, wait_extra, wait_ns, contig, xmap, swz);
}

cudaError_t launch_guide_pack(const void* codes, int64_t nchunks, uint32_t* guide,
                              int sm_count, cudaStream_t st) {
  const Plan p = plan_for((const void*)k_guide_pack,
                          steps_of(nchunks, (int64_t)kThreads * kPackPerThread), sm_count);
  k_guide_pack<<<p.grid, kThreads, 0, st>>>((const uint8_t*)codes, (uint32_t)nchunks,
                                            p.steps_per_cta, (uint8_t*)guide);
  return cudaGetLastError();
}

cudaError_t launch_guide_unpack(const void* x_ref, const uint32_t* guide, const void* bs_r,
                                const float* gs_r, int64_t nchunks, int32_t cpr,
                                const SegParam& seg_r, void* codes, int sm_count,
                                cudaStream_t st) {
  const Plan p = plan_for((const void*)k_guide_unpack, steps_of(nchunks, kThreads), sm_count);
  k_guide_unpack<<<p.grid, kThreads, 0, st>>>(
      (const uint8_t*)x_ref, (const uint8_t*)guide, (const uint8_t*)bs_r, gs_r,
      (uint32_t)nchunks, FastDivU((uint32_t)cpr), p.steps_per_cta, seg_r, (uint8_t*)codes);
  return cudaGetLastError();
}

cudaError_t launch_ste_backward(const void* g, const uint32_t* mask, int64_t nchunks, void* out,
                                int sm_count, cudaStream_t st) {
  const Plan p = plan_for((const void*)k_ste_backward,
                          steps_of(nchunks, (int64_t)kThreads * kSteChunks), sm_count);
  k_ste_backward<<<p.grid, kThreads, 0, st>>>((const uint8_t*)g, (const uint8_t*)mask,
                                              (uint32_t)nchunks, p.steps_per_cta, (uint8_t*)out);
  return cudaGetLastError();
}

cudaError_t dbg_set_ranges_kernels(const DbgRanges& r, cudaStream_t st) {
  return dbg_set_here(r, st);
}
unsigned long long dbg_take_kernels() { return dbg_take_here(); }

}  // namespace tfp4
