// trace_kernels.cu - sm_103a kernels of the guided-NVFP4 hot path of TRACE.
//
// Sources: "Alibaba Qwen Proposes TRACE for 5.4x Faster FP4 RL Rollouts",
// section "TRACE Core Concept" (rollout records FP4 results; training-side
// fake quantisation picks the adjacent E2M1 point closer to the rollout's;
// a compact record of mantissa bit + scale sets the direction) and the
// worked example of section "Why Does FP4 Rollout 'Break' RL Training?".
//
// Work decomposition.  Every kernel streams a flat sequence of 32-element
// "chunks" (two 16-element NVFP4 blocks, one STE mask word).  Rows hold
// cols/32 chunks, so a chunk never straddles a row or a segment.  A CTA of
// 256 threads handles a "step" of 256 consecutive chunks (16 KiB of bf16),
// one chunk per thread, and owns a contiguous range of steps; the next
// step's loads are issued before the current step is computed.  Segments
// are looked up once per step (uniform across the CTA); only a step that
// straddles a segment boundary resolves segments per thread.
//
// Arithmetic.  All of it is binary32 with round-to-nearest-even (explicit
// __f*_rn intrinsics so nothing is contracted into an FMA; no flush to zero),
// in the same operation order as the method's definition:
//   gs = amax / 2688;  bs = e4m3(bamax / (gs * 6));  S = dec(bs) * gs;
//   inv = 1 / S (0 if S == 0 or the reciprocal overflows);  t = |x| * inv.
// E2M1 rounding uses directed-rounding adds against a constant C whose ulp
// equals the E2M1 spacing of t's binade (C = 1.5 * 2^(22+e), 2^e the binade
// of max(t, 1), t clamped to 6): fl_rz(t + C) - C, fl_rp(t + C) - C and
// fl_rn(t + C) - C are exactly the lower, upper and nearest E2M1 points
// (ties go to the even index because C is an even number of ulps), and the
// last significand bit of fl_rz(t + C) is the parity of the lower index.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <unordered_map>

#include "trace_internal.h"

namespace tfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kWaveSegs = 256;  // segments per wave of the fused rollout kernel
constexpr uint32_t kAbs2 = 0x7FFF7FFFu;

// ---------------------------------------------------------------------------
// memory access
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_stream2(const void* p) {
  uint2 v;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_stream_u16(const void* p) {
  unsigned short v;
  asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(void* p, uint32_t a, uint32_t b, uint32_t c,
                                          uint32_t d) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void st_stream2(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void st_stream1(void* p, uint32_t a) {
  asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}

__device__ __forceinline__ void st_stream_u16(void* p, uint32_t a) {
  asm volatile("st.global.cs.u16 [%0], %1;" ::"l"(p), "h"((unsigned short)a) : "memory");
}

struct Chunk {
  uint32_t w[16];  // 32 bf16: element 2i in the low half of w[i]
};

__device__ __forceinline__ void load_chunk(Chunk& c, const uint8_t* base, uint32_t chunk) {
  const uint8_t* p = base + (uint64_t)chunk * 64u;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = ld_stream(p + 16 * q);
    c.w[4 * q + 0] = v.x;
    c.w[4 * q + 1] = v.y;
    c.w[4 * q + 2] = v.z;
    c.w[4 * q + 3] = v.w;
  }
}

// ---------------------------------------------------------------------------
// segments
// ---------------------------------------------------------------------------

// Largest s with off[s] <= row (off[n] = rows > row); with empty segments the
// non-empty one is found.
__device__ __forceinline__ int seg_search(const SegParam& p, uint32_t row) {
  int lo = 0, hi = p.n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((uint32_t)p.off[mid] <= row) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ int seg_advance(const SegParam& p, int s, uint32_t row) {
  while ((uint32_t)p.off[s + 1] <= row) ++s;
  return s;
}

// Per-step segment resolution: `cur` follows the step's first row; update()
// returns true when the whole step lies inside segment `cur`.
struct StepSeg {
  int cur;
  __device__ __forceinline__ bool update(const SegParam& p, uint32_t r0, uint32_t r1) {
    cur = seg_advance(p, cur, r0);
    return (uint32_t)p.off[cur + 1] > r1;
  }
};

// ---------------------------------------------------------------------------
// scales
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Eight words of masked bf16 magnitudes -> binary32 bits of their maximum.
__device__ __forceinline__ float block_amax8(const uint32_t* a) {
  uint32_t m0 = max_u16x2(a[0], a[1]);
  const uint32_t m1 = max_u16x2(a[2], a[3]);
  const uint32_t m2 = max_u16x2(a[4], a[5]);
  const uint32_t m3 = max_u16x2(a[6], a[7]);
  m0 = max_u16x2(max_u16x2(m0, m1), max_u16x2(m2, m3));
  const uint32_t hi = m0 >> 16, lo = m0 & 0xFFFFu;
  return __uint_as_float((hi > lo ? hi : lo) << 16);
}

// E4M3 code -> binary32: placing the 7 magnitude bits at bit 20 gives the
// value times 2^-120 (normal and subnormal codes alike); scaling by 2^120 is
// exact.
__device__ __forceinline__ float e4m3_decode(uint32_t code) {
  return __fmul_rn(__uint_as_float(code << 20), 0x1p120f);
}

__device__ __forceinline__ float global_scale_of(uint32_t amax_bits) {
  const float amax = __uint_as_float(amax_bits);
  if (!(amax > 0.0f)) return 0.0f;
  const float gs = __fdiv_rn(amax, 2688.0f);
  return gs > 0.0f ? gs : 0.0f;
}

struct PairScale {
  uint32_t codes;  // byte 0: block 0, byte 1: block 1
  float S[2];
  float inv[2];
};

__device__ __forceinline__ void real_scale(uint32_t code, float gs, float& S, float& inv) {
  S = __fmul_rn(e4m3_decode(code), gs);
  float r = 0.0f;
  if (S > 0.0f) {
    r = __frcp_rn(S);
    if (r == __int_as_float(0x7F800000)) r = 0.0f;  // reciprocal overflow: flush
  }
  inv = r;
}

// Two binary32 values -> two E4M3 codes (RNE, satfinite): byte 0 = lo.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  unsigned short c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(hi), "f"(lo));
  return c;
}

// Both blocks' E4M3 scales from their maxima and the segment scale.
//
// The method divides: q = bamax / (gs * 6), rounded once.  An IEEE division
// costs about twenty integer-pipe instructions, so the quotient is first
// formed as q' = bamax * fl(1 / (gs * 6)), which lies within 2.5 ulp of q.
// E4M3 encoding is monotone, so when q' * (1 - 2^-21) and q' * (1 + 2^-21)
// (a bracket around q) encode to the same code, that code is the code of q.
// Otherwise -- q within a few ulps of an E4M3 rounding boundary, or a
// reciprocal that overflows -- the correctly rounded division decides.
// E4M3 codes of both blocks given den = gs * 6 and rden = fl(1 / den).
__device__ __forceinline__ uint32_t pair_codes(float bamax0, float bamax1, float gs, float den,
                                               float rden) {
  uint32_t codes = 0;
  if (gs > 0.0f) {
    bool exact = !(rden < __int_as_float(0x7F800000));
    if (!exact) {
      const float q0 = __fmul_rn(bamax0, rden), q1 = __fmul_rn(bamax1, rden);
      const uint32_t lo = e4m3x2(__fmul_rn(q0, 1.0f - 0x1p-21f), __fmul_rn(q1, 1.0f - 0x1p-21f));
      const uint32_t hi = e4m3x2(__fmul_rn(q0, 1.0f + 0x1p-21f), __fmul_rn(q1, 1.0f + 0x1p-21f));
      codes = lo;
      exact = lo != hi;
    }
    if (exact) codes = e4m3x2(__fdiv_rn(bamax0, den), __fdiv_rn(bamax1, den));
  }
  return codes;
}

__device__ __forceinline__ PairScale pair_scale(float bamax0, float bamax1, float gs) {
  const float den = __fmul_rn(gs, 6.0f);
  const uint32_t codes = pair_codes(bamax0, bamax1, gs, den, gs > 0.0f ? __frcp_rn(den) : 0.0f);
  PairScale p;
  p.codes = codes;
  real_scale(codes & 0xFFu, gs, p.S[0], p.inv[0]);
  real_scale(codes >> 8, gs, p.S[1], p.inv[1]);
  return p;
}

// STE threshold of a block in bf16 magnitude bits, doubled into two 16-bit
// lanes with the lane top bits set: |x| > 6 * S exactly when the bf16 |x|
// exceeds 6 * S rounded down to bf16 (truncation), so for a word of two
// magnitudes, bit 15 / 31 of thr2 - |x| is set exactly when the element is
// kept (no borrow crosses the lanes).
__device__ __forceinline__ uint32_t ste_threshold2(float S) {
  const uint32_t thr = S > 0.0f ? (__float_as_uint(__fmul_rn(6.0f, S)) >> 16) : 0x7FFFu;
  return (thr | 0x8000u) * 0x00010001u;
}

// Per-segment table in shared memory, indexed by E4M3 code: the block's real
// scale, its reciprocal (flush rule applied) and STE threshold.  A segment's
// blocks take one of at most 127 scales, so the reciprocals are formed once
// per segment instead of once per block.  Codes above 0x7E never come out of
// the quantiser; a stored code is masked to 7 bits before the lookup.
struct ScaleTab {
  float2 sinv[128];
  uint32_t thr2[128];
};

__device__ __forceinline__ void build_tab(ScaleTab& t, float gs) {
  for (int c = threadIdx.x; c < 128; c += blockDim.x) {
    float S, inv;
    real_scale((uint32_t)c, gs, S, inv);
    t.sinv[c] = make_float2(S, inv);
    t.thr2[c] = ste_threshold2(S);
  }
}

// Real scales of two stored E4M3 codes (the rollout side's record).
__device__ __forceinline__ PairScale pair_scale_stored(uint32_t codes, float gs) {
  PairScale p;
  p.codes = codes;
  real_scale(codes & 0x7Fu, gs, p.S[0], p.inv[0]);
  real_scale((codes >> 8) & 0x7Fu, gs, p.S[1], p.inv[1]);
  return p;
}

// ---------------------------------------------------------------------------
// packed binary32 pairs (f32x2 instructions: one issue slot for two lanes)
// ---------------------------------------------------------------------------

struct F2 {
  float x, y;
};

#define TFP4_F2_OP(name, inst)                                                      \
  __device__ __forceinline__ F2 name(F2 a, F2 b) {                                   \
    F2 d;                                                                           \
    asm("{ .reg .b64 A, B, D; mov.b64 A, {%2, %3}; mov.b64 B, {%4, %5}; " inst       \
        " D, A, B; mov.b64 {%0, %1}, D; }"                                          \
        : "=f"(d.x), "=f"(d.y)                                                      \
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));                                  \
    return d;                                                                       \
  }
TFP4_F2_OP(add2_rn, "add.rn.f32x2")
TFP4_F2_OP(add2_rz, "add.rz.f32x2")
TFP4_F2_OP(add2_rp, "add.rp.f32x2")
TFP4_F2_OP(sub2_rn, "sub.rn.f32x2")
TFP4_F2_OP(mul2_rn, "mul.rn.f32x2")
#undef TFP4_F2_OP

__device__ __forceinline__ F2 fma2_rn(F2 a, F2 b, F2 c) {
  F2 d;
  asm("{ .reg .b64 A, B, C, D; mov.b64 A, {%2, %3}; mov.b64 B, {%4, %5}; "
      "mov.b64 C, {%6, %7}; fma.rn.f32x2 D, A, B, C; mov.b64 {%0, %1}, D; }"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ F2 splat(float v) { return F2{v, v}; }

// Multiply-add on the FMA pipe (IMAD): a * b + c, wrapping.
__device__ __forceinline__ uint32_t imad(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ float fma_sat(float a, float b, float c) {
  float d;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ---------------------------------------------------------------------------
// E2M1
// ---------------------------------------------------------------------------

// Two signed binary32 values -> one byte of two E2M1 nibbles (lo = first).
// Hardware RTN, ties to even, saturating at +-6, sign kept.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b8 b; cvt.rn.satfinite.e2m1x2.f32 b, %1, %2; cvt.u32.u8 %0, b; }"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// The rounding constant for t in [0, 6]: 1.5 * 2^(22 + e) with 2^e the
// binade of max(t, 1).
__device__ __forceinline__ float magic_of(float tc) {
  uint32_t e = __float_as_uint(tc) & 0x7F800000u;
  e = e > 0x3F800000u ? e : 0x3F800000u;
  return __uint_as_float(e + 0x0B400000u);
}

// The same constant for a pair of clamped values.  Two exact formulations:
// TFP4_MAGIC_FMA = 1 builds it on the FMA pipe from two saturating
// indicators, b1 = [tc > 2] and b2 = [tc > 4] (sat(tc * 2^30 - 2^31) is 0 for
// tc <= 2 and 1 otherwise: the next binary32 above 2 is 2 + 2^-22), then
// C = K * (1 + b1) * (1 + b2), K = 1.5 * 2^22; otherwise it takes the
// exponent field with integer operations.  At tc = 2 or 4 both constants put
// the (on-grid) value on the grid, so the boundary side does not matter.
#ifndef TFP4_MAGIC_FMA
#define TFP4_MAGIC_FMA 1
#endif
__device__ __forceinline__ F2 magic_pair(F2 tc) {
#if TFP4_MAGIC_FMA
  const float k = 0x1.8p22f;
  const F2 b1 = {fma_sat(tc.x, 0x1p30f, -0x1p31f), fma_sat(tc.y, 0x1p30f, -0x1p31f)};
  const F2 b2 = {fma_sat(tc.x, 0x1p30f, -0x1p32f), fma_sat(tc.y, 0x1p30f, -0x1p32f)};
  const F2 m1 = fma2_rn(b1, splat(k), splat(k));
  return fma2_rn(b2, m1, m1);
#else
  return F2{magic_of(tc.x), magic_of(tc.y)};
#endif
}

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
    if (m) atomicMax(dst, m);
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
      if (c < nchunks && m) atomicMax(amax_bits + seg_advance(seg, ss.cur, cpr.div(c)), m);
    }
    cur = nxt;
  }
  if (open >= 0) cta_flush_max(run, amax_bits + open, red);

  // The last CTA to finish turns maxima into global scales and re-zeroes the
  // maxima for the next call.  No CTA ever waits for another.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t ticket = atomicAdd(done, 1u);
    is_last = (ticket == gridDim.x - 1);
  }
  __syncthreads();
  if (is_last) {
    __threadfence();
    for (int s = threadIdx.x; s < seg.n; s += kThreads) {
      const uint32_t a = atomicExch(amax_bits + s, 0u);
      gs_out[s] = global_scale_of(a);
    }
    if (threadIdx.x == 0) atomicExch(done, 0u);
  }
}

// ---------------------------------------------------------------------------
// compact word helpers
// ---------------------------------------------------------------------------

// Eight nibbles -> the 8 bits found at nibble bit `b` (0: index LSB, 3: sign).
__device__ __forceinline__ uint32_t gather_nibble_bit(uint32_t w, int b) {
  uint32_t v = (w >> b) & 0x11111111u;
  v = (v | (v >> 3)) & 0x03030303u;
  v = (v | (v >> 6)) & 0x000F000Fu;
  v = (v | (v >> 12)) & 0x000000FFu;
  return v;
}

// Sixteen nibbles (one block, two words) -> compact word.
__device__ __forceinline__ uint32_t compact_word(uint32_t c0, uint32_t c1) {
  const uint32_t sgn = gather_nibble_bit(c0, 3) | (gather_nibble_bit(c1, 3) << 8);
  const uint32_t lsb = gather_nibble_bit(c0, 0) | (gather_nibble_bit(c1, 0) << 8);
  return sgn | (lsb << 16);
}

// ---------------------------------------------------------------------------
// a2: rollout quantisation
// ---------------------------------------------------------------------------

// One chunk (two blocks) -> 16 code bytes, two block-scale codes and two
// compact words, given the segment's global scale g.
__device__ __forceinline__ void quant_chunk(const Chunk& cur, float g, uint32_t c,
                                            uint8_t* __restrict__ codes, uint8_t* __restrict__ bs,
                                            uint8_t* __restrict__ guide) {
  uint32_t a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = cur.w[i] & kAbs2;
  const PairScale ps = pair_scale(block_amax8(a), block_amax8(a + 8), g);
  uint32_t out[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float inv = ps.inv[q >> 1];
    uint32_t word = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t w = cur.w[4 * q + k];
      // signed x * inv keeps the input's sign in the nibble
      const uint32_t b = e2m1x2(__fmul_rn(__uint_as_float(w << 16), inv),
                                __fmul_rn(__uint_as_float(w & 0xFFFF0000u), inv));
      word |= b << (8 * k);
    }
    out[q] = word;
  }
  st_stream(codes + (uint64_t)c * 16u, out[0], out[1], out[2], out[3]);
  st_stream_u16(bs + (uint64_t)c * 2u, ps.codes);
  if (guide)
    st_stream2(guide + (uint64_t)c * 8u, compact_word(out[0], out[1]), compact_word(out[2], out[3]));
}

__global__ void __launch_bounds__(kThreads)
    k_rollout_quant(const uint8_t* __restrict__ x, uint32_t nchunks, FastDivU cpr,
                    uint32_t steps_per_cta, const __grid_constant__ SegParam seg,
                    const float* __restrict__ gs, uint8_t* __restrict__ codes,
                    uint8_t* __restrict__ bs, uint8_t* __restrict__ guide) {
  const uint32_t nsteps = (nchunks + kThreads - 1) / kThreads;
  uint32_t step = blockIdx.x * steps_per_cta;
  const uint32_t step_end = min(step + steps_per_cta, nsteps);
  StepSeg ss;
  ss.cur = step < step_end ? seg_search(seg, cpr.div(step * kThreads)) : 0;

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
    if (c < nchunks) {
      const int s = uniform ? ss.cur : seg_advance(seg, ss.cur, cpr.div(c));
      quant_chunk(cur, gs[s], c, codes, bs, guide);
    }
    cur = nxt;
  }
}

// ---------------------------------------------------------------------------
// a1 + a2 fused: segment amax and quantisation in one cooperative launch
// ---------------------------------------------------------------------------
//
// The segments are grouped into waves of whole segments small enough to stay
// in L2 (host-planned, WaveParam, at most kWaveSegs segments each).  The
// 256-chunk steps of the call are dealt round-robin to the CTAs, one CTA
// per SM.  In each CTA one producer thread stages steps into shared memory
// with TMA bulk copies (cp.async.bulk, completion on mbarriers) on two
// rings (a second thread watches the cross-CTA wave counters for it):
//   - the amax ring streams this CTA's steps from HBM; four amax warps fold
//     per-segment maxima into shared memory and, at the end of each wave,
//     into amax_bits, then count the CTA done with that wave (wave_cnt);
//   - the quantiser ring re-reads the same steps of an earlier wave, from
//     L2, once every CTA has counted that wave; eight quantiser warps turn
//     each staged chunk into codes, block scales and compact words with
//     gs = amax/2688.
// The amax stream leads the quantiser by a bounded number of steps, which
// bounds what L2 must hold, and otherwise never waits, so HBM streaming and
// quantisation overlap.
//
// The launch is cooperative (all CTAs co-resident).  Every wait is bounded:
// the producer gives up the cross-CTA waits once nothing has moved for the
// time limit (setting *err, the outputs are then undefined), every mbarrier
// wait has the same limit, and the producer waits for its own copies in
// flight before the CTA exits.

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

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

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// One thread: true once *p >= target; false after limit_ns (or a fixed
// number of polls, whichever comes first).
__device__ __noinline__ bool wait_at_least(const uint32_t* p, uint32_t target, uint64_t limit_ns) {
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

// First step of wave-local steps [0, nst) that CTA b owns when steps are
// dealt round-robin over the whole call, the wave's first step being global
// step `base`.
__device__ __forceinline__ uint32_t first_owned(uint32_t base, uint32_t b, uint32_t G) {
  const uint32_t r = base % G;
  return b >= r ? b - r : b + G - r;
}

// ---- TMA bulk copies and mbarriers -------------------------------------------


__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Non-blocking: has the phase with this parity completed?
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for a phase; false (and *err set) once limit_ns has passed.
__device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                       uint32_t* err) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 22); ++it) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 15u) == 15u && global_ns() - t0 > limit_ns) break;
  }
  atomicOr(err, 2u);
  return false;
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// bytes (a multiple of 16) from global src to shared dst, completing on bar
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

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
__device__ __forceinline__ uint32_t quad_max2(uint4 v) {
  return max_u16x2(max_u16x2(v.x & kAbs2, v.y & kAbs2), max_u16x2(v.z & kAbs2, v.w & kAbs2));
}

__device__ __forceinline__ uint32_t max2_bits(uint32_t m) {
  const uint32_t hi = m >> 16, lo = m & 0xFFFFu;
  return (hi > lo ? hi : lo) << 16;
}

// Step cursor over the waves: the k-th owned step of wave w, dealt
// round-robin over the whole call (global step base + k goes to CTA
// (base + k) mod G).
struct WaveCursor {
  int w;
  uint32_t base, k, nst, c0, c1;
  __device__ __forceinline__ void enter(const SegParam& seg, const WaveParam& wv, uint32_t cpr_u,
                                        uint32_t b, uint32_t G) {
    // skip waves in which this CTA owns no step
    while (w < wv.n) {
      c0 = (uint32_t)seg.off[wv.seg0[w]] * cpr_u;
      c1 = (uint32_t)seg.off[wv.seg0[w + 1]] * cpr_u;
      nst = (c1 - c0 + kThreads - 1) / kThreads;
      k = first_owned(base, b, G);
      if (k < nst) return;
      base += nst;
      ++w;
    }
  }
  // advances to the next owned step; returns the wave it left when a wave ends
  __device__ __forceinline__ void next(const SegParam& seg, const WaveParam& wv, uint32_t cpr_u,
                                       uint32_t b, uint32_t G) {
    k += G;
    if (k >= nst) {
      base += nst;
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
#define TFP4_FUSED_SLOTS_A 6
#endif
#ifndef TFP4_FUSED_SLOTS_Q
#define TFP4_FUSED_SLOTS_Q 6
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
// warp 0: copies; warp 1: watches the wave counters; then the amax warps
// and the quantiser groups
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

struct FusedSmem {
  alignas(128) uint8_t a[kSlotsA][kStepBytes];
  alignas(128) uint8_t q[kSlotsQ][kStepBytes];
  uint64_t full_a[kSlotsA], empty_a[kSlotsA], full_q[kSlotsQ], empty_q[kSlotsQ];
  uint32_t smax[kWaveSegs];
};
constexpr size_t kFusedSmemBytes = sizeof(FusedSmem) + 128;

#ifndef TFP4_FUSED_EVICT_FIRST
#define TFP4_FUSED_EVICT_FIRST 1
#endif

__global__ void __launch_bounds__(kFusedThreads, 1)
    k_rollout_fused(const uint8_t* __restrict__ x, uint32_t cpr_u, FastDivU cpr,
                    const __grid_constant__ SegParam seg, const __grid_constant__ WaveParam wv,
                    float* __restrict__ gs_out, uint8_t* __restrict__ codes,
                    uint8_t* __restrict__ bs, uint8_t* __restrict__ guide,
                    uint32_t* __restrict__ amax_bits, uint32_t* __restrict__ wave_cnt,
                    uint32_t* __restrict__ done, uint32_t* __restrict__ err,
                    uint32_t wait_extra, uint64_t wait_ns) {
  extern __shared__ uint8_t smem_raw[];
  FusedSmem& sm = *reinterpret_cast<FusedSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  __shared__ int is_last;
  __shared__ int ready_w;  // highest wave whose maxima are complete in every CTA
  const uint32_t G = gridDim.x, b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    ready_w = -1;
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
    // ---- producer: one thread issues every copy ----
    if (lane == 0) {
      uint64_t evict_first;
      asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(evict_first));
      WaveCursor ca = {0, 0, 0, 0, 0, 0}, cq = {0, 0, 0, 0, 0, 0};
      ca.enter(seg, wv, cpr_u, b, G);
      cq.enter(seg, wv, cpr_u, b, G);
      uint32_t na = 0, nq = 0;  // copies issued into each ring
      bool broken = false;
      uint64_t idle_since = 0;
      while (ca.w < wv.n || cq.w < wv.n) {
        bool progress = false;
        // quantiser stream: wave cq.w once every CTA has counted it
        if (cq.w < wv.n) {
          const uint32_t slot = nq % kSlotsQ, use = nq / kSlotsQ;
          if ((broken || ld_acquire_cta(&ready_w) >= cq.w) &&
              (use == 0 || mbar_test(&sm.empty_q[slot], (use - 1) & 1u))) {
            // the consumers' generic-proxy reads of the slot come before
            // the copy's async-proxy writes
            fence_proxy_async();
            const uint32_t bytes = cq.step_chunks() * 64u;
            mbar_expect_tx(&sm.full_q[slot], bytes);
#if TFP4_FUSED_EVICT_FIRST
            bulk_load_hint(sm.q[slot], x + (uint64_t)cq.step_chunk() * 64u, bytes,
                           &sm.full_q[slot], evict_first);
#else
            bulk_load(sm.q[slot], x + (uint64_t)cq.step_chunk() * 64u, bytes, &sm.full_q[slot]);
#endif
            ++nq;
            cq.next(seg, wv, cpr_u, b, G);
            progress = true;
          }
        }
        // amax stream: through the quantiser's wave, then at most
        // kLeadSteps ahead of it
        if (ca.w < wv.n && (ca.w <= cq.w || na - nq < kLeadSteps)) {
          const uint32_t slot = na % kSlotsA, use = na / kSlotsA;
          if (use == 0 || mbar_test(&sm.empty_a[slot], (use - 1) & 1u)) {
            fence_proxy_async();
            const uint32_t bytes = ca.step_chunks() * 64u;
            mbar_expect_tx(&sm.full_a[slot], bytes);
            bulk_load(sm.a[slot], x + (uint64_t)ca.step_chunk() * 64u, bytes, &sm.full_a[slot]);
            ++na;
            ca.next(seg, wv, cpr_u, b, G);
            progress = true;
          }
        }
        if (progress) {
          idle_since = 0;
        } else {
          const uint64_t t = global_ns();
          if (idle_since == 0) {
            idle_since = t;
          } else if (t - idle_since > wait_ns) {
            // nothing moved for the whole limit: give up the cross-CTA waits
            if (broken) break;
            atomicOr(err, 1u);
            broken = true;
            idle_since = 0;
          }
          __nanosleep(32);
        }
      }
      // no copy may still be in flight when the CTA exits
      for (uint32_t i = 0; i < kSlotsA && i < na; ++i) {
        const uint32_t n = na - 1 - i, slot = n % kSlotsA;
        mbar_wait(&sm.full_a[slot], (n / kSlotsA) & 1u, wait_ns, err);
      }
      for (uint32_t i = 0; i < kSlotsQ && i < nq; ++i) {
        const uint32_t n = nq - 1 - i, slot = n % kSlotsQ;
        mbar_wait(&sm.full_q[slot], (n / kSlotsQ) & 1u, wait_ns, err);
      }
    }
  } else if (warp == 1) {
    // ---- watcher: publishes, wave by wave, that every CTA has counted it,
    // and writes the global scales of the waves w with w mod G == b ----
    if (lane == 0) {
      bool broken = false;
      for (int w = 0; w < wv.n; ++w) {
        if (!broken && !wait_at_least(wave_cnt + w, G + wait_extra, wait_ns)) {
          atomicOr(err, 1u);
          broken = true;
        }
        if (b == (uint32_t)w % G) {
          for (int s = wv.seg0[w]; s < wv.seg0[w + 1]; ++s)
            gs_out[s] = global_scale_of(ld_l2(amax_bits + s));
        }
        st_release_cta(&ready_w, w);
      }
    }
  } else if (warp < kFirstAmaxWarp + kAmaxWarps) {
    // ---- amax warps: per-segment maxima of each staged step ----
    const int t = threadIdx.x - 32 * kFirstAmaxWarp;  // 0..127
    WaveCursor c = {0, 0, 0, 0, 0, 0};
    c.enter(seg, wv, cpr_u, b, G);
    StepSeg ss;
    ss.cur = 0;
    uint32_t n = 0;
    bool broken = false;
    // every CTA counts itself done with every wave; waves in which it owns
    // no step are counted as soon as the cursor passes them
    int counted = 0;
    if (t == 0)
      for (; counted < c.w; ++counted) red_release_add(wave_cnt + counted, 1u);
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
#pragma unroll
        for (int j = 0; j < kStepBytes / 16 / (32 * kAmaxWarps); ++j) {
          const uint32_t u = t + 32 * kAmaxWarps * j;
          if (u < nu) m = max_u16x2(m, quad_max2(st4[u]));
        }
        const uint32_t mw = __reduce_max_sync(0xFFFFFFFFu, max2_bits(m));
        if (lane == 0) {
          mbar_arrive(&sm.empty_a[slot]);
          if (mw) atomicMax(&sm.smax[ss.cur - s0], mw);
        }
      } else {
        for (int j = 0; j < kStepBytes / 16 / (32 * kAmaxWarps); ++j) {
          const uint32_t u = t + 32 * kAmaxWarps * j;
          if (u < nu) {
            const uint32_t m = max2_bits(quad_max2(st4[u]));
            if (m) atomicMax(&sm.smax[seg_advance(seg, ss.cur, cpr.div(cs + u / 4)) - s0], m);
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
            atomicMax(amax_bits + s0 + i, m);
            sm.smax[i] = 0u;
          }
        }
        amax_warps_sync();
        if (t == 0)
          for (; counted < c.w; ++counted) red_release_add(wave_cnt + counted, 1u);
      }
    }
  } else {
    // ---- quantiser warps: one chunk of each staged step per thread ----
    const int qt = threadIdx.x - 32 * (kFirstAmaxWarp + kAmaxWarps);
    const int group = qt / (32 * kQuantWarps), t = qt % (32 * kQuantWarps);  // t: 0..255
    WaveCursor c = {0, 0, 0, 0, 0, 0};
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
        smem_chunk(ch, sm.q[slot], t);
        const uint32_t cidx = cs + t;
        const int s = uniform ? ss.cur : seg_advance(seg, ss.cur, cpr.div(cidx));
        if (s != gseg) {
          gseg = s;
          g = global_scale_of(ld_acquire(amax_bits + s));
        }
        quant_chunk(ch, g, cidx, codes, bs, guide);
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

  // The last CTA to finish re-zeroes the maxima and the wave counters for
  // the next call (every CTA has finished reading them by then).
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t ticket = atomicAdd(done, 1u);
    is_last = (ticket == G - 1);
  }
  __syncthreads();
  if (is_last) {
    __threadfence();
    for (int s = threadIdx.x; s < seg.n; s += kFusedThreads) amax_bits[s] = 0u;
    for (int w = threadIdx.x; w < wv.n; w += kFusedThreads) wave_cnt[w] = 0u;
    if (threadIdx.x == 0) *done = 0u;
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

// Rollout-frame decode of a pair from the compact record: for each element
// the bracket member of t_r whose index parity equals its stored bit (a
// point bracket ignores the bit).  gw is the block's compact word and j0 the
// first element's index: the parity of the lower member (bit 0 of the
// rz-sum) is moved up to the stored bit's position (16 + j) by a multiply
// and compared there.  Returns the two E2M1 magnitudes.
__device__ __forceinline__ F2 decode_pair(F2 tr, uint32_t gw, int j0) {
  const F2 tc = {fminf(tr.x, 6.0f), fminf(tr.y, 6.0f)};
  const F2 C = magic_pair(tc);
  const F2 uz = add2_rz(tc, C), up = add2_rp(tc, C);
  const uint32_t b0 = 1u << (16 + j0), b1 = 1u << (17 + j0);
  const uint32_t m0 = (imad(__float_as_uint(uz.x), b0, 0u) ^ gw) & b0;
  const uint32_t m1 = (imad(__float_as_uint(uz.y), b1, 0u) ^ gw) & b1;
  const F2 us = {m0 ? up.x : uz.x, m1 ? up.y : uz.y};
  return sub2_rn(us, C);
}

// Two elements of one bf16x2 word -> one byte of rollout codes.  j0 is the
// index of the word's low element inside its 16-element block.
__device__ __forceinline__ uint32_t unpack_pair(uint32_t w, float inv, uint32_t gw, int j0) {
  const uint32_t a = w & kAbs2;
  const F2 ax = {__uint_as_float(a << 16), __uint_as_float(a & 0xFFFF0000u)};
  const F2 g = decode_pair(mul2_rn(ax, splat(inv)), gw, j0);
  // signs from the record; E2M1 conversion of exact grid points gives indices
  const float g0 = __uint_as_float(__float_as_uint(g.x) | ((gw << (31 - j0)) & 0x80000000u));
  const float g1 = __uint_as_float(__float_as_uint(g.y) | ((gw << (30 - j0)) & 0x80000000u));
  return e2m1x2(g0, g1);
}

__global__ void __launch_bounds__(kThreads)
    k_guide_unpack(const uint8_t* __restrict__ x, const uint8_t* __restrict__ guide,
                   const uint8_t* __restrict__ bs_r, const float* __restrict__ gs_r,
                   uint32_t nchunks, FastDivU cpr, uint32_t steps_per_cta,
                   const __grid_constant__ SegParam seg, uint8_t* __restrict__ codes) {
  const uint32_t nsteps = (nchunks + kThreads - 1) / kThreads;
  uint32_t step = blockIdx.x * steps_per_cta;
  const uint32_t step_end = min(step + steps_per_cta, nsteps);
  StepSeg ss;
  ss.cur = step < step_end ? seg_search(seg, cpr.div(step * kThreads)) : 0;

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
    if (c < nchunks) {
      const int s = uniform ? ss.cur : seg_advance(seg, ss.cur, cpr.div(c));
      const PairScale ps = pair_scale_stored(bcur, gs_r[s]);
      uint32_t out[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int b = q >> 1;
        const uint32_t gw = b ? gcur.y : gcur.x;
        uint32_t word = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j0 = (q & 1) * 8 + 2 * k;
          word |= unpack_pair(cur.w[4 * q + k], ps.inv[b], gw, j0) << (8 * k);
        }
        out[q] = word;
      }
      st_stream(codes + (uint64_t)c * 16u, out[0], out[1], out[2], out[3]);
    }
    cur = nxt;
    gcur = gnxt;
    bcur = bnxt;
  }
}

// ---------------------------------------------------------------------------
// a5 + a6: training-side guided fake quantisation
// ---------------------------------------------------------------------------

// Signed E2M1 values of a byte's two nibbles (hardware E2M1 -> f16 decode).
__device__ __forceinline__ void e2m1x2_values(uint32_t byte, float& v0, float& v1) {
  uint32_t h;
  asm("{ .reg .b8 b; cvt.u8.u32 b, %1; cvt.rn.f16x2.e2m1x2 %0, b; }" : "=r"(h) : "r"(byte));
  const unsigned short lo = (unsigned short)(h & 0xFFFFu), hi = (unsigned short)(h >> 16);
  asm("cvt.f32.f16 %0, %1;" : "=f"(v0) : "h"(lo));
  asm("cvt.f32.f16 %0, %1;" : "=f"(v1) : "h"(hi));
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

struct Counters {
  uint32_t mm_rtn, mm_g, h_rtn[4], h_g[4];
};

// exact signed grid value -> signed E2M1 index (+0 and -0 both give 0)
__device__ __forceinline__ int signed_index(float g_signed) {
  const uint32_t n = e2m1x2(g_signed, 0.0f) & 0xFu;
  const int m = (int)(n & 7u);
  return (n & 8u) ? -m : m;
}

__device__ __forceinline__ void count(Counters& k, int k_r, int k_rtn, int k_g) {
  int d0 = k_rtn - k_r, d1 = k_g - k_r;
  d0 = d0 < 0 ? -d0 : d0;
  d1 = d1 < 0 ? -d1 : d1;
  k.mm_rtn += d0 != 0;
  k.mm_g += d1 != 0;
  k.h_rtn[0] += d0 == 0;
  k.h_rtn[1] += d0 == 1;
  k.h_rtn[2] += d0 == 2;
  k.h_rtn[3] += d0 >= 3;
  k.h_g[0] += d1 == 0;
  k.h_g[1] += d1 == 1;
  k.h_g[2] += d1 == 2;
  k.h_g[3] += d1 >= 3;
}

__device__ __forceinline__ float fmul_sat(float a, float b) {
  float d;
  asm("mul.rn.sat.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// Training side of one pair of elements.  ax holds |x|; St holds the
// training scale carrying each element's sign, vr the rollout's
// reconstructed values with the rollout's signs, so the candidates
// v_c = G[c] * St are the signed values the method compares and the chosen
// one is the signed output.  ym receives the chosen signed values; with
// WANT_G, gsel / grtn receive the chosen and the RTN E2M1 magnitudes.
//
// The choice: hi wins when |d_hi| < |d_lo|, or on equality when RTN is hi.
// diff = |d_lo| - |d_hi| is exact in sign (and +0 only on equality), and
// RTN-is-hi is bits(s_rn) - bits(s_rz), 0 or 1, so hi <=> bits(diff) +
// rtn_hi - 1 >= 0 as a signed integer; the select is done on the bit
// patterns: y = v_hi - lo * (v_hi - v_lo) with lo = 0 or 1.
template <bool GUIDED, bool WANT_G>
__device__ __forceinline__ void train_pair(F2 ax, float inv_t, F2 St, F2 vr, F2& ym, F2& gsel,
                                           F2& grtn) {
  const F2 t = mul2_rn(ax, splat(inv_t));
  const F2 tc = {fminf(t.x, 6.0f), fminf(t.y, 6.0f)};
  const F2 C = magic_pair(tc);
  const F2 sn = add2_rn(tc, C);
  if (!GUIDED) {
    const F2 g = sub2_rn(sn, C);
    ym = mul2_rn(g, St);
    gsel = g;
    grtn = g;
    return;
  }
  const F2 sz = add2_rz(tc, C), sp = add2_rp(tc, C);
  const F2 glo = sub2_rn(sz, C), ghi = sub2_rn(sp, C);
  const F2 vlo = mul2_rn(glo, St), vhi = mul2_rn(ghi, St);
  const F2 dlo = sub2_rn(vlo, vr), dhi = sub2_rn(vhi, vr);
  const float diff0 = __fsub_rn(fabsf(dlo.x), fabsf(dhi.x));
  const float diff1 = __fsub_rn(fabsf(dlo.y), fabsf(dhi.y));
#if TFP4_SELECT_IMAD
  // lo = key >> 31 as the high word of key * 2; v_lo - v_hi on bit patterns
  const uint32_t k0 = __float_as_uint(diff0) + __float_as_uint(sn.x) + ~__float_as_uint(sz.x);
  const uint32_t k1 = __float_as_uint(diff1) + __float_as_uint(sn.y) + ~__float_as_uint(sz.y);
  const uint32_t lo0 = __umulhi(k0, 2u), lo1 = __umulhi(k1, 2u);
  const uint32_t h0 = __float_as_uint(vhi.x), h1 = __float_as_uint(vhi.y);
  ym = F2{__uint_as_float(imad(lo0, imad(h0, 0xFFFFFFFFu, __float_as_uint(vlo.x)), h0)),
          __uint_as_float(imad(lo1, imad(h1, 0xFFFFFFFFu, __float_as_uint(vlo.y)), h1))};
#else
  const uint32_t lo0 = (__float_as_uint(diff0) + __float_as_uint(sn.x) + ~__float_as_uint(sz.x)) >> 31;
  const uint32_t lo1 = (__float_as_uint(diff1) + __float_as_uint(sn.y) + ~__float_as_uint(sz.y)) >> 31;
  const uint32_t h0 = __float_as_uint(vhi.x), h1 = __float_as_uint(vhi.y);
  ym = F2{__uint_as_float(imad(lo0, __float_as_uint(vlo.x) - h0, h0)),
          __uint_as_float(imad(lo1, __float_as_uint(vlo.y) - h1, h1))};
#endif
  if (WANT_G) {
    gsel = F2{lo0 ? glo.x : ghi.x, lo1 ? glo.y : ghi.y};
    grtn = F2{sn.x != sz.x ? ghi.x : glo.x, sn.y != sz.y ? ghi.y : glo.y};
  }
}

// Spreads the 16 low bits of v to the even bit positions.
__device__ __forceinline__ uint32_t spread16(uint32_t v) {
  v = (v | (v << 8)) & 0x00FF00FFu;
  v = (v | (v << 4)) & 0x0F0F0F0Fu;
  v = (v | (v << 2)) & 0x33333333u;
  v = (v | (v << 1)) & 0x55555555u;
  return v;
}

#ifndef TFP4_FQ_PREFETCH
#define TFP4_FQ_PREFETCH 0
#endif
#ifndef TFP4_FQ_MIN_CTAS
#define TFP4_FQ_MIN_CTAS 4
#endif
template <int KIND, bool MASK, bool CODES, bool STATS>
__global__ void __launch_bounds__(kThreads, TFP4_FQ_MIN_CTAS)
    k_fakequant(const uint8_t* __restrict__ x, uint32_t nchunks, FastDivU cpr,
                uint32_t steps_per_cta, const __grid_constant__ SegParam seg_t,
                const float* __restrict__ gs_t, const __grid_constant__ SegParam seg_r,
                const uint8_t* __restrict__ guide, const uint8_t* __restrict__ bs_r,
                const float* __restrict__ gs_r, uint8_t* __restrict__ y,
                uint8_t* __restrict__ mask, uint8_t* __restrict__ codes_t,
                trace_stats_t* __restrict__ stats) {
  constexpr bool GUIDED = KIND != TRACE_GUIDE_NONE;
  const uint32_t nsteps = (nchunks + kThreads - 1) / kThreads;
  uint32_t step = blockIdx.x * steps_per_cta;
  const uint32_t step_end = min(step + steps_per_cta, nsteps);
  StepSeg st, sr;
  st.cur = 0;
  sr.cur = 0;
  if (step < step_end) {
    const uint32_t r0 = cpr.div(step * kThreads);
    st.cur = seg_search(seg_t, r0);
    if (GUIDED) sr.cur = seg_search(seg_r, r0);
  }
  Counters cnt = {};
  uint32_t n_done = 0;
  __shared__ ScaleTab tab_t, tab_r;
  int tseg = -1, rseg = -1;                 // segments the tables hold
  float seg_gs = 0.0f, seg_den = 0.0f, seg_rden = 0.0f;

  Chunk cur, nxt;
  uint4 gcur = make_uint4(0, 0, 0, 0), gnxt = make_uint4(0, 0, 0, 0);
  uint32_t bcur = 0, bnxt = 0;
  if (step < step_end) {
    const uint32_t c = step * kThreads + threadIdx.x;
    if (c < nchunks) {
      load_chunk(cur, x, c);
      if (KIND == TRACE_GUIDE_COMPACT) {
        const uint2 v = ld_stream2(guide + (uint64_t)c * 8u);
        gcur.x = v.x;
        gcur.y = v.y;
      } else if (KIND == TRACE_GUIDE_FULL) {
        gcur = ld_stream(guide + (uint64_t)c * 16u);
      }
      if (GUIDED) bcur = ld_stream_u16(bs_r + (uint64_t)c * 2u);
    }
  }
  for (; step < step_end; ++step) {
    const uint32_t c0 = step * kThreads;
    const uint32_t c = c0 + threadIdx.x;
    if (TFP4_FQ_PREFETCH && step + 1 < step_end) {
      const uint32_t cn = c + kThreads;
      if (cn < nchunks) {
        load_chunk(nxt, x, cn);
        if (KIND == TRACE_GUIDE_COMPACT) {
          const uint2 v = ld_stream2(guide + (uint64_t)cn * 8u);
          gnxt.x = v.x;
          gnxt.y = v.y;
        } else if (KIND == TRACE_GUIDE_FULL) {
          gnxt = ld_stream(guide + (uint64_t)cn * 16u);
        }
        if (GUIDED) bnxt = ld_stream_u16(bs_r + (uint64_t)cn * 2u);
      }
    }
    const uint32_t r0 = cpr.div(c0), r1 = cpr.div(min(c0 + kThreads, nchunks) - 1);
    const bool uni_t = st.update(seg_t, r0, r1);
    const bool uni_r = GUIDED ? sr.update(seg_r, r0, r1) : true;
    // refresh the scale tables when the (uniform) segment changes
    const bool new_t = uni_t && st.cur != tseg;
    const bool new_r = GUIDED && uni_r && sr.cur != rseg;
    if (new_t || new_r) {
      __syncthreads();
      if (new_t) {
        tseg = st.cur;
        seg_gs = gs_t[tseg];
        seg_den = __fmul_rn(seg_gs, 6.0f);
        seg_rden = seg_gs > 0.0f ? __frcp_rn(seg_den) : 0.0f;
        build_tab(tab_t, seg_gs);
      }
      if (new_r) {
        rseg = sr.cur;
        build_tab(tab_r, gs_r[rseg]);
      }
      __syncthreads();
    }
    if (c < nchunks) {
      int s_t = st.cur, s_r = sr.cur;
      if (!uni_t || !uni_r) {
        const uint32_t row = cpr.div(c);
        if (!uni_t) s_t = seg_advance(seg_t, st.cur, row);
        if (GUIDED && !uni_r) s_r = seg_advance(seg_r, sr.cur, row);
      }
      uint32_t a[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) a[i] = cur.w[i] & kAbs2;
      PairScale pt, pr = {};
      uint32_t thr2[2];
      if (uni_t) {
        pt.codes = pair_codes(block_amax8(a), block_amax8(a + 8), seg_gs, seg_den, seg_rden);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const uint32_t code = (pt.codes >> (8 * b)) & 0xFFu;
          const float2 e = tab_t.sinv[code];
          pt.S[b] = e.x;
          pt.inv[b] = e.y;
          thr2[b] = tab_t.thr2[code];
        }
      } else {
        pt = pair_scale(block_amax8(a), block_amax8(a + 8), gs_t[s_t]);
        thr2[0] = ste_threshold2(pt.S[0]);
        thr2[1] = ste_threshold2(pt.S[1]);
      }
      if (GUIDED) {
        if (uni_r) {
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const float2 e = tab_r.sinv[(bcur >> (8 * b)) & 0x7Fu];
            pr.S[b] = e.x;
            pr.inv[b] = e.y;
          }
        } else {
          pr = pair_scale_stored(bcur, gs_r[s_r]);
        }
      }

      uint32_t ybits[4];
      uint32_t cbytes[16];
      uint32_t kept = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int b = i >> 3;        // block of this word
        const int j0 = (i & 7) * 2;  // index of its low element in the block
        const uint32_t w = cur.w[i];
        const F2 ax = {__uint_as_float(imad(a[i], 0x10000u, 0u)), __uint_as_float(a[i] & 0xFFFF0000u)};
        const uint32_t sx0 = imad(w, 0x10000u, 0u) & 0x80000000u, sx1 = w & 0x80000000u;
        const uint32_t Stb = __float_as_uint(pt.S[b]);
        const F2 St = {__uint_as_float(Stb | sx0), __uint_as_float(Stb | sx1)};
        F2 vr = {0.0f, 0.0f};
        F2 grs = {0.0f, 0.0f};  // signed rollout magnitudes (statistics)
        if (KIND == TRACE_GUIDE_COMPACT) {
          const uint32_t gw = b ? gcur.y : gcur.x;
          const F2 gr = decode_pair(mul2_rn(ax, splat(pr.inv[b])), gw, j0);
          const uint32_t sr0 = imad(gw, 1u << (31 - j0), 0u) & 0x80000000u;
          const uint32_t sr1 = imad(gw, 1u << (30 - j0), 0u) & 0x80000000u;
          const uint32_t Sb = __float_as_uint(pr.S[b]);
          vr = mul2_rn(gr, F2{__uint_as_float(Sb | sr0), __uint_as_float(Sb | sr1)});
          if (STATS) grs = F2{__uint_as_float(__float_as_uint(gr.x) | sr0),
                              __uint_as_float(__float_as_uint(gr.y) | sr1)};
        } else if (KIND == TRACE_GUIDE_FULL) {
          const uint32_t gword = (i < 4) ? gcur.x : (i < 8) ? gcur.y : (i < 12) ? gcur.z : gcur.w;
          float g0, g1;
          e2m1x2_values((gword >> (8 * (i & 3))) & 0xFFu, g0, g1);
          vr = mul2_rn(F2{g0, g1}, splat(pr.S[b]));
          if (STATS) grs = F2{g0, g1};
        }
        F2 ym, gsel, grtn;
        train_pair<GUIDED, CODES || STATS>(ax, pt.inv[b], St, vr, ym, gsel, grtn);
        ybits[i & 3] = bf16x2_rn(ym.x, ym.y);
        if ((i & 3) == 3)
          st_stream(y + (uint64_t)c * 64u + 16 * (i >> 2), ybits[0], ybits[1], ybits[2], ybits[3]);
        if (MASK) kept = (kept >> 1) | (imad(a[i], 0xFFFFFFFFu, thr2[b]) & 0x80008000u);
        if (CODES || STATS) {
          const float g0 = __uint_as_float(__float_as_uint(gsel.x) | sx0);
          const float g1 = __uint_as_float(__float_as_uint(gsel.y) | sx1);
          if (CODES) cbytes[i] = e2m1x2(g0, g1);
          if (STATS && GUIDED) {
            count(cnt, signed_index(grs.x),
                  signed_index(__uint_as_float(__float_as_uint(grtn.x) | sx0)), signed_index(g0));
            count(cnt, signed_index(grs.y),
                  signed_index(__uint_as_float(__float_as_uint(grtn.y) | sx1)), signed_index(g1));
          }
        }
      }
      // word i left its two bits at positions i and 16 + i: interleave
      if (MASK) kept = spread16(kept & 0xFFFFu) | (spread16(kept >> 16) << 1);
      if (MASK) st_stream1(mask + (uint64_t)c * 4u, kept);
      if (CODES) {
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          o[q] = cbytes[4 * q] | (cbytes[4 * q + 1] << 8) | (cbytes[4 * q + 2] << 16) |
                 (cbytes[4 * q + 3] << 24);
        st_stream(codes_t + (uint64_t)c * 16u, o[0], o[1], o[2], o[3]);
      }
      if (STATS) n_done += 32;
    }
    if (TFP4_FQ_PREFETCH) {
      cur = nxt;
      gcur = gnxt;
      bcur = bnxt;
    } else if (step + 1 < step_end) {
      const uint32_t cn = c + kThreads;
      if (cn < nchunks) {
        load_chunk(cur, x, cn);
        if (KIND == TRACE_GUIDE_COMPACT) {
          const uint2 v = ld_stream2(guide + (uint64_t)cn * 8u);
          gcur.x = v.x;
          gcur.y = v.y;
        } else if (KIND == TRACE_GUIDE_FULL) {
          gcur = ld_stream(guide + (uint64_t)cn * 16u);
        }
        if (GUIDED) bcur = ld_stream_u16(bs_r + (uint64_t)cn * 2u);
      }
    }
  }
  if (STATS) {
    const uint32_t v[11] = {n_done,       cnt.mm_rtn,   cnt.mm_g,     cnt.h_rtn[0],
                            cnt.h_rtn[1], cnt.h_rtn[2], cnt.h_rtn[3], cnt.h_g[0],
                            cnt.h_g[1],   cnt.h_g[2],   cnt.h_g[3]};
    unsigned long long* dst = reinterpret_cast<unsigned long long*>(stats);
#pragma unroll
    for (int k = 0; k < 11; ++k) {
      if (!GUIDED && k > 0) break;
      const uint32_t tot = __reduce_add_sync(0xFFFFFFFFu, v[k]);
      if ((threadIdx.x & 31) == 0 && tot) atomicAdd(dst + k, (unsigned long long)tot);
    }
  }
}

// ---------------------------------------------------------------------------
// straight-through backward: grad_in = grad_out where the mask bit is 1, +0
// elsewhere.  One chunk (32 elements, one mask word) per thread per step;
// each mask bit pair becomes a 0xFFFF / 0x0000 lane mask for a bf16x2 word.
// ---------------------------------------------------------------------------

constexpr int kSteChunks = 2;  // chunks per thread per step (bytes in flight)

__global__ void __launch_bounds__(kThreads)
    k_ste_backward(const uint8_t* __restrict__ g, const uint8_t* __restrict__ mask,
                   uint32_t nchunks, uint32_t steps_per_cta, uint8_t* __restrict__ out) {
  constexpr uint32_t kStep = kThreads * kSteChunks;
  const uint32_t nsteps = (nchunks + kStep - 1) / kStep;
  uint32_t step = blockIdx.x * steps_per_cta;
  const uint32_t step_end = min(step + steps_per_cta, nsteps);
  for (; step < step_end; ++step) {
    Chunk v[kSteChunks];
    uint32_t m[kSteChunks];
#pragma unroll
    for (int k = 0; k < kSteChunks; ++k) {
      const uint32_t c = step * kStep + k * kThreads + threadIdx.x;
      if (c < nchunks) {
        load_chunk(v[k], g, c);
        unsigned int mw;
        asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(mw) : "l"(mask + (uint64_t)c * 4u));
        m[k] = mw;
      }
    }
#pragma unroll
    for (int k = 0; k < kSteChunks; ++k) {
      const uint32_t c = step * kStep + k * kThreads + threadIdx.x;
      if (c < nchunks) {
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          // bits 2i, 2i+1 -> lane masks (0 - bit keeps all 16 lane bits)
          const uint32_t lo = (0u - ((m[k] >> (2 * i)) & 1u)) & 0x0000FFFFu;
          const uint32_t hi = (0u - ((m[k] >> (2 * i + 1)) & 1u)) & 0xFFFF0000u;
          o[i] = v[k].w[i] & (lo | hi);
        }
        uint8_t* p = out + (uint64_t)c * 64u;
#pragma unroll
        for (int q = 0; q < 4; ++q) st_stream(p + 16 * q, o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// launch planning: persistent grids of (occupancy x SM count) CTAs, each
// owning a contiguous range of steps
// ---------------------------------------------------------------------------

struct Plan {
  int grid;
  uint32_t steps_per_cta;
};

int occupancy_of(const void* kernel) {
  static std::mutex mu;
  static std::unordered_map<const void*, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(kernel);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0) != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  if (n < 1) n = 1;
  cache[kernel] = n;
  return n;
}

Plan plan_for(const void* kernel, int64_t nsteps, int sm_count) {
  int64_t g = (int64_t)sm_count * occupancy_of(kernel);
  if (nsteps < g) g = nsteps;
  if (g < 1) g = 1;
  Plan p;
  p.grid = (int)g;
  p.steps_per_cta = (uint32_t)((nsteps + g - 1) / g);
  return p;
}

int64_t steps_of(int64_t nchunks, int64_t per_step) { return (nchunks + per_step - 1) / per_step; }

template <int KIND, bool MASK, bool CODES, bool STATS>
cudaError_t fq_launch(const FakequantArgs& a, const SegParam& seg_t, const SegParam& seg_r,
                      int sm_count, cudaStream_t st) {
  auto kern = k_fakequant<KIND, MASK, CODES, STATS>;
  const Plan p = plan_for((const void*)kern, steps_of(a.nchunks, kThreads), sm_count);
  kern<<<p.grid, kThreads, 0, st>>>((const uint8_t*)a.x, (uint32_t)a.nchunks,
                                    FastDivU((uint32_t)a.cpr), p.steps_per_cta, seg_t, a.gs_t,
                                    seg_r, (const uint8_t*)a.guide, (const uint8_t*)a.bs_r,
                                    a.gs_r, (uint8_t*)a.y, (uint8_t*)a.mask,
                                    (uint8_t*)a.codes_t, a.stats);
  return cudaGetLastError();
}

template <int KIND>
cudaError_t fq_dispatch(const FakequantArgs& a, const SegParam& t, const SegParam& r, int sm,
                        cudaStream_t st) {
  const int sel = ((a.mask != nullptr) << 2) | ((a.codes_t != nullptr) << 1) | (a.stats != nullptr);
  switch (sel) {
    case 0: return fq_launch<KIND, false, false, false>(a, t, r, sm, st);
    case 1: return fq_launch<KIND, false, false, true>(a, t, r, sm, st);
    case 2: return fq_launch<KIND, false, true, false>(a, t, r, sm, st);
    case 3: return fq_launch<KIND, false, true, true>(a, t, r, sm, st);
    case 4: return fq_launch<KIND, true, false, false>(a, t, r, sm, st);
    case 5: return fq_launch<KIND, true, false, true>(a, t, r, sm, st);
    case 6: return fq_launch<KIND, true, true, false>(a, t, r, sm, st);
    default: return fq_launch<KIND, true, true, true>(a, t, r, sm, st);
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
                                 uint32_t* guide, int sm_count, cudaStream_t st) {
  const Plan p = plan_for((const void*)k_rollout_quant, steps_of(nchunks, kThreads), sm_count);
  k_rollout_quant<<<p.grid, kThreads, 0, st>>>((const uint8_t*)x, (uint32_t)nchunks,
                                               FastDivU((uint32_t)cpr), p.steps_per_cta, seg, gs,
                                               (uint8_t*)codes, (uint8_t*)bs, (uint8_t*)guide);
  return cudaGetLastError();
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

cudaError_t launch_rollout_fused(const void* x, int64_t nchunks, int32_t cpr, const SegParam& seg,
                                 const WaveParam& wv, const Scratch& s, float* gs_out,
                                 void* codes, void* bs, uint32_t* guide, int sm_count,
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
  return cudaLaunchKernelEx(&cfg, k_rollout_fused, (const uint8_t*)x, (uint32_t)cpr,
                            FastDivU((uint32_t)cpr), seg, wv, gs_out, (uint8_t*)codes,
                            (uint8_t*)bs, (uint8_t*)guide, s.amax_bits, s.wave_cnt, s.done,
                            s.err, wait_extra, wait_ns);
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

cudaError_t launch_fakequant(const FakequantArgs& a, const SegParam& seg_t,
                             const SegParam& seg_r, int sm_count, cudaStream_t st) {
  switch (a.kind) {
    case TRACE_GUIDE_FULL: return fq_dispatch<TRACE_GUIDE_FULL>(a, seg_t, seg_r, sm_count, st);
    case TRACE_GUIDE_COMPACT:
      return fq_dispatch<TRACE_GUIDE_COMPACT>(a, seg_t, seg_r, sm_count, st);
    default: return fq_dispatch<TRACE_GUIDE_NONE>(a, seg_t, seg_r, sm_count, st);
  }
}

}  // namespace tfp4
