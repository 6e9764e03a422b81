// trace_device.cuh - device helpers shared by the sm_103a kernels of the
// guided-NVFP4 hot path of TRACE (trace_kernels.cu, trace_fakequant.cu),
// and the launch planning both use.  Internal; not part of the ABI.
//
// Sources: "Alibaba Qwen Proposes TRACE for 5.4x Faster FP4 RL Rollouts",
// section "TRACE Core Concept" (rollout records FP4 results; training-side
// fake quantisation picks the adjacent E2M1 point closer to the rollout's;
// a compact record of mantissa bit + scale sets the direction) and the
// worked example of section "Why Does FP4 Rollout 'Break' RL Training?".
//
// Work decomposition.  Kernels stream a flat sequence of 32-element
// "chunks" (two 16-element NVFP4 blocks, one STE mask word).  Rows hold
// cols/32 chunks, so a chunk never straddles a row or a segment.  A CTA of
// 256 threads handles a "step" of 256 consecutive chunks (16 KiB of bf16),
// one chunk per thread, and owns a contiguous range of steps; the next
// step's loads are issued before the current step is computed.  Segments
// are looked up once per step (uniform across the CTA); only a step that
// straddles a segment boundary resolves segments per thread.  Two kernels
// differ: the fused rollout kernel stages steps with TMA copies and splits
// its CTA into producer, amax and quantiser warps, and the STE backward
// gives each thread one 16-byte word of eight elements per instruction.
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
#pragma once

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

// Debug builds: every global access of the helpers below (and the direct
// accesses marked TFP4_OK in the kernels) is checked against the ranges the
// API registered for the call; one outside them is counted and skipped.
#ifdef TRACE_DEBUG_BOUNDS
__device__ DbgRanges g_dbg_ranges;
__device__ unsigned long long g_dbg_violations;
__device__ __noinline__ bool dbg_ok(const void* p, uint32_t bytes) {
  const uint64_t a = reinterpret_cast<uint64_t>(p);
  for (uint32_t i = 0; i < g_dbg_ranges.n && i < (uint32_t)kDbgRanges; ++i)
    if (a >= g_dbg_ranges.lo[i] && a + bytes <= g_dbg_ranges.hi[i]) return true;
  atomicAdd(&g_dbg_violations, 1ull);
  return false;
}
#define TFP4_OK(p, bytes) dbg_ok((const void*)(p), (bytes))
#else
#define TFP4_OK(p, bytes) true
#endif

// A float from global memory (0 if a debug build finds it out of range).
__device__ __forceinline__ float ldf(const float* p) { return TFP4_OK(p, 4) ? *p : 0.0f; }

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v = make_uint4(0, 0, 0, 0);
  if (!TFP4_OK(p, 16)) return v;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_stream2(const void* p) {
  uint2 v = make_uint2(0, 0);
  if (!TFP4_OK(p, 8)) return v;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_stream_u16(const void* p) {
  unsigned short v = 0;
  if (!TFP4_OK(p, 2)) return v;
  asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(void* p, uint32_t a, uint32_t b, uint32_t c,
                                          uint32_t d) {
  if (!TFP4_OK(p, 16)) return;
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void st_stream2(void* p, uint32_t a, uint32_t b) {
  if (!TFP4_OK(p, 8)) return;
  asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void st_stream1(void* p, uint32_t a) {
  if (!TFP4_OK(p, 4)) return;
  asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}

__device__ __forceinline__ void st_stream_u16(void* p, uint32_t a) {
  if (!TFP4_OK(p, 2)) return;
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

// Lane-wise max(|a|, |b|) of two bf16 pairs.  The lanes' sign bits come
// out as the xor of the inputs' signs, so every consumer masks them; the
// magnitudes are exact for finite inputs.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// A pair of bf16 lanes (signs ignored) -> binary32 bits of the larger |lane|.
__device__ __forceinline__ uint32_t absmax_lanes_bits(uint32_t m) {
  return (absmax_bf16x2(m, m >> 16) << 16) & 0x7FFF0000u;
}

// The two block maxima of a chunk (bf16 abs-max on the raw words).
__device__ __forceinline__ void chunk_bamax(const Chunk& cur, float& b0, float& b1) {
  uint32_t m[2];
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const uint32_t* w = cur.w + 8 * b;
    const uint32_t m01 = absmax_bf16x2(absmax_bf16x2(w[0], w[1]), absmax_bf16x2(w[2], w[3]));
    const uint32_t m23 = absmax_bf16x2(absmax_bf16x2(w[4], w[5]), absmax_bf16x2(w[6], w[7]));
    m[b] = absmax_lanes_bits(absmax_bf16x2(m01, m23));
  }
  b0 = __uint_as_float(m[0]);
  b1 = __uint_as_float(m[1]);
}

// E4M3 code -> binary32: placing the 7 magnitude bits at bit 20 gives the
// value times 2^-120 (normal and subnormal codes alike); scaling by 2^120 is
// exact.
__device__ __forceinline__ float e4m3_decode(uint32_t code) {
  return __fmul_rn(__uint_as_float(code << 20), 0x1p120f);
}

// Per-thread maximum of |x| over one segment, folded into the segment's word
// (binary32 bits of a non-negative float, so unsigned order is float order)
// by one atomic per warp, then reset; called by whole warps.
__device__ __forceinline__ void flush_seg_max(uint32_t& m, uint32_t* dst) {
  const uint32_t wm = __reduce_max_sync(0xFFFFFFFFu, m);
  if ((threadIdx.x & 31u) == 0 && wm && TFP4_OK(dst, 4)) atomicMax(dst, wm);
  m = 0u;
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

__device__ __forceinline__ F2 fma2_rz(F2 a, F2 b, F2 c) {
  F2 d;
  asm("{ .reg .b64 A, B, C, D; mov.b64 A, {%2, %3}; mov.b64 B, {%4, %5}; "
      "mov.b64 C, {%6, %7}; fma.rz.f32x2 D, A, B, C; mov.b64 {%0, %1}, D; }"
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

// Four pairs -> one word of eight E2M1 nibbles, pair k in byte k (first
// value of a pair in the low nibble).
__device__ __forceinline__ uint32_t e2m1x8(F2 p0, F2 p1, F2 p2, F2 p3) {
  uint32_t r;
  asm("{ .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3}; }"
      : "=r"(r)
      : "f"(p0.x), "f"(p0.y), "f"(p1.x), "f"(p1.y), "f"(p2.x), "f"(p2.y), "f"(p3.x),
        "f"(p3.y));
  return r;
}

// The rounding constant for a pair of clamped values t in [0, 6]:
// C = 1.5 * 2^(22 + e) with 2^e the binade of max(t, 1), on the FMA pipe in
// three instructions.  u = fl_rz(t * m + 2^23) with m = 0.5 - 2^-25 holds
// F = floor(t * m) in its low significand bits (t * m < 3 stays below one
// ulp of 2^23 times 3), and F is e: t * m < 1 for t < 2, < 2 for t < 4, and
// 6 * m < 3; only t = 2 and t = 4 exactly fall one binade low, where either
// constant puts the on-grid value on the grid.  bits(u) * 2^23 adds F to the
// exponent field of K = 1.5 * 2^22 (bits(2^23) * 2^23 vanishes mod 2^32).
__device__ __forceinline__ F2 magic_pair(F2 tc) {
  const F2 u = fma2_rz(tc, splat(0x1.fffffep-2f), splat(0x1p23f));
  return F2{__uint_as_float(imad(__float_as_uint(u.x), 1u << 23, 0x4AC00000u)),
            __uint_as_float(imad(__float_as_uint(u.y), 1u << 23, 0x4AC00000u))};
}

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


// ---------------------------------------------------------------------------
// launch planning: persistent grids of (occupancy x SM count) CTAs, each
// owning a contiguous range of steps
// ---------------------------------------------------------------------------

struct Plan {
  int grid;
  uint32_t steps_per_cta;
};

// Host side of this translation unit's debug table.
inline cudaError_t dbg_set_here(const DbgRanges& r, cudaStream_t st) {
#ifdef TRACE_DEBUG_BOUNDS
  return cudaMemcpyToSymbolAsync(g_dbg_ranges, &r, sizeof(r), 0, cudaMemcpyHostToDevice, st);
#else
  (void)r;
  (void)st;
  return cudaSuccess;
#endif
}

inline unsigned long long dbg_take_here() {
#ifdef TRACE_DEBUG_BOUNDS
  unsigned long long v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_dbg_violations, sizeof(v)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_dbg_violations, &zero, sizeof(zero)) != cudaSuccess) {
    cudaGetLastError();
    return ~0ull;
  }
  return v;
#else
  return 0;
#endif
}

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

}  // namespace
}  // namespace tfp4
