// trace_fakequant.cu - the training-side guided fake quantiser (sm_103a):
// training scales, the guided E2M1 choice against the rollout record,
// bf16 output, STE mask, optional codes and mismatch counters.
//
// Source: "Alibaba Qwen Proposes TRACE for 5.4x Faster FP4 RL Rollouts",
// section "TRACE Core Concept" (first design: guided rounding; second
// design: the compact record sets the direction).
#include "trace_device.cuh"

namespace tfp4 {
namespace {

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

// A packed product that an add or subtract consumes is formed by this.  The
// code generator may fuse a packed multiply into the packed add that follows
// it (it did so for the distances below, even with explicit round-to-nearest
// on both instructions), which skips the product's own rounding and changes
// near-tie decisions.  An explicit FMA with a -0 addend known only at run
// time (a kernel argument) is the rounded product itself (adding -0 changes
// no value, +0 included) and cannot be fused into anything further.
__device__ __forceinline__ F2 mul2_kept(F2 a, F2 b, float nzero) {
  return fma2_rn(a, b, splat(nzero));
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
__device__ __forceinline__ void train_pair(F2 ax, float inv_t, F2 St, F2 vr, float nzero, F2& ym,
                                           F2& gsel, F2& grtn) {
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
  const F2 vlo = mul2_kept(glo, St, nzero), vhi = mul2_kept(ghi, St, nzero);
  const F2 dlo = sub2_rn(vlo, vr), dhi = sub2_rn(vhi, vr);
  const float diff0 = __fsub_rn(fabsf(dlo.x), fabsf(dhi.x));
  const float diff1 = __fsub_rn(fabsf(dlo.y), fabsf(dhi.y));
  const uint32_t lo0 = (__float_as_uint(diff0) + __float_as_uint(sn.x) + ~__float_as_uint(sz.x)) >> 31;
  const uint32_t lo1 = (__float_as_uint(diff1) + __float_as_uint(sn.y) + ~__float_as_uint(sz.y)) >> 31;
  const uint32_t h0 = __float_as_uint(vhi.x), h1 = __float_as_uint(vhi.y);
  ym = F2{__uint_as_float(imad(lo0, __float_as_uint(vlo.x) - h0, h0)),
          __uint_as_float(imad(lo1, __float_as_uint(vlo.y) - h1, h1))};
  if (WANT_G) {
    gsel = F2{lo0 ? glo.x : ghi.x, lo1 ? glo.y : ghi.y};
    grtn = F2{sn.x != sz.x ? ghi.x : glo.x, sn.y != sz.y ? ghi.y : glo.y};
  }
}

// STE mask bits of a chunk.  Word i (elements 2i, 2i + 1) yields
// X = (thr2 - |x|pair) & 0x80008000, its two kept bits at 15 and 31.  One
// 64-bit multiply-add per word moves them to their interleaved place:
// X * (2^(2k + 15) + 2^(2k)), k = i mod 8, puts bit 15 at 2k + 30 and bit 31
// at 2k + 31; the two other partial products land at 2k + 15 (below bit 30)
// and 2k + 46 (above bit 45), every one at its own position for k = 0..7,
// so the sum has no carries and bits 30..45 of the two accumulators (words
// 0..7 and 8..15) are the mask word's two halves in element order.
__device__ __forceinline__ void mask_gather(uint64_t& acc, uint32_t X, int k) {
  asm("mad.wide.u32 %0, %1, %2, %0;" : "+l"(acc) : "r"(X), "r"((1u << (2 * k + 15)) + (1u << (2 * k))));
}
__device__ __forceinline__ uint32_t mask_word(uint64_t acc0, uint64_t acc1) {
  return ((uint32_t)(acc0 >> 30) & 0xFFFFu) | ((uint32_t)(acc1 >> 30) << 16);
}

// ---------------------------------------------------------------------------
// The guided choice without distances (the fast form)
// ---------------------------------------------------------------------------
//
// Let rho = S_r / S_t.  The method compares d_c = |G[c] S_t - v_r| for the
// two candidates lo < hi = lo + 1 of t in binary32.  In exact arithmetic,
// with equal signs, hi is closer exactly when G[m_r] rho > (G[lo] + G[hi])/2.
// Over every adjacent pair of the E2M1 grid that midpoint lies at least
// 7/6 G[lo] above G[lo] and at most 7/8 G[hi] below G[hi], so whenever
// 7/8 < rho < 7/6 the rollout index alone decides: hi if m_r > lo (that is,
// m_r >= hi), else lo; with opposite signs lo always wins (the smaller
// magnitude is nearer a value of the other sign); a point bracket has one
// candidate.  The margins used below (0.876, 1.165) leave at least 2^-9 of
// relative room between the two distances, far above the few binary32
// rounding errors of the products and differences, and the scales are kept
// at or above 2^-100 so that every product is a normal number.  No tie can
// occur inside that window, so the RTN fallback never applies there.
//
// Which side of lo the rollout index lies on needs no rollout-frame bracket.
// The decoded index is the member of the bracket of t_r = |x| * inv_r whose
// parity is the stored bit, so with glo = G[lo], ghi = G[hi] of the
// training side:  t_r < glo or t_r == glo gives m_r <= lo;  t_r >= ghi gives
// m_r >= hi;  glo < t_r < ghi gives m_r = lo or hi by the stored bit.  All
// of that is read off t_r rounded down and up to the training side's grid
// spacing s (the rounding constant C of t):  uz = fl_rz(t_r + C) and
// up = fl_rp(t_r + C) are C + s floor(t_r / s) and C + s ceil(t_r / s), the
// member us of {uz, up} whose significand parity equals the stored bit is
// the decoded point relative to that grid, and the chosen candidate is
// us clamped to [C + glo, C + ghi].  An opposite rollout sign is carried by
// t_r itself (x is given the relative sign first): t_r < 0 gives us <= C,
// which clamps to lo.  For the full record the stored index's value is
// clamped the same way (rounded toward zero onto the grid of C).
//
// The form is exact wherever it is taken; blocks whose ratio lies outside
// the window (rare: about one block in 10^4 to 10^5 on the workloads) send
// their warp through the distance comparison.
constexpr float kRhoLo = 0.876f, kRhoHi = 1.165f, kScaleMin = 0x1p-100f;

__device__ __forceinline__ bool fast_block(float S_t, float S_r) {
  return S_t >= kScaleMin && S_r > __fmul_rn(kRhoLo, S_t) && S_r < __fmul_rn(kRhoHi, S_t);
}

// A compact word's sixteen sign bits rearranged so that the signs of
// elements 2k and 2k + 1 land at bits 15 and 31 after a left shift by
// 15 - 2k: even elements at bit j, odd elements at bit j + 15.
__device__ __forceinline__ uint32_t sign_spread(uint32_t gw) {
  return (gw & 0x5555u) | ((gw & 0xAAAAu) << 15);
}

// The two bf16 lanes of a word as binary32 (signs kept).
__device__ __forceinline__ F2 lanes(uint32_t w) {
  return F2{__uint_as_float(imad(w, 0x10000u, 0u)), __uint_as_float(w & 0xFFFF0000u)};
}

// Training bracket of a pair in the frame of its rounding constant:
// C, sz = C + glo, sp = C + ghi (t may carry any sign; |t| is bracketed).
__device__ __forceinline__ void train_bracket(F2 t, F2& C, F2& sz, F2& sp) {
  const F2 tc = {fminf(fabsf(t.x), 6.0f), fminf(fabsf(t.y), 6.0f)};
  C = magic_pair(tc);
  sz = add2_rz(tc, C);
  sp = add2_rp(tc, C);
}

// sat(4 a): 0 for a <= 0, 1 for a >= 1/4.
__device__ __forceinline__ float sat4(float a) {
  float d;
  asm("mul.rn.sat.f32 %0, %1, 0f40800000;" : "=f"(d) : "f"(a));
  return d;
}
#ifndef TFP4_FQ_MIN_CTAS
#define TFP4_FQ_MIN_CTAS 4
#endif
// AMAX: also the training segments' maxima of x into amax_out (zeroed by the
// caller), for a later call scaled by them (delayed scaling).
template <int KIND, bool MASK, bool CODES, bool STATS, bool AMAX = false>
__global__ void __launch_bounds__(kThreads, TFP4_FQ_MIN_CTAS)
    k_fakequant(const uint8_t* __restrict__ x, uint32_t nchunks, FastDivU cpr,
                uint32_t steps_per_cta, const __grid_constant__ SegParam seg_t,
                const float* __restrict__ gs_t, const __grid_constant__ SegParam seg_r,
                const uint8_t* __restrict__ guide, const uint8_t* __restrict__ bs_r,
                const float* __restrict__ gs_r, uint8_t* __restrict__ y,
                uint8_t* __restrict__ mask, uint8_t* __restrict__ codes_t,
                trace_stats_t* __restrict__ stats, float nzero, uint32_t* __restrict__ amax_out) {
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
  uint32_t mseg = 0u;                       // AMAX: this thread's maximum in segment aseg
  int aseg = -1;
  float seg_gs = 0.0f, seg_den = 0.0f, seg_rden = 0.0f;

  // the next step's inputs are loaded at the end of the current step
  Chunk cur = {};
  uint4 gcur = make_uint4(0, 0, 0, 0);
  uint32_t bcur = 0;
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
    const uint32_t r0 = cpr.div(c0), r1 = cpr.div(min(c0 + kThreads, nchunks) - 1);
    const bool uni_t = st.update(seg_t, r0, r1);
    const bool uni_r = GUIDED ? sr.update(seg_r, r0, r1) : true;
    if (AMAX && uni_t && st.cur != aseg) {
      if (aseg >= 0) flush_seg_max(mseg, amax_out + aseg);
      aseg = st.cur;
    }
    // refresh the scale tables when the (uniform) segment changes
    const bool new_t = uni_t && st.cur != tseg;
    const bool new_r = GUIDED && uni_r && sr.cur != rseg;
    if (new_t || new_r) {
      __syncthreads();
      if (new_t) {
        tseg = st.cur;
        seg_gs = ldf(gs_t + tseg);
        seg_den = __fmul_rn(seg_gs, 6.0f);
        seg_rden = seg_gs > 0.0f ? __frcp_rn(seg_den) : 0.0f;
        build_tab(tab_t, seg_gs);
      }
      if (new_r) {
        rseg = sr.cur;
        build_tab(tab_r, ldf(gs_r + rseg));
      }
      __syncthreads();
    }
    // scales of both blocks (threads past the end compute on stale data
    // and store nothing)
    PairScale pt, pr = {};
    uint32_t thr2[2];
    {
      int s_t = st.cur, s_r = sr.cur;
      if (!uni_t || !uni_r) {
        const uint32_t row = cpr.div(min(c, nchunks - 1));
        if (!uni_t) s_t = seg_advance(seg_t, st.cur, row);
        if (GUIDED && !uni_r) s_r = seg_advance(seg_r, sr.cur, row);
      }
      float bam0, bam1;
      chunk_bamax(cur, bam0, bam1);
      if (AMAX && c < nchunks) {
        const uint32_t mb = max(__float_as_uint(bam0), __float_as_uint(bam1));
        if (uni_t)
          mseg = max(mseg, mb);
        else if (mb && TFP4_OK(amax_out + s_t, 4))
          atomicMax(amax_out + s_t, mb);
      }
      if (uni_t) {
        pt.codes = pair_codes(bam0, bam1, seg_gs, seg_den, seg_rden);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          // codes of non-negative block maxima are at most 0x7F (NaN); the
          // mask keeps the table index in range whatever the input holds
          const uint32_t code = (pt.codes >> (8 * b)) & 0x7Fu;
          const float2 e = tab_t.sinv[code];
          pt.S[b] = e.x;
          pt.inv[b] = e.y;
          thr2[b] = tab_t.thr2[code];
        }
      } else {
        pt = pair_scale(bam0, bam1, ldf(gs_t + s_t));
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
          pr = pair_scale_stored(bcur, ldf(gs_r + s_r));
        }
      }
    }
    // the fast form when every block of the warp's chunks allows it
    bool fast = false;
    if (GUIDED && !STATS)
      fast = __all_sync(0xFFFFFFFFu, c >= nchunks || (fast_block(pt.S[0], pr.S[0]) &&
                                                       fast_block(pt.S[1], pr.S[1])));
    if (c < nchunks) {
      uint32_t ybits[4];
      uint32_t cbytes[16];
      uint64_t kacc[2] = {0, 0};
      if (fast) {
        uint32_t U[2] = {0u, 0u};
        if (KIND == TRACE_GUIDE_COMPACT) {
          U[0] = sign_spread(gcur.x);
          U[1] = sign_spread(gcur.y);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int b = i >> 3;        // block of this word
          const int j0 = (i & 7) * 2;  // index of its low element in the block
          const uint32_t w = cur.w[i];
          F2 C, sz, sp, us;
          if (KIND == TRACE_GUIDE_COMPACT) {
            // x with the relative sign (training xor rollout) in both lanes
            const uint32_t rel = w ^ (imad(U[b], 1u << (15 - j0), 0u) & 0x80008000u);
            const F2 xl = lanes(rel);
            train_bracket(mul2_rn(xl, splat(pt.inv[b])), C, sz, sp);
            const F2 tr = mul2_kept(xl, splat(pr.inv[b]), nzero);
            const F2 uz = add2_rz(tr, C), up = add2_rp(tr, C);
            const uint32_t gw = b ? gcur.y : gcur.x;
            const uint32_t b0 = 1u << (16 + j0), b1 = 1u << (17 + j0);
            const uint32_t m0 = (imad(__float_as_uint(uz.x), b0, 0u) ^ gw) & b0;
            const uint32_t m1 = (imad(__float_as_uint(uz.y), b1, 0u) ^ gw) & b1;
            us = F2{m0 ? up.x : uz.x, m1 ? up.y : uz.y};
          } else {
            train_bracket(mul2_rn(lanes(w), splat(pt.inv[b])), C, sz, sp);
            const uint32_t gword =
                (i < 4) ? gcur.x : (i < 8) ? gcur.y : (i < 12) ? gcur.z : gcur.w;
            uint32_t h;  // the stored pair's values (f16x2), relative sign
            asm("{ .reg .b8 q; cvt.u8.u32 q, %1; cvt.rn.f16x2.e2m1x2 %0, q; }"
                : "=r"(h)
                : "r"((gword >> (8 * (i & 3))) & 0xFFu));
            h ^= w & 0x80008000u;
            float g0, g1;
            asm("cvt.f32.f16 %0, %1;" : "=f"(g0) : "h"((unsigned short)(h & 0xFFFFu)));
            asm("cvt.f32.f16 %0, %1;" : "=f"(g1) : "h"((unsigned short)(h >> 16)));
            us = add2_rz(F2{g0, g1}, C);
          }
          // the chosen point g: us clamped to [sz, sp], minus C.  With the
          // compact record the clamp is two min/max per element (measured
          // faster than the form below); with the full record it runs on the
          // FMA pipe: us - sz is a multiple of the grid spacing (>= 0.5) or
          // <= 0, so h = sat(4 (us - sz)) is exactly 1 or 0, and
          // g = glo + h (ghi - glo).
          F2 g;
          if (KIND == TRACE_GUIDE_COMPACT) {
            const F2 yc = {fminf(fmaxf(us.x, sz.x), sp.x), fminf(fmaxf(us.y, sz.y), sp.y)};
            g = sub2_rn(yc, C);
          } else {
            const F2 dl = sub2_rn(us, sz);
            g = fma2_rn(F2{sat4(dl.x), sat4(dl.y)}, sub2_rn(sp, sz), sub2_rn(sz, C));
          }
          const F2 ym = mul2_rn(g, splat(pt.S[b]));
          ybits[i & 3] = bf16x2_rn(ym.x, ym.y) | (w & 0x80008000u);
          if ((i & 3) == 3)
            st_stream(y + (uint64_t)c * 64u + 16 * (i >> 2), ybits[0], ybits[1], ybits[2], ybits[3]);
          if (MASK) mask_gather(kacc[b], imad(w & kAbs2, 0xFFFFFFFFu, thr2[b]) & 0x80008000u, i & 7);
          if (CODES)
            cbytes[i] = e2m1x2(__uint_as_float(__float_as_uint(g.x) | (imad(w, 0x10000u, 0u) & 0x80000000u)),
                               __uint_as_float(__float_as_uint(g.y) | (w & 0x80000000u)));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int b = i >> 3;        // block of this word
          const int j0 = (i & 7) * 2;  // index of its low element in the block
          const uint32_t w = cur.w[i];
          const uint32_t a = w & kAbs2;
          const F2 ax = {__uint_as_float(imad(a, 0x10000u, 0u)), __uint_as_float(a & 0xFFFF0000u)};
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
            vr = mul2_kept(gr, F2{__uint_as_float(Sb | sr0), __uint_as_float(Sb | sr1)}, nzero);
            if (STATS) grs = F2{__uint_as_float(__float_as_uint(gr.x) | sr0),
                                __uint_as_float(__float_as_uint(gr.y) | sr1)};
          } else if (KIND == TRACE_GUIDE_FULL) {
            const uint32_t gword = (i < 4) ? gcur.x : (i < 8) ? gcur.y : (i < 12) ? gcur.z : gcur.w;
            float g0, g1;
            e2m1x2_values((gword >> (8 * (i & 3))) & 0xFFu, g0, g1);
            vr = mul2_kept(F2{g0, g1}, splat(pr.S[b]), nzero);
            if (STATS) grs = F2{g0, g1};
          }
          F2 ym, gsel, grtn;
          train_pair<GUIDED, CODES || STATS>(ax, pt.inv[b], St, vr, nzero, ym, gsel, grtn);
          ybits[i & 3] = bf16x2_rn(ym.x, ym.y);
          if ((i & 3) == 3)
            st_stream(y + (uint64_t)c * 64u + 16 * (i >> 2), ybits[0], ybits[1], ybits[2], ybits[3]);
          if (MASK) mask_gather(kacc[b], imad(a, 0xFFFFFFFFu, thr2[b]) & 0x80008000u, i & 7);
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
      }
      if (MASK) st_stream1(mask + (uint64_t)c * 4u, mask_word(kacc[0], kacc[1]));
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
    if (step + 1 < step_end) {
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
  if (AMAX && aseg >= 0) flush_seg_max(mseg, amax_out + aseg);
  if (STATS) {
    const uint32_t v[11] = {n_done,       cnt.mm_rtn,   cnt.mm_g,     cnt.h_rtn[0],
                            cnt.h_rtn[1], cnt.h_rtn[2], cnt.h_rtn[3], cnt.h_g[0],
                            cnt.h_g[1],   cnt.h_g[2],   cnt.h_g[3]};
    unsigned long long* dst = reinterpret_cast<unsigned long long*>(stats);
#pragma unroll
    for (int k = 0; k < 11; ++k) {
      if (!GUIDED && k > 0) break;
      const uint32_t tot = __reduce_add_sync(0xFFFFFFFFu, v[k]);
      if ((threadIdx.x & 31) == 0 && tot && TFP4_OK(dst + k, 8))
        atomicAdd(dst + k, (unsigned long long)tot);
    }
  }
}

template <int KIND, bool MASK, bool CODES, bool STATS, bool AMAX = false>
cudaError_t fq_launch(const FakequantArgs& a, const SegParam& seg_t, const SegParam& seg_r,
                      int sm_count, cudaStream_t st) {
  auto kern = k_fakequant<KIND, MASK, CODES, STATS, AMAX>;
  const Plan p = plan_for((const void*)kern, steps_of(a.nchunks, kThreads), sm_count);
  kern<<<p.grid, kThreads, 0, st>>>((const uint8_t*)a.x, (uint32_t)a.nchunks,
                                    FastDivU((uint32_t)a.cpr), p.steps_per_cta, seg_t, a.gs_t,
                                    seg_r, (const uint8_t*)a.guide, (const uint8_t*)a.bs_r,
                                    a.gs_r, (uint8_t*)a.y, (uint8_t*)a.mask,
                                    (uint8_t*)a.codes_t, a.stats, -0.0f, a.amax_out);
  return cudaGetLastError();
}

template <int KIND>
cudaError_t fq_dispatch(const FakequantArgs& a, const SegParam& t, const SegParam& r, int sm,
                        cudaStream_t st) {
  const int sel = ((a.mask != nullptr) << 2) | ((a.codes_t != nullptr) << 1) | (a.stats != nullptr);
  if (a.amax_out) {
    // delayed scaling: y and the mask (or y alone)
    if (sel == 4) return fq_launch<KIND, true, false, false, true>(a, t, r, sm, st);
    if (sel == 0) return fq_launch<KIND, false, false, false, true>(a, t, r, sm, st);
    return cudaErrorInvalidValue;
  }
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

cudaError_t launch_fakequant(const FakequantArgs& a, const SegParam& seg_t,
                             const SegParam& seg_r, int sm_count, cudaStream_t st) {
  switch (a.kind) {
    case TRACE_GUIDE_FULL: return fq_dispatch<TRACE_GUIDE_FULL>(a, seg_t, seg_r, sm_count, st);
    case TRACE_GUIDE_COMPACT:
      return fq_dispatch<TRACE_GUIDE_COMPACT>(a, seg_t, seg_r, sm_count, st);
    default: return fq_dispatch<TRACE_GUIDE_NONE>(a, seg_t, seg_r, sm_count, st);
  }
}

cudaError_t dbg_set_ranges_fakequant(const DbgRanges& r, cudaStream_t st) {
  return dbg_set_here(r, st);
}
unsigned long long dbg_take_fakequant() { return dbg_take_here(); }

}  // namespace tfp4
