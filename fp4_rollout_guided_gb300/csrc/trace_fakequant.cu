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

// Spreads the 16 low bits of v to the even bit positions.
__device__ __forceinline__ uint32_t spread16(uint32_t v) {
  v = (v | (v << 8)) & 0x00FF00FFu;
  v = (v | (v << 4)) & 0x0F0F0F0Fu;
  v = (v | (v << 2)) & 0x33333333u;
  v = (v | (v << 1)) & 0x55555555u;
  return v;
}

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

  // the next step's inputs are loaded at the end of the current step
  Chunk cur;
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
