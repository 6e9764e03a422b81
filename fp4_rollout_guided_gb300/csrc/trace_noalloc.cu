// trace_noalloc.cu - trace_rollout_quant_noalloc: the rollout-side quantiser
// for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc: code running inside a custom device
// allocator or memory pool (allocating from there would recurse), runtimes
// that have pre-reserved every byte of device memory for their own arena,
// and real-time loops that forbid allocation on the hot path.  Those callers
// cannot create a trace_handle_t either, because trace_create allocates the
// handle's scratch.  This entry point needs no handle: its only scratch (the
// per-segment maxima and the amax kernel's completion ticket) lives in a
// fixed, file-scope device array that every GPU loading the library holds
// until the process exits.
//
// The first call on a device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress and caches it together
// with the identity of the calling thread's current CUDA context; make that
// first call before any stream capture.  A later call reuses the cached
// address while the current context is the same one, and looks it up again
// when it is not (after cudaDeviceReset, or with another context made
// current on the device), so an address from a destroyed or foreign context
// is never used.  All calls on a device share the one array: each call
// clears the part it needs with cudaMemsetAsync on its own stream, and calls
// that overlap on the GPU (for example on two streams at once) race on it.
//
// The call always runs the two-kernel rollout path (the amax pass, then the
// quantiser), so x is read twice; the fused single-read kernel needs the
// per-wave counters and error word of a handle.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string.h>

#include <mutex>

#include "trace_fp4.h"
#include "trace_internal.h"

namespace {

// amax words for TRACE_NOALLOC_MAX_SEGMENTS segments, then the ticket.
constexpr int kWords = TRACE_NOALLOC_MAX_SEGMENTS + 64;
static __device__ __align__(256) uint32_t g_noalloc_scratch[kWords];

constexpr int kMaxDevices = 64;

struct DeviceSlot {
  bool ready = false;            // device checked, sm_count known
  uint32_t* scratch = nullptr;   // device address of the array ...
  unsigned long long ctx = 0;    // ... in this context (0: unknown, look up every call)
  int sm_count = 0;
};

std::mutex g_mu;
DeviceSlot g_slots[kMaxDevices];

// Identity of the calling thread's current context (driver entry points
// looked up once through the runtime); 0 when there is none or the driver
// cannot tell, in which case the address is looked up on every call.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    cudaGetLastError();
  });
  if (!get_cur || !get_id) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_cur(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// With the device current: check the device once, and resolve the scratch
// array's device address whenever the current context is not the one the
// cached address belongs to.
trace_status_t setup(int dev, DeviceSlot** out) {
  if (dev < 0 || dev >= kMaxDevices) return TRACE_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceSlot& s = g_slots[dev];
  if (!s.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return TRACE_ERR_UNSUPPORTED_DEVICE;
    }
    if (major != 10 || minor != 3) return TRACE_ERR_UNSUPPORTED_DEVICE;
    s.sm_count = sms;
    s.ready = true;
  }
  const unsigned long long ctx = current_context_id();
  if (s.scratch == nullptr || ctx == 0 || ctx != s.ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      s.scratch = nullptr;
      return TRACE_ERR_CUDA;
    }
    s.scratch = (uint32_t*)p;
    // the lookup above made a context current if there was none
    s.ctx = ctx != 0 ? ctx : current_context_id();
  }
  *out = &s;
  return TRACE_OK;
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

}  // namespace

extern "C" {

trace_status_t trace_rollout_quant_noalloc(const void* x_bf16, int64_t rows, int64_t cols,
                                           trace_segments_t seg, void* codes_u8,
                                           void* bs_e4m3, float* gs_f32,
                                           uint32_t* guide_bits, trace_stream_t stream) {
  // shape and pointer rules of trace_rollout_quant
  if (rows < 0 || cols <= 0 || cols % 32 != 0 || rows >= (int64_t(1) << 31))
    return TRACE_ERR_INVALID_ARG;
  if (rows > 0 && cols / 32 > (int64_t(1) << 31) / rows) return TRACE_ERR_INVALID_ARG;
  const int64_t nchunks = rows * (cols / 32);
  if (nchunks >= (int64_t(1) << 31)) return TRACE_ERR_INVALID_ARG;
  const bool empty = rows == 0;
  for (const void* p : {x_bf16, (const void*)codes_u8, (const void*)bs_e4m3}) {
    if (!p && !empty) return TRACE_ERR_INVALID_ARG;
    if (p && !aligned(p, 16)) return TRACE_ERR_ALIGNMENT;
  }
  if (guide_bits && !aligned(guide_bits, 16)) return TRACE_ERR_ALIGNMENT;
  if (!gs_f32) return TRACE_ERR_INVALID_ARG;
  if (!aligned(gs_f32, 4)) return TRACE_ERR_ALIGNMENT;

  // the segment table, limited by the fixed scratch
  static thread_local tfp4::SegParam sp;
  if (!seg.row_offsets) {
    sp.n = 1;
    sp.off[0] = 0;
    sp.off[1] = (int32_t)rows;
  } else {
    if (seg.n_seg < 1 || seg.n_seg > TRACE_NOALLOC_MAX_SEGMENTS) return TRACE_ERR_INVALID_ARG;
    const int64_t* o = seg.row_offsets;
    if (o[0] != 0 || o[seg.n_seg] != rows) return TRACE_ERR_INVALID_ARG;
    for (int32_t s = 0; s < seg.n_seg; ++s)
      if (o[s + 1] < o[s]) return TRACE_ERR_INVALID_ARG;
    sp.n = seg.n_seg;
    for (int32_t s = 0; s <= seg.n_seg; ++s) sp.off[s] = (int32_t)o[s];
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return TRACE_ERR_UNSUPPORTED_DEVICE;
  }
  DeviceSlot* slot = nullptr;
  trace_status_t st = setup(dev, &slot);
  if (st != TRACE_OK) return st;

  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  if (nchunks == 0) {
    e = cudaMemsetAsync(gs_f32, 0, sizeof(float) * sp.n, s);
  } else {
    tfp4::Scratch sc;
    sc.amax_bits = slot->scratch;
    sc.done = slot->scratch + TRACE_NOALLOC_MAX_SEGMENTS;
    sc.gs_train = nullptr;
    // the maxima start at zero and the ticket at zero for this call
    e = cudaMemsetAsync(slot->scratch, 0, sizeof(uint32_t) * kWords, s);
#ifdef TRACE_DEBUG_BOUNDS
    if (e == cudaSuccess) {
      tfp4::DbgRanges r;
      memset(&r, 0, sizeof(r));
      const void* p[6] = {x_bf16, codes_u8, bs_e4m3, gs_f32, guide_bits, slot->scratch};
      const int64_t n[6] = {rows * cols * 2, rows * cols / 2, rows * cols / 16,
                            (int64_t)sizeof(float) * sp.n, rows * cols / 4,
                            (int64_t)sizeof(uint32_t) * kWords};
      for (int i = 0; i < 6; ++i)
        if (p[i]) {
          r.lo[r.n] = (uint64_t)p[i];
          r.hi[r.n] = (uint64_t)p[i] + (uint64_t)n[i];
          ++r.n;
        }
      e = tfp4::dbg_set_ranges(r, s);
    }
#endif
    const int32_t cpr = (int32_t)(cols / 32);
    if (e == cudaSuccess)
      e = tfp4::launch_amax(x_bf16, nchunks, cpr, sp, sc, gs_f32, slot->sm_count, s);
    if (e == cudaSuccess)
      e = tfp4::launch_rollout_quant(x_bf16, nchunks, cpr, sp, gs_f32, codes_u8, bs_e4m3,
                                     tfp4::MmaOut{nullptr, 0}, guide_bits, slot->sm_count, s);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return TRACE_ERR_CUDA;
  }
  return TRACE_OK;
}

}  // extern "C"
