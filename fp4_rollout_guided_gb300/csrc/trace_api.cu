// trace_api.cu - the C ABI declared in include/trace_fp4.h: handle life
// cycle, argument validation, scratch ordering, the built-in profiler, and
// the calls that enqueue the kernels of trace_kernels.cu and trace_fakequant.cu.
//
// Method: "Alibaba Qwen Proposes TRACE for 5.4x Faster FP4 RL Rollouts",
// section "TRACE Core Concept" (rollout-side record, training-side guided
// rounding, compact record of mantissa bit and scale).
#include <cuda_runtime.h>
#include <stdint.h>

#include <string.h>

#include <initializer_list>
#include <mutex>
#include <new>
#include <vector>

#include "trace_fp4.h"
#include "trace_internal.h"

namespace {

constexpr int kMaxTimed = 4096;

struct TimedLaunch {
  int kernel;
  cudaEvent_t start, stop;
};

}  // namespace

struct trace_ctx {
  int device = 0;
  int sm_count = 0;
  tfp4::Scratch scratch = {};
  cudaEvent_t order = nullptr;  // orders calls on the handle's scratch
  int last_error = 0;
  bool profiling = false;
  bool fused_amax = true;
  int64_t wave_bytes = int64_t(32) << 20;
  uint64_t wait_ns = 1000000000ull;
  uint32_t wait_extra = 0;
  float* gemm_scalars = nullptr;  // alpha, beta of the NVFP4 GEMM (device)
  void* lt = nullptr;          // cuBLASLt handle of the NVFP4 GEMM
  void* gemm_ws = nullptr;     // its workspace
  size_t gemm_ws_bytes = 0;
  std::vector<TimedLaunch> timed;
  std::vector<cudaEvent_t> spare;  // recycled timing events
  const void* scratch_base = nullptr;  // the one scratch allocation
  size_t scratch_bytes = 0;
  bool dbg_shrink = false;  // debug builds: register outputs 16 bytes short
  int gemm = TRACE_GEMM_TC256;  // form of trace_nvfp4_gemm
};

namespace {

// Debug builds: registers the byte ranges the call's launches may touch
// (its buffers, and the handle's scratch), stream-ordered before them.
// Outputs are registered 16 bytes short while the test option asks for it.
struct DbgBuf {
  const void* p;
  int64_t bytes;
  bool out;
};
cudaError_t dbg_register(const trace_ctx* h, cudaStream_t st, std::initializer_list<DbgBuf> bufs,
                         const void* extra = nullptr, int64_t extra_bytes = 0) {
#ifdef TRACE_DEBUG_BOUNDS
  tfp4::DbgRanges r;
  memset(&r, 0, sizeof(r));
  auto add = [&](const void* p, int64_t n) {
    if (p && n > 0 && r.n < (uint32_t)tfp4::kDbgRanges) {
      r.lo[r.n] = (uint64_t)p;
      r.hi[r.n] = (uint64_t)p + (uint64_t)n;
      ++r.n;
    }
  };
  for (const DbgBuf& b : bufs) add(b.p, b.bytes - ((b.out && h && h->dbg_shrink) ? 16 : 0));
  if (h) add(h->scratch_base, (int64_t)h->scratch_bytes);
  add(extra, extra_bytes);
  return tfp4::dbg_set_ranges(r, st);
#else
  (void)h;
  (void)st;
  (void)bufs;
  (void)extra;
  (void)extra_bytes;
  return cudaSuccess;
#endif
}

// Makes the handle's device current for the duration of a call.
class DeviceGuard {
 public:
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&old_) == cudaSuccess && old_ != dev) {
      if (cudaSetDevice(dev) == cudaSuccess) switched_ = true;
    }
  }
  ~DeviceGuard() {
    if (switched_) cudaSetDevice(old_);
  }

 private:
  int old_ = -1;
  bool switched_ = false;
};

trace_status_t cuda_fail(trace_ctx* h, cudaError_t e) {
  if (h) h->last_error = (int)e;
  cudaGetLastError();  // clear the sticky-free error state for the next call
  return TRACE_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// Shape rules shared by every call.
trace_status_t check_shape(int64_t rows, int64_t cols) {
  if (rows < 0 || cols <= 0 || cols % 32 != 0) return TRACE_ERR_INVALID_ARG;
  if (rows >= (int64_t(1) << 31)) return TRACE_ERR_INVALID_ARG;
  if (rows > 0 && cols / 32 > (int64_t(1) << 31) / rows) return TRACE_ERR_INVALID_ARG;
  if (rows * (cols / 32) >= (int64_t(1) << 31)) return TRACE_ERR_INVALID_ARG;
  return TRACE_OK;
}

// A tensor pointer must be non-null and 16-byte aligned, except that an
// empty input (rows == 0) may pass null pointers for its empty tensors.
trace_status_t check_tensor(const void* p, bool empty = false) {
  if (!p) return empty ? TRACE_OK : TRACE_ERR_INVALID_ARG;
  if (!aligned(p, 16)) return TRACE_ERR_ALIGNMENT;
  return TRACE_OK;
}

// Host segment table -> kernel parameter (validated, narrowed to int32).
trace_status_t make_segments(const trace_segments_t& in, int64_t rows, tfp4::SegParam* out) {
  if (!in.row_offsets) {
    out->n = 1;
    out->off[0] = 0;
    out->off[1] = (int32_t)rows;
    return TRACE_OK;
  }
  if (in.n_seg < 1 || in.n_seg > TRACE_MAX_SEGMENTS) return TRACE_ERR_INVALID_ARG;
  const int64_t* o = in.row_offsets;
  if (o[0] != 0 || o[in.n_seg] != rows) return TRACE_ERR_INVALID_ARG;
  for (int32_t s = 0; s < in.n_seg; ++s)
    if (o[s + 1] < o[s]) return TRACE_ERR_INVALID_ARG;
  out->n = in.n_seg;
  for (int32_t s = 0; s <= in.n_seg; ++s) out->off[s] = (int32_t)o[s];
  return TRACE_OK;
}

cudaEvent_t take_event(trace_ctx* h) {
  if (!h->spare.empty()) {
    cudaEvent_t e = h->spare.back();
    h->spare.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return e;
}

// Runs one launcher, bracketed by timing events when profiling is on.
template <typename F>
cudaError_t timed(trace_ctx* h, int kernel, cudaStream_t st, F&& launch) {
  if (!h->profiling || (int)h->timed.size() >= kMaxTimed) return launch();
  cudaEvent_t a = take_event(h), b = take_event(h);
  if (!a || !b) {
    if (a) h->spare.push_back(a);
    if (b) h->spare.push_back(b);
    return launch();
  }
  cudaEventRecord(a, st);
  const cudaError_t e = launch();
  cudaEventRecord(b, st);
  h->timed.push_back({kernel, a, b});
  return e;
}

// Orders this call after the previous user of the handle's scratch.
cudaError_t begin_call(trace_ctx* h, cudaStream_t st) { return cudaStreamWaitEvent(st, h->order, 0); }
cudaError_t end_call(trace_ctx* h, cudaStream_t st) { return cudaEventRecord(h->order, st); }

}  // namespace

extern "C" {

int trace_version(void) { return 300; }

const char* trace_status_string(trace_status_t s) {
  switch (s) {
    case TRACE_OK: return "ok";
    case TRACE_ERR_INVALID_ARG: return "invalid argument";
    case TRACE_ERR_ALIGNMENT: return "tensor pointer not 16-byte aligned";
    case TRACE_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case TRACE_ERR_CUDA: return "CUDA error";
    case TRACE_ERR_OOM: return "out of device memory";
    case TRACE_ERR_TIMEOUT: return "device wait timed out";
    case TRACE_ERR_LIBRARY: return "cuBLASLt missing or refused the operation";
  }
  return "unknown status";
}

int trace_last_cuda_error(trace_handle_t h) { return h ? h->last_error : 0; }

trace_status_t trace_create(trace_handle_t* out, int device) {
  if (!out) return TRACE_ERR_INVALID_ARG;
  *out = nullptr;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || device < 0 || device >= count) {
    cudaGetLastError();
    return TRACE_ERR_UNSUPPORTED_DEVICE;
  }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) {
    cudaGetLastError();
    return TRACE_ERR_UNSUPPORTED_DEVICE;
  }
  if (prop.major != 10 || prop.minor != 3) return TRACE_ERR_UNSUPPORTED_DEVICE;
  trace_ctx* h = new (std::nothrow) trace_ctx;
  if (!h) return TRACE_ERR_OOM;
  h->device = device;
  h->sm_count = prop.multiProcessorCount;
  DeviceGuard g(device);
  // one allocation: amax words, ticket (padded to 256 B), training scales,
  // wave counters, error word (padded to 256 B), GEMM alpha/beta (256 B)
  const size_t seg_bytes = sizeof(uint32_t) * TRACE_MAX_SEGMENTS;
  const size_t bytes = seg_bytes + 256 + seg_bytes + seg_bytes + 256 + 256;
  char* base = nullptr;
  if (cudaMalloc(&base, bytes) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return TRACE_ERR_OOM;
  }
  if (cudaMemset(base, 0, bytes) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->order, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(base);
    delete h;
    return TRACE_ERR_CUDA;
  }
  h->scratch_base = base;
  h->scratch_bytes = bytes;
  h->scratch.amax_bits = (uint32_t*)base;
  h->scratch.done = (uint32_t*)(base + seg_bytes);
  h->scratch.gs_train = (float*)(base + seg_bytes + 256);
  h->scratch.wave_cnt = (uint32_t*)(base + 2 * seg_bytes + 256);
  h->scratch.err = (uint32_t*)(base + 3 * seg_bytes + 256);
  h->gemm_scalars = (float*)(base + 3 * seg_bytes + 512);
  *out = h;
  return TRACE_OK;
}

trace_status_t trace_destroy(trace_handle_t h) {
  if (!h) return TRACE_OK;
  DeviceGuard g(h->device);
  for (auto& t : h->timed) {
    cudaEventDestroy(t.start);
    cudaEventDestroy(t.stop);
  }
  for (auto e : h->spare) cudaEventDestroy(e);
  if (h->order) cudaEventDestroy(h->order);
  tfp4::lt_destroy(h->lt);
  if (h->gemm_ws) cudaFree(h->gemm_ws);
  cudaFree(h->scratch.amax_bits);
  cudaGetLastError();
  delete h;
  return TRACE_OK;
}

trace_status_t trace_set_option(trace_handle_t h, trace_option_t opt, int64_t value) {
  if (!h) return TRACE_ERR_INVALID_ARG;
  switch (opt) {
    case TRACE_OPT_FUSED_AMAX:
      if (value != 0 && value != 1) return TRACE_ERR_INVALID_ARG;
      h->fused_amax = value != 0;
      return TRACE_OK;
    case TRACE_OPT_WAVE_BYTES:
      if (value < 4096 || value > (int64_t(40) << 20)) return TRACE_ERR_INVALID_ARG;
      h->wave_bytes = value;
      return TRACE_OK;
    case TRACE_OPT_WAIT_LIMIT_NS:
      if (value < 1000000 || value > 10000000000ll) return TRACE_ERR_INVALID_ARG;
      h->wait_ns = (uint64_t)value;
      return TRACE_OK;
    case TRACE_OPT_WAIT_EXTRA:
      if (value != 0 && value != 1) return TRACE_ERR_INVALID_ARG;
      h->wait_extra = (uint32_t)value;
      return TRACE_OK;
    case TRACE_OPT_GEMM:
      if (value != TRACE_GEMM_TC256 && value != TRACE_GEMM_CUBLASLT && value != TRACE_GEMM_TC128 &&
          value != TRACE_GEMM_TC_PAIR)
        return TRACE_ERR_INVALID_ARG;
      h->gemm = (int)value;
      return TRACE_OK;
    case TRACE_OPT_DEBUG_SHRINK:
#ifdef TRACE_DEBUG_BOUNDS
      if (value != 0 && value != 1) return TRACE_ERR_INVALID_ARG;
      h->dbg_shrink = value != 0;
      return TRACE_OK;
#else
      return TRACE_ERR_INVALID_ARG;
#endif
  }
  return TRACE_ERR_INVALID_ARG;
}

trace_status_t trace_device_status(trace_handle_t h, trace_stream_t stream) {
  if (!h) return TRACE_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t word = 0;
  cudaError_t e = cudaStreamWaitEvent(st, h->order, 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&word, h->scratch.err, sizeof(word),
                                            cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->scratch.err, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  return word ? TRACE_ERR_TIMEOUT : TRACE_OK;
}

}  // extern "C"

namespace {

// trace_rollout_quant and trace_rollout_quant_mma: block scales row-major
// (bs_e4m3) and/or in the tensor-core tile layout (bs_mma).  With amax_prev
// (trace_rollout_quant_delayed) the global scales come from those maxima,
// one kernel, and amax_out receives this tensor's maxima.
trace_status_t rollout_quant_impl(trace_handle_t h, const void* x_bf16, int64_t rows,
                                  int64_t cols, trace_segments_t seg, void* codes_u8,
                                  void* bs_e4m3, void* bs_mma, float* gs_f32,
                                  uint32_t* guide_bits, trace_stream_t stream,
                                  const float* amax_prev = nullptr, float* amax_out = nullptr) {
  if (!h) return TRACE_ERR_INVALID_ARG;
  trace_status_t s = check_shape(rows, cols);
  if (s != TRACE_OK) return s;
  const bool empty = rows == 0;
  for (const void* p : {x_bf16, (const void*)codes_u8})
    if ((s = check_tensor(p, empty)) != TRACE_OK) return s;
  if (!bs_e4m3 && !bs_mma && !empty) return TRACE_ERR_INVALID_ARG;
  if (bs_e4m3 && (s = check_tensor(bs_e4m3, empty)) != TRACE_OK) return s;
  if (bs_mma && (s = check_tensor(bs_mma, empty)) != TRACE_OK) return s;
  if (guide_bits && (s = check_tensor(guide_bits)) != TRACE_OK) return s;
  if (!gs_f32) return TRACE_ERR_INVALID_ARG;
  if (!aligned(gs_f32, 4)) return TRACE_ERR_ALIGNMENT;
  if ((amax_prev && !aligned(amax_prev, 4)) || (amax_out && !aligned(amax_out, 4)))
    return TRACE_ERR_ALIGNMENT;
  static thread_local tfp4::SegParam sp;
  if ((s = make_segments(seg, rows, &sp)) != TRACE_OK) return s;

  DeviceGuard g(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = begin_call(h, st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  const int64_t nchunks = rows * (cols / 32);
  const int32_t cpr = (int32_t)(cols / 32);
  const tfp4::MmaOut mma{(uint8_t*)bs_mma, (uint32_t)((cols / 16 + 3) / 4)};
  if (e == cudaSuccess)
    e = dbg_register(h, st, {{x_bf16, rows * cols * 2, false}, {codes_u8, rows * cols / 2, true},
                             {bs_e4m3, rows * cols / 16, true},
                             {bs_mma, bs_mma ? tfp4::mma_scales_bytes(rows, cols) : 0, true},
                             {gs_f32, (int64_t)sizeof(float) * sp.n, true},
                             {guide_bits, rows * cols / 4, true},
                             {amax_prev, amax_prev ? (int64_t)sizeof(float) * sp.n : 0, false},
                             {amax_out, amax_out ? (int64_t)sizeof(float) * sp.n : 0, true}});
  // the tile layout's padding (rows past a multiple of 128, scale columns
  // past a multiple of 4) is zero
  if (bs_mma && (rows % 128 != 0 || (cols / 16) % 4 != 0))
    e = cudaMemsetAsync(bs_mma, 0, (size_t)tfp4::mma_scales_bytes(rows, cols), st);
  if (e == cudaSuccess && amax_out)
    e = cudaMemsetAsync(amax_out, 0, sizeof(float) * sp.n, st);
  if (e == cudaSuccess && amax_prev) {
    e = timed(h, TRACE_KERNEL_ROLLOUT_DELAYED, st, [&] {
      return tfp4::launch_rollout_quant_delayed(x_bf16, nchunks, cpr, sp, amax_prev, gs_f32,
                                                codes_u8, bs_e4m3, mma, guide_bits, amax_out,
                                                h->sm_count, st);
    });
  } else if (e == cudaSuccess && nchunks == 0) {
    e = cudaMemsetAsync(gs_f32, 0, sizeof(float) * sp.n, st);
  } else if (e == cudaSuccess) {
    static thread_local tfp4::WaveParam wv;
    bool fused = h->fused_amax && tfp4::plan_waves(sp, (int32_t)cols, h->wave_bytes, &wv);
    if (fused) {
      e = timed(h, TRACE_KERNEL_ROLLOUT_FUSED, st, [&] {
        return tfp4::launch_rollout_fused(x_bf16, nchunks, cpr, sp, wv, h->scratch, gs_f32,
                                          codes_u8, bs_e4m3, mma, guide_bits, h->sm_count,
                                          h->wait_extra, h->wait_ns, st);
      });
      // a device that cannot hold the whole grid at once takes the two-kernel path
      if (e == cudaErrorCooperativeLaunchTooLarge) {
        cudaGetLastError();
        fused = false;
        e = cudaSuccess;
      }
    }
    if (!fused) {
      e = timed(h, TRACE_KERNEL_AMAX, st, [&] {
        return tfp4::launch_amax(x_bf16, nchunks, cpr, sp, h->scratch, gs_f32, h->sm_count, st);
      });
      if (e == cudaSuccess)
        e = timed(h, TRACE_KERNEL_ROLLOUT_QUANT, st, [&] {
          return tfp4::launch_rollout_quant(x_bf16, nchunks, cpr, sp, gs_f32, codes_u8, bs_e4m3,
                                            mma, guide_bits, h->sm_count, st);
        });
    }
  }
  const cudaError_t e2 = end_call(h, st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  if (e2 != cudaSuccess) return cuda_fail(h, e2);
  return TRACE_OK;
}

}  // namespace

extern "C" {

trace_status_t trace_rollout_quant(trace_handle_t h, const void* x_bf16, int64_t rows,
                                   int64_t cols, trace_segments_t seg, void* codes_u8,
                                   void* bs_e4m3, float* gs_f32, uint32_t* guide_bits,
                                   trace_stream_t stream) {
  if (!bs_e4m3 && rows > 0) return TRACE_ERR_INVALID_ARG;
  return rollout_quant_impl(h, x_bf16, rows, cols, seg, codes_u8, bs_e4m3, nullptr, gs_f32,
                            guide_bits, stream);
}

trace_status_t trace_rollout_quant_mma(trace_handle_t h, const void* x_bf16, int64_t rows,
                                       int64_t cols, trace_segments_t seg, void* codes_u8,
                                       void* bs_e4m3, void* bs_mma, float* gs_f32,
                                       uint32_t* guide_bits, trace_stream_t stream) {
  return rollout_quant_impl(h, x_bf16, rows, cols, seg, codes_u8, bs_e4m3, bs_mma, gs_f32,
                            guide_bits, stream);
}

trace_status_t trace_rollout_quant_delayed(trace_handle_t h, const void* x_bf16, int64_t rows,
                                           int64_t cols, trace_segments_t seg,
                                           const float* amax_prev, void* codes_u8,
                                           void* bs_e4m3, float* gs_f32, uint32_t* guide_bits,
                                           float* amax_out, trace_stream_t stream) {
  if (!amax_prev || (!bs_e4m3 && rows > 0)) return TRACE_ERR_INVALID_ARG;
  return rollout_quant_impl(h, x_bf16, rows, cols, seg, codes_u8, bs_e4m3, nullptr, gs_f32,
                            guide_bits, stream, amax_prev, amax_out);
}

trace_status_t trace_guide_pack(trace_handle_t h, const void* codes_u8, int64_t rows,
                                int64_t cols, uint32_t* guide_bits, trace_stream_t stream) {
  if (!h) return TRACE_ERR_INVALID_ARG;
  trace_status_t s = check_shape(rows, cols);
  if (s != TRACE_OK) return s;
  const bool empty = rows == 0;
  if ((s = check_tensor(codes_u8, empty)) != TRACE_OK) return s;
  if ((s = check_tensor(guide_bits, empty)) != TRACE_OK) return s;
  const int64_t nchunks = rows * (cols / 32);
  if (nchunks == 0) return TRACE_OK;
  DeviceGuard g(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = dbg_register(h, st, {{codes_u8, rows * cols / 2, false},
                                       {guide_bits, rows * cols / 4, true}});
  if (e == cudaSuccess)
    e = timed(h, TRACE_KERNEL_GUIDE_PACK, st, [&] {
      return tfp4::launch_guide_pack(codes_u8, nchunks, guide_bits, h->sm_count, st);
    });
  if (e != cudaSuccess) return cuda_fail(h, e);
  return TRACE_OK;
}

trace_status_t trace_guide_unpack(trace_handle_t h, const void* x_ref_bf16,
                                  const uint32_t* guide_bits, const void* bs_r,
                                  const float* gs_r, trace_segments_t seg_r, int64_t rows,
                                  int64_t cols, void* codes_u8, trace_stream_t stream) {
  if (!h) return TRACE_ERR_INVALID_ARG;
  trace_status_t s = check_shape(rows, cols);
  if (s != TRACE_OK) return s;
  const bool empty = rows == 0;
  for (const void* p : {x_ref_bf16, (const void*)guide_bits, bs_r, (const void*)codes_u8})
    if ((s = check_tensor(p, empty)) != TRACE_OK) return s;
  if (!gs_r) return TRACE_ERR_INVALID_ARG;
  if (!aligned(gs_r, 4)) return TRACE_ERR_ALIGNMENT;
  static thread_local tfp4::SegParam sp;
  if ((s = make_segments(seg_r, rows, &sp)) != TRACE_OK) return s;
  const int64_t nchunks = rows * (cols / 32);
  if (nchunks == 0) return TRACE_OK;
  DeviceGuard g(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = dbg_register(h, st, {{x_ref_bf16, rows * cols * 2, false},
                                       {guide_bits, rows * cols / 4, false},
                                       {bs_r, rows * cols / 16, false},
                                       {gs_r, (int64_t)sizeof(float) * sp.n, false},
                                       {codes_u8, rows * cols / 2, true}});
  if (e == cudaSuccess)
    e = timed(h, TRACE_KERNEL_GUIDE_UNPACK, st, [&] {
      return tfp4::launch_guide_unpack(x_ref_bf16, guide_bits, bs_r, gs_r, nchunks,
                                       (int32_t)(cols / 32), sp, codes_u8, h->sm_count, st);
    });
  if (e != cudaSuccess) return cuda_fail(h, e);
  return TRACE_OK;
}

}  // extern "C"

namespace {

// The training-side fake quantiser; gs_t == nullptr: the call first runs the
// amax pass over x into the handle's training scales, or with amax_prev
// (delayed scaling) turns those maxima into them, and amax_out then receives
// x's own maxima from the fake-quant kernel itself.
trace_status_t train_fakequant_impl(trace_ctx* h, const void* x_bf16, int64_t rows, int64_t cols,
                                    trace_segments_t seg_t, const float* gs_t,
                                    trace_guide_kind_t kind, const void* guide, const void* bs_r,
                                    const float* gs_r, trace_segments_t seg_r, void* y_bf16,
                                    uint32_t* ste_mask, void* codes_t_u8,
                                    trace_stats_t* stats_dev, trace_stream_t stream,
                                    const float* amax_prev = nullptr, float* amax_out = nullptr) {
  if (!h) return TRACE_ERR_INVALID_ARG;
  trace_status_t s = check_shape(rows, cols);
  if (s != TRACE_OK) return s;
  if (kind != TRACE_GUIDE_NONE && kind != TRACE_GUIDE_FULL && kind != TRACE_GUIDE_COMPACT)
    return TRACE_ERR_INVALID_ARG;
  const bool empty = rows == 0;
  if ((s = check_tensor(x_bf16, empty)) != TRACE_OK) return s;
  if ((s = check_tensor(y_bf16, empty)) != TRACE_OK) return s;
  if (ste_mask && (s = check_tensor(ste_mask)) != TRACE_OK) return s;
  if (codes_t_u8 && (s = check_tensor(codes_t_u8)) != TRACE_OK) return s;
  if (stats_dev && !aligned(stats_dev, 8)) return TRACE_ERR_ALIGNMENT;
  if (gs_t && !aligned(gs_t, 4)) return TRACE_ERR_ALIGNMENT;
  if ((amax_prev && !aligned(amax_prev, 4)) || (amax_out && !aligned(amax_out, 4)))
    return TRACE_ERR_ALIGNMENT;
  if (amax_out && (codes_t_u8 || stats_dev)) return TRACE_ERR_INVALID_ARG;
  static thread_local tfp4::SegParam spt, spr;
  if ((s = make_segments(seg_t, rows, &spt)) != TRACE_OK) return s;
  if (kind != TRACE_GUIDE_NONE) {
    if ((s = check_tensor(guide, empty)) != TRACE_OK) return s;
    if ((s = check_tensor(bs_r, empty)) != TRACE_OK) return s;
    if (!gs_r) return TRACE_ERR_INVALID_ARG;
    if (!aligned(gs_r, 4)) return TRACE_ERR_ALIGNMENT;
    if ((s = make_segments(seg_r, rows, &spr)) != TRACE_OK) return s;
  } else {
    spr.n = 1;
    spr.off[0] = 0;
    spr.off[1] = (int32_t)rows;
  }
  const int64_t nchunks = rows * (cols / 32);
  if (nchunks == 0 && !amax_out) return TRACE_OK;

  DeviceGuard g(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = begin_call(h, st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  const int32_t cpr = (int32_t)(cols / 32);
  if (e == cudaSuccess && amax_out)
    e = cudaMemsetAsync(amax_out, 0, sizeof(float) * spt.n, st);
  if (e == cudaSuccess)
    e = dbg_register(h, st, {{x_bf16, rows * cols * 2, false}, {y_bf16, rows * cols * 2, true},
                             {ste_mask, rows * cols / 8, true}, {codes_t_u8, rows * cols / 2, true},
                             {stats_dev, (int64_t)sizeof(trace_stats_t), true},
                             {guide, kind == TRACE_GUIDE_FULL ? rows * cols / 2 : rows * cols / 4,
                              false},
                             {bs_r, rows * cols / 16, false},
                             {gs_r, (int64_t)sizeof(float) * spr.n, false},
                             {gs_t, (int64_t)sizeof(float) * spt.n, false},
                             {amax_prev, amax_prev ? (int64_t)sizeof(float) * spt.n : 0, false},
                             {amax_out, amax_out ? (int64_t)sizeof(float) * spt.n : 0, true},
                             {h->scratch.gs_train, (int64_t)sizeof(float) * spt.n, true}});
  if (e == cudaSuccess && amax_prev) {
    e = tfp4::launch_scales_from_amax(amax_prev, spt.n, h->scratch.gs_train, st);
    gs_t = h->scratch.gs_train;
  }
  if (e == cudaSuccess && !gs_t) {
    e = timed(h, TRACE_KERNEL_AMAX, st, [&] {
      return tfp4::launch_amax(x_bf16, nchunks, cpr, spt, h->scratch, h->scratch.gs_train,
                               h->sm_count, st);
    });
    gs_t = h->scratch.gs_train;
  }
  if (e == cudaSuccess) {
    tfp4::FakequantArgs a;
    a.x = x_bf16;
    a.nchunks = nchunks;
    a.cpr = cpr;
    a.gs_t = gs_t;
    a.kind = (int)kind;
    a.guide = guide;
    a.bs_r = bs_r;
    a.gs_r = gs_r;
    a.y = y_bf16;
    a.mask = ste_mask;
    a.codes_t = codes_t_u8;
    a.stats = stats_dev;
    a.amax_out = reinterpret_cast<uint32_t*>(amax_out);
    if (nchunks > 0)
      e = timed(h, TRACE_KERNEL_FAKEQUANT, st,
                [&] { return tfp4::launch_fakequant(a, spt, spr, h->sm_count, st); });
  }
  const cudaError_t e2 = end_call(h, st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  if (e2 != cudaSuccess) return cuda_fail(h, e2);
  return TRACE_OK;
}

}  // namespace

extern "C" {

trace_status_t trace_train_fakequant(trace_handle_t h, const void* x_bf16, int64_t rows,
                                     int64_t cols, trace_segments_t seg_t,
                                     trace_guide_kind_t kind, const void* guide,
                                     const void* bs_r, const float* gs_r,
                                     trace_segments_t seg_r, void* y_bf16, uint32_t* ste_mask,
                                     void* codes_t_u8, trace_stats_t* stats_dev,
                                     trace_stream_t stream) {
  return train_fakequant_impl(h, x_bf16, rows, cols, seg_t, nullptr, kind, guide, bs_r, gs_r,
                              seg_r, y_bf16, ste_mask, codes_t_u8, stats_dev, stream);
}

trace_status_t trace_train_fakequant_gs(trace_handle_t h, const void* x_bf16, int64_t rows,
                                        int64_t cols, trace_segments_t seg_t, const float* gs_t,
                                        trace_guide_kind_t kind, const void* guide,
                                        const void* bs_r, const float* gs_r,
                                        trace_segments_t seg_r, void* y_bf16,
                                        uint32_t* ste_mask, void* codes_t_u8,
                                        trace_stats_t* stats_dev, trace_stream_t stream) {
  if (!gs_t) return TRACE_ERR_INVALID_ARG;
  return train_fakequant_impl(h, x_bf16, rows, cols, seg_t, gs_t, kind, guide, bs_r, gs_r,
                              seg_r, y_bf16, ste_mask, codes_t_u8, stats_dev, stream);
}

trace_status_t trace_train_fakequant_delayed(trace_handle_t h, const void* x_bf16, int64_t rows,
                                             int64_t cols, trace_segments_t seg_t,
                                             const float* amax_prev_t, trace_guide_kind_t kind,
                                             const void* guide, const void* bs_r,
                                             const float* gs_r, trace_segments_t seg_r,
                                             void* y_bf16, uint32_t* ste_mask, float* amax_out_t,
                                             trace_stream_t stream) {
  if (!amax_prev_t) return TRACE_ERR_INVALID_ARG;
  return train_fakequant_impl(h, x_bf16, rows, cols, seg_t, nullptr, kind, guide, bs_r, gs_r,
                              seg_r, y_bf16, ste_mask, nullptr, nullptr, stream, amax_prev_t,
                              amax_out_t);
}

trace_status_t trace_segment_amax(trace_handle_t h, const void* x_bf16, int64_t rows,
                                  int64_t cols, trace_segments_t seg, float* gs_f32,
                                  trace_stream_t stream) {
  if (!h) return TRACE_ERR_INVALID_ARG;
  trace_status_t s = check_shape(rows, cols);
  if (s != TRACE_OK) return s;
  if ((s = check_tensor(x_bf16, rows == 0)) != TRACE_OK) return s;
  if (!gs_f32) return TRACE_ERR_INVALID_ARG;
  if (!aligned(gs_f32, 4)) return TRACE_ERR_ALIGNMENT;
  static thread_local tfp4::SegParam sp;
  if ((s = make_segments(seg, rows, &sp)) != TRACE_OK) return s;
  DeviceGuard g(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = begin_call(h, st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  const int64_t nchunks = rows * (cols / 32);
  if (e == cudaSuccess)
    e = dbg_register(h, st, {{x_bf16, rows * cols * 2, false},
                             {gs_f32, (int64_t)sizeof(float) * sp.n, true}});
  if (e != cudaSuccess) {
  } else if (nchunks == 0) {
    e = cudaMemsetAsync(gs_f32, 0, sizeof(float) * sp.n, st);
  } else {
    e = timed(h, TRACE_KERNEL_AMAX, st, [&] {
      return tfp4::launch_amax(x_bf16, nchunks, (int32_t)(cols / 32), sp, h->scratch, gs_f32,
                               h->sm_count, st);
    });
  }
  const cudaError_t e2 = end_call(h, st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  if (e2 != cudaSuccess) return cuda_fail(h, e2);
  return TRACE_OK;
}

trace_status_t trace_ste_backward(trace_handle_t h, const void* grad_out_bf16,
                                  const uint32_t* ste_mask, int64_t rows, int64_t cols,
                                  void* grad_in_bf16, trace_stream_t stream) {
  if (!h) return TRACE_ERR_INVALID_ARG;
  trace_status_t s = check_shape(rows, cols);
  if (s != TRACE_OK) return s;
  const bool empty = rows == 0;
  for (const void* p : {grad_out_bf16, (const void*)ste_mask, (const void*)grad_in_bf16})
    if ((s = check_tensor(p, empty)) != TRACE_OK) return s;
  const int64_t nchunks = rows * (cols / 32);
  if (nchunks == 0) return TRACE_OK;
  DeviceGuard g(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = dbg_register(h, st, {{grad_out_bf16, rows * cols * 2, false},
                                       {ste_mask, rows * cols / 8, false},
                                       {grad_in_bf16, rows * cols * 2, true}});
  if (e == cudaSuccess)
    e = timed(h, TRACE_KERNEL_STE_BACKWARD, st, [&] {
      return tfp4::launch_ste_backward(grad_out_bf16, ste_mask, nchunks, grad_in_bf16,
                                       h->sm_count, st);
    });
  if (e != cudaSuccess) return cuda_fail(h, e);
  return TRACE_OK;
}

// ---- guide transport -------------------------------------------------------

static_assert(sizeof(trace_record_header_t) == 64, "record header is 64 bytes");

static uint64_t align256(uint64_t v) { return (v + 255u) & ~uint64_t(255); }

// Full record: one 4-bit code per element; compact: one 32-bit word (16 sign
// bits, 16 index-parity bits) per 16 elements.
static uint64_t record_guide_bytes(const trace_record_header_t& hd) {
  return hd.kind == TRACE_GUIDE_FULL ? (uint64_t)hd.rows * (uint64_t)(hd.cols / 2)
                                     : (uint64_t)hd.rows * (uint64_t)(hd.cols / 16) * 4;
}

static uint64_t record_bs_bytes(const trace_record_header_t& hd) {
  return (uint64_t)hd.rows * (uint64_t)(hd.cols / 16);
}

static bool record_layout(trace_guide_kind_t kind, int64_t rows, int64_t cols, int32_t n_seg,
                          trace_record_header_t* hd) {
  if (kind != TRACE_GUIDE_FULL && kind != TRACE_GUIDE_COMPACT) return false;
  if (check_shape(rows, cols) != TRACE_OK) return false;
  if (n_seg < 1 || n_seg > TRACE_MAX_SEGMENTS) return false;
  memset(hd, 0, sizeof(*hd));
  hd->kind = (uint32_t)kind;
  hd->rows = rows;
  hd->cols = cols;
  const uint64_t guide_bytes = record_guide_bytes(*hd), bs_bytes = record_bs_bytes(*hd);
  hd->magic = TRACE_RECORD_MAGIC;
  hd->version = 1;
  hd->n_seg = n_seg;
  hd->guide_offset = 256;
  hd->bs_offset = align256(hd->guide_offset + guide_bytes);
  hd->gs_offset = align256(hd->bs_offset + bs_bytes);
  hd->seg_offset = align256(hd->gs_offset + sizeof(float) * (uint64_t)n_seg);
  return true;
}

static uint64_t record_end(const trace_record_header_t& hd) {
  return hd.seg_offset + sizeof(int64_t) * ((uint64_t)hd.n_seg + 1);
}

extern "C" size_t trace_record_size(trace_guide_kind_t kind, int64_t rows, int64_t cols,
                                    int32_t n_seg) {
  trace_record_header_t hd;
  if (!record_layout(kind, rows, cols, n_seg, &hd)) return 0;
  return (size_t)record_end(hd);
}

extern "C" trace_status_t trace_record_export(trace_handle_t h, trace_guide_kind_t kind,
                                              const void* guide, const void* bs,
                                              const float* gs, int64_t rows, int64_t cols,
                                              trace_segments_t seg, void* host_dst,
                                              size_t dst_bytes, trace_stream_t stream) {
  if (!h || !host_dst) return TRACE_ERR_INVALID_ARG;
  const int32_t n_seg = seg.row_offsets ? seg.n_seg : 1;
  trace_record_header_t hd;
  if (!record_layout(kind, rows, cols, n_seg, &hd)) return TRACE_ERR_INVALID_ARG;
  if (dst_bytes < record_end(hd)) return TRACE_ERR_INVALID_ARG;
  static thread_local tfp4::SegParam sp;
  trace_status_t s = make_segments(seg, rows, &sp);
  if (s != TRACE_OK) return s;
  const bool empty = rows == 0;
  if ((s = check_tensor(guide, empty)) != TRACE_OK) return s;
  if ((s = check_tensor(bs, empty)) != TRACE_OK) return s;
  if (!gs) return TRACE_ERR_INVALID_ARG;
  uint8_t* dst = (uint8_t*)host_dst;
  memset(dst, 0, 256);
  memcpy(dst, &hd, sizeof(hd));
  int64_t* offs = (int64_t*)(dst + hd.seg_offset);
  for (int32_t i = 0; i <= n_seg; ++i) offs[i] = sp.off[i];
  DeviceGuard g(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  const uint64_t guide_bytes = record_guide_bytes(hd), bs_bytes = record_bs_bytes(hd);
  cudaError_t e = cudaSuccess;
  if (guide_bytes) e = cudaMemcpyAsync(dst + hd.guide_offset, guide, guide_bytes, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && bs_bytes)
    e = cudaMemcpyAsync(dst + hd.bs_offset, bs, bs_bytes, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(dst + hd.gs_offset, gs, sizeof(float) * n_seg, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  return TRACE_OK;
}

extern "C" trace_status_t trace_record_info(const void* host_src, size_t src_bytes,
                                            trace_record_header_t* out) {
  if (!host_src || !out || src_bytes < sizeof(trace_record_header_t)) return TRACE_ERR_INVALID_ARG;
  trace_record_header_t hd;
  memcpy(&hd, host_src, sizeof(hd));
  trace_record_header_t ref;
  if (hd.magic != TRACE_RECORD_MAGIC || hd.version != 1) return TRACE_ERR_INVALID_ARG;
  if (!record_layout((trace_guide_kind_t)hd.kind, hd.rows, hd.cols, hd.n_seg, &ref))
    return TRACE_ERR_INVALID_ARG;
  if (ref.guide_offset != hd.guide_offset || ref.bs_offset != hd.bs_offset ||
      ref.gs_offset != hd.gs_offset || ref.seg_offset != hd.seg_offset)
    return TRACE_ERR_INVALID_ARG;
  if (src_bytes < record_end(hd)) return TRACE_ERR_INVALID_ARG;
  const int64_t* offs = (const int64_t*)((const uint8_t*)host_src + hd.seg_offset);
  if (offs[0] != 0 || offs[hd.n_seg] != hd.rows) return TRACE_ERR_INVALID_ARG;
  for (int32_t i = 0; i < hd.n_seg; ++i)
    if (offs[i + 1] < offs[i]) return TRACE_ERR_INVALID_ARG;
  *out = hd;
  return TRACE_OK;
}

extern "C" trace_status_t trace_record_import(trace_handle_t h, const void* host_src,
                                              size_t src_bytes, void* guide, void* bs, float* gs,
                                              trace_stream_t stream) {
  if (!h) return TRACE_ERR_INVALID_ARG;
  trace_record_header_t hd;
  trace_status_t s = trace_record_info(host_src, src_bytes, &hd);
  if (s != TRACE_OK) return s;
  const bool empty = hd.rows == 0;
  if ((s = check_tensor(guide, empty)) != TRACE_OK) return s;
  if ((s = check_tensor(bs, empty)) != TRACE_OK) return s;
  if (!gs) return TRACE_ERR_INVALID_ARG;
  const uint64_t guide_bytes = record_guide_bytes(hd), bs_bytes = record_bs_bytes(hd);
  const uint8_t* src = (const uint8_t*)host_src;
  DeviceGuard g(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  if (guide_bytes) e = cudaMemcpyAsync(guide, src + hd.guide_offset, guide_bytes, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && bs_bytes)
    e = cudaMemcpyAsync(bs, src + hd.bs_offset, bs_bytes, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(gs, src + hd.gs_offset, sizeof(float) * hd.n_seg, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  return TRACE_OK;
}

// ---- f4: tensor-core scale layout and the NVFP4 GEMM -------------------------

extern "C" size_t trace_block_scales_mma_bytes(int64_t rows, int64_t cols) {
  if (check_shape(rows, cols) != TRACE_OK) return 0;
  const int64_t b = tfp4::mma_scales_bytes(rows, cols);
  return b < 0 ? 0 : (size_t)b;
}

extern "C" trace_status_t trace_block_scales_mma(trace_handle_t h, const void* bs_e4m3,
                                                 int64_t rows, int64_t cols, void* out,
                                                 trace_stream_t stream) {
  if (!h) return TRACE_ERR_INVALID_ARG;
  trace_status_t s = check_shape(rows, cols);
  if (s != TRACE_OK) return s;
  const bool empty = rows == 0;
  if (!bs_e4m3 && !empty) return TRACE_ERR_INVALID_ARG;
  if ((s = check_tensor(out, empty)) != TRACE_OK) return s;
  DeviceGuard g(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  const cudaError_t e = timed(h, TRACE_KERNEL_MMA_SCALES, st, [&] {
    return tfp4::launch_mma_scales(bs_e4m3, rows, cols, out, h->sm_count, st);
  });
  if (e != cudaSuccess) return cuda_fail(h, e);
  return TRACE_OK;
}

extern "C" trace_status_t trace_nvfp4_gemm(trace_handle_t h, const void* a_codes,
                                           const void* a_scales_mma, const float* a_gs,
                                           const void* b_codes, const void* b_scales_mma,
                                           const float* b_gs, int64_t m, int64_t n, int64_t k,
                                           void* d, trace_out_t d_type, trace_stream_t stream) {
  if (!h) return TRACE_ERR_INVALID_ARG;
  if (m <= 0 || n <= 0 || k <= 0 || k % 32) return TRACE_ERR_INVALID_ARG;
  if (check_shape(m, k) != TRACE_OK || check_shape(n, k) != TRACE_OK) return TRACE_ERR_INVALID_ARG;
  if (d_type != TRACE_OUT_F32 && d_type != TRACE_OUT_BF16) return TRACE_ERR_INVALID_ARG;
  trace_status_t s;
  for (const void* p : {a_codes, a_scales_mma, b_codes, b_scales_mma, (const void*)d})
    if ((s = check_tensor(p)) != TRACE_OK) return s;
  if (!a_gs || !b_gs) return TRACE_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  if (h->gemm != TRACE_GEMM_CUBLASLT) {
    cudaError_t e = begin_call(h, st);
    if (e == cudaSuccess)
      e = timed(h, TRACE_KERNEL_NVFP4_GEMM, st, [&] {
        return tfp4::launch_nvfp4_gemm_tc(a_codes, a_scales_mma, a_gs, b_codes, b_scales_mma,
                                          b_gs, m, n, k, d, d_type == TRACE_OUT_BF16,
                                          h->gemm == TRACE_GEMM_TC128    ? tfp4::kGemmTile128
                                          : h->gemm == TRACE_GEMM_TC_PAIR ? tfp4::kGemmTilePair
                                                                          : tfp4::kGemmTile256,
                                          h->scratch.err, h->wait_ns, h->sm_count, st);
      });
    const cudaError_t e2 = end_call(h, st);
    if (e != cudaSuccess) return cuda_fail(h, e);
    if (e2 != cudaSuccess) return cuda_fail(h, e2);
    return TRACE_OK;
  }
  if (!tfp4::lt_available()) return TRACE_ERR_LIBRARY;
  if (!h->gemm_ws) {
    const size_t ws = size_t(32) << 20;
    if (cudaMalloc(&h->gemm_ws, ws) != cudaSuccess) {
      cudaGetLastError();
      h->gemm_ws = nullptr;
      return TRACE_ERR_OOM;
    }
    h->gemm_ws_bytes = ws;
  }
  cudaError_t e = begin_call(h, st);
  if (e == cudaSuccess) e = tfp4::launch_gemm_scalars(a_gs, b_gs, h->gemm_scalars, st);
  if (e != cudaSuccess) return cuda_fail(h, e);
  int rc = 0;
  e = timed(h, TRACE_KERNEL_NVFP4_GEMM, st, [&] {
    rc = tfp4::lt_nvfp4_gemm(&h->lt, h->gemm_ws, h->gemm_ws_bytes, a_codes, a_scales_mma,
                             b_codes, b_scales_mma, h->gemm_scalars, m, n, k, d,
                             d_type == TRACE_OUT_BF16, st);
    return cudaSuccess;
  });
  const cudaError_t e2 = end_call(h, st);
  if (rc != 0) {
    h->last_error = rc;
    return TRACE_ERR_LIBRARY;
  }
  if (e != cudaSuccess) return cuda_fail(h, e);
  if (e2 != cudaSuccess) return cuda_fail(h, e2);
  return TRACE_OK;
}

trace_status_t trace_profile_enable(trace_handle_t h, int enable) {
  if (!h) return TRACE_ERR_INVALID_ARG;
  h->profiling = enable != 0;
  return TRACE_OK;
}

trace_status_t trace_profile_collect(trace_handle_t h, trace_kernel_time_t* out) {
  if (!h || !out) return TRACE_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  for (int k = 0; k < TRACE_KERNEL_COUNT; ++k) {
    out[k].launches = 0;
    out[k].total_ms = 0.0;
  }
  cudaError_t first = cudaSuccess;
  for (auto& t : h->timed) {
    float ms = 0.0f;
    cudaError_t e = cudaEventSynchronize(t.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t.start, t.stop);
    if (e == cudaSuccess) {
      out[t.kernel].launches += 1;
      out[t.kernel].total_ms += ms;
    } else if (first == cudaSuccess) {
      first = e;
    }
    h->spare.push_back(t.start);
    h->spare.push_back(t.stop);
  }
  h->timed.clear();
  if (first != cudaSuccess) return cuda_fail(h, first);
  return TRACE_OK;
}

}  // extern "C"

namespace tfp4 {

cudaError_t dbg_set_ranges(const DbgRanges& r, cudaStream_t st) {
  cudaError_t e = dbg_set_ranges_kernels(r, st);
  if (e == cudaSuccess) e = dbg_set_ranges_fakequant(r, st);
  return e;
}

unsigned long long dbg_take_violations() {
  const unsigned long long a = dbg_take_kernels(), b = dbg_take_fakequant();
  return (a == ~0ull || b == ~0ull) ? ~0ull : a + b;
}

}  // namespace tfp4

extern "C" trace_status_t trace_debug_bounds(trace_handle_t h, int* checked,
                                             uint64_t* violations) {
  if (!h || !checked || !violations) return TRACE_ERR_INVALID_ARG;
#ifdef TRACE_DEBUG_BOUNDS
  DeviceGuard g(h->device);
  *checked = 1;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(h, e);
  const unsigned long long v = tfp4::dbg_take_violations();
  if (v == ~0ull) return cuda_fail(h, cudaGetLastError());
  *violations = v;
#else
  *checked = 0;
  *violations = 0;
#endif
  return TRACE_OK;
}
