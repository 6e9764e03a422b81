/*
 * trace_fp4.h - C ABI of libtrace_fp4.so, the GB300 (sm_103a) hot path of
 * TRACE: rollout-side NVFP4 quantisation with a compact guidance record, and
 * training-side rollout-guided FP4 fake quantisation.
 *
 * Sources (page title, section):
 *   [EN] "Alibaba Qwen Proposes TRACE for 5.4x Faster FP4 RL Rollouts"
 *     - "Why Does FP4 Rollout 'Break' RL Training?", worked example after
 *       Fig. 1: nearly equal train/rollout values that share a global and a
 *       block scale can round to different E2M1 points (60.24 -> 3,
 *       59.76 -> 2, gap amplified to 24).
 *     - "TRACE Core Concept", first design (before Fig. 3): rollout records the
 *       FP4 results of routed-expert activations and KV states; training-side
 *       fake quantisation picks, of the two adjacent E2M1 points, the one
 *       closer to the rollout's actual point instead of plain RTN.
 *     - "TRACE Core Concept", second design (after Fig. 3): full records are
 *       costly to move GPU -> CPU -> disk -> GPU; over 99% of mismatches are
 *       one codebook entry apart, so a little mantissa information plus the
 *       scale suffices to set the rounding direction.
 *   Number formats: OCP Microscaling Formats v1.0 (FP4 E2M1, FP8 E4M3);
 *   NVFP4 two-level scaling (FP32 tensor scale, E4M3 scale per 16 values).
 *
 * Common conventions
 *   - Tensors are row-major [rows, cols] with cols % 32 == 0 and cols > 0;
 *     rows == 0 is an empty, valid input whose tensor pointers may be NULL
 *     (trace_rollout_quant still writes gs = 0 for every segment).
 *     rows * cols / 32 must stay below
 *     2^31 and rows below 2^31.  A "block" is 16 consecutive elements of a row.
 *   - bf16 values are passed as raw 16-bit patterns.
 *   - Packed E2M1 codes: uint8 [rows, cols/2]; element 2i is the low nibble
 *     of byte i; nibble = (sign << 3) | m, m = 0..7 indexes the magnitudes
 *     {0, 0.5, 1, 1.5, 2, 3, 4, 6}.  The sign is always the input's sign.
 *   - Block scales: uint8 E4M3 codes [rows, cols/16], plain row-major;
 *     trace_rollout_quant_mma can also write them in the tensor-core tile
 *     layout of block-scaled GEMMs.
 *   - Global scales: float [n_seg], gs = amax / (6 * 448) per segment.
 *   - Compact guide: uint32 [rows, cols/16]; for element j of a block, bit j
 *     is its sign and bit 16+j the low bit of its E2M1 index (the single
 *     mantissa bit).
 *   - STE mask: uint32 [rows, cols/32]; bit j of word w covers element 32w+j
 *     of the row and is 0 exactly when the element was clipped by the top
 *     code (S > 0 and |x| > 6*S), else 1.
 *   - Segments: a host array of n_seg + 1 int64 row offsets with [0] == 0,
 *     [n_seg] == rows, non-decreasing (empty segments allowed), at most
 *     TRACE_MAX_SEGMENTS segments.  row_offsets == NULL means one segment
 *     over all rows.  The table travels in the kernel's parameter block; the
 *     caller may free it as soon as the call returns.
 *   - All tensor pointers are caller-owned DEVICE pointers on the handle's
 *     device, 16-byte aligned (host pointers only where a call says so).
 *     Calls enqueue work on `stream` and never synchronise the host, except
 *     trace_device_status and the first trace_nvfp4_gemm of a handle (which
 *     allocates its workspace).  Global scales never leave the device unless
 *     a record is exported.
 *   - Errors: argument errors return before anything is enqueued.  A failed
 *     launch returns TRACE_ERR_CUDA and the raw cudaError_t is available from
 *     trace_last_cuda_error.  Nothing aborts and no exception crosses the ABI.
 *   - Threading: one host thread at a time per handle.  Calls through one
 *     handle on different streams are ordered on the handle's scratch with
 *     an internal event, so they run one after another on the GPU.  Work
 *     that should run concurrently uses one handle per stream (each has its
 *     own scratch).
 *   - Inputs must be finite; NaN/Inf inputs give unspecified codes but never
 *     fault.
 *
 * Arithmetic (shared by every entry point; each step is binary32 with round
 * to nearest even, no fused multiply-add, subnormals kept):
 *   amax  = max |x| over the segment;  gs = amax / 2688 (0 if amax == 0)
 *   bs    = E4M3_rne_satfinite(block_amax / (gs * 6))   (0 if gs == 0)
 *   S     = decode(bs) * gs;  inv = 1 / S, or 0 when S == 0 or 1/S overflows
 *   t     = |x| * inv;  RTN index = nearest E2M1 magnitude, ties to the even
 *           index, t > 6 -> 7;  bracket {lo, hi} = the adjacent points of t
 */
#ifndef TRACE_FP4_H
#define TRACE_FP4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TRACE_API __attribute__((visibility("default")))
#else
#define TRACE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct trace_ctx* trace_handle_t;
typedef struct CUstream_st* trace_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  TRACE_OK = 0,
  TRACE_ERR_INVALID_ARG = 1,        /* null pointer, bad shape or segment table */
  TRACE_ERR_ALIGNMENT = 2,          /* a tensor pointer is not 16-byte aligned   */
  TRACE_ERR_UNSUPPORTED_DEVICE = 3, /* no device, or not compute capability 10.3 */
  TRACE_ERR_CUDA = 4,               /* a CUDA call failed; see trace_last_cuda_error */
  TRACE_ERR_OOM = 5,                /* device scratch could not be allocated     */
  TRACE_ERR_TIMEOUT = 6,            /* a bounded device wait gave up (reported by
                                       trace_device_status)                      */
  TRACE_ERR_LIBRARY = 7             /* cuBLASLt is missing or refused the GEMM;
                                       its status is in trace_last_cuda_error     */
} trace_status_t;

typedef enum {
  TRACE_GUIDE_NONE = 0,    /* plain RTN fake quantisation                    */
  TRACE_GUIDE_FULL = 1,    /* guide = rollout codes uint8 [rows, cols/2]     */
  TRACE_GUIDE_COMPACT = 2  /* guide = compact words uint32 [rows, cols/16]   */
} trace_guide_kind_t;

#define TRACE_MAX_SEGMENTS 4000

typedef struct {
  const int64_t* row_offsets; /* host array [n_seg + 1], or NULL for one segment */
  int32_t n_seg;              /* ignored when row_offsets == NULL                */
} trace_segments_t;

/* Train/rollout code agreement counters, accumulated (never cleared) by
 * trace_train_fakequant.  Signed index k = sign ? -m : m (so +0 == -0); a
 * mismatch is k_train != k_rollout.  hist_* count |dk| = 0, 1, 2, >= 3.
 * With TRACE_GUIDE_NONE only n_elems advances. */
typedef struct {
  uint64_t n_elems;
  uint64_t mismatch_rtn;
  uint64_t mismatch_guided;
  uint64_t hist_rtn[4];
  uint64_t hist_guided[4];
} trace_stats_t;

/* Kernel identifiers for the built-in profiler. */
typedef enum {
  TRACE_KERNEL_AMAX = 0,
  TRACE_KERNEL_ROLLOUT_QUANT = 1,
  TRACE_KERNEL_GUIDE_PACK = 2,
  TRACE_KERNEL_GUIDE_UNPACK = 3,
  TRACE_KERNEL_FAKEQUANT = 4,
  TRACE_KERNEL_STE_BACKWARD = 5,
  TRACE_KERNEL_ROLLOUT_FUSED = 6, /* amax + quantisation in one launch */
  TRACE_KERNEL_MMA_SCALES = 7,    /* block scales -> tensor-core tile layout */
  TRACE_KERNEL_NVFP4_GEMM = 8,    /* the GEMM (the tcgen05 kernel, or all of
                                     cuBLASLt's kernels)                     */
  TRACE_KERNEL_ROLLOUT_DELAYED = 9, /* quantisation with given maxima        */
  TRACE_KERNEL_COUNT = 10
} trace_kernel_id_t;

typedef struct {
  uint64_t launches; /* launches timed since the last collect        */
  double total_ms;   /* summed CUDA-event time of those launches     */
} trace_kernel_time_t;

/* Creates a handle on `device`: checks for compute capability 10.3 and
 * allocates the device scratch (per-segment amax words, a completion ticket,
 * per-segment training global scales, wave counters and an error word of
 * the fused rollout kernel).  *out is NULL on failure. */
TRACE_API trace_status_t trace_create(trace_handle_t* out, int device);

/* Frees the handle.  The caller must have finished (synchronised) all work
 * enqueued through it.  NULL is accepted. */
TRACE_API trace_status_t trace_destroy(trace_handle_t h);

/* Static text for a status code. */
TRACE_API const char* trace_status_string(trace_status_t s);

/* Raw cudaError_t of the last TRACE_ERR_CUDA on this handle (0 if none). */
TRACE_API int trace_last_cuda_error(trace_handle_t h);

/* Library version as major*10000 + minor*100 + patch. */
TRACE_API int trace_version(void);

/* Per-handle options (trace_set_option returns TRACE_ERR_INVALID_ARG for an
 * unknown option or a value out of range). */
typedef enum {
  TRACE_OPT_FUSED_AMAX = 0,    /* 1 (default): fuse amax into trace_rollout_quant
                                  where segments fit; 0: always two kernels   */
  TRACE_OPT_WAVE_BYTES = 1,    /* target bytes of x per wave of the fused kernel,
                                  4 KiB .. 40 MiB (default 32 MiB)            */
  TRACE_OPT_WAIT_LIMIT_NS = 2, /* limit of each in-kernel wait, 1 ms .. 10 s
                                  (default 1 s)                               */
  TRACE_OPT_WAIT_EXTRA = 3,    /* test hook, 0 (default) or 1: each wait also
                                  expects an arrival that never comes, so every
                                  wait runs out at its limit                  */
  TRACE_OPT_DEBUG_SHRINK = 4,  /* test hook of builds with TRACE_DEBUG_BOUNDS
                                  (see trace_debug_bounds), 0 (default) or 1:
                                  every output buffer is registered 16 bytes
                                  short, so the kernels' last stores into it
                                  are counted as out of range and skipped.
                                  Other builds return TRACE_ERR_INVALID_ARG. */
  TRACE_OPT_GEMM = 5           /* form of trace_nvfp4_gemm: TRACE_GEMM_TC256
                                  (default), TRACE_GEMM_TC128,
                                  TRACE_GEMM_TC_PAIR or TRACE_GEMM_CUBLASLT   */
} trace_option_t;

/* Values of TRACE_OPT_GEMM. */
enum {
  TRACE_GEMM_TC256 = 0,    /* hand-written tcgen05 kernel, 128 x 256 output tiles */
  TRACE_GEMM_CUBLASLT = 1, /* cuBLASLt's block-scaled GEMM                        */
  TRACE_GEMM_TC128 = 2,    /* hand-written tcgen05 kernel, 128 x 128 output tiles */
  TRACE_GEMM_TC_PAIR = 3   /* hand-written tcgen05 kernel, 256 x 256 output tiles
                              on SM pairs (two-CTA clusters)                      */
};
TRACE_API trace_status_t trace_set_option(trace_handle_t h, trace_option_t opt, int64_t value);

/* Synchronises `stream`, then reports and clears the handle's device-side
 * error word: TRACE_ERR_TIMEOUT if an in-kernel wait of an earlier call ran
 * out, else TRACE_OK. */
TRACE_API trace_status_t trace_device_status(trace_handle_t h, trace_stream_t stream);

/* Rollout-side quantisation ([EN] "TRACE Core Concept", first and second
 * designs): per-segment amax and global scale, per-block E4M3 scale, per-
 * element RTN E2M1 code, and (if guide_bits != NULL) the compact guide words.
 *   x_bf16     [rows, cols] bf16
 *   codes_u8   [rows, cols/2] out
 *   bs_e4m3    [rows, cols/16] out
 *   gs_f32     [n_seg] out (device)
 *   guide_bits [rows, cols/16] out, nullable
 * When every segment holds at most 40 MiB of x (and TRACE_OPT_FUSED_AMAX is
 * on) this is one cooperative kernel that reads x from HBM once: segments
 * are taken in L2-sized waves, amax first, then quantisation from L2.  A
 * wait inside it that runs out (TRACE_OPT_WAIT_LIMIT_NS) leaves the outputs
 * undefined and is reported by trace_device_status.  Otherwise two kernels:
 * a streaming amax pass, then the quantiser. */
TRACE_API trace_status_t trace_rollout_quant(trace_handle_t h, const void* x_bf16, int64_t rows,
                                   int64_t cols, trace_segments_t seg, void* codes_u8,
                                   void* bs_e4m3, float* gs_f32, uint32_t* guide_bits,
                                   trace_stream_t stream);

/* Full codes -> compact guide words ([EN] "TRACE Core Concept", second
 * design): keeps each element's sign and index low bit.  Integer only.
 *   codes_u8 [rows, cols/2] in; guide_bits [rows, cols/16] out. */
TRACE_API trace_status_t trace_guide_pack(trace_handle_t h, const void* codes_u8, int64_t rows,
                                int64_t cols, uint32_t* guide_bits, trace_stream_t stream);

/* Compact guide words + reference values -> full rollout codes ([EN] "TRACE
 * Core Concept", second design: the reference value narrows the candidates).
 * For each element t = |x_ref| * inv_r in the rollout's own scale frame
 * (S_r = decode(bs_r) * gs_r[segment]); of the two adjacent E2M1 points the
 * one whose index low bit equals the stored bit is decoded; a point bracket
 * needs no bit.  The sign comes from the guide.
 *   x_ref_bf16 [rows, cols]; guide_bits [rows, cols/16]; bs_r [rows, cols/16];
 *   gs_r [n_seg_r] (device); codes_u8 [rows, cols/2] out. */
TRACE_API trace_status_t trace_guide_unpack(trace_handle_t h, const void* x_ref_bf16,
                                  const uint32_t* guide_bits, const void* bs_r,
                                  const float* gs_r, trace_segments_t seg_r, int64_t rows,
                                  int64_t cols, void* codes_u8, trace_stream_t stream);

/* Training-side rollout-guided fake quantisation ([EN] "TRACE Core Concept",
 * first design).  The training tensor uses its own scales (segments seg_t).
 * Each element is restricted to its bracket {lo, hi}; the candidate whose
 * dequantised value (with the training scale) is closer to the rollout's
 * reconstructed value (rollout code with the rollout scale; decoded from the
 * compact word against x itself when kind == COMPACT) is chosen; equal
 * distances, a point bracket or kind == NONE give RTN.
 *   x_bf16 [rows, cols]
 *   guide: codes uint8 [rows, cols/2] (FULL) or words uint32 [rows, cols/16]
 *          (COMPACT); ignored for NONE
 *   bs_r [rows, cols/16], gs_r [n_seg_r] (device), seg_r: the rollout's
 *          scales; ignored for NONE
 *   y_bf16 [rows, cols] out: +-G[m] * S_t rounded to bf16
 *   ste_mask [rows, cols/32] out, nullable
 *   codes_t_u8 [rows, cols/2] out, nullable: the chosen training codes
 *   stats_dev: device trace_stats_t, nullable, accumulated atomically
 * Two kernels: the amax pass over x, then the fused fake quantiser. */
TRACE_API trace_status_t trace_train_fakequant(trace_handle_t h, const void* x_bf16, int64_t rows,
                                     int64_t cols, trace_segments_t seg_t,
                                     trace_guide_kind_t kind, const void* guide,
                                     const void* bs_r, const float* gs_r,
                                     trace_segments_t seg_r, void* y_bf16, uint32_t* ste_mask,
                                     void* codes_t_u8, trace_stats_t* stats_dev,
                                     trace_stream_t stream);

/* trace_train_fakequant with the training scales supplied: the fake
 * quantiser alone.  gs_t [n_seg_t] (device) holds one global scale per
 * training segment, as trace_segment_amax writes them for the same x and
 * seg_t; with those scales the outputs equal trace_train_fakequant's bit for
 * bit.  Lets the training-side amax pass run earlier, for instance on another
 * handle and stream while the rollout-side calls run.  gs_t == NULL is an
 * argument error. */
TRACE_API trace_status_t trace_train_fakequant_gs(trace_handle_t h, const void* x_bf16,
                                                  int64_t rows, int64_t cols,
                                                  trace_segments_t seg_t, const float* gs_t,
                                                  trace_guide_kind_t kind, const void* guide,
                                                  const void* bs_r, const float* gs_r,
                                                  trace_segments_t seg_r, void* y_bf16,
                                                  uint32_t* ste_mask, void* codes_t_u8,
                                                  trace_stats_t* stats_dev,
                                                  trace_stream_t stream);

/* The training-side fake quantiser with delayed scaling: as
 * trace_train_fakequant_gs with gs_t[s] = amax_prev_t[s] / 2688 (binary32;
 * a maximum that is not positive gives 0), but with the maxima given instead
 * of the scales and, if amax_out_t != NULL, x's own training-segment maxima
 * returned by the fake-quant kernel itself (bit-exact with a separate amax
 * pass) for the next call, so that x is read once.  Delayed scaling is a
 * deployment option of this library, not the pages' definition (see
 * trace_rollout_quant_delayed).  y and the STE mask (which may be NULL) only:
 * no training codes, no counters.  The handle's training-scale scratch holds
 * the scales, so calls through one handle run one after another.
 *   amax_prev_t [n_seg_t] device; amax_out_t [n_seg_t] out (device, may be
 *   NULL; zero rows zeroes it).  Other arguments as trace_train_fakequant. */
TRACE_API trace_status_t trace_train_fakequant_delayed(
    trace_handle_t h, const void* x_bf16, int64_t rows, int64_t cols, trace_segments_t seg_t,
    const float* amax_prev_t, trace_guide_kind_t kind, const void* guide, const void* bs_r,
    const float* gs_r, trace_segments_t seg_r, void* y_bf16, uint32_t* ste_mask,
    float* amax_out_t, trace_stream_t stream);

/* Per-segment amax and global scale alone ([EN] "TRACE Core Concept": one
 * FP32 global scale per segment, gs = amax / (448 * 6)); the first pass of
 * trace_rollout_quant's two-kernel form and of trace_train_fakequant.
 *   x_bf16 [rows, cols]; gs_f32 [n_seg] out (device); an empty or all-zero
 *   segment gets 0.  One streaming kernel (no wait on other CTAs). */
TRACE_API trace_status_t trace_segment_amax(trace_handle_t h, const void* x_bf16, int64_t rows,
                                            int64_t cols, trace_segments_t seg, float* gs_f32,
                                            trace_stream_t stream);

/* Backward of the fake quantiser through the straight-through estimator
 * (the article's title names quantization-aware training, which trains
 * through the fake quantiser): grad_in = grad_out where the element's mask
 * bit (from trace_train_fakequant) is 1, +0 where it is 0.
 *   grad_out_bf16 [rows, cols]; ste_mask [rows, cols/32];
 *   grad_in_bf16 [rows, cols] out (may alias grad_out_bf16). */
TRACE_API trace_status_t trace_ste_backward(trace_handle_t h, const void* grad_out_bf16,
                                            const uint32_t* ste_mask, int64_t rows,
                                            int64_t cols, void* grad_in_bf16,
                                            trace_stream_t stream);

/* Guide transport ([EN] "TRACE Core Concept", second design: rollout
 * records travel GPU -> CPU -> CPU cache -> disk -> back to the GPU, which is
 * why the compact record exists).  A record is one byte buffer: a 64-byte
 * header, then 256-byte-aligned sections: the guide (full codes
 * [rows, cols/2] or compact words [rows, cols/16]), the block scales
 * [rows, cols/16], the global scales [n_seg] and the row offsets
 * [n_seg + 1] (int64).  The buffer can be written to disk as is. */
#define TRACE_RECORD_MAGIC 0x31475254u /* "TRG1" little-endian */
typedef struct {
  uint32_t magic;      /* TRACE_RECORD_MAGIC                              */
  uint32_t version;    /* 1                                               */
  uint32_t kind;       /* TRACE_GUIDE_FULL or TRACE_GUIDE_COMPACT          */
  int32_t n_seg;
  int64_t rows, cols;
  uint64_t guide_offset, bs_offset, gs_offset, seg_offset; /* from the start */
} trace_record_header_t;

/* Bytes of a record for this shape (0 for bad arguments). */
TRACE_API size_t trace_record_size(trace_guide_kind_t kind, int64_t rows, int64_t cols,
                                   int32_t n_seg);

/* Writes the header and the row offsets into host_dst at once and enqueues
 * device -> host copies of the guide, block scales and global scales on
 * `stream` (pinned host memory makes them asynchronous).  host_dst must hold
 * trace_record_size(...) bytes and stay valid until the stream passes the
 * copies.  seg.row_offsets == NULL means one segment. */
TRACE_API trace_status_t trace_record_export(trace_handle_t h, trace_guide_kind_t kind,
                                             const void* guide, const void* bs,
                                             const float* gs, int64_t rows, int64_t cols,
                                             trace_segments_t seg, void* host_dst,
                                             size_t dst_bytes, trace_stream_t stream);

/* Validates a record's header (magic, version, kind, sizes against
 * src_bytes) and copies it out; returns TRACE_ERR_INVALID_ARG for a damaged
 * or truncated record.  The row offsets are at host_src + header.seg_offset. */
TRACE_API trace_status_t trace_record_info(const void* host_src, size_t src_bytes,
                                           trace_record_header_t* out);

/* Enqueues host -> device copies of a validated record's guide, block scales
 * and global scales into caller-owned device buffers of the record's shape. */
TRACE_API trace_status_t trace_record_import(trace_handle_t h, const void* host_src,
                                             size_t src_bytes, void* guide, void* bs,
                                             float* gs, trace_stream_t stream);

/* ---- f4: the rollout codes as operands of an NVFP4 tensor-core GEMM -----
 * ([EN] "TRACE Core Concept": rollout runs weights and activations in
 * NVFP4.)  Block-scaled tensor-core GEMMs take E4M3 block scales in NVIDIA's
 * tile layout (cuBLAS documentation, "1D block scaling factors layout"):
 * 512-byte tiles of 128 rows x 4 scale columns (64 elements), tiles running
 * along the scale columns, the scale of (r, c) inside a tile at byte
 * 16 * (r mod 32) + 4 * (r div 32) + c, rows padded to a multiple of 128
 * and scale columns to a multiple of 4 with zeros. */

/* Bytes of that layout for an operand [rows, cols] (0 for a bad shape). */
TRACE_API size_t trace_block_scales_mma_bytes(int64_t rows, int64_t cols);

/* Rearranges row-major block scales bs_e4m3 [rows, cols/16] (as written by
 * trace_rollout_quant) into the tile layout at out (16-byte aligned,
 * trace_block_scales_mma_bytes(rows, cols) bytes, padding written as 0). */
TRACE_API trace_status_t trace_block_scales_mma(trace_handle_t h, const void* bs_e4m3,
                                                int64_t rows, int64_t cols, void* out,
                                                trace_stream_t stream);

/* trace_rollout_quant that also (or only) writes the block scales in the
 * tile layout: bs_e4m3 [rows, cols/16] row-major and bs_mma
 * (trace_block_scales_mma_bytes(rows, cols) bytes, 16-byte aligned) may
 * each be NULL, not both.  The scales are written from the quantiser's
 * registers, so the layout costs no extra pass. */
TRACE_API trace_status_t trace_rollout_quant_mma(trace_handle_t h, const void* x_bf16,
                                                 int64_t rows, int64_t cols,
                                                 trace_segments_t seg, void* codes_u8,
                                                 void* bs_e4m3, void* bs_mma, float* gs_f32,
                                                 uint32_t* guide_bits, trace_stream_t stream);

/* Rollout-side quantisation with delayed scaling: the same codes, block
 * scales and compact words as trace_rollout_quant, but each segment's global
 * scale comes from a given maximum, gs = amax_prev[s] / 2688 (binary32, the
 * division trace_rollout_quant applies to the segment's own maximum), so x is
 * read once, by one kernel, with no pass over the segment first.  The pages
 * define gs from the segment's own maximum ([EN] "TRACE Core Concept");
 * taking it from an earlier step, such as the same activations one rollout
 * step before, is a deployment option of this library: elements whose
 * magnitude exceeds amax_prev saturate (block scale 448, code magnitude 6),
 * exactly as the oracle with that maximum given.
 *   amax_prev  [n_seg] device, the maxima to scale by (a maximum that is not
 *              positive gives gs = 0: the segment quantises to zero)
 *   gs_f32     [n_seg] out (device), the global scales used
 *   amax_out   [n_seg] out (device, may be NULL): this tensor's segment
 *              maxima, bit-exact with trace_segment_amax, for the next call
 * Other arguments, layouts and errors as trace_rollout_quant.  amax_prev and
 * amax_out must not overlap. */
TRACE_API trace_status_t trace_rollout_quant_delayed(trace_handle_t h, const void* x_bf16,
                                                     int64_t rows, int64_t cols,
                                                     trace_segments_t seg,
                                                     const float* amax_prev, void* codes_u8,
                                                     void* bs_e4m3, float* gs_f32,
                                                     uint32_t* guide_bits, float* amax_out,
                                                     trace_stream_t stream);

typedef enum { TRACE_OUT_F32 = 0, TRACE_OUT_BF16 = 1 } trace_out_t;

/* NVFP4 GEMM over rollout codes: d [m, n] (row-major) =
 *   fl32(a_gs[0] * b_gs[0]) * sum_k A[i, k] * B[j, k],
 * A [m, k] and B [n, k] given as codes ([rows, k/2], element 2i in the low
 * nibble) and block scales in the tile layout, a_gs / b_gs device pointers
 * to one global scale each (a single segment per operand).  Block-scaled
 * E2M1 products with FP32 accumulation on the tensor cores, in the form
 * TRACE_OPT_GEMM selects: the library's own tcgen05 kernel (default; no
 * allocation, a wait inside it that runs out is reported by
 * trace_device_status) or cuBLASLt (loaded at the first such call; the
 * handle then keeps its cuBLASLt handle and a 32 MiB workspace).  k must be
 * a multiple of 32; d, the codes and the tile-layout scales 16-byte
 * aligned.  The cuBLASLt form returns TRACE_ERR_LIBRARY if cuBLASLt is
 * missing or refuses the shape. */
TRACE_API trace_status_t trace_nvfp4_gemm(trace_handle_t h, const void* a_codes,
                                          const void* a_scales_mma, const float* a_gs,
                                          const void* b_codes, const void* b_scales_mma,
                                          const float* b_gs, int64_t m, int64_t n, int64_t k,
                                          void* d, trace_out_t d_type, trace_stream_t stream);

/* Rollout-side quantisation without a handle and without any device
 * allocation.  The paper has no counterpart: this is a deployment variant of
 * trace_rollout_quant with the same arguments, layouts and results (bit for
 * bit).  It always runs the two-kernel path (amax pass, then quantiser), so
 * x is read twice; the handle's fused kernel reads it once.
 *
 * It is for callers that must not call cudaMalloc (code running inside a
 * device allocator or memory pool, runtimes that pre-reserve all device
 * memory for their own arena, allocation-free real-time loops); such callers
 * cannot create a handle either, since trace_create allocates scratch.  The
 * scratch this call needs (per-segment maxima and a completion ticket) is a
 * fixed array in the library's device image, held by every GPU that loads
 * the library until the process exits, sized for at most
 * TRACE_NOALLOC_MAX_SEGMENTS segments; more segments return
 * TRACE_ERR_INVALID_ARG before anything is enqueued.
 *
 * It works on the current device.  Its first call on a device resolves the
 * array's device address (cudaGetSymbolAddress) and caches it with the
 * identity of the current CUDA context, so make that first call before any
 * stream capture; a call made under another context (after cudaDeviceReset,
 * or with a different context current) resolves the address again.  rows ==
 * 0 writes n_seg zero global scales and launches no kernel.  Every call
 * clears the part of the array it uses on `stream`; all calls on one device
 * share the array, so calls that overlap on the GPU (e.g. on two streams at
 * once) race. */
#define TRACE_NOALLOC_MAX_SEGMENTS 1024
TRACE_API trace_status_t trace_rollout_quant_noalloc(const void* x_bf16, int64_t rows,
                                                     int64_t cols, trace_segments_t seg,
                                                     void* codes_u8, void* bs_e4m3,
                                                     float* gs_f32, uint32_t* guide_bits,
                                                     trace_stream_t stream);

/* Bounds checking of debug builds.  A library compiled with
 * -DTRACE_DEBUG_BOUNDS registers, before every launch of a call, the byte
 * ranges of the call's buffers and of the handle's scratch (stream-ordered),
 * and its hot-path kernels check every global access against them: an access
 * outside them is counted and skipped (never a trap).  This call waits for
 * the device (cudaDeviceSynchronize), sets *checked to 1 and *violations to
 * the accesses counted since the previous call, and clears the count.  In
 * other builds it sets *checked = 0, *violations = 0.  No counterpart in the
 * paper: it stands in for a device-side memory checker. */
TRACE_API trace_status_t trace_debug_bounds(trace_handle_t h, int* checked, uint64_t* violations);

/* Built-in profiler.  While enabled, every kernel launch through the handle
 * is bracketed by CUDA events on its own stream.  trace_profile_collect
 * waits for the recorded events, writes per-kernel launch counts and summed
 * milliseconds into out[TRACE_KERNEL_COUNT] and clears the record.  At most
 * 4096 launches are kept between collects; later ones are not timed. */
TRACE_API trace_status_t trace_profile_enable(trace_handle_t h, int enable);
TRACE_API trace_status_t trace_profile_collect(trace_handle_t h, trace_kernel_time_t* out);

#ifdef __cplusplus
}
#endif

#endif /* TRACE_FP4_H */
