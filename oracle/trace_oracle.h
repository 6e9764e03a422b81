/*
 * trace_oracle.h - the CPU oracle for the guided-NVFP4 hot path of TRACE.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded C
 * restatement of what the rollout-side NVFP4 quantiser and the training-side
 * rollout-guided fake quantiser compute.  Only the test suite, the smoke check
 * and the CPU-baseline leg of the benchmark may load it.  It shares no code,
 * header, table or constant with the CUDA library, and the CUDA library never
 * calls it.
 *
 * Sources (cited by page title and section):
 *   [EN] "Alibaba Qwen Proposes TRACE for 5.4x Faster FP4 RL Rollouts"
 *        (todayforai.com): section "Why Does FP4 Rollout 'Break' RL Training?"
 *        (worked example after Fig. 1), section "TRACE Core Concept"
 *        (guided rounding after its first heading; compact record after Fig. 3).
 *   [ZH] the same article in Chinese (yktworld.com), same sections.
 *   Number formats: OCP Microscaling Formats (MX) v1.0, sections on FP4 E2M1
 *   and FP8 E4M3; IEEE 754 binary32 round-to-nearest-even; bfloat16 as the
 *   upper half of binary32.  The NVFP4 two-level scale (FP32 tensor scale,
 *   E4M3 scale per 16 elements) is NVIDIA's published NVFP4 convention.
 *
 * Layouts (all row-major, cols % 32 == 0, a "block" is 16 consecutive
 * elements of a row):
 *   x        uint16 [rows, cols]      bfloat16 bit patterns
 *   codes    uint8  [rows, cols/2]    element 2i in the low nibble of byte i,
 *                                     nibble = (sign << 3) | m, m in 0..7
 *   bs       uint8  [rows, cols/16]   E4M3 block scale codes
 *   gs       float  [n_seg]           FP32 global scale per segment
 *   guide    uint32 [rows, cols/16]   bit j = sign of element j of the block,
 *                                     bit 16+j = m & 1 of element j
 *   y        uint16 [rows, cols]      bfloat16 dequantised output
 *   mask     uint32 [rows, cols/32]   bit j of word w = element 32w+j kept
 *                                     by the straight-through estimator
 *   segments int64 [n_seg+1]          row offsets, [0] = 0, [n_seg] = rows,
 *                                     non-decreasing; NULL means one segment
 *
 * Every function returns 0 on success and a negative value on a bad argument.
 */
#ifndef TRACE_ORACLE_H
#define TRACE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* guide kinds for orc_train_fakequant */
#define ORC_GUIDE_NONE 0
#define ORC_GUIDE_FULL 1     /* guide = rollout codes, uint8 [rows, cols/2]   */
#define ORC_GUIDE_COMPACT 2  /* guide = sign/LSB words, uint32 [rows, cols/16] */

/* statistics layout (uint64 [11]) */
#define ORC_STAT_N 0
#define ORC_STAT_MISMATCH_RTN 1
#define ORC_STAT_MISMATCH_GUIDED 2
#define ORC_STAT_HIST_RTN 3      /* 4 buckets: |dk| = 0, 1, 2, >=3 */
#define ORC_STAT_HIST_GUIDED 7   /* 4 buckets */
#define ORC_STAT_COUNT 11

/* ---- number formats ---------------------------------------------------- */
float orc_bf16_to_f32(uint16_t h);
uint16_t orc_f32_to_bf16(float f);
uint8_t orc_e4m3_encode(float v);
float orc_e4m3_decode(uint8_t c);
float orc_e2m1_value(int m);                 /* magnitude of index m, 0..7 */
int orc_e2m1_rtn(float t);                   /* t >= 0 -> nearest index     */
void orc_e2m1_bracket(float t, int* lo, int* hi);

/* ---- scalar pieces of the method --------------------------------------- */
float orc_global_scale(float amax);
uint8_t orc_block_scale(float bamax, float gs);
void orc_scale_pair(uint8_t bs, float gs, float* S, float* inv);
int orc_unpack_index(float t_ref, int lsb);
int orc_guided_index(float x, float S_t, float inv_t, int have_guide,
                     int nib_r, float S_r);

/* array forms of the scalar pieces, for exhaustive sweeps */
void orc_e2m1_rtn_array(const float* t, int64_t n, uint8_t* m_out);
void orc_e2m1_bracket_array(const float* t, int64_t n, uint8_t* lo, uint8_t* hi);
void orc_e4m3_encode_array(const float* v, int64_t n, uint8_t* out);
void orc_f32_to_bf16_array(const float* v, int64_t n, uint16_t* out);

/* ---- the hot path -------------------------------------------------------- */
int orc_segment_amax(const uint16_t* x, int64_t rows, int64_t cols,
                     const int64_t* seg, int32_t n_seg, float* amax);

int orc_rollout_quant(const uint16_t* x, int64_t rows, int64_t cols,
                      const int64_t* seg, int32_t n_seg, uint8_t* codes,
                      uint8_t* bs, float* gs, uint32_t* guide);

/* Same as orc_rollout_quant, but the per-segment maxima come from amax_in
 * [n_seg] instead of the rows themselves.  This lets a test check a sample
 * of rows of a large segment whose maximum was taken separately. */
int orc_rollout_quant_given(const uint16_t* x, int64_t rows, int64_t cols,
                            const int64_t* seg, int32_t n_seg, const float* amax_in,
                            uint8_t* codes, uint8_t* bs, float* gs, uint32_t* guide);

int orc_guide_pack(const uint8_t* codes, int64_t rows, int64_t cols,
                   uint32_t* guide);

int orc_guide_unpack(const uint16_t* x_ref, const uint32_t* guide,
                     const uint8_t* bs_r, const float* gs_r,
                     const int64_t* seg_r, int32_t n_seg_r, int64_t rows,
                     int64_t cols, uint8_t* codes);

int orc_train_fakequant(const uint16_t* x, int64_t rows, int64_t cols,
                        const int64_t* seg_t, int32_t n_seg_t, int kind,
                        const void* guide, const uint8_t* bs_r,
                        const float* gs_r, const int64_t* seg_r,
                        int32_t n_seg_r, uint16_t* y, uint32_t* mask,
                        uint8_t* codes_t, uint64_t* stats);

/* Straight-through backward of the fake quantiser: the incoming gradient
 * passes where the element's mask bit is 1 and becomes +0 where it is 0.
 *   g, out  uint16 [rows, cols] bf16 patterns;  mask uint32 [rows, cols/32] */
int orc_ste_backward(const uint16_t* g, const uint32_t* mask, int64_t rows, int64_t cols,
                     uint16_t* out);

/* Same as orc_train_fakequant with the training maxima taken from
 * amax_t_in [n_seg_t] (see orc_rollout_quant_given). */
int orc_train_fakequant_given(const uint16_t* x, int64_t rows, int64_t cols,
                              const int64_t* seg_t, int32_t n_seg_t,
                              const float* amax_t_in, int kind, const void* guide,
                              const uint8_t* bs_r, const float* gs_r,
                              const int64_t* seg_r, int32_t n_seg_r, uint16_t* y,
                              uint32_t* mask, uint8_t* codes_t, uint64_t* stats);

/* ---- block scales for tensor cores, and the NVFP4 GEMM that uses them ----
 *
 * Block-scaled tensor-core GEMMs (cuBLASLt scale mode VEC16_UE4M3; NVIDIA's
 * cuBLAS documentation, "1D block scaling factors layout") take the E4M3
 * block scales of an operand [rows, cols] in tiles of 128 rows x 4 scale
 * columns (64 elements of the inner dimension), 512 bytes per tile, tiles
 * ordered along the scale columns first.  Inside a tile the scale of
 * (row r, scale column c) is byte 16 * (r mod 32) + 4 * (r div 32) + c.
 * Rows are padded to a multiple of 128 and scale columns to a multiple of 4
 * with zero bytes. */
int64_t orc_mma_scales_bytes(int64_t rows, int64_t cols);
int orc_mma_scales(const uint8_t* bs, int64_t rows, int64_t cols, uint8_t* out);

/* The NVFP4 GEMM a rollout engine runs on these operands ([EN] "TRACE Core
 * Concept": rollout runs weights and activations in FP4):
 *   d [m, n] = fl32(a_gs * b_gs) * sum_k A[i, k] * B[j, k]
 * with A [m, k] and B [n, k] given as codes + row-major block scales (one
 * global scale each), element value = E2M1(code) * E4M3(bs) and the sum taken
 * in double (each product has at most 14 significant bits). */
int orc_nvfp4_gemm(const uint8_t* a_codes, const uint8_t* a_bs, float a_gs,
                   const uint8_t* b_codes, const uint8_t* b_bs, float b_gs,
                   int64_t m, int64_t n, int64_t k, double* d);

#ifdef __cplusplus
}
#endif

#endif /* TRACE_ORACLE_H */
