// trace_gemm.cu - the consumer side of the rollout codes: block scales in
// the tensor-core tile layout, and the NVFP4 GEMM that takes codes + scales
// as they come out of the rollout quantiser.
//
// Source: "Alibaba Qwen Proposes TRACE for 5.4x Faster FP4 RL Rollouts",
// sections on FP4 rollout (weights and activations in NVFP4 during
// rollout); the scale tile layout is NVIDIA's documented interface of
// block-scaled tensor-core GEMMs (cuBLAS, "1D block scaling factors
// layout"): 512-byte tiles of 128 rows x 4 scale columns, tiles running along
// the scale columns, (r, c) inside a tile at 16 (r mod 32) + 4 (r div 32) + c,
// zero padding.
//
// The contraction itself is a plain library GEMM (cuBLASLt, block-scaled
// E2M1 x E2M1 with UE4M3 scales, FP32 accumulation), loaded with dlopen at
// the first call so that the library loads where cuBLASLt is absent.
#include <cublasLt.h>
#include <cuda_runtime.h>
#include <dlfcn.h>
#include <stdint.h>

#include <mutex>
#include <type_traits>

#include "trace_internal.h"

namespace tfp4 {
namespace {

// One thread per 16-byte line of the tiled layout: line L of tile T holds
// rows 32 j + (L mod 32), j = 0..3, scale columns 4 (T mod tiles) + c.
__global__ void __launch_bounds__(256)
    k_mma_scales(const uint8_t* __restrict__ bs, int32_t rows, int32_t sc, int32_t tiles_per_row,
                 uint32_t lines, uint8_t* __restrict__ out) {
  for (uint32_t L = blockIdx.x * blockDim.x + threadIdx.x; L < lines;
       L += gridDim.x * blockDim.x) {
    const uint32_t tile = L >> 5, i = L & 31u;
    const int32_t r0 = (int32_t)(tile / tiles_per_row) * 128 + (int32_t)i;
    const int32_t c0 = (int32_t)(tile % tiles_per_row) * 4;
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int32_t r = r0 + 32 * j;
      uint32_t v = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int32_t col = c0 + c;
        if (r < rows && col < sc) v |= (uint32_t)bs[(int64_t)r * sc + col] << (8 * c);
      }
      w[j] = v;
    }
    *reinterpret_cast<uint4*>(out + (uint64_t)L * 16u) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// alpha = fl32(gs_a * gs_b), beta = 0 for the GEMM (device pointer mode).
__global__ void k_gemm_scalars(const float* gs_a, const float* gs_b, float* out) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    out[0] = __fmul_rn(gs_a[0], gs_b[0]);
    out[1] = 0.0f;
  }
}

// ---- cuBLASLt, resolved at first use ---------------------------------------

struct LtApi {
  decltype(&cublasLtCreate) create = nullptr;
  decltype(&cublasLtDestroy) destroy = nullptr;
  decltype(&cublasLtMatmulDescCreate) desc_create = nullptr;
  decltype(&cublasLtMatmulDescDestroy) desc_destroy = nullptr;
  decltype(&cublasLtMatmulDescSetAttribute) desc_set = nullptr;
  decltype(&cublasLtMatrixLayoutCreate) layout_create = nullptr;
  decltype(&cublasLtMatrixLayoutDestroy) layout_destroy = nullptr;
  decltype(&cublasLtMatmulPreferenceCreate) pref_create = nullptr;
  decltype(&cublasLtMatmulPreferenceDestroy) pref_destroy = nullptr;
  decltype(&cublasLtMatmulPreferenceSetAttribute) pref_set = nullptr;
  decltype(&cublasLtMatmulAlgoGetHeuristic) heuristic = nullptr;
  decltype(&cublasLtMatmul) matmul = nullptr;
  bool ok = false;
};

const LtApi& lt_api() {
  static LtApi api;
  static std::once_flag once;
  std::call_once(once, [] {
    void* so = dlopen("libcublasLt.so.13", RTLD_NOW | RTLD_LOCAL);
#ifdef TRACE_CUDA_LIB_DIR
    if (!so) so = dlopen(TRACE_CUDA_LIB_DIR "/libcublasLt.so.13", RTLD_NOW | RTLD_LOCAL);
#endif
    if (!so) return;
    auto get = [so](auto& fn, const char* name) {
      fn = reinterpret_cast<std::remove_reference_t<decltype(fn)>>(dlsym(so, name));
      return fn != nullptr;
    };
    api.ok = get(api.create, "cublasLtCreate") && get(api.destroy, "cublasLtDestroy") &&
             get(api.desc_create, "cublasLtMatmulDescCreate") &&
             get(api.desc_destroy, "cublasLtMatmulDescDestroy") &&
             get(api.desc_set, "cublasLtMatmulDescSetAttribute") &&
             get(api.layout_create, "cublasLtMatrixLayoutCreate") &&
             get(api.layout_destroy, "cublasLtMatrixLayoutDestroy") &&
             get(api.pref_create, "cublasLtMatmulPreferenceCreate") &&
             get(api.pref_destroy, "cublasLtMatmulPreferenceDestroy") &&
             get(api.pref_set, "cublasLtMatmulPreferenceSetAttribute") &&
             get(api.heuristic, "cublasLtMatmulAlgoGetHeuristic") &&
             get(api.matmul, "cublasLtMatmul");
  });
  return api;
}

}  // namespace

int64_t mma_scales_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols <= 0 || cols % 32) return -1;
  return (rows + 127) / 128 * 128 * ((cols / 16 + 3) / 4 * 4);
}

cudaError_t launch_mma_scales(const void* bs, int64_t rows, int64_t cols, void* out, int sm_count,
                              cudaStream_t st) {
  const int64_t bytes = mma_scales_bytes(rows, cols);
  const int32_t sc = (int32_t)(cols / 16);
  const int32_t tiles_per_row = (sc + 3) / 4;
  const uint32_t lines = (uint32_t)(bytes / 16);
  if (lines == 0) return cudaSuccess;
  int64_t grid = (lines + 255) / 256;
  if (grid > 8LL * sm_count) grid = 8LL * sm_count;
  k_mma_scales<<<(unsigned)grid, 256, 0, st>>>((const uint8_t*)bs, (int32_t)rows, sc,
                                               tiles_per_row, lines, (uint8_t*)out);
  return cudaGetLastError();
}

bool lt_available() { return lt_api().ok; }

void lt_destroy(void* lt) {
  if (lt && lt_api().ok) lt_api().destroy((cublasLtHandle_t)lt);
}

// d [m, n] (row-major, fp32 or bf16) = alpha * sum_k a[i, k] b[j, k].  In
// cuBLASLt's column-major terms: D (n x m) = op_T(W) op_N(X) with W = b
// stored as k x n and X = a stored as k x m, both with leading dimension k.
int lt_nvfp4_gemm(void** lt, void* workspace, size_t ws_bytes, const void* a_codes,
                  const void* a_scales, const void* b_codes, const void* b_scales,
                  const float* alpha_beta, int64_t m, int64_t n, int64_t k, void* d, int d_bf16,
                  cudaStream_t st) {
  const LtApi& api = lt_api();
  if (!api.ok) return -1;
  if (!*lt) {
    cublasLtHandle_t h = nullptr;
    if (api.create(&h) != CUBLAS_STATUS_SUCCESS) return -2;
    *lt = h;
  }
  cublasLtHandle_t h = (cublasLtHandle_t)*lt;
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, ld = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  int rc = 0;
  cublasStatus_t s = api.desc_create(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F);
  const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
  const int32_t mode = CUBLASLT_MATMUL_MATRIX_SCALE_VEC16_UE4M3;
  const cublasLtPointerMode_t pm = CUBLASLT_POINTER_MODE_DEVICE;
  const void* sa = b_scales;  // cuBLASLt's A is our b (weights-side operand)
  const void* sb = a_scales;
  if (s == CUBLAS_STATUS_SUCCESS) s = api.desc_set(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof(ta));
  if (s == CUBLAS_STATUS_SUCCESS) s = api.desc_set(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb));
  if (s == CUBLAS_STATUS_SUCCESS)
    s = api.desc_set(op, CUBLASLT_MATMUL_DESC_A_SCALE_MODE, &mode, sizeof(mode));
  if (s == CUBLAS_STATUS_SUCCESS)
    s = api.desc_set(op, CUBLASLT_MATMUL_DESC_B_SCALE_MODE, &mode, sizeof(mode));
  if (s == CUBLAS_STATUS_SUCCESS)
    s = api.desc_set(op, CUBLASLT_MATMUL_DESC_A_SCALE_POINTER, &sa, sizeof(sa));
  if (s == CUBLAS_STATUS_SUCCESS)
    s = api.desc_set(op, CUBLASLT_MATMUL_DESC_B_SCALE_POINTER, &sb, sizeof(sb));
  if (s == CUBLAS_STATUS_SUCCESS)
    s = api.desc_set(op, CUBLASLT_MATMUL_DESC_POINTER_MODE, &pm, sizeof(pm));
  if (s == CUBLAS_STATUS_SUCCESS) s = api.layout_create(&la, CUDA_R_4F_E2M1, k, n, k);
  if (s == CUBLAS_STATUS_SUCCESS) s = api.layout_create(&lb, CUDA_R_4F_E2M1, k, m, k);
  if (s == CUBLAS_STATUS_SUCCESS)
    s = api.layout_create(&ld, d_bf16 ? CUDA_R_16BF : CUDA_R_32F, n, m, n);
  if (s == CUBLAS_STATUS_SUCCESS) s = api.pref_create(&pref);
  if (s == CUBLAS_STATUS_SUCCESS)
    s = api.pref_set(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes, sizeof(ws_bytes));
  cublasLtMatmulHeuristicResult_t heur = {};
  int found = 0;
  if (s == CUBLAS_STATUS_SUCCESS) s = api.heuristic(h, op, la, lb, ld, ld, pref, 1, &heur, &found);
  if (s == CUBLAS_STATUS_SUCCESS && found < 1) s = CUBLAS_STATUS_NOT_SUPPORTED;
  if (s == CUBLAS_STATUS_SUCCESS)
    s = api.matmul(h, op, alpha_beta, b_codes, la, a_codes, lb, alpha_beta + 1, d, ld, d, ld,
                   &heur.algo, workspace, ws_bytes, st);
  if (s != CUBLAS_STATUS_SUCCESS) rc = (int)s;
  if (pref) api.pref_destroy(pref);
  if (ld) api.layout_destroy(ld);
  if (lb) api.layout_destroy(lb);
  if (la) api.layout_destroy(la);
  if (op) api.desc_destroy(op);
  return rc;
}

cudaError_t launch_gemm_scalars(const float* gs_a, const float* gs_b, float* out,
                                cudaStream_t st) {
  k_gemm_scalars<<<1, 32, 0, st>>>(gs_a, gs_b, out);
  return cudaGetLastError();
}

}  // namespace tfp4
