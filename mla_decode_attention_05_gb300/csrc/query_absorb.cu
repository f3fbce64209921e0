// Query absorption: the 576-value query rows the decode kernel reads, from
// the query part of the fused projection output (vLLM kimi_k3
// specialized-decode "mla.query" page, MlaQuery.kernel / MlaQuery.tiled):
//   xq   = RMSNorm(q_a) x w_qa, rounded to bf16            (1536 values)
//   qb_h = bf16(W_QB[h] . xq)                               (192 rows per head:
//                                                            128 no-PE, 64 RoPE)
//   q_h  = [ bf16(qb_h[0:128] . W_UK[h]) | qb_h[128:192] ]  (512 latent + 64)
// The RMSNorm is this library's own kernel with the same exact arithmetic as
// the KV insert (sum of squares exact, then IEEE fp32 steps):
//   S = sum x_i^2 (exact, rounded once to fp32), mean = fp32(fp32(S / 1536)
//   + eps), r = fp32(1 / fp32(sqrt(mean))) (0 if mean == 0),
//   xq_i = bf16(fp32(fp32(x_i * w_i) * r)).
// The two contractions are plain bf16 GEMMs with fp32 accumulation (one
// GEMM for Q_B, one strided-batched GEMM over heads for W_UK), run by cuBLAS,
// which this file loads at the first call (dlopen) so that the rest of the
// library does not depend on it; the RoPE rows are copied by a small kernel.
#include <cublas_v2.h>
#include <dlfcn.h>

#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "exact_sum.cuh"

namespace mla {
namespace {

constexpr int D_QA = 1536;
constexpr int QB_ROWS = 192;
constexpr int D_NOPE = 128;
constexpr int kWarps = 8;
constexpr int kChunks = D_QA / 8 / 32;  // 16-byte chunks per lane: 6

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// One warp per token.  Lane l holds 16-byte chunks l, l + 32, ..., l + 160 of
// the row, so every warp-wide load and store covers 512 contiguous bytes.
__global__ void __launch_bounds__(kWarps * 32)
    qa_norm_kernel(const __nv_bfloat16 *q_a, int ld_qa, const __nv_bfloat16 *w_qa, float eps, int N,
                   __nv_bfloat16 *xq) {
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (j >= N) return;
  const uint4 *xr = reinterpret_cast<const uint4 *>(q_a + (size_t)j * ld_qa);
  const uint4 *wr = reinterpret_cast<const uint4 *>(w_qa);
  LaneBf16<4 * kChunks> x;
  uint4 w4[kChunks];
#pragma unroll
  for (int c = 0; c < kChunks; c++) {
    const uint4 v = __ldg(xr + 32 * c + lane);
    x.w[4 * c] = v.x;
    x.w[4 * c + 1] = v.y;
    x.w[4 * c + 2] = v.z;
    x.w[4 * c + 3] = v.w;
    w4[c] = __ldg(wr + 32 * c + lane);
  }
  const float S = sum_sq_rn<4 * kChunks>(x);
  const float mean = __fadd_rn(__fdiv_rn(S, (float)D_QA), eps);
  const float r = mean > 0.f ? __fdiv_rn(1.f, __fsqrt_rn(mean)) : 0.f;
  uint4 *dst = reinterpret_cast<uint4 *>(xq + (size_t)j * D_QA);
#pragma unroll
  for (int c = 0; c < kChunks; c++) {
    const uint32_t ww[4] = {w4[c].x, w4[c].y, w4[c].z, w4[c].w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const uint32_t xv = x.w[4 * c + k];
      const float x0 = __uint_as_float(xv << 16), x1 = __uint_as_float(xv & 0xFFFF0000u);
      const float w0 = __uint_as_float(ww[k] << 16), w1 = __uint_as_float(ww[k] & 0xFFFF0000u);
      __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(__fmul_rn(x0, w0), r), __fmul_rn(__fmul_rn(x1, w1), r));
      o[k] = *reinterpret_cast<uint32_t *>(&b2);
    }
    dst[32 * c + lane] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// q[n][h][512 + i] = qb[n][h * 192 + 128 + i], i < 64: one thread per 16 bytes.
__global__ void rope_copy_kernel(const __nv_bfloat16 *qb, __nv_bfloat16 *q, int NH) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= NH * 8) return;
  const int row = i >> 3, c = i & 7;
  const uint4 v = *reinterpret_cast<const uint4 *>(qb + (size_t)row * QB_ROWS + D_NOPE + 8 * c);
  *reinterpret_cast<uint4 *>(q + (size_t)row * D_QK + D_V + 8 * c) = v;
}

// cuBLAS, loaded at first use (the C entry points, by name).
using GemmExFn = cublasStatus_t (*)(cublasHandle_t, cublasOperation_t, cublasOperation_t, int, int, int, const void *,
                                    const void *, cudaDataType, int, const void *, cudaDataType, int, const void *,
                                    void *, cudaDataType, int, cublasComputeType_t, cublasGemmAlgo_t);
using GemmSbFn = cublasStatus_t (*)(cublasHandle_t, cublasOperation_t, cublasOperation_t, int, int, int, const void *,
                                    const void *, cudaDataType, int, long long, const void *, cudaDataType, int,
                                    long long, const void *, void *, cudaDataType, int, long long, int,
                                    cublasComputeType_t, cublasGemmAlgo_t);
struct Cublas {
  cublasStatus_t (*create)(cublasHandle_t *) = nullptr;
  cublasStatus_t (*set_stream)(cublasHandle_t, cudaStream_t) = nullptr;
  GemmExFn gemm = nullptr;
  GemmSbFn gemm_sb = nullptr;
  bool ok = false;
};

std::mutex g_mu;

const Cublas *cublas() {
  static Cublas cb;
  static bool tried = false;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!tried) {
    tried = true;
    void *h = dlopen("libcublas.so.13", RTLD_NOW | RTLD_GLOBAL);
    if (!h) h = dlopen("libcublas.so", RTLD_NOW | RTLD_GLOBAL);
    if (h) {
      cb.create = reinterpret_cast<decltype(cb.create)>(dlsym(h, "cublasCreate_v2"));
      cb.set_stream = reinterpret_cast<decltype(cb.set_stream)>(dlsym(h, "cublasSetStream_v2"));
      cb.gemm = reinterpret_cast<decltype(cb.gemm)>(dlsym(h, "cublasGemmEx"));
      cb.gemm_sb = reinterpret_cast<decltype(cb.gemm_sb)>(dlsym(h, "cublasGemmStridedBatchedEx"));
      cb.ok = cb.create && cb.set_stream && cb.gemm && cb.gemm_sb;
    }
  }
  return cb.ok ? &cb : nullptr;
}

// One handle per thread and device, created on first use and kept for the
// life of the thread.
constexpr int kMaxDevices = 64;
thread_local cublasHandle_t t_handle[kMaxDevices] = {};

int fail(int code, const char *msg) {
  set_last_error(msg);
  return code;
}

}  // namespace
}  // namespace mla

size_t mla_query_absorb_workspace_bytes(int N, int H) {
  if (N < 0 || H < 1 || H > MLA_MAX_HEADS) return 0;
  return mla::round256((size_t)N * mla::D_QA * 2) + mla::round256((size_t)N * H * mla::QB_ROWS * 2) + 256;
}

int mla_query_absorb(const void *q_a, int ld_qa, const void *w_qa, float eps, const void *w_qb, const void *w_uk,
                     int N, int H, void *q, void *workspace, size_t workspace_bytes, mla_stream_t stream) {
  using namespace mla;
  if (N < 0) return fail(MLA_ERR_INVALID_ARG, "N must be >= 0");
  if (H < 1 || H > MLA_MAX_HEADS) return fail(MLA_ERR_INVALID_ARG, "H must be in [1, 128]");
  if (ld_qa < D_QA || ld_qa % 8) return fail(MLA_ERR_INVALID_ARG, "ld_qa must be >= 1536 and a multiple of 8");
  if (!(eps >= 0.f) || eps > 3.0e38f) return fail(MLA_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (N == 0) {
    set_last_error("");
    return MLA_OK;
  }
  if (!q_a || !w_qa || !w_qb || !w_uk || !q || !workspace) return fail(MLA_ERR_INVALID_ARG, "null pointer");
  auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!a16(q_a) || !a16(w_qa) || !a16(w_qb) || !a16(w_uk) || !a16(q) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(MLA_ERR_INVALID_ARG, "q_a, w_qa, w_qb, w_uk, q must be 16-byte aligned, workspace 256-byte aligned");
  if (workspace_bytes < mla_query_absorb_workspace_bytes(N, H))
    return fail(MLA_ERR_WORKSPACE, "workspace smaller than mla_query_absorb_workspace_bytes(N, H)");
  const Cublas *cb = cublas();
  if (!cb) return fail(MLA_ERR_UNSUPPORTED, "cuBLAS (libcublas.so.13) could not be loaded");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(MLA_ERR_CUDA, "cudaGetDevice failed");
  cublasHandle_t &hd = t_handle[dev];
  if (!hd && cb->create(&hd) != CUBLAS_STATUS_SUCCESS) {
    hd = nullptr;
    return fail(MLA_ERR_CUDA, "cublasCreate failed");
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (cb->set_stream(hd, s) != CUBLAS_STATUS_SUCCESS) return fail(MLA_ERR_CUDA, "cublasSetStream failed");

  __nv_bfloat16 *xq = static_cast<__nv_bfloat16 *>(workspace);
  __nv_bfloat16 *qb = reinterpret_cast<__nv_bfloat16 *>(static_cast<uint8_t *>(workspace) +
                                                         round256((size_t)N * D_QA * 2));
  __nv_bfloat16 *qo = static_cast<__nv_bfloat16 *>(q);
  qa_norm_kernel<<<(N + kWarps - 1) / kWarps, kWarps * 32, 0, s>>>(
      static_cast<const __nv_bfloat16 *>(q_a), ld_qa, static_cast<const __nv_bfloat16 *>(w_qa), eps, N, xq);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, cudaGetErrorString(e));
  const float one = 1.f, zero = 0.f;
  // Q_B: qb[n][h*192 + p] = sum_k W_QB[h*192 + p][k] xq[n][k]; column-major
  // view: qb^T (H*192 x N) = W_QB^T^T (op T of the 1536 x H*192 matrix) * xq^T
  if (cb->gemm(hd, CUBLAS_OP_T, CUBLAS_OP_N, H * QB_ROWS, N, D_QA, &one, w_qb, CUDA_R_16BF, D_QA, xq, CUDA_R_16BF,
               D_QA, &zero, qb, CUDA_R_16BF, H * QB_ROWS, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) !=
      CUBLAS_STATUS_SUCCESS)
    return fail(MLA_ERR_CUDA, "cublasGemmEx (Q_B) failed");
  // W_UK per head: q[n][h][l] = sum_p qb[n][h*192 + p] W_UK[h][p][l], p < 128;
  // column-major per head: (512 x N, ld H*576) = W_UK[h] (512 x 128, ld 512)
  // * qb_nope (128 x N, ld H*192)
  if (cb->gemm_sb(hd, CUBLAS_OP_N, CUBLAS_OP_N, D_V, N, D_NOPE, &one, w_uk, CUDA_R_16BF, D_V,
                  (long long)D_NOPE * D_V, qb, CUDA_R_16BF, H * QB_ROWS, QB_ROWS, &zero, qo, CUDA_R_16BF, H * D_QK,
                  D_QK, H, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
    return fail(MLA_ERR_CUDA, "cublasGemmStridedBatchedEx (W_UK) failed");
  const int nh = N * H;
  rope_copy_kernel<<<(nh * 8 + 255) / 256, 256, 0, s>>>(qb, qo, nh);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, cudaGetErrorString(e));
  set_last_error("");
  return MLA_OK;
}
