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
// Q_B (qb_kernel) and W_UK with the RoPE-row copy (wuk_kernel) are tcgen05
// GEMMs of this library with fp32 accumulation in tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "exact_sum.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int D_QA = 1536;
constexpr int QB_ROWS = 192;
constexpr int D_NOPE = 128;
constexpr int kWarps = 8;
constexpr int kChunks = D_QA / 8 / 32;  // 16-byte chunks per lane: 6

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

std::mutex g_mu_enc;

// One warp per token.  Lane l holds 16-byte chunks l, l + 32, ..., l + 160 of
// the row, so every warp-wide load and store covers 512 contiguous bytes.
__global__ void __launch_bounds__(kWarps * 32)
    qa_norm_kernel(const __nv_bfloat16 *q_a, int ld_qa, const __nv_bfloat16 *w_qa, float eps, int N,
                   __nv_bfloat16 *xq) {
  grid_dep_trigger();  // the Q_B kernel may start its weight loads meanwhile
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
  const float r = mean > 0.f ? __frcp_rn(__fsqrt_rn(mean)) : 0.f;
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

// ---- Q_B: one CTA per 128 rows of W_QB (and per block of up to 256 tokens)
//
// qb[n][row] = bf16(sum_k W_QB[row][k] * xq[n][k]) is computed transposed,
// D[row][n], so that the weight rows fill the MMA's M = 128 (a decode batch
// has too few tokens to fill M) and the tokens are its N: A = 128 rows of
// W_QB and B = the tokens' xq rows, both K-major, arrive as 128-byte swizzled
// TMA boxes of 64 k-values (A 128 rows = 16 KB, B ntile rows) into a ring of
// stages; D (128 x ntile fp32) sits in TMEM.  The step streams 75.5 MB of
// weights for 128 heads, so it is bound by HBM: two CTAs share each SM and
// every CTA keeps its ring of about 96 KB in flight.  Thread 0 loads, thread
// 32 issues the MMAs (4 per stage), and the four warps read D back (lane =
// weight row), round to bf16 and write it to shared memory as [token][128
// rows], which one TMA store puts into qb (clipped at N and H * 192).
constexpr int kQbThreads = 128;
constexpr uint32_t kQbABytes = 128 * 128;   // 64 k-values x 128 weight rows (bf16)
constexpr uint32_t kQbRingBytes = 98304;    // ring budget per CTA (two CTAs per SM)
constexpr int kQbKSteps = D_QA / 64;        // 24
constexpr uint64_t kQbWaitNs = 2000000000ull;

__host__ __device__ inline uint32_t qb_stage_bytes(int ntile) { return kQbABytes + (uint32_t)ntile * 128; }
__host__ __device__ inline int qb_stages(int ntile) {
  const int st = (int)(kQbRingBytes / qb_stage_bytes(ntile));
  return st > 4 ? 4 : st;
}
__host__ inline uint32_t qb_smem_bytes(int ntile) {
  return (uint32_t)qb_stages(ntile) * qb_stage_bytes(ntile) + 128 + 1024;  // + barriers, alignment slack
}

__global__ void __launch_bounds__(kQbThreads, 2)
    qb_kernel(const __grid_constant__ CUtensorMap w_map, const __grid_constant__ CUtensorMap x_map,
              const __grid_constant__ CUtensorMap o_map, int ntile, unsigned int *status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int stages = qb_stages(ntile);
  const uint32_t stage_bytes = qb_stage_bytes(ntile);
  uint64_t *full = reinterpret_cast<uint64_t *>(base + stages * stage_bytes);
  uint64_t *empty = full + stages;
  uint64_t *done = empty + stages;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * 128, n0 = blockIdx.y * ntile;
  int abort_flag = 0;  // the waits below give up only on their time limit
  __shared__ int gave_up;  // a load or MMA wait of this CTA ran out
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    gave_up = 0;
    for (int s = 0; s < stages; s++) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(done), 1);
    fence_mbar_init_cluster();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t ring = smem_u32(base);
  grid_dep_trigger();  // the W_UK kernel may start its own weight loads
  if (threadIdx.x == 0) {  // loads
    const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_normal();
    // The weights do not depend on the kernel before this one (the q_a
    // RMSNorm): the first stages' weight boxes go out before waiting for it.
    for (int k = 0; k < stages; k++) {
      mbar_arrive_expect_tx(smem_u32(&full[k]), stage_bytes);
      tma_load_2d(ring + k * stage_bytes, &w_map, smem_u32(&full[k]), 64 * k, m0, pol_w);
    }
    grid_dep_wait();
    for (int k = 0; k < kQbKSteps; k++) {
      const int s = k % stages;
      const uint32_t dst = ring + s * stage_bytes;
      if (k >= stages) {
        if (!mbar_wait<false>(smem_u32(&empty[s]), ((k / stages) - 1) & 1, &abort_flag, kQbWaitNs)) {
          atomicOr(status, MLA_STATUS_WAIT_TIMEOUT);
          gave_up = 1;
          break;
        }
        mbar_arrive_expect_tx(smem_u32(&full[s]), stage_bytes);
        tma_load_2d(dst, &w_map, smem_u32(&full[s]), 64 * k, m0, pol_w);
      }
      tma_load_2d(dst + kQbABytes, &x_map, smem_u32(&full[s]), 64 * k, n0, pol_x);
    }
  } else if (threadIdx.x == 32) {  // MMAs
    const uint32_t idesc = idesc_bf16_f32(128, ntile, false, false);
    bool ok = true;
    for (int k = 0; k < kQbKSteps && ok; k++) {
      const int s = k % stages;
      ok = mbar_wait<false>(smem_u32(&full[s]), (k / stages) & 1, &abort_flag, kQbWaitNs);
      if (!ok) break;
      tc_fence_after();
      const uint32_t a = ring + s * stage_bytes, b = a + kQbABytes;
#pragma unroll
      for (int kk = 0; kk < 4; kk++)
        mma_ss(tmem, smem_desc_sw128(a + kk * 32, 16, 1024), smem_desc_sw128(b + kk * 32, 16, 1024), idesc,
               (k | kk) ? 1u : 0u);
      mma_commit(smem_u32(&empty[s]));
    }
    if (ok) {
      mma_commit(smem_u32(done));
    } else {
      atomicOr(status, MLA_STATUS_WAIT_TIMEOUT);
      gave_up = 1;
      mbar_arrive(smem_u32(done));  // release the readers; they see the flag below
    }
  }
  const bool ok = mbar_wait<false>(smem_u32(done), 0, &abort_flag, kQbWaitNs);
  if (!ok && lane == 0) atomicOr(status, MLA_STATUS_WAIT_TIMEOUT);
  tc_fence_after();
  // D (lane = weight row r, column = token) -> bf16 [token][128] in the ring,
  // which every MMA has finished reading
  const int r = warp * 32 + lane;
  for (int c = 0; c < ntile; c += 32) {
    uint32_t v[32];
    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c, v);  // warp-wide
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; j++) {
      if (c + j < ntile) {
        const __nv_bfloat16 hb = __float2bfloat16_rn(__uint_as_float(v[j]));
        *reinterpret_cast<__nv_bfloat16 *>(base + (size_t)(c + j) * 256 + r * 2) = hb;
      }
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  // did every wait of this CTA complete?
  const bool all_ok = __syncthreads_and(ok && *(volatile int *)&gave_up == 0);
  if (threadIdx.x == 0 && all_ok) {
    tma_store_2d(&o_map, ring, m0, n0);
    bulk_store_commit_wait_read();
  }
  if (!all_ok) {  // a wait gave up: let copies or MMAs still in flight land before the CTA exits
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 2000000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ---- W_UK and the RoPE rows: one CTA per (head, 256 latent columns, block
// of 128 tokens) -----------------------------------------------------------
//
// q[n][h][l] = bf16(sum_{p<128} qb[n][h*192 + p] * W_UK[h][p][l]) as one
// tcgen05 GEMM per CTA: M = 128 token rows (rows past N read as zeros), N =
// 256 latent columns, K = 128.  A = the tokens' no-PE rows of qb, K-major;
// B = the CTA's 256 columns of W_UK[h], read MN-major: both arrive as
// 128-byte swizzled TMA boxes of 64 columns x 128 rows (16 KB).  D (128 x
// 256 fp32) takes 256 TMEM columns and two CTAs share an SM, so a decode
// batch (up to 128 tokens, 128 heads) runs in one wave: each CTA's chain of
// load, MMA and store is paid once.  The CTAs of the first column half copy
// the tokens' 64 RoPE values of qb after the latent columns while their
// loads are in flight; four warps then read their 32 rows of D back, round
// to bf16 and store them.
constexpr int kWukThreads = 128;
constexpr uint32_t kBoxBytes = 128 * 128;               // 64 bf16 columns x 128 rows
constexpr uint32_t OFF_W = 0;                           // 4 boxes: latent columns col0 + 64j
constexpr uint32_t OFF_A = 4 * kBoxBytes;               // 2 boxes: no-PE rows 0..63, 64..127
constexpr uint32_t OFF_WBAR = OFF_A + 2 * kBoxBytes;    // full, done, tmem base
constexpr uint32_t kWukSmem = OFF_WBAR + 64 + 1024;     // + slack for the 1024-byte alignment
constexpr uint32_t IDESC_WUK = idesc_bf16_f32(128, 256, false, true);
constexpr uint64_t kWukWaitNs = 2000000000ull;

__global__ void __launch_bounds__(kWukThreads, 1)
    wuk_kernel(const __grid_constant__ CUtensorMap w_map, const __grid_constant__ CUtensorMap a_map,
               const __nv_bfloat16 *qb, __nv_bfloat16 *q, int N, int H, unsigned int *status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *full = reinterpret_cast<uint64_t *>(base + OFF_WBAR);
  uint64_t *done = full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, col0 = blockIdx.y * 256, n0 = blockIdx.z * 128;
  int abort_flag = 0;  // the waits below give up only on their time limit
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    mbar_init(smem_u32(full), 1);
    mbar_init(smem_u32(done), 1);
    fence_mbar_init_cluster();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sw = smem_u32(base + OFF_W), sa = smem_u32(base + OFF_A);
  const int n = n0 + warp * 32 + lane;
  __nv_bfloat16 *qrow = q + ((size_t)n * H + h) * D_QK;
  if (threadIdx.x == 0) {
    const uint64_t pol = policy_evict_first();
    mbar_arrive_expect_tx(smem_u32(full), 6 * kBoxBytes);
    for (int j = 0; j < 4; j++) tma_load_2d(sw + j * kBoxBytes, &w_map, smem_u32(full), col0 + 64 * j, 128 * h, pol);
    grid_dep_wait();  // qb is written by the Q_B kernel before this one
    for (int j = 0; j < 2; j++)
      tma_load_2d(sa + j * kBoxBytes, &a_map, smem_u32(full), h * 192 + 64 * j, n0, policy_evict_normal());
    if (mbar_wait<false>(smem_u32(full), 0, &abort_flag, kWukWaitNs)) {
      tc_fence_after();
      for (int k = 0; k < 8; k++) {
        const uint64_t ad = smem_desc_sw128(sa + (k >> 2) * kBoxBytes + (k & 3) * 32, 16, 1024);
        const uint64_t bd = smem_desc_sw128(sw + k * 16 * 128, kBoxBytes, 1024);
        mma_ss(tmem, ad, bd, IDESC_WUK, k ? 1u : 0u);
      }
      mma_commit(smem_u32(done));
    } else {
      atomicOr(status, MLA_STATUS_WAIT_TIMEOUT);
      mbar_arrive(smem_u32(done));  // nothing was issued: release the waiters
    }
  }
  grid_dep_wait();  // (every thread: the RoPE rows below read qb)
  if (n < N && col0 == 0) {  // the RoPE rows, while the loads and MMAs run
    const uint4 *src = reinterpret_cast<const uint4 *>(qb + (size_t)n * H * QB_ROWS + h * QB_ROWS + D_NOPE);
    uint4 *dst = reinterpret_cast<uint4 *>(qrow + D_V);
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; j++) v[j] = src[j];
#pragma unroll
    for (int j = 0; j < 8; j++) dst[j] = v[j];
  }
  const bool ok = mbar_wait<false>(smem_u32(done), 0, &abort_flag, kWukWaitNs);
  if (!ok && lane == 0) atomicOr(status, MLA_STATUS_WAIT_TIMEOUT);
  tc_fence_after();
  const bool live = ok && n < N;
  for (int c = 0; c < 8; c++) {
    uint32_t v[32];
    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + 32 * c, v);  // warp-wide
    tmem_wait_ld();
    if (!live) continue;
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; j++) {
      __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
      w[j] = *reinterpret_cast<uint32_t *>(&b2);
    }
    uint4 *d4 = reinterpret_cast<uint4 *>(qrow + col0 + 32 * c);
#pragma unroll
    for (int j = 0; j < 4; j++) d4[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  }
  if (!ok) {  // a wait gave up: let copies or MMAs still in flight land before the CTA exits
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 2000000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  std::lock_guard<std::mutex> lock(g_mu_enc);
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult qr;
    void *f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// A 2-D bf16 tensor map [rows][cols] (row stride ld elements) with boxes of
// box_cols x box_rows, 128-byte swizzled (or not swizzled).
bool make_map(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint64_t ld, uint32_t box_cols = 64,
              uint32_t box_rows = 128, bool swizzle = true) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

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
  cudaStream_t s = (cudaStream_t)stream;
  __nv_bfloat16 *xq = static_cast<__nv_bfloat16 *>(workspace);
  __nv_bfloat16 *qb = reinterpret_cast<__nv_bfloat16 *>(static_cast<uint8_t *>(workspace) +
                                                         round256((size_t)N * D_QA * 2));
  __nv_bfloat16 *qo = static_cast<__nv_bfloat16 *>(q);
  qa_norm_kernel<<<(N + kWarps - 1) / kWarps, kWarps * 32, 0, s>>>(
      static_cast<const __nv_bfloat16 *>(q_a), ld_qa, static_cast<const __nv_bfloat16 *>(w_qa), eps, N, xq);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, cudaGetErrorString(e));
  // Q_B (tokens in blocks of up to 256) and W_UK + the RoPE rows
  const int ntile = N >= 256 ? 256 : (N + 15) / 16 * 16;
  CUtensorMap wq_map, x_map, o_map, w_map, a_map;
  if (!make_map(&wq_map, w_qb, D_QA, (uint64_t)H * QB_ROWS, D_QA) ||
      !make_map(&x_map, xq, D_QA, (uint64_t)N, D_QA, 64, (uint32_t)ntile) ||
      !make_map(&o_map, qb, (uint64_t)H * QB_ROWS, (uint64_t)N, (uint64_t)H * QB_ROWS, 128, (uint32_t)ntile, false) ||
      !make_map(&w_map, w_uk, D_V, (uint64_t)H * D_NOPE, D_V) ||
      !make_map(&a_map, qb, (uint64_t)H * QB_ROWS, (uint64_t)N, (uint64_t)H * QB_ROWS))
    return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  unsigned int *st = nullptr;
  if (status_word(&st) != MLA_OK) return fail(MLA_ERR_CUDA, "device status word unavailable");
  e = cudaFuncSetAttribute(qb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)qb_smem_bytes(256));
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, cudaGetErrorString(e));
  // Q_B and W_UK are programmatic dependents of the kernel before each: they
  // set up and start their weight loads while it finishes, and read its
  // output only after griddepcontrol.wait.
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((H * QB_ROWS + 127) / 128, (N + ntile - 1) / ntile);
  cfg.blockDim = dim3(kQbThreads);
  cfg.dynamicSmemBytes = qb_smem_bytes(ntile);
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, qb_kernel, wq_map, x_map, o_map, ntile, st);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, cudaGetErrorString(e));
  e = cudaFuncSetAttribute(wuk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWukSmem);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, cudaGetErrorString(e));
  cfg.gridDim = dim3(H, D_V / 256, (N + 127) / 128);
  cfg.blockDim = dim3(kWukThreads);
  cfg.dynamicSmemBytes = kWukSmem;
  e = cudaLaunchKernelEx(&cfg, wuk_kernel, w_map, a_map, (const __nv_bfloat16 *)qb, qo, N, H, st);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, cudaGetErrorString(e));
  set_last_error("");
  return MLA_OK;
}
