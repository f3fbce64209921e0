// KV insert: RMSNorm of each new token's latent row, then the write of the
// normalised row and its RoPE'd key into the paged cache (vLLM kimi_k3
// specialized-decode "mla.query" page, MlaQuery.insert: page and offset are
// slot // page_size and slot % page_size; k_pe follows the 512 latent values).
//
// Arithmetic, per token with a live slot (every step after S is one IEEE
// fp32 operation, round to nearest even):
//   S    = sum x_i^2, exact, then rounded once to fp32
//   mean = fp32(fp32(S * 2^-9) + eps)
//   r    = fp32(1 / fp32(sqrt(mean)))         (0 when mean == 0)
//   n_i  = bf16(fp32(fp32(x_i * w_i) * r))
// S is exact because a bf16 square is an 8-bit integer squared times a power
// of two: the 512 squares are added as integers in a fixed-point frame
// aligned to the largest one (exact_sum.cuh), so the sum does not depend on
// the order of additions and every code below is a function of the inputs.
//
// One warp per token, a persistent grid of warps striding over the tokens.
// Each warp keeps its next kStages - 1 tokens (latent row, k_pe, slot) in
// flight into a ring in shared memory with cp.async while it processes the
// current one.
// Lane l holds latent values 16l .. 16l + 15, so the 8 lanes 8t .. 8t+7 hold
// FP8 scale tile t (values 128t .. 128t + 127) and every lane stores one
// 16-byte piece of the latent part of the row.
#include <cuda_fp8.h>

#include "common.cuh"
#include "exact_sum.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;
constexpr int kBlocksPerSm = 4;

template <int N>
__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[N], int at) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; k++) {
    f[at + 2 * k] = __uint_as_float(w[k] << 16);
    f[at + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

// Two values -> two e4m3 codes (first value in the low byte), saturating.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return e4m3x2(a, b) | (e4m3x2(c, d) << 16);
}

constexpr int kStages = 4;
constexpr int kStageBytes = 1024 + 128 + 16;  // latent row, k_pe, slot (8 bytes, padded)
constexpr int kSmemBytes = kWarps * kStages * kStageBytes;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Start the copies of token j into a stage (nothing past the last token);
// every call commits one group, so the group count per stage stays fixed.
__device__ __forceinline__ void issue_token(const KvInsertParams &p, int j, int lane, uint32_t stage) {
  if (j < p.N) {
    const uint8_t *x = reinterpret_cast<const uint8_t *>(p.kv_c + (size_t)j * p.ld_kv) + 32 * lane;
    cp_async16(stage + 32 * lane, x);
    cp_async16(stage + 32 * lane + 16, x + 16);
    if (lane < 8) cp_async16(stage + 1024 + 16 * lane, p.k_pe + (size_t)j * p.ld_pe + 8 * lane);
    if (lane == 0) cp_async8(stage + 1152, p.slots + j);
  }
  cp_async_commit();
}

// Tile scale s = max(fp32(amax / 448), 2^-126) and inv = fp32(1 / s) for a
// bf16 amax > 0.  amax = m * 2^E with m its 8-bit significand (1..255), and
// scaling by a power of two commutes with rounding while the result stays
// normal, so s and inv are fp32(m / 448) and fp32(1 / fp32(m / 448)) (tables
// built at kernel start with those same divisions) with E added to, or taken
// from, the exponent.  A quotient below 2^-126 is the floor, whose
// reciprocal is 2^126.
__device__ __forceinline__ void tile_scale(float amax, const uint32_t *sc_tab, const uint32_t *inv_tab, float &sc,
                                           float &inv) {
  const uint32_t a = __float_as_uint(amax);
  const int e = (int)((a >> 23) & 0xFFu);
  const uint32_t m = ((a >> 16) & 0x7Fu) | (e ? 0x80u : 0u);
  const int E = e ? e - 134 : -133;
  const uint32_t sb = sc_tab[m];
  if ((int)(sb >> 23) + E >= 1) {
    sc = __uint_as_float(sb + ((uint32_t)E << 23));
    inv = __uint_as_float(inv_tab[m] - ((uint32_t)E << 23));
  } else {
    sc = 0x1p-126f;
    inv = 0x1p126f;
  }
}

struct Token {
  uint4 xa, xb, pe;
  long long slot;
};

__device__ __forceinline__ void insert_token(const KvInsertParams &p, const Token &tk, const float (&w)[16],
                                             int lane, const uint32_t *sc_tab, const uint32_t *inv_tab) {
  const long long slot = tk.slot;
  if (slot < 0 || slot >= p.n_slots) {
    if (slot != -1 && lane == 0) atomicOr(p.status, MLA_STATUS_BAD_PAGE);
    return;
  }
  const LaneBf16<8> xr = {{tk.xa.x, tk.xa.y, tk.xa.z, tk.xa.w, tk.xb.x, tk.xb.y, tk.xb.z, tk.xb.w}};
  const uint32_t *xw = xr.w;
  const float S = sum_sq_rn<8>(xr);
  const float mean = __fadd_rn(__fmul_rn(S, 1.f / 512.f), p.eps);
  const float r = mean > 0.f ? __frcp_rn(__fsqrt_rn(mean)) : 0.f;

  // n_i = bf16(fp32(fp32(x_i * w_i) * r)), kept as packed bf16 pairs
  uint32_t nb[8];
#pragma unroll
  for (int k = 0; k < 8; k++) {
    const float x0 = __uint_as_float(xw[k] << 16), x1 = __uint_as_float(xw[k] & 0xFFFF0000u);
    __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(__fmul_rn(x0, w[2 * k]), r),
                                              __fmul_rn(__fmul_rn(x1, w[2 * k + 1]), r));
    nb[k] = *reinterpret_cast<uint32_t *>(&b2);
  }

  if (p.kv_format == MLA_KV_BF16) {
    uint8_t *row = p.cache + (size_t)slot * (D_QK * 2);
    uint4 *dst = reinterpret_cast<uint4 *>(row) + 2 * lane;
    dst[0] = make_uint4(nb[0], nb[1], nb[2], nb[3]);
    dst[1] = make_uint4(nb[4], nb[5], nb[6], nb[7]);
    if (lane < 8) reinterpret_cast<uint4 *>(row + D_V * 2)[lane] = tk.pe;
    return;
  }
  float n[16];
#pragma unroll
  for (int k = 0; k < 8; k++) {
    n[2 * k] = __uint_as_float(nb[k] << 16);
    n[2 * k + 1] = __uint_as_float(nb[k] & 0xFFFF0000u);
  }
  if (p.kv_format == MLA_KV_FP8_E4M3) {
    uint8_t *row = p.cache + (size_t)slot * FP8_ROW;
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(n[i]));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    // s = fp32(amax / 448), at least the smallest normal 2^-126 (so 1 / s
    // stays finite); 1 for an all-zero tile
    float sc = 1.f, inv = 1.f;
    if (amax > 0.f) tile_scale(amax, sc_tab, inv_tab, sc, inv);
    uint32_t c[4];
#pragma unroll
    for (int k = 0; k < 4; k++)
      c[k] = e4m3x4(__fmul_rn(n[4 * k], inv), __fmul_rn(n[4 * k + 1], inv), __fmul_rn(n[4 * k + 2], inv),
                    __fmul_rn(n[4 * k + 3], inv));
    reinterpret_cast<uint4 *>(row)[lane] = make_uint4(c[0], c[1], c[2], c[3]);
    if (lane < 8) reinterpret_cast<uint4 *>(row + D_V)[lane] = tk.pe;
    const float s1 = __shfl_sync(0xffffffffu, sc, 8);
    const float s2 = __shfl_sync(0xffffffffu, sc, 16);
    const float s3 = __shfl_sync(0xffffffffu, sc, 24);
    if (lane == 0) reinterpret_cast<float4 *>(p.kv_scales)[slot] = make_float4(sc, s1, s2, s3);
  } else {  // MLA_KV_FP8_E4M3_TENSOR
    uint8_t *row = p.cache + (size_t)slot * D_QK;
    const float ksi = __ldg(p.k_scale_inv);
    uint32_t c[4];
#pragma unroll
    for (int k = 0; k < 4; k++)
      c[k] = e4m3x4(__fmul_rn(n[4 * k], ksi), __fmul_rn(n[4 * k + 1], ksi), __fmul_rn(n[4 * k + 2], ksi),
                    __fmul_rn(n[4 * k + 3], ksi));
    reinterpret_cast<uint4 *>(row)[lane] = make_uint4(c[0], c[1], c[2], c[3]);
    if (lane < 8) {
      float f[8];
      unpack8(tk.pe, f, 0);
      reinterpret_cast<uint2 *>(row + D_V)[lane] =
          make_uint2(e4m3x4(__fmul_rn(f[0], ksi), __fmul_rn(f[1], ksi), __fmul_rn(f[2], ksi), __fmul_rn(f[3], ksi)),
                     e4m3x4(__fmul_rn(f[4], ksi), __fmul_rn(f[5], ksi), __fmul_rn(f[6], ksi), __fmul_rn(f[7], ksi)));
    }
  }
}

__global__ void __launch_bounds__(kWarps * 32, kBlocksPerSm) kv_insert_kernel(KvInsertParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ uint32_t sc_tab[256], inv_tab[256];  // fp32(m / 448), fp32(1 / that), m = 0..255
  static_assert(kWarps * 32 == 256, "one table entry per thread");
  {
    const float q = __fdiv_rn((float)threadIdx.x, 448.f);
    sc_tab[threadIdx.x] = __float_as_uint(q);
    inv_tab[threadIdx.x] = __float_as_uint(__fdiv_rn(1.f, q));  // m = 0: unused
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int first = blockIdx.x * kWarps + warp;
  const int stride = gridDim.x * kWarps;
  if (first >= p.N) return;
  uint8_t *ring = smem + warp * kStages * kStageBytes;
  const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
  float w[16];
  const uint4 *wr = reinterpret_cast<const uint4 *>(p.w_kva) + 2 * lane;
  unpack8(__ldg(wr), w, 0);
  unpack8(__ldg(wr + 1), w, 8);
#pragma unroll
  for (int s = 0; s < kStages - 1; s++) issue_token(p, first + s * stride, lane, ring_s + s * kStageBytes);
  int st = 0;
  for (int j = first; j < p.N; j += stride) {
    const int ahead = st == 0 ? kStages - 1 : st - 1;  // the stage freed last iteration
    issue_token(p, j + (kStages - 1) * stride, lane, ring_s + ahead * kStageBytes);
    cp_async_wait<kStages - 1>();  // this token's group has landed (for this lane's copies)
    __syncwarp();                  // ... and lane 0's slot copy is visible to all lanes
    const uint8_t *cur = ring + st * kStageBytes;
    Token tk;
    tk.xa = *reinterpret_cast<const uint4 *>(cur + 32 * lane);
    tk.xb = *reinterpret_cast<const uint4 *>(cur + 32 * lane + 16);
    tk.pe = lane < 8 ? *reinterpret_cast<const uint4 *>(cur + 1024 + 16 * lane) : make_uint4(0u, 0u, 0u, 0u);
    tk.slot = *reinterpret_cast<const long long *>(cur + 1152);
    __syncwarp();  // every lane has read the stage before it is refilled
    insert_token(p, tk, w, lane, sc_tab, inv_tab);
    st = st + 1 == kStages ? 0 : st + 1;
  }
  cp_async_wait<0>();
}

}  // namespace

cudaError_t launch_kv_insert(const KvInsertParams &p, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int need = (p.N + kWarps - 1) / kWarps;
  const int blocks = need < sms * kBlocksPerSm ? need : sms * kBlocksPerSm;
  static_assert(kSmemBytes <= 48 * 1024, "dynamic shared memory above the default limit");
  kv_insert_kernel<<<blocks, kWarps * 32, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
