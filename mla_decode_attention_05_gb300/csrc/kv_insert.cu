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
// of two: the 512 squares are added as integers in a 128-bit fixed-point
// accumulator aligned to the largest one, so the sum does not depend on the
// order of additions and every code below is a function of the inputs.
//
// One warp per token.  Lane l holds latent values 16l .. 16l + 15, so the
// 8 lanes 8t .. 8t+7 hold FP8 scale tile t (values 128t .. 128t + 127) and
// every lane stores one 16-byte piece of the latent part of the row.
#include <cuda_fp8.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;

template <int N>
__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[N], int at) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; k++) {
    f[at + 2 * k] = __uint_as_float(w[k] << 16);
    f[at + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t ca = __nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3);
  const uint32_t cb = __nv_cvt_float_to_fp8(b, __NV_SATFINITE, __NV_E4M3);
  const uint32_t cc = __nv_cvt_float_to_fp8(c, __NV_SATFINITE, __NV_E4M3);
  const uint32_t cd = __nv_cvt_float_to_fp8(d, __NV_SATFINITE, __NV_E4M3);
  return ca | (cb << 8) | (cc << 16) | (cd << 24);
}

// The 16 bf16 values of this lane: value = m * 2^(ee - 134) with m the
// 8-bit significand (hidden bit included) and ee the biased exponent (1 for
// subnormals).
__device__ __forceinline__ void split_bf16(uint32_t h, uint32_t &m, int &ee) {
  const int e = (h >> 7) & 0xFF;
  m = (h & 0x7Fu) | (e ? 0x80u : 0u);
  ee = e ? e : 1;
}

// Position of the largest square in the accumulator: 512 squares below 2^16
// each, placed at bit 102 at most, stay below 2^127.
constexpr int kAccTop = 102;

// sum of the squares of the warp's 512 bf16 values (finite), rounded once
// to fp32 (ties to even).
__device__ float exact_sum_sq_rn(const uint32_t (&xw)[8]) {
  int emax = 0;
#pragma unroll
  for (int i = 0; i < 16; i++) {
    uint32_t m;
    int ee;
    split_bf16((xw[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu, m, ee);
    if (m) emax = max(emax, ee);
  }
  emax = (int)__reduce_max_sync(0xffffffffu, (unsigned)emax);
  if (emax == 0) return 0.f;  // all zeros
  unsigned __int128 acc = 0;
  bool sticky = false;
#pragma unroll
  for (int i = 0; i < 16; i++) {
    uint32_t m;
    int ee;
    split_bf16((xw[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu, m, ee);
    const uint32_t t = m * m;
    const int sh = kAccTop - 2 * (emax - ee);
    if (sh >= 0) {
      acc += (unsigned __int128)t << sh;
    } else if (sh > -32) {  // below the accumulator: keep what fits, note the rest
      acc += t >> -sh;
      sticky |= (t & ((1u << -sh) - 1u)) != 0u;
    } else {
      sticky |= t != 0u;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t lo = __shfl_xor_sync(0xffffffffu, (unsigned long long)acc, o);
    const uint64_t hi = __shfl_xor_sync(0xffffffffu, (unsigned long long)(acc >> 64), o);
    acc += ((unsigned __int128)hi << 64) | lo;
  }
  // A nonzero remainder far below the rounding position only matters as a
  // sticky bit.
  if (__any_sync(0xffffffffu, sticky)) acc |= 1u;
  // S = acc * 2^e0; round acc to 24 significant bits (or to the fp32
  // subnormal quantum 2^-149)
  const int e0 = 2 * emax - 268 - kAccTop;
  const uint64_t hi = (uint64_t)(acc >> 64);
  const int lead = hi ? 127 - __clzll((long long)hi) : 63 - __clzll((long long)(uint64_t)acc);
  const int q = max(lead - 23, -149 - e0);
  if (q <= 0) return ldexpf((float)(uint32_t)acc, e0);  // exact: acc < 2^24
  if (q >= lead + 2) return 0.f;                         // below half the smallest subnormal
  unsigned __int128 keep = acc >> q;
  const unsigned __int128 rem = acc & (((unsigned __int128)1 << q) - 1);
  const unsigned __int128 half = (unsigned __int128)1 << (q - 1);
  if (rem > half || (rem == half && (keep & 1))) keep += 1;
  return ldexpf((float)(uint32_t)keep, q + e0);  // keep <= 2^24: exact; overflow -> inf
}

__global__ void __launch_bounds__(kWarps * 32) kv_insert_kernel(KvInsertParams p) {
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (j >= p.N) return;
  const long long slot = p.slots[j];
  if (slot < 0 || slot >= p.n_slots) {
    if (slot != -1 && lane == 0) atomicOr(p.status, MLA_STATUS_BAD_PAGE);
    return;
  }
  const uint4 *xr = reinterpret_cast<const uint4 *>(p.kv_c + (size_t)j * p.ld_kv) + 2 * lane;
  const uint4 *wr = reinterpret_cast<const uint4 *>(p.w_kva) + 2 * lane;
  const uint4 xa = __ldg(xr), xb = __ldg(xr + 1);
  uint4 pe = make_uint4(0u, 0u, 0u, 0u);
  if (lane < 8) pe = __ldg(reinterpret_cast<const uint4 *>(p.k_pe + (size_t)j * p.ld_pe) + lane);
  float x[16], w[16];
  unpack8(xa, x, 0);
  unpack8(xb, x, 8);
  unpack8(__ldg(wr), w, 0);
  unpack8(__ldg(wr + 1), w, 8);

  const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
  const float S = exact_sum_sq_rn(xw);
  const float mean = __fadd_rn(__fmul_rn(S, 1.f / 512.f), p.eps);
  const float r = mean > 0.f ? __fdiv_rn(1.f, __fsqrt_rn(mean)) : 0.f;

  float n[16];
#pragma unroll
  for (int i = 0; i < 16; i++)
    n[i] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__fmul_rn(x[i], w[i]), r)));

  uint8_t *row;
  if (p.kv_format == MLA_KV_BF16) {
    row = p.cache + (size_t)slot * (D_QK * 2);
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 8; k++) {
      __nv_bfloat162 b2 = __floats2bfloat162_rn(n[2 * k], n[2 * k + 1]);  // exact: n is bf16
      h[k] = *reinterpret_cast<uint32_t *>(&b2);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(row) + 2 * lane;
    dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
    dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
    if (lane < 8) reinterpret_cast<uint4 *>(row + D_V * 2)[lane] = pe;
  } else if (p.kv_format == MLA_KV_FP8_E4M3) {
    row = p.cache + (size_t)slot * FP8_ROW;
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(n[i]));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    const float inv = __fdiv_rn(1.f, sc);
    uint32_t c[4];
#pragma unroll
    for (int k = 0; k < 4; k++)
      c[k] = e4m3x4(__fmul_rn(n[4 * k], inv), __fmul_rn(n[4 * k + 1], inv), __fmul_rn(n[4 * k + 2], inv),
                    __fmul_rn(n[4 * k + 3], inv));
    reinterpret_cast<uint4 *>(row)[lane] = make_uint4(c[0], c[1], c[2], c[3]);
    if (lane < 8) reinterpret_cast<uint4 *>(row + D_V)[lane] = pe;
    const float s1 = __shfl_sync(0xffffffffu, sc, 8);
    const float s2 = __shfl_sync(0xffffffffu, sc, 16);
    const float s3 = __shfl_sync(0xffffffffu, sc, 24);
    if (lane == 0) reinterpret_cast<float4 *>(p.kv_scales)[slot] = make_float4(sc, s1, s2, s3);
  } else {  // MLA_KV_FP8_E4M3_TENSOR
    row = p.cache + (size_t)slot * D_QK;
    const float ksi = __ldg(p.k_scale_inv);
    uint32_t c[4];
#pragma unroll
    for (int k = 0; k < 4; k++)
      c[k] = e4m3x4(__fmul_rn(n[4 * k], ksi), __fmul_rn(n[4 * k + 1], ksi), __fmul_rn(n[4 * k + 2], ksi),
                    __fmul_rn(n[4 * k + 3], ksi));
    reinterpret_cast<uint4 *>(row)[lane] = make_uint4(c[0], c[1], c[2], c[3]);
    if (lane < 8) {
      float f[8];
      unpack8(pe, f, 0);
      reinterpret_cast<uint2 *>(row + D_V)[lane] =
          make_uint2(e4m3x4(__fmul_rn(f[0], ksi), __fmul_rn(f[1], ksi), __fmul_rn(f[2], ksi), __fmul_rn(f[3], ksi)),
                     e4m3x4(__fmul_rn(f[4], ksi), __fmul_rn(f[5], ksi), __fmul_rn(f[6], ksi), __fmul_rn(f[7], ksi)));
    }
  }
}

}  // namespace

cudaError_t launch_kv_insert(const KvInsertParams &p, cudaStream_t stream) {
  const int blocks = (p.N + kWarps - 1) / kWarps;
  kv_insert_kernel<<<blocks, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
