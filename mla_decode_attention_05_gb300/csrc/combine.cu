// Split-KV combine: merges the partial outputs of an item processed by
// several workers.  With partial results (O_s, L_s) over disjoint key sets,
// L = log2 sum_s 2^{L_s} and O = sum_s 2^{L_s - L} O_s (partials are stored
// normalised and in base 2); a partial over no key has L_s = -inf and
// weight 0.  One warp per query row, 16 output values per lane.
#include "common.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ void acc_add(float4 (&acc)[4], const float4 (&v)[4], float w) {
#pragma unroll
  for (int k = 0; k < 4; k++) {
    acc[k].x = fmaf(w, v[k].x, acc[k].x);
    acc[k].y = fmaf(w, v[k].y, acc[k].y);
    acc[k].z = fmaf(w, v[k].z, acc[k].z);
    acc[k].w = fmaf(w, v[k].w, acc[k].w);
  }
}

// Lane l of the warp of row r holds output values 4*(32k + l) .. +3, k < 4:
// every 16-byte load and 8-byte store of the warp covers one contiguous
// 512 / 256-byte span.  The chain of dependent loads is kept short: the
// item's geometry is arithmetic (no sequence length is read), and the
// partial O of the first two splits is loaded together with the LSEs,
// before their maximum is known; lane s holds the LSE of split s (s < 32).
__global__ void __launch_bounds__(kWarps * 32, 3)
combine_kernel(DecodeParams p) {
  grid_dep_wait();  // the decode kernel's partials are complete
  const int i = blockIdx.x;
  const int base = p.num_splits[i];
  const int ns = p.num_splits[i + 1] - base;
  if (ns <= 1) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int b, row0, rows;
  if (p.topk_len > 0) {
    b = i / p.T;
    row0 = (i % p.T) * p.H;
    rows = p.H;
  } else {
    b = i / p.n_mt;
    row0 = (i % p.n_mt) * M_TILE;
    rows = min(M_TILE, p.T * p.H - row0);
  }
  const int r = blockIdx.y * kWarps + warp;
  if (r >= rows) return;
  const float *lse_r = p.ws_lse + (size_t)base * M_TILE + r;                        // split s at [s * M_TILE]
  const float4 *o_r = reinterpret_cast<const float4 *>(p.ws_o + ((size_t)base * M_TILE + r) * D_V);
  constexpr size_t kSplitStride4 = (size_t)M_TILE * D_V / 4;                        // float4s per split slot
  const float lse_l = lane < ns ? __ldcg(lse_r + (size_t)lane * M_TILE) : -INFINITY;
  float4 v[2][4];
#pragma unroll
  for (int s = 0; s < 2; s++)
#pragma unroll
    for (int k = 0; k < 4; k++)
      v[s][k] = s < ns ? __ldcg(o_r + s * kSplitStride4 + 32 * k + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
  float m = lse_l;
  for (int s = 32 + lane; s < ns; s += 32) m = fmaxf(m, __ldcg(lse_r + (size_t)s * M_TILE));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; k++) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  float sum = 0.f;
  if (m != -INFINITY) {
#pragma unroll
    for (int s = 0; s < 2; s++) {
      const float l = __shfl_sync(0xffffffffu, lse_l, s);
      const float w = (s < ns && l != -INFINITY) ? exp2f(l - m) : 0.f;
      sum += w;
      acc_add(acc, v[s], w);
    }
    for (int s = 2; s < ns; s++) {  // more than two splits: one at a time
      const float l = s < 32 ? __shfl_sync(0xffffffffu, lse_l, s) : __ldcg(lse_r + (size_t)s * M_TILE);
      const float w = l == -INFINITY ? 0.f : exp2f(l - m);
      float4 u[4];
#pragma unroll
      for (int k = 0; k < 4; k++) u[k] = __ldcg(o_r + s * kSplitStride4 + 32 * k + lane);
      sum += w;
      acc_add(acc, u, w);
    }
  }
  const int R = row0 + r;
  const int t = R / p.H, h = R % p.H;
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  uint2 *dst = reinterpret_cast<uint2 *>(p.out + (((size_t)b * p.T + t) * p.H + h) * D_V);
#pragma unroll
  for (int k = 0; k < 4; k++) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x * inv, acc[k].y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z * inv, acc[k].w * inv);
    dst[32 * k + lane] = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
  }
  if (lane == 0)
    p.lse[((size_t)b * p.H + h) * p.T + t] = sum > 0.f ? (m + log2f(sum)) * LN2 : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const DecodeParams &p, cudaStream_t stream) {
  // launched as a programmatic dependent of the decode kernel: its blocks
  // are scheduled while the decode kernel runs and wait for it in
  // grid_dep_wait()
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_items, M_TILE / kWarps);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace mla
