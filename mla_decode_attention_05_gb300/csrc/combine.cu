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
// 512 / 256-byte span.  Two splits are loaded at a time.
__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(DecodeParams p) {
  grid_dep_wait();  // the decode kernel's partials are complete
  const int i = blockIdx.x;
  const int base = p.num_splits[i];
  const int ns = p.num_splits[i + 1] - base;
  if (ns <= 1) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Item it = item_at(i, p.seqlens, p.H, p.T, p.topk_len, p.causal, p.n_mt, p.status);
  const int r = blockIdx.y * kWarps + warp;
  if (r >= it.rows) return;
  float m = -INFINITY;
  for (int s = lane; s < ns; s += 32)
    m = fmaxf(m, __ldcg(p.ws_lse + (size_t)(base + s) * M_TILE + r));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; k++) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  float sum = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < ns; s += 2) {
      const bool two = s + 1 < ns;  // every split slot holds a written partial
      const float l0 = __ldcg(p.ws_lse + (size_t)(base + s) * M_TILE + r);
      const float l1 = two ? __ldcg(p.ws_lse + (size_t)(base + s + 1) * M_TILE + r) : -INFINITY;
      const float4 *src0 = reinterpret_cast<const float4 *>(p.ws_o + ((size_t)(base + s) * M_TILE + r) * D_V);
      const float4 *src1 = src0 + (M_TILE * D_V) / 4;
      float4 v0[4], v1[4];
#pragma unroll
      for (int k = 0; k < 4; k++) v0[k] = __ldcg(src0 + 32 * k + lane);
#pragma unroll
      for (int k = 0; k < 4; k++) v1[k] = two ? __ldcg(src1 + 32 * k + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float w0 = l0 == -INFINITY ? 0.f : exp2f(l0 - m);
      const float w1 = l1 == -INFINITY ? 0.f : exp2f(l1 - m);
      sum += w0 + w1;
      acc_add(acc, v0, w0);
      acc_add(acc, v1, w1);
    }
  }
  const int R = it.row0 + r;
  const int t = R / p.H, h = R % p.H;
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  uint2 *dst = reinterpret_cast<uint2 *>(p.out + (((size_t)it.b * p.T + t) * p.H + h) * D_V);
#pragma unroll
  for (int k = 0; k < 4; k++) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x * inv, acc[k].y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z * inv, acc[k].w * inv);
    dst[32 * k + lane] = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
  }
  if (lane == 0)
    p.lse[((size_t)it.b * p.H + h) * p.T + t] = sum > 0.f ? (m + log2f(sum)) * LN2 : -INFINITY;
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
