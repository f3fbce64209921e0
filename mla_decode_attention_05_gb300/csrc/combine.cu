// Split-KV combine: merges the partial outputs of an item processed by
// several workers.  With partial results (O_s, L_s) over disjoint key sets,
// L = log2 sum_s 2^{L_s} and O = sum_s 2^{L_s - L} O_s (partials are stored
// normalised and in base 2); a partial over no key has L_s = -inf and
// weight 0.  One warp per query row, 16 output values per lane.
#include "common.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(DecodeParams p) {
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
    m = fmaxf(m, p.ws_lse[(size_t)(base + s) * M_TILE + r]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; k++) acc[k] = 0.f;
  float sum = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < ns; s++) {
      float ls = p.ws_lse[(size_t)(base + s) * M_TILE + r];
      if (ls == -INFINITY) continue;
      float w = exp2f(ls - m);
      sum += w;
      const float2 *src = reinterpret_cast<const float2 *>(
          p.ws_o + ((size_t)(base + s) * M_TILE + r) * D_V);
#pragma unroll
      for (int k = 0; k < 8; k++) {
        float2 v = src[lane + 32 * k];
        acc[2 * k] = fmaf(w, v.x, acc[2 * k]);
        acc[2 * k + 1] = fmaf(w, v.y, acc[2 * k + 1]);
      }
    }
  }
  const int R = it.row0 + r;
  const int t = R / p.H, h = R % p.H;
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(
      p.out + (((size_t)it.b * p.T + t) * p.H + h) * D_V);
#pragma unroll
  for (int k = 0; k < 8; k++)
    dst[lane + 32 * k] = __floats2bfloat162_rn(acc[2 * k] * inv, acc[2 * k + 1] * inv);
  if (lane == 0)
    p.lse[((size_t)it.b * p.H + h) * p.T + t] = sum > 0.f ? (m + log2f(sum)) * LN2 : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const DecodeParams &p, cudaStream_t stream) {
  dim3 grid(p.n_items, M_TILE / kWarps);
  combine_kernel<<<grid, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
