// Split-KV combine: merges the partial outputs of an item processed by
// several workers.  With partial results (O_s, L_s) over disjoint key sets,
// L = log2 sum_s 2^{L_s} and O = sum_s 2^{L_s - L} O_s (partials are stored
// normalised and in base 2); a partial over no key has L_s = -inf and
// weight 0.  One lane per query row, one warp per 32 output columns.
#include "common.cuh"

namespace mla {
namespace {

// Block (item, row group y, column half z), 8 warps: warp w takes output
// columns [256z + 32w, 256z + 32w + 32) (chunks 32z + 4w .. +3 of the
// chunk-major partials) of 32 query rows, one row per lane, so every load of
// a chunk covers 1 KB of contiguous memory (32 rows x 8 floats).  The chain
// of dependent loads is kept short: the partials of the first two splits are
// loaded together with the LSEs, before their maximum is known, and later
// splits are loaded two at a time.
constexpr int kWarps = 8;
constexpr int kChunks = 4;  // chunks of 8 columns per warp

// 32-byte load (sm_100 family), L2 only: the partials were written by other
// SMs.  The address must be 32-byte aligned.
__device__ __forceinline__ void ld_cg_v8(float (&v)[8], const float *ptr) {
  uint32_t u[8];
  asm volatile("ld.global.cg.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7])
               : "l"(ptr));
#pragma unroll
  for (int j = 0; j < 8; j++) v[j] = __uint_as_float(u[j]);
}

__device__ __forceinline__ void load_chunks(float (&v)[kChunks][8], const DecodeParams &p, size_t slot, int chunk0,
                                            int r) {
  const float *src = p.ws_o + ((slot * 64 + chunk0) * M_TILE + r) * 8;
#pragma unroll
  for (int k = 0; k < kChunks; k++) ld_cg_v8(v[k], src + (size_t)k * M_TILE * 8);
}

__device__ __forceinline__ void st_v8(__nv_bfloat16 *ptr, const uint32_t (&w)[kChunks * 4], int o) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[o]), "r"(w[o + 1]),
               "r"(w[o + 2]), "r"(w[o + 3]), "r"(w[o + 4]), "r"(w[o + 5]), "r"(w[o + 6]), "r"(w[o + 7])
               : "memory");
}

__device__ __forceinline__ void acc_add(float (&acc)[kChunks * 8], const float (&v)[kChunks][8], float w) {
#pragma unroll
  for (int k = 0; k < kChunks; k++)
#pragma unroll
    for (int j = 0; j < 8; j++) acc[8 * k + j] = fmaf(w, v[k][j], acc[8 * k + j]);
}

__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(DecodeParams p) {
  // the schedule was complete before any decode block began its pieces, so
  // it is read before waiting for the decode kernel
  const int i = blockIdx.x;
  const int base = p.num_splits[i];
  const int ns = p.num_splits[i + 1] - base;
  if (ns <= 1) return;
  grid_dep_wait();  // the decode kernel's partials are complete
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int b, row0, rows;
  if (p.topk_len > 0) {
    b = i / p.T;
    row0 = (i % p.T) * p.H;
    rows = p.H;
  } else {
    b = i % p.B;
    row0 = (i / p.B) * M_TILE;
    rows = min(M_TILE, p.T * p.H - row0);
  }
  if (blockIdx.y * 32 >= rows) return;  // whole block
  const int r = blockIdx.y * 32 + lane;
  const int chunk0 = blockIdx.z * 32 + warp * kChunks;
  const float *lse_r = p.ws_lse + (size_t)base * M_TILE + r;  // split s at [s * M_TILE]
  float va[kChunks][8], vb[kChunks][8];
  load_chunks(va, p, base, chunk0, r);
  load_chunks(vb, p, base + 1, chunk0, r);
  float l4[4];  // the LSEs of the first four splits stay in registers
#pragma unroll
  for (int s = 0; s < 4; s++) l4[s] = s < ns ? __ldcg(lse_r + (size_t)s * M_TILE) : -INFINITY;
  float m = fmaxf(fmaxf(l4[0], l4[1]), fmaxf(l4[2], l4[3]));
  for (int s = 4; s < ns; s++) m = fmaxf(m, __ldcg(lse_r + (size_t)s * M_TILE));
  float acc[kChunks * 8];
#pragma unroll
  for (int k = 0; k < kChunks * 8; k++) acc[k] = 0.f;
  float sum = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < ns; s += 2) {
      if (s > 0) {
        load_chunks(va, p, base + s, chunk0, r);
        if (s + 1 < ns) load_chunks(vb, p, base + s + 1, chunk0, r);
      }
      const float la = s < 4 ? (s == 0 ? l4[0] : l4[2]) : __ldcg(lse_r + (size_t)s * M_TILE);
      const float wa = la == -INFINITY ? 0.f : exp2f(la - m);
      sum += wa;
      acc_add(acc, va, wa);
      if (s + 1 < ns) {
        const float lb = s < 4 ? (s == 0 ? l4[1] : l4[3]) : __ldcg(lse_r + (size_t)(s + 1) * M_TILE);
        const float wb = lb == -INFINITY ? 0.f : exp2f(lb - m);
        sum += wb;
        acc_add(acc, vb, wb);
      }
    }
  }
  if (r >= rows) return;
  const int R = row0 + r;
  const int t = R / p.H, h = R % p.H;
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  __nv_bfloat16 *dst = p.out + (((size_t)b * p.T + t) * p.H + h) * D_V + chunk0 * 8;
  uint32_t wv[kChunks * 4];
#pragma unroll
  for (int e = 0; e < kChunks * 4; e++) {
    __nv_bfloat162 pr = __floats2bfloat162_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv);
    wv[e] = *reinterpret_cast<uint32_t *>(&pr);
  }
  if (p.out_v8) {  // 32-byte stores (the 64 bytes of this lane start 64-byte aligned)
    st_v8(dst, wv, 0);
    st_v8(dst + 16, wv, 8);
  } else {
#pragma unroll
    for (int k = 0; k < kChunks; k++)
      reinterpret_cast<uint4 *>(dst)[k] = make_uint4(wv[4 * k], wv[4 * k + 1], wv[4 * k + 2], wv[4 * k + 3]);
  }
  if (warp == 0 && blockIdx.z == 0)
    p.lse[((size_t)b * p.H + h) * p.T + t] = sum > 0.f ? (m + log2f(sum)) * LN2 : -INFINITY;
}

}  // namespace

cudaError_t launch_combine(const DecodeParams &p, cudaStream_t stream) {
  // launched as a programmatic dependent of the decode kernel: its blocks
  // are scheduled while the decode kernel runs and wait for it in
  // grid_dep_wait()
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_items, M_TILE / 32, 2);
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
