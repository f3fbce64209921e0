// MLA decode, plain-SIMT form: one warp per query row, the 64-key tile of
// the shared latent cache staged once per CTA in shared memory as bf16 (FP8
// rows are dequantised on the way in).  Online softmax over tiles in base 2.
//
// Each CTA serves one worker (blockIdx.x) of the split-KV partition and
// eight query rows (blockIdx.y) of every item that worker processes.
#include "common.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct SmemSimt {
  __nv_bfloat162 kv[PAGE][D_QK / 2];  // 73728 B
  int tok[PAGE];                      // logical token of each row, -1 = none
  int page[PAGE];
};

// Resolve the 64 rows of key tile `tile` of item `it`, then copy them into
// shared memory (zeros for rows that take no part).
__device__ void stage_tile(const DecodeParams &p, const Item &it, int t_item,
                           int tile, int sk, SmemSimt &sm, bool record) {
  const int tid = threadIdx.x;
  if (tid < PAGE) {
    int n = -1, pg = -1;
    if (p.topk_len > 0) {
      int slot = tile * PAGE + tid;
      if (slot < p.topk_len) {
        int id = p.topk[((size_t)it.b * p.T + t_item) * p.topk_len + slot];
        if (id >= sk || id < -1) {
          atomicOr(p.status, MLA_STATUS_BAD_TOPK);
          id = -1;
        }
        n = id;
      }
    } else {
      int pos = tile * PAGE + tid;
      if (pos < it.kv_len) n = pos;
    }
    if (n >= 0) {
      int j = n / PAGE;
      if (j >= p.max_pages) {
        atomicOr(p.status, MLA_STATUS_BAD_SEQLEN);
        n = -1;
      } else {
        pg = p.block_table[(size_t)it.b * p.max_pages + j];
        if (pg < 0 || pg >= p.num_pages) {
          atomicOr(p.status, MLA_STATUS_BAD_PAGE);
          n = -1;
        }
      }
    }
    sm.tok[tid] = n;
    sm.page[tid] = pg;
    if (record && p.gathered != nullptr) {
      int slot = tile * PAGE + tid;
      if (slot < p.topk_len)
        p.gathered[((size_t)it.b * p.T + t_item) * p.topk_len + slot] = n;
    }
  }
  __syncthreads();
  if (p.kv_format == MLA_KV_BF16) {
    constexpr int kChunks = D_QK * 2 / 16;  // 72 x 16 B per row
    for (int c = tid; c < PAGE * kChunks; c += kThreads) {
      int r = c / kChunks, k = c % kChunks;
      uint4 v = make_uint4(0, 0, 0, 0);
      int n = sm.tok[r];
      if (n >= 0) {
        const uint8_t *row = p.kv + ((size_t)sm.page[r] * PAGE + (n % PAGE)) * (D_QK * 2);
        v = __ldg(reinterpret_cast<const uint4 *>(row) + k);
      }
      reinterpret_cast<uint4 *>(&sm.kv[r][0])[k] = v;
    }
  } else {
    constexpr int kChunks = 40;  // 32 x 16 e4m3 bytes + 8 x 16 RoPE bytes
    for (int c = tid; c < PAGE * kChunks; c += kThreads) {
      int r = c / kChunks, k = c % kChunks;
      int n = sm.tok[r];
      uint4 *dst = reinterpret_cast<uint4 *>(&sm.kv[r][0]);
      if (n < 0) {
        if (k < 32) {
          dst[2 * k] = make_uint4(0, 0, 0, 0);
          dst[2 * k + 1] = make_uint4(0, 0, 0, 0);
        } else {
          dst[64 + (k - 32)] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      size_t rowi = (size_t)sm.page[r] * PAGE + (n % PAGE);
      const uint8_t *row = p.kv + rowi * FP8_ROW;
      uint4 v = __ldg(reinterpret_cast<const uint4 *>(row) + k);
      if (k >= 32) {  // RoPE: 64 bf16 stored after the 512 e4m3 bytes
        dst[64 + (k - 32)] = v;
        continue;
      }
      float sc = __ldg(p.kv_scales + rowi * 4 + k / 8);
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 4; i++) {
#pragma unroll
        for (int h = 0; h < 2; h++) {
          uint32_t b0 = (w[i] >> (16 * h)) & 0xFFu, b1 = (w[i] >> (16 * h + 8)) & 0xFFu;
          __nv_bfloat162 pr = __floats2bfloat162_rn(e4m3_to_float(b0) * sc, e4m3_to_float(b1) * sc);
          o[2 * i + h] = *reinterpret_cast<uint32_t *>(&pr);
        }
      }
      dst[2 * k] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[2 * k + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
  __syncthreads();
}

__device__ inline float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ inline float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__global__ void __launch_bounds__(kThreads, 1)
decode_simt_kernel(DecodeParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SmemSimt &sm = *reinterpret_cast<SmemSimt *>(smem_raw);
  const int part = blockIdx.x;
  const int rg = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t *md = p.tile_md + (size_t)part * MD_STRIDE;
  const int a = md[0], bt = md[1], z = md[2], et = md[3], fp = md[4], at_start = md[5];

  for (int i = a; i <= z; i++) {
    Item it = item_at(i, p.seqlens, p.H, p.T, p.topk_len, p.causal, p.n_mt, p.status);
    int t0 = (i == a) ? bt : 0;
    int t1 = (i == z) ? et : it.ntiles;
    int piece = (i == a) ? fp : 0;
    bool empty_owned = (it.ntiles == 0) && (i > a || at_start);
    if (!(t1 > t0 || empty_owned)) continue;
    if (rg * kWarps >= it.rows) continue;  // no rows of this item here
    const int sk = clamp_seqlen(p.seqlens[it.b], p.status);
    const int t_item = (p.topk_len > 0) ? (i % p.T) : 0;
    const int r = rg * kWarps + warp;      // row within the item
    const bool active = r < it.rows;
    const int R = it.row0 + (active ? r : 0);
    const int t = R / p.H, h = R % p.H;
    const int my_len = row_kv_len(sk, p.T, t, p.causal);

    float qf[18];
    {
      const __nv_bfloat162 *qr = reinterpret_cast<const __nv_bfloat162 *>(
          p.q + (((size_t)it.b * p.T + t) * p.H + h) * D_QK);
#pragma unroll
      for (int k = 0; k < 9; k++) {
        float2 f = __bfloat1622float2(qr[lane + 32 * k]);
        qf[2 * k] = f.x;
        qf[2 * k + 1] = f.y;
      }
    }
    float o[16];
#pragma unroll
    for (int k = 0; k < 16; k++) o[k] = 0.f;
    float m = -INFINITY, l = 0.f;

    for (int tile = t0; tile < t1; tile++) {
      stage_tile(p, it, t_item, tile, sk, sm, rg == 0);
      float sa = -INFINITY, sb = -INFINITY;
      for (int n = 0; n < PAGE; n++) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 9; k++) {
          float2 kf = __bfloat1622float2(sm.kv[n][lane + 32 * k]);
          acc = fmaf(qf[2 * k], kf.x, acc);
          acc = fmaf(qf[2 * k + 1], kf.y, acc);
        }
        acc = warp_sum(acc);
        bool valid = sm.tok[n] >= 0;
        if (p.topk_len == 0) valid = valid && (tile * PAGE + n < my_len);
        float s = valid ? acc * p.scale_log2 : -INFINITY;
        if (lane == (n & 31)) {
          if (n < 32) sa = s; else sb = s;
        }
      }
      float mt = warp_max(fmaxf(sa, sb));
      float m_new = fmaxf(m, mt);
      float pa = 0.f, pb = 0.f, alpha = 1.f;
      if (m_new != -INFINITY) {
        alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
        pa = (sa == -INFINITY) ? 0.f : exp2f(sa - m_new);
        pb = (sb == -INFINITY) ? 0.f : exp2f(sb - m_new);
        m = m_new;
      }
      l = l * alpha + warp_sum(pa + pb);
#pragma unroll
      for (int k = 0; k < 16; k++) o[k] *= alpha;
      for (int n = 0; n < PAGE; n++) {
        float pn = __shfl_sync(0xffffffffu, n < 32 ? pa : pb, n & 31);
        if (pn == 0.f) continue;  // uniform across the warp
#pragma unroll
        for (int k = 0; k < 8; k++) {
          float2 vf = __bfloat1622float2(sm.kv[n][lane + 32 * k]);
          o[2 * k] = fmaf(pn, vf.x, o[2 * k]);
          o[2 * k + 1] = fmaf(pn, vf.y, o[2 * k + 1]);
        }
      }
      __syncthreads();  // the tile buffer is rewritten next iteration
    }

    if (!active) continue;
    const int nsplit = p.num_splits[i + 1] - p.num_splits[i];
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
    const float lse2 = (l > 0.f) ? m + log2f(l) : -INFINITY;
    if (nsplit <= 1) {
      __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(
          p.out + (((size_t)it.b * p.T + t) * p.H + h) * D_V);
#pragma unroll
      for (int k = 0; k < 8; k++)
        dst[lane + 32 * k] = __floats2bfloat162_rn(o[2 * k] * inv, o[2 * k + 1] * inv);
      if (lane == 0) p.lse[((size_t)it.b * p.H + h) * p.T + t] = lse2 * LN2;
    } else {
      size_t slot = (size_t)p.num_splits[i] + piece;
      float2 *dst = reinterpret_cast<float2 *>(p.ws_o + (slot * M_TILE + r) * D_V);
#pragma unroll
      for (int k = 0; k < 8; k++) dst[lane + 32 * k] = make_float2(o[2 * k] * inv, o[2 * k + 1] * inv);
      if (lane == 0) p.ws_lse[slot * M_TILE + r] = lse2;
    }
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, cudaStream_t stream,
                          cudaEvent_t ev_before, cudaEvent_t ev_after) {
  const size_t smem = sizeof(SmemSimt);
  cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_parts, M_TILE / kWarps);
  if (ev_before) cudaEventRecord(ev_before, stream);
  decode_simt_kernel<<<grid, kThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (ev_after) cudaEventRecord(ev_after, stream);
  return e;
}

}  // namespace mla
