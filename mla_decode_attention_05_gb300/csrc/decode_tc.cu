// MLA decode on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// One worker of the split-KV partition = one cluster of two CTAs (a pair of
// SMs).  Heads are packed into the MMA M dimension (STAGE_D2.md "Strategy A":
// Q reshaped to (T*n_h, d), one M tile of 128 query rows, row = t*H + h), so
// each 64-token key tile is read from HBM once per (item, split) for all
// heads.  The 576 latent dims are divided between the two CTAs:
//
//   rank 0: QK dims [0,256) + the RoPE block [512,576); V dims [0,256)
//   rank 1: QK dims [256,512);                          V dims [256,512)
//
// so that every KV byte is staged exactly once per pair and every flop is
// done once: each CTA forms a partial S over its dims (the RoPE block being
// one more block of the reduction, FlashMLA issue #169 "dual gemm"), the
// two partial S tiles are swapped through distributed shared memory and
// summed (the same sum on both sides), both CTAs run the same online softmax,
// and each accumulates its half of O = P V in its own TMEM.  This is the
// pair-level form of the dual-GEMM idea of FlashMLA issue #169 (the
// reduction dimension cut in halves whose partial S are added before the
// softmax), chosen because a 128 x 512 fp32 O accumulator alone fills all of
// one SM's tensor memory.
//
// Per CTA (256 threads):
//   warp 0        producer: TMA of the CTA's column blocks of each page
//                 (dense / causal bf16), or, in the gather form, with warps
//                 2-3: row gather (top-k) and FP8 dequantisation into the
//                 same swizzled layout
//   warp 1        TMEM allocation and the single MMA-issuing thread
//   warps 4-7     softmax / epilogue: thread = query row = TMEM lane
//
// TMEM (512 columns x 128 lanes): O half [0,256), S [256,320), Q part
// [320,480) (A operand of QK read straight from TMEM).
// Shared memory: 3 KV stages of 5 blocks x (64 tokens x 128 B, 128-byte
// swizzle), 2 P buffers (128 x 64 bf16, A operand of PV), 2 exchange
// buffers for the peer's partial S (128 x 64 fp32).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <cstring>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kThreads = 256;
constexpr int kStages = 3;
constexpr int kBlkBytes = PAGE * 128;             // 64 tokens x 64 dims bf16
constexpr int kMaxBlocks = 5;
constexpr int kStageBytes = kMaxBlocks * kBlkBytes;  // 40 KB
constexpr int kPBytes = M_TILE * 128;             // 128 rows x 64 tokens bf16
constexpr int kXchBytes = M_TILE * PAGE * 4;      // 128 rows x 64 fp32
constexpr int kProducers = 96;                    // gather form: warps 0, 2, 3
constexpr uint64_t kWaitNs = 2000000000ull;       // bounded waits: 2 s
constexpr float kRescaleThreshold = 8.0f;         // log2 units

constexpr uint32_t TM_O = 0;
constexpr uint32_t TM_S = 256;
constexpr uint32_t TM_Q = 320;
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 256, false, true);

struct Smem {
  uint8_t kv[kStages][kStageBytes];
  uint8_t p[2][kPBytes];
  uint8_t xch[2][kXchBytes];
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full, s_free, o_done, q_ready;
  uint64_t p_full[2];   // per P buffer: a phase can never run two ahead
  uint64_t p_empty[2];
  uint64_t xch_full[2];
  uint64_t peer_free[2];
  uint32_t mask[kStages][2];     // valid rows of each stage (bits)
  long long rowoff[kStages][PAGE];  // gather form: row index in the pool, -1 = none
  uint32_t tmem_base;
  int abort;
};

// First dim of column block kb of CTA `rank`.
__device__ __forceinline__ int block_dim(uint32_t rank, int kb) {
  return rank == 0 ? (kb < 4 ? kb * 64 : D_V) : D_V / 2 + kb * 64;
}

struct Ctx {
  const DecodeParams *p;
  Smem *sm;
  uint32_t rank, peer;
  int nblk;
  int part;
};

__device__ __forceinline__ bool wait_or_abort(const Ctx &c, uint64_t *bar, uint32_t parity) {
  if (mbar_wait<false>(smem_u32(bar), parity, &c.sm->abort, kWaitNs)) return true;
  atomicOr(c.p->status, MLA_STATUS_WAIT_TIMEOUT);
  c.sm->abort = 1;
  return false;
}

__device__ __forceinline__ bool wait_cluster_or_abort(const Ctx &c, uint64_t *bar, uint32_t parity) {
  if (mbar_wait<true>(smem_u32(bar), parity, &c.sm->abort, kWaitNs)) return true;
  atomicOr(c.p->status, MLA_STATUS_WAIT_TIMEOUT);
  c.sm->abort = 1;
  return false;
}

// Walk the pieces of this worker: f(item_index, item, t0, t1, piece, empty).
template <class F>
__device__ __forceinline__ bool for_each_piece(const DecodeParams &p, int part, F &&f) {
  const int32_t *md = p.tile_md + (size_t)part * MD_STRIDE;
  const int a = md[0], bt = md[1], z = md[2], et = md[3], fp = md[4], at_start = md[5];
  for (int i = a; i <= z; i++) {
    Item it = item_at(i, p.seqlens, p.H, p.T, p.topk_len, p.causal, p.n_mt, p.status);
    int t0 = (i == a) ? bt : 0;
    int t1 = (i == z) ? et : it.ntiles;
    bool empty_owned = (it.ntiles == 0) && (i > a || at_start);
    if (!(t1 > t0 || empty_owned)) continue;
    if (!f(i, it, t0, t1, (i == a) ? fp : 0, it.ntiles == 0)) return false;
  }
  return true;
}

// ---- producer: TMA of whole pages ------------------------------------------------

__device__ void producer_tma(const Ctx &c, const CUtensorMap *map) {
  const DecodeParams &p = *c.p;
  Smem &sm = *c.sm;
  const uint64_t pol = policy_evict_first();
  uint32_t g = 0;
  for_each_piece(p, c.part, [&](int, const Item &it, int t0, int t1, int, bool empty) {
    if (empty) return true;
    for (int tile = t0; tile < t1; tile++, g++) {
      const int s = g % kStages;
      if (!wait_or_abort(c, &sm.kv_empty[s], ((g / kStages) & 1) ^ 1)) return false;
      int page = -1;
      if (tile < p.max_pages) {
        page = p.block_table[(size_t)it.b * p.max_pages + tile];
        if (page < 0 || page >= p.num_pages) {
          atomicOr(p.status, MLA_STATUS_BAD_PAGE);
          page = -1;
        }
      } else {
        atomicOr(p.status, MLA_STATUS_BAD_SEQLEN);
      }
      const int nvalid = min(PAGE, it.kv_len - tile * PAGE);
      uint64_t m = 0;
      if (page >= 0) m = nvalid >= 64 ? ~0ull : ((1ull << nvalid) - 1ull);
      sm.mask[s][0] = (uint32_t)m;
      sm.mask[s][1] = (uint32_t)(m >> 32);
      const uint32_t bar = smem_u32(&sm.kv_full[s]);
      mbar_arrive_expect_tx(bar, (uint32_t)(c.nblk * kBlkBytes));
      const uint32_t dst = smem_u32(&sm.kv[s][0]);
      for (int kb = 0; kb < c.nblk; kb++)
        tma_load_3d(dst + kb * kBlkBytes, map, bar, block_dim(c.rank, kb), 0, page < 0 ? 0 : page, pol);
    }
    return true;
  });
}

// ---- producer: row gather / FP8 dequantisation -----------------------------------

// 16 e4m3 bytes x scale -> 16 bf16 (two 16-byte chunks).
__device__ __forceinline__ void dequant16(uint4 v, float sc, uint4 &lo, uint4 &hi) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; i++) {
#pragma unroll
    for (int h = 0; h < 2; h++) {
      uint16_t pair = (uint16_t)(w[i] >> (16 * h));
      uint32_t f16x2;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f16x2) : "h"(pair));
      __half2 hv = *reinterpret_cast<__half2 *>(&f16x2);
      float2 f = __half22float2(hv);
      __nv_bfloat162 b = __floats2bfloat162_rn(f.x * sc, f.y * sc);
      o[2 * i + h] = *reinterpret_cast<uint32_t *>(&b);
    }
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ void producer_gather(const Ctx &c, int pi /* 0..95 */) {
  const DecodeParams &p = *c.p;
  Smem &sm = *c.sm;
  const bool fp8 = p.kv_format == MLA_KV_FP8_E4M3;
  const size_t row_bytes = fp8 ? FP8_ROW : D_QK * 2;
  // units per row: fp8 -> 16 e4m3 chunks (+ 8 RoPE chunks on rank 0);
  // bf16 -> 32 latent chunks (+ 8 RoPE chunks on rank 0)
  const int n_main = fp8 ? 16 : 32;
  const int n_units = n_main + (c.rank == 0 ? 8 : 0);
  uint32_t g = 0;
  for_each_piece(p, c.part, [&](int idx, const Item &it, int t0, int t1, int, bool empty) {
    if (empty) return true;
    const int t_item = (p.topk_len > 0) ? (idx % p.T) : 0;
    const int sk = clamp_seqlen(p.seqlens[it.b], p.status);
    for (int tile = t0; tile < t1; tile++, g++) {
      const int s = g % kStages;
      if (!wait_or_abort(c, &sm.kv_empty[s], ((g / kStages) & 1) ^ 1)) return false;
      // 1. resolve the 64 rows of this tile (producer threads 0..63)
      if (pi < PAGE) {
        int n = -1;
        if (p.topk_len > 0) {
          const int slot = tile * PAGE + pi;
          if (slot < p.topk_len) {
            int id = p.topk[((size_t)it.b * p.T + t_item) * p.topk_len + slot];
            if (id >= sk || id < -1) {
              atomicOr(p.status, MLA_STATUS_BAD_TOPK);
              id = -1;
            }
            n = id;
          }
        } else {
          const int pos = tile * PAGE + pi;
          if (pos < it.kv_len) n = pos;
        }
        long long off = -1;
        if (n >= 0) {
          const int j = n / PAGE;
          if (j >= p.max_pages) {
            atomicOr(p.status, MLA_STATUS_BAD_SEQLEN);
            n = -1;
          } else {
            const int pg = p.block_table[(size_t)it.b * p.max_pages + j];
            if (pg < 0 || pg >= p.num_pages) {
              atomicOr(p.status, MLA_STATUS_BAD_PAGE);
              n = -1;
            } else {
              off = (long long)pg * PAGE + (n % PAGE);
            }
          }
        }
        sm.rowoff[s][pi] = off;
        const uint32_t bits = __ballot_sync(0xffffffffu, off >= 0);
        if ((pi & 31) == 0) sm.mask[s][pi >> 5] = bits;
        if (c.rank == 0 && p.gathered != nullptr && p.topk_len > 0) {
          const int slot = tile * PAGE + pi;
          if (slot < p.topk_len) p.gathered[((size_t)it.b * p.T + t_item) * p.topk_len + slot] = n;
        }
      }
      named_bar_sync(1, kProducers);
      // 2. copy / dequantise into the swizzled stage
      const uint32_t stage = smem_u32(&sm.kv[s][0]);
      for (int w = pi; w < PAGE * n_units; w += kProducers) {
        const int i = w / n_units, u = w % n_units;
        const long long off = sm.rowoff[s][i];
        const uint8_t *row = p.kv + (size_t)(off < 0 ? 0 : off) * row_bytes;
        if (u < n_main) {
          if (fp8) {
            // e4m3 chunk u of this CTA's 256 latent bytes -> dims 16u..16u+15
            uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
            if (off >= 0) {
              const uint4 v = __ldg(reinterpret_cast<const uint4 *>(row + c.rank * 256) + u);
              const float sc = __ldg(p.kv_scales + (size_t)off * 4 + c.rank * 2 + u / 8);
              dequant16(v, sc, lo, hi);
            }
            const int kb = u / 4, ch = 2 * (u % 4);
            const uint32_t base = stage + kb * kBlkBytes + i * 128;
            st_shared_v4(base + (((ch) ^ (i & 7)) << 4), lo);
            st_shared_v4(base + (((ch + 1) ^ (i & 7)) << 4), hi);
          } else {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (off >= 0) v = __ldg(reinterpret_cast<const uint4 *>(row + c.rank * 512) + u);
            const int kb = u / 8, ch = u % 8;
            st_shared_v4(stage + kb * kBlkBytes + i * 128 + ((ch ^ (i & 7)) << 4), v);
          }
        } else {
          // RoPE (rank 0): 64 bf16 after the latent part of the row
          const int ch = u - n_main;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (off >= 0) v = __ldg(reinterpret_cast<const uint4 *>(row + (fp8 ? D_V : 2 * D_V)) + ch);
          st_shared_v4(stage + 4 * kBlkBytes + i * 128 + ((ch ^ (i & 7)) << 4), v);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&sm.kv_full[s]));
    }
    return true;
  });
}

// ---- MMA issuer (one thread) ------------------------------------------------------
//
// Per tile g:  QK(g): S = Q_part . K_part^T  (M=128, N=64, K = 64 per block,
// A = Q from TMEM, B = the K-major swizzled key block), commit -> s_full;
// then PV(g-1): O_half (+)= P(g-1) . V_half (M=128, N=256, K=64 tokens,
// A = P from shared memory, B = the same stage read MN-major as V), commit
// -> kv_empty, p_empty, o_done.  QK of the next tile is issued before PV of
// the current one so the tensor pipe has work while the softmax runs.

__device__ void mma_issuer(const Ctx &c, uint32_t tmem) {
  const DecodeParams &p = *c.p;
  Smem &sm = *c.sm;
  const uint32_t kv0 = smem_u32(&sm.kv[0][0]);
  const uint32_t p0 = smem_u32(&sm.p[0][0]);
  uint32_t g = 0;
  uint32_t qn = 0;
  auto issue_pv = [&](uint32_t gg, bool first) -> bool {
    const int s = gg % kStages;
    const int b = gg & 1;
    if (!wait_or_abort(c, &sm.p_full[b], (gg >> 1) & 1)) return false;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
      const uint64_t a = smem_desc_sw128(p0 + b * kPBytes + kk * 32, 16, 1024);
      const uint64_t v = smem_desc_sw128(kv0 + s * kStageBytes + kk * 2048, kBlkBytes, 1024);
      mma_ss(tmem + TM_O, a, v, IDESC_PV, (first && kk == 0) ? 0u : 1u);
    }
    mma_commit(smem_u32(&sm.kv_empty[s]));
    mma_commit(smem_u32(&sm.p_empty[b]));
    mma_commit(smem_u32(&sm.o_done));
    return true;
  };
  for_each_piece(p, c.part, [&](int, const Item &, int t0, int t1, int, bool empty) {
    if (empty) return true;
    if (!wait_or_abort(c, &sm.q_ready, qn & 1)) return false;
    qn++;
    tc_fence_after();
    const uint32_t gfirst = g;
    for (int tile = t0; tile < t1; tile++, g++) {
      const int s = g % kStages;
      if (!wait_or_abort(c, &sm.kv_full[s], (g / kStages) & 1)) return false;
      if (!wait_or_abort(c, &sm.s_free, (g & 1) ^ 1)) return false;
      tc_fence_after();
      const uint32_t kvs = kv0 + s * kStageBytes;
      for (int kb = 0; kb < c.nblk; kb++) {
#pragma unroll
        for (int kk = 0; kk < 4; kk++) {
          const uint64_t kd = smem_desc_sw128(kvs + kb * kBlkBytes + kk * 32, 16, 1024);
          mma_ts(tmem + TM_S, tmem + TM_Q + kb * 32 + kk * 8, kd, IDESC_QK, (kb | kk) != 0 ? 1u : 0u);
        }
      }
      mma_commit(smem_u32(&sm.s_full));
      if (g > gfirst && !issue_pv(g - 1, g - 1 == gfirst)) return false;
    }
    return issue_pv(g - 1, g - 1 == gfirst);
  });
}

// ---- softmax / epilogue (warps 4-7, thread = query row = TMEM lane) ---------------

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Query row r (this CTA's dims) -> TMEM columns TM_Q.. as bf16 pairs.
__device__ __forceinline__ void load_q(const Ctx &c, uint32_t lane_tmem, const Item &it, int r,
                                       bool row_ok) {
  const DecodeParams &p = *c.p;
  const int R = it.row0 + (row_ok ? r : 0);
  const int t = R / p.H, h = R % p.H;
  const uint4 *src = reinterpret_cast<const uint4 *>(p.q + (((size_t)it.b * p.T + t) * p.H + h) * D_QK);
  for (int kb = 0; kb < c.nblk; kb++) {
    const int d0 = block_dim(c.rank, kb);  // 64 dims = 8 x 16 B
    uint32_t v[32];
#pragma unroll
    for (int j = 0; j < 8; j++) {
      uint4 x = row_ok ? __ldg(src + d0 / 8 + j) : make_uint4(0, 0, 0, 0);
      v[4 * j] = x.x;
      v[4 * j + 1] = x.y;
      v[4 * j + 2] = x.z;
      v[4 * j + 3] = x.w;
    }
    tmem_st32(lane_tmem + TM_Q + kb * 32, v);
  }
  tmem_wait_st();
}

__device__ void softmax_role(const Ctx &c, uint32_t tmem, int q, int lane) {
  const DecodeParams &p = *c.p;
  Smem &sm = *c.sm;
  const int r = q * 32 + lane;
  const uint32_t lt = tmem + ((uint32_t)(q * 32) << 16);
  const uint32_t xch_peer = mapa(smem_u32(&sm.xch[0][0]), c.peer);
  const uint32_t xfull_peer = mapa(smem_u32(&sm.xch_full[0]), c.peer);
  const uint32_t pfree_peer = mapa(smem_u32(&sm.peer_free[0]), c.peer);
  const uint32_t xch_mine = smem_u32(&sm.xch[0][0]);
  const uint32_t p_mine = smem_u32(&sm.p[0][0]);
  const int sw = r & 7;
  uint32_t g = 0;
  for_each_piece(p, c.part, [&](int idx, const Item &it, int t0, int t1, int piece, bool empty) {
    const bool row_ok = r < it.rows;
    const int R = it.row0 + (row_ok ? r : 0);
    const int t = R / p.H, h = R % p.H;
    const int nsplit = p.num_splits[idx + 1] - p.num_splits[idx];
    const size_t slot = (size_t)p.num_splits[idx] + piece;
    __nv_bfloat16 *orow = p.out + (((size_t)it.b * p.T + t) * p.H + h) * D_V + c.rank * 256;
    if (empty) {  // no key at all: O = 0, LSE = -inf
      if (row_ok) {
        uint4 *o4 = reinterpret_cast<uint4 *>(orow);
        for (int j = 0; j < 32; j++) o4[j] = make_uint4(0, 0, 0, 0);
        if (c.rank == 0) p.lse[((size_t)it.b * p.H + h) * p.T + t] = -INFINITY;
      }
      return true;
    }
    load_q(c, lt, it, r, row_ok);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm.q_ready));
    const int sk = clamp_seqlen(p.seqlens[it.b], p.status);
    const int my_len = (p.topk_len > 0) ? 0x7fffffff : row_kv_len(sk, p.T, t, p.causal);
    float m_ref = -INFINITY, l = 0.f;
    for (int tile = t0; tile < t1; tile++, g++) {
      const int s = g % kStages;
      const int b = g & 1;
      const uint32_t u = g >> 1;
      // 1. own partial S -> registers, release the S columns
      if (!wait_or_abort(c, &sm.s_full, g & 1)) return false;
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld32(lt + TM_S, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(lt + TM_S + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.s_free));
      // 2. swap partial S with the peer CTA
      if (!wait_cluster_or_abort(c, &sm.peer_free[b], (u & 1) ^ 1)) return false;
      {
        const uint32_t dst = xch_peer + b * kXchBytes + r * 256;
        const uint32_t bar = xfull_peer + b * 8;
#pragma unroll
        for (int j = 0; j < 16; j++)
          st_async_v4(dst + ((j ^ sw) << 4), make_uint4(sr[4 * j], sr[4 * j + 1], sr[4 * j + 2], sr[4 * j + 3]),
                      bar);
      }
      if (lane == 0) mbar_arrive_expect_tx(smem_u32(&sm.xch_full[b]), 32 * 256);
      if (!wait_cluster_or_abort(c, &sm.xch_full[b], u & 1)) return false;
      float sv[64];
      {
        const uint32_t src = xch_mine + b * kXchBytes + r * 256;
#pragma unroll
        for (int j = 0; j < 16; j++) {
          const uint4 v = ld_shared_v4(src + ((j ^ sw) << 4));
          sv[4 * j] = __uint_as_float(sr[4 * j]) + __uint_as_float(v.x);
          sv[4 * j + 1] = __uint_as_float(sr[4 * j + 1]) + __uint_as_float(v.y);
          sv[4 * j + 2] = __uint_as_float(sr[4 * j + 2]) + __uint_as_float(v.z);
          sv[4 * j + 3] = __uint_as_float(sr[4 * j + 3]) + __uint_as_float(v.w);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(pfree_peer + b * 8);
      // 3. mask, scale, running max
      if (!wait_or_abort(c, &sm.kv_full[s], (g / kStages) & 1)) return false;
      uint64_t mk = (uint64_t)sm.mask[s][0] | ((uint64_t)sm.mask[s][1] << 32);
      const int lim = my_len - tile * PAGE;
      if (lim <= 0) mk = 0;
      else if (lim < 64) mk &= (1ull << lim) - 1ull;
      float mt = -INFINITY;
#pragma unroll
      for (int n = 0; n < 64; n++) {
        sv[n] = ((mk >> n) & 1ull) ? sv[n] * p.scale_log2 : -INFINITY;
        mt = fmaxf(mt, sv[n]);
      }
      bool resc = false;
      float alpha = 1.f;
      if (mt > m_ref + kRescaleThreshold) {
        if (m_ref != -INFINITY) {
          alpha = exp2f(m_ref - mt);
          resc = true;
        }
        m_ref = mt;
        l *= alpha;
      }
      // 4. P = 2^(s - m_ref) -> bf16 row of the P buffer (128-byte swizzle)
      if (!wait_or_abort(c, &sm.p_empty[b], (u & 1) ^ 1)) return false;
      float psum = 0.f;
      const bool live = m_ref != -INFINITY;
      const uint32_t prow = p_mine + b * kPBytes + r * 128;
#pragma unroll
      for (int ch = 0; ch < 8; ch++) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int n = ch * 8 + 2 * e;
          const float p0 = (live && sv[n] != -INFINITY) ? exp2f(sv[n] - m_ref) : 0.f;
          const float p1 = (live && sv[n + 1] != -INFINITY) ? exp2f(sv[n + 1] - m_ref) : 0.f;
          psum += p0 + p1;
          w[e] = pack_bf16(p0, p1);
        }
        st_shared_v4(prow + ((ch ^ sw) << 4), make_uint4(w[0], w[1], w[2], w[3]));
      }
      l += psum;
      fence_proxy_async_smem();
      // 5. rare: the reference max moved by more than the threshold -> O *= alpha
      if (__any_sync(0xffffffffu, resc)) {
        if (!wait_or_abort(c, &sm.o_done, (g - 1) & 1)) return false;
        tc_fence_after();
        for (int cc = 0; cc < 8; cc++) {
          uint32_t o[32];
          tmem_ld32(lt + TM_O + cc * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e++) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(lt + TM_O + cc * 32, o);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.p_full[b]));
    }
    // 6. epilogue: O / l (and LSE) for the final output, or the split partial
    if (!wait_or_abort(c, &sm.o_done, (g - 1) & 1)) return false;
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse2 = l > 0.f ? m_ref + log2f(l) : -INFINITY;
    float *wrow = p.ws_o + (slot * M_TILE + r) * D_V + c.rank * 256;
    for (int cc = 0; cc < 8; cc++) {
      uint32_t o[32];
      tmem_ld32(lt + TM_O + cc * 32, o);
      tmem_wait_ld();
      if (!row_ok) continue;
      if (nsplit <= 1) {
        uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 32);
#pragma unroll
        for (int j = 0; j < 4; j++) {
          const int e = 8 * j;
          dst[j] = make_uint4(pack_bf16(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv),
                              pack_bf16(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv),
                              pack_bf16(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv),
                              pack_bf16(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv));
        }
      } else {
        float4 *dst = reinterpret_cast<float4 *>(wrow + cc * 32);
#pragma unroll
        for (int j = 0; j < 8; j++)
          dst[j] = make_float4(__uint_as_float(o[4 * j]) * inv, __uint_as_float(o[4 * j + 1]) * inv,
                               __uint_as_float(o[4 * j + 2]) * inv, __uint_as_float(o[4 * j + 3]) * inv);
      }
    }
    if (row_ok && c.rank == 0) {
      if (nsplit <= 1)
        p.lse[((size_t)it.b * p.H + h) * p.T + t] = lse2 * LN2;
      else
        p.ws_lse[slot * M_TILE + r] = lse2;
    }
    return true;
  });
}

// ---- kernel ---------------------------------------------------------------------

template <bool kGather>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw + pad);
  const uint32_t rank = cluster_ctarank();
  const Ctx c{&p, &sm, rank, rank ^ 1u, rank == 0 ? 5 : 4, (int)cluster_id_x()};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(smem_u32(&sm.kv_full[s]), kGather ? kProducers : 1);
      mbar_init(smem_u32(&sm.kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&sm.s_full), 1);
    mbar_init(smem_u32(&sm.s_free), 4);
    mbar_init(smem_u32(&sm.o_done), 1);
    mbar_init(smem_u32(&sm.q_ready), 4);
    for (int b = 0; b < 2; b++) {
      mbar_init(smem_u32(&sm.p_full[b]), 4);
      mbar_init(smem_u32(&sm.p_empty[b]), 1);
      mbar_init(smem_u32(&sm.xch_full[b]), 4);
      mbar_init(smem_u32(&sm.peer_free[b]), 4);
    }
    sm.abort = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), TM_COLS);
    tmem_relinquish();
  }
  if (!kGather && threadIdx.x == 0) prefetch_tensormap(&kv_map);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote arrive / st.async
  const uint32_t tmem = sm.tmem_base;

  if (kGather) {
    if (warp == 0 || warp == 2 || warp == 3) producer_gather(c, warp == 0 ? lane : (warp - 1) * 32 + lane);
  } else if (warp == 0 && lane == 0) {
    producer_tma(c, &kv_map);
  }
  if (warp == 1 && lane == 0) mma_issuer(c, tmem);
  if (warp >= 4) softmax_role(c, tmem, warp - 4, lane);

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (sm.abort) {  // a bounded wait gave up: let copies / MMAs in flight drain
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 2000000ull) {
    }
  }
  cluster_sync();  // the peer no longer writes into this CTA's shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void *f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, cudaStream_t stream, cudaEvent_t ev_before,
                          cudaEvent_t ev_after) {
  const bool gather = p.kv_format != MLA_KV_BF16 || p.topk_len > 0;
  CUtensorMap map;
  memset(&map, 0, sizeof map);
  if (!gather) {
    // The page pool as a 3-D tensor [num_pages][64 tokens][576 dims] of
    // bf16; one box = 64 dims x 64 tokens of one page, 128-byte swizzle.
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {(cuuint64_t)D_QK, (cuuint64_t)PAGE, (cuuint64_t)p.num_pages};
    cuuint64_t strides[2] = {(cuuint64_t)D_QK * 2, (cuuint64_t)D_QK * 2 * PAGE};
    cuuint32_t box[3] = {64, (cuuint32_t)PAGE, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint8_t *>(p.kv), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  const size_t smem = sizeof(Smem) + 1024;
  auto kern = gather ? decode_tc_kernel<true> : decode_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(2 * p.num_parts);
  if (ev_before) cudaEventRecord(ev_before, stream);
  kern<<<grid, kThreads, smem, stream>>>(map, p);
  e = cudaGetLastError();
  if (ev_after) cudaEventRecord(ev_after, stream);
  return e;
}

}  // namespace mla
