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
  uint64_t s_full, s_free, p_full, o_done, q_ready;
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
