// MLA decode on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// One worker of the split-KV partition = one cluster of two CTAs (a pair of
// SMs).  Heads are packed into the MMA M dimension (STAGE_D2.md "Strategy A":
// Q reshaped to (T*n_h, d), one M tile of 128 query rows, row = t*H + h), so
// each 64-token key tile is read from HBM once per (item, split) for all
// heads.  A 128 x 512 fp32 O accumulator fills all of one SM's tensor memory,
// so the two CTAs of the pair split the work by stage rather than by data:
//
//   rank 0 ("S engine"): S = Q K^T over all 576 dims (the RoPE block is just
//          one more block of the reduction, FlashMLA issue #169 "dual gemm"),
//          Q resident in TMEM as the A operand, S double-buffered in TMEM;
//          the online softmax (conditional rescaling); P in bf16 plus the
//          per-row rescale factors go to rank 1.
//   rank 1 ("O engine"): O (+)= P V over the 512 latent dims, O resident in
//          TMEM; applies the rare O rescales; normalises and writes O.
//
// Only P crosses between the SMs, never a partial S.  P travels through L2:
// the softmax threads of rank 0 write P and the per-row rescale factors into
// a small per-worker ring in the workspace, and rank 1 bulk-copies each slot
// into shared memory.  P is stored chunk-major, [8 chunks of 8 tokens][128
// rows][16 bytes], so each warp store covers 512 contiguous bytes, and that
// same image is the A operand of rank 1's MMA (K-major, no swizzle: core
// matrices of 8 rows x 16 bytes, 2048 bytes apart along K, 128 along M).  The direct SM-to-SM
// path (DSMEM) is several times narrower than that per SM.
//
// Per CTA, 384 threads:
//   warp 0      producer: TMA of the page (rank 0: all 9 column blocks, with
//               an L2 prefetch of the page PF tiles ahead; rank 1: the 8 V
//               blocks), or with warp 3 the row gather / FP8 dequantisation
//   warp 1      TMEM allocation and the MMA-issuing thread
//   warp 2      rank 0: publishes written P slots to rank 1;
//               rank 1: P loader (ring slot -> shared memory)
//   warps 4-11  rank 0: softmax, two threads per query row (TMEM lane):
//               warps 4-7 take tokens 0-31 of each tile, warps 8-11 32-63
//               rank 1: O rescale and epilogue, warps 4-7 on O columns
//               0-255, warps 8-11 on 256-511
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <cstring>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kThreads = 384;
constexpr int kSoftmaxWarps = 8;
constexpr int kBlkBytes = PAGE * 128;             // 64 tokens x 64 dims bf16, 128-byte swizzle
constexpr int kStages0 = 3;                       // rank 0: K stages of 9 blocks
constexpr int kStages1 = 3;                       // rank 1: V stages of 8 blocks
constexpr int kStage0Bytes = 9 * kBlkBytes;       // 73728
constexpr int kStage1Bytes = 8 * kBlkBytes;       // 65536
constexpr int kPBytes = M_TILE * 128;             // P tile: 128 rows x 64 tokens bf16
constexpr int kMetaBytes = 1056;                  // alpha[128], ell[128], flags[8]
constexpr int kSlotBytes = kPBytes + kMetaBytes;  // one P message (P_SLOT_BYTES apart)
static_assert(kSlotBytes <= P_SLOT_BYTES, "P ring slot");
constexpr int kMaskRing = 8;
constexpr int kPrefetch = 3;                      // rank 0: L2 prefetch distance (tiles)
constexpr uint64_t kWaitNs = 2000000000ull;       // bounded waits: 2 s
constexpr float kRescaleThreshold = 8.0f;         // log2 units

// shared memory map (byte offsets from a 1024-aligned base)
constexpr uint32_t OFF_KV = 0;
constexpr uint32_t OFF_RCV_P = kStages1 * kStage1Bytes;            // rank 1: 196608
constexpr uint32_t OFF_RCV_META = OFF_RCV_P + 2 * kPBytes;         // rank 1: 229376
constexpr uint32_t OFF_BARS = OFF_RCV_META + 2 * kMetaBytes;       // 231488
constexpr uint32_t OFF_LPART = kStages0 * kStage0Bytes;            // rank 0: float[2][128]

// TMEM columns
constexpr uint32_t TM_Q = 0;      // rank 0: 288 columns (576 bf16 per row)
constexpr uint32_t TM_S = 320;    // rank 0: two S buffers of 64 columns (64-aligned)
constexpr uint32_t TM_O = 0;      // rank 1: 512 columns
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 256, false, true);

struct Bars {
  uint64_t kv_full[3], kv_empty[3];
  uint64_t s_full[2], s_free[2];
  uint64_t mfull[kMaskRing];
  uint64_t gfree[P_RING];   // rank 0: ring slot copied out by rank 1
  uint64_t pwritten[P_RING];// rank 0: the 8 softmax warps wrote ring slot
  uint64_t q_ready;
  uint64_t p_full[P_RING];  // rank 1: ring slot published by rank 0
  uint64_t p_land[2];       // rank 1: slot copied into shared buffer b
  uint64_t p_empty[2];
  // O updates, per P buffer: the epilogue warps can run up to two tiles ahead
  // of the PV MMAs, so a single barrier could be two phases behind a waiter
  uint64_t o_done[2];
  uint64_t o_ready[2];   // per P buffer, so a phase can never run two ahead
  uint32_t mask[kMaskRing][2];
  uint32_t tmem_base;
  int abort;
};
static_assert(OFF_BARS + sizeof(Bars) <= 232448, "shared memory budget");
static_assert(OFF_LPART + 2 * M_TILE * 4 <= OFF_BARS, "rank 0 map");
static_assert(OFF_RCV_P % 1024 == 0, "P tiles need 1024-byte alignment");

struct Meta {
  float alpha[M_TILE];
  float ell[M_TILE];
  uint32_t flags[kSoftmaxWarps];  // per softmax warp: any row rescaled in this tile
};
static_assert(sizeof(Meta) == kMetaBytes, "meta size");

struct Ctx {
  const DecodeParams *p;
  uint8_t *base;   // shared memory base (1024-aligned)
  Bars *bars;
  uint32_t rank;
  int part;
};

__device__ __forceinline__ bool wait_or_abort(const Ctx &c, uint64_t *bar, uint32_t parity) {
  if (mbar_wait<false>(smem_u32(bar), parity, &c.bars->abort, kWaitNs)) return true;
  atomicOr(c.p->status, MLA_STATUS_WAIT_TIMEOUT);
  c.bars->abort = 1;
  return false;
}

__device__ __forceinline__ bool wait_cluster_or_abort(const Ctx &c, uint64_t *bar, uint32_t parity) {
  if (mbar_wait<true>(smem_u32(bar), parity, &c.bars->abort, kWaitNs)) return true;
  atomicOr(c.p->status, MLA_STATUS_WAIT_TIMEOUT);
  c.bars->abort = 1;
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

// Page of key tile `tile` of sequence b, or -1 (status bit set) if the
// block table entry is outside the pool.
__device__ __forceinline__ int page_of(const DecodeParams &p, int b, int tile) {
  if (tile >= p.max_pages) {
    atomicOr(p.status, MLA_STATUS_BAD_SEQLEN);
    return -1;
  }
  const int page = __ldg(p.block_table + (size_t)b * p.max_pages + tile);
  if (page < 0 || page >= p.num_pages) {
    atomicOr(p.status, MLA_STATUS_BAD_PAGE);
    return -1;
  }
  return page;
}

__device__ __forceinline__ void prefetch_l2_bulk(const void *gaddr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(gaddr)), "r"(bytes)
               : "memory");
}

// ---- producer: TMA of whole pages ------------------------------------------------
//
// rank 0 loads all 576 dims (9 blocks) of each page into a 2-stage ring and
// prefetches the page kPrefetch tiles ahead into L2; it also publishes the
// validity mask of each tile.  rank 1 loads the 512 V dims (8 blocks) into a
// 3-stage ring.

__device__ void producer_tma(const Ctx &c, const CUtensorMap *map) {
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  // rank 1 is the last reader of each page
  const uint64_t pol = c.rank == 0 ? policy_evict_normal() : policy_evict_first();
  const int nstage = c.rank == 0 ? kStages0 : kStages1;
  const int nblk = c.rank == 0 ? 9 : 8;
  const uint32_t stage_bytes = c.rank == 0 ? kStage0Bytes : kStage1Bytes;
  const uint32_t kv0 = smem_u32(c.base + OFF_KV);
  uint32_t g = 0;
  for_each_piece(p, c.part, [&](int, const Item &it, int t0, int t1, int, bool empty) {
    if (empty) return true;
    if (c.rank == 0) {
      for (int k = 0; k < kPrefetch && t0 + k < t1; k++) {
        const int pg = (t0 + k < p.max_pages) ? __ldg(p.block_table + (size_t)it.b * p.max_pages + t0 + k) : -1;
        if (pg >= 0 && pg < p.num_pages)
          prefetch_l2_bulk(p.kv + (size_t)pg * PAGE * D_QK * 2, PAGE * D_QK * 2);
      }
    }
    for (int tile = t0; tile < t1; tile++, g++) {
      const uint32_t s = g % nstage;
      if (!wait_or_abort(c, &br.kv_empty[s], ((g / nstage) & 1) ^ 1)) return false;
      const int page = page_of(p, it.b, tile);
      if (c.rank == 0) {
        const int ahead = tile + kPrefetch;
        if (ahead < t1) {
          const int pg = (ahead < p.max_pages) ? __ldg(p.block_table + (size_t)it.b * p.max_pages + ahead) : -1;
          if (pg >= 0 && pg < p.num_pages)
            prefetch_l2_bulk(p.kv + (size_t)pg * PAGE * D_QK * 2, PAGE * D_QK * 2);
        }
        const int nvalid = min(PAGE, it.kv_len - tile * PAGE);
        uint64_t m = 0;
        if (page >= 0) m = nvalid >= 64 ? ~0ull : ((1ull << nvalid) - 1ull);
        const uint32_t mi = g % kMaskRing;
        br.mask[mi][0] = (uint32_t)m;
        br.mask[mi][1] = (uint32_t)(m >> 32);
        mbar_arrive(smem_u32(&br.mfull[mi]));
      }
      const uint32_t bar = smem_u32(&br.kv_full[s]);
      mbar_arrive_expect_tx(bar, (uint32_t)nblk * kBlkBytes);
      const uint32_t dst = kv0 + s * stage_bytes;
      for (int kb = 0; kb < nblk; kb++)
        tma_load_3d(dst + kb * kBlkBytes, map, bar, kb * 64, 0, page < 0 ? 0 : page, pol);
    }
    return true;
  });
}

// ---- producer: row gather / FP8 dequantisation (warps 0 and 3) --------------------

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

constexpr int kGatherThreads = 64;

// Thread pi (0..63) of the gather warps owns row pi of every tile: it
// resolves the row (top-k index or position, block table, bounds checks),
// loads it with 16-byte loads and writes it, dequantised to bf16, into the
// CTA's column blocks of the stage.
__device__ void producer_gather(const Ctx &c, int pi) {
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  const bool fp8 = p.kv_format == MLA_KV_FP8_E4M3;
  const int nstage = c.rank == 0 ? kStages0 : kStages1;
  const uint32_t stage_bytes = c.rank == 0 ? kStage0Bytes : kStage1Bytes;
  const uint32_t kv0 = smem_u32(c.base + OFF_KV);
  const int sw = pi & 7;
  uint32_t g = 0;
  for_each_piece(p, c.part, [&](int idx, const Item &it, int t0, int t1, int, bool empty) {
    if (empty) return true;
    const int t_item = (p.topk_len > 0) ? (idx % p.T) : 0;
    const int sk = clamp_seqlen(p.seqlens[it.b], p.status);
    for (int tile = t0; tile < t1; tile++, g++) {
      const uint32_t s = g % nstage;
      if (!wait_or_abort(c, &br.kv_empty[s], ((g / nstage) & 1) ^ 1)) return false;
      int n = -1;
      if (p.topk_len > 0) {
        const int slot = tile * PAGE + pi;
        if (slot < p.topk_len) {
          int id = __ldg(p.topk + ((size_t)it.b * p.T + t_item) * p.topk_len + slot);
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
      size_t row = 0;
      bool ok = false;
      if (n >= 0) {
        const int pg = page_of(p, it.b, n / PAGE);
        if (pg < 0) {
          n = -1;
        } else {
          row = (size_t)pg * PAGE + (n % PAGE);
          ok = true;
        }
      }
      const uint32_t bits = __ballot_sync(0xffffffffu, ok);
      if (c.rank == 0) {
        const uint32_t mi = g % kMaskRing;
        if ((pi & 31) == 0) br.mask[mi][pi >> 5] = bits;
        if (p.gathered != nullptr && p.topk_len > 0) {
          const int slot = tile * PAGE + pi;
          if (slot < p.topk_len) p.gathered[((size_t)it.b * p.T + t_item) * p.topk_len + slot] = n;
        }
      }
      const uint32_t dst = kv0 + s * stage_bytes + pi * 128;
      if (fp8) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.kv + row * FP8_ROW);
        const float *sc = p.kv_scales + row * 4;
        // 512 e4m3 values = 32 chunks of 16 -> 64 bf16 chunks in blocks 0..7
#pragma unroll 2
        for (int q8 = 0; q8 < 4; q8++) {
          uint4 v[8];
#pragma unroll
          for (int j = 0; j < 8; j++) v[j] = ok ? __ldg(src + q8 * 8 + j) : make_uint4(0, 0, 0, 0);
          const float scale = ok ? __ldg(sc + q8) : 0.f;
#pragma unroll
          for (int j = 0; j < 8; j++) {
            uint4 lo, hi;
            dequant16(v[j], scale, lo, hi);
            const int u = q8 * 8 + j;             // dims 16u .. 16u+15
            const int kb = u / 4, ch = 2 * (u % 4);
            st_shared_v4(dst + kb * kBlkBytes + ((ch ^ sw) << 4), lo);
            st_shared_v4(dst + kb * kBlkBytes + (((ch + 1) ^ sw) << 4), hi);
          }
        }
        if (c.rank == 0) {  // RoPE: 64 bf16 after the 512 e4m3 bytes -> block 8
          uint4 v[8];
#pragma unroll
          for (int j = 0; j < 8; j++) v[j] = ok ? __ldg(src + 32 + j) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int j = 0; j < 8; j++) st_shared_v4(dst + 8 * kBlkBytes + ((j ^ sw) << 4), v[j]);
        }
      } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.kv + row * (D_QK * 2));
        const int nb = c.rank == 0 ? 9 : 8;
        for (int kb = 0; kb < nb; kb++) {
          uint4 v[8];
#pragma unroll
          for (int j = 0; j < 8; j++) v[j] = ok ? __ldg(src + kb * 8 + j) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int j = 0; j < 8; j++) st_shared_v4(dst + kb * kBlkBytes + ((j ^ sw) << 4), v[j]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&br.kv_full[s]));
      if (c.rank == 0) {
        __syncwarp();
        if ((pi & 31) == 0) mbar_arrive(smem_u32(&br.mfull[g % kMaskRing]));
      }
    }
    return true;
  });
}

// ---- rank 0: QK MMA issuer ----------------------------------------------------------
//
// Per tile g: S[g&1] = Q . K^T (M=128, N=64 tokens, K=576 in 36 steps of 16;
// A = Q from TMEM, B = the K-major swizzled key blocks), commit -> s_full,
// kv_empty.  S is double-buffered, so QK(g+1) overlaps the softmax of g.

__device__ void mma_qk(const Ctx &c, uint32_t tmem) {
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  const uint32_t kv0 = smem_u32(c.base + OFF_KV);
  uint32_t g = 0, qn = 0;
  for_each_piece(p, c.part, [&](int, const Item &, int t0, int t1, int, bool empty) {
    if (empty) return true;
    if (!wait_or_abort(c, &br.q_ready, qn & 1)) return false;
    qn++;
    tc_fence_after();
    for (int tile = t0; tile < t1; tile++, g++) {
      const uint32_t s = g % kStages0, b = g & 1, u = g >> 1;
      if (!wait_or_abort(c, &br.kv_full[s], (g / kStages0) & 1)) return false;
      if (!wait_or_abort(c, &br.s_free[b], (u & 1) ^ 1)) return false;
      tc_fence_after();
      // One base descriptor per tile; block kb / step kk only move its
      // start-address field (16-byte units: 512 per 8 KB block, 2 per 32 B),
      // which stays below 2^14 for every address of the shared map.
      const uint64_t kd0 = smem_desc_sw128(kv0 + s * kStage0Bytes, 16, 1024);
      const uint32_t d = tmem + TM_S + b * 64;
      mma_ts(d, tmem + TM_Q, kd0, IDESC_QK, 0u);
#pragma unroll
      for (int i = 1; i < 36; i++) {
        const int kb = i >> 2, kk = i & 3;
        mma_ts(d, tmem + TM_Q + kb * 32 + kk * 8, kd0 + (uint64_t)(kb * 512 + kk * 2), IDESC_QK, 1u);
      }
      mma_commit(smem_u32(&br.s_full[b]));
      mma_commit(smem_u32(&br.kv_empty[s]));
    }
    return true;
  });
}

// ---- rank 1: PV MMA issuer ----------------------------------------------------------
//
// Per tile g: O[:, 0:256) and O[:, 256:512) (+)= P(g) . V(g) (M=128, N=256,
// K=64 tokens in 4 steps; A = P from shared memory, K-major; B = the V
// blocks of the stage read MN-major).  The first tile of a piece overwrites
// O.  Waits for the epilogue warps' o_ready (rescale applied / previous
// piece read out).

__device__ void mma_pv(const Ctx &c, uint32_t tmem) {
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  const uint32_t kv0 = smem_u32(c.base + OFF_KV);
  const uint32_t pbuf = smem_u32(c.base + OFF_RCV_P);
  uint32_t g = 0;
  for_each_piece(p, c.part, [&](int, const Item &, int t0, int t1, int, bool empty) {
    if (empty) return true;
    const uint32_t gfirst = g;
    for (int tile = t0; tile < t1; tile++, g++) {
      const uint32_t s = g % kStages1, b = g & 1, u = g >> 1;
      if (!wait_or_abort(c, &br.kv_full[s], (g / kStages1) & 1)) return false;
      if (!wait_or_abort(c, &br.p_land[b], u & 1)) return false;
      if (!wait_or_abort(c, &br.o_ready[b], u & 1)) return false;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; kk++) {
        const uint64_t a = smem_desc_noswz(pbuf + b * kPBytes + kk * 2 * 2048, 2048, 128);
#pragma unroll
        for (int nh = 0; nh < 2; nh++) {
          const uint64_t v = smem_desc_sw128(kv0 + s * kStage1Bytes + nh * 4 * kBlkBytes + kk * 2048, kBlkBytes, 1024);
          mma_ss(tmem + TM_O + nh * 256, a, v, IDESC_PV, (g == gfirst && kk == 0) ? 0u : 1u);
        }
      }
      mma_commit(smem_u32(&br.kv_empty[s]));
      mma_commit(smem_u32(&br.p_empty[b]));
      mma_commit(smem_u32(&br.o_done[b]));
    }
    return true;
  });
}

// ---- rank 1: P loader ----------------------------------------------------------------
//
// Per tile g: wait for rank 0's four softmax warps to have written ring slot
// g % P_RING, and for shared buffer g & 1 to be free (PV(g-2) done); bulk
// copy the slot (P tile + meta) into the buffer; once it has landed, hand the
// slot back to rank 0.

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ const uint8_t *ring_slot(const DecodeParams &p, int part, uint32_t g) {
  return p.ws_p + ((size_t)part * P_RING + (g % P_RING)) * P_SLOT_BYTES;
}

__device__ void p_loader(const Ctx &c) {
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  const uint32_t rcv_p = smem_u32(c.base + OFF_RCV_P), rcv_m = smem_u32(c.base + OFF_RCV_META);
  const uint32_t gfree0 = mapa(smem_u32(&br.gfree[0]), 0);
  uint32_t g = 0;
  for_each_piece(p, c.part, [&](int, const Item &, int t0, int t1, int, bool empty) {
    if (empty) return true;
    for (int tile = t0; tile < t1; tile++, g++) {
      const uint32_t b = g & 1, u = g >> 1, gs = g % P_RING;
      if (!wait_cluster_or_abort(c, &br.p_full[gs], (g / P_RING) & 1)) return false;
      if (!wait_or_abort(c, &br.p_empty[b], (u & 1) ^ 1)) return false;
      fence_proxy_async_global();
      const uint8_t *slot = ring_slot(p, c.part, g);
      const uint32_t land = smem_u32(&br.p_land[b]);
      mbar_arrive_expect_tx(land, kSlotBytes);
      bulk_g2s(rcv_p + b * kPBytes, slot, kPBytes, land);
      bulk_g2s(rcv_m + b * kMetaBytes, slot + kPBytes, kMetaBytes, land);
      if (!wait_or_abort(c, &br.p_land[b], u & 1)) return false;
      mbar_arrive_remote(gfree0 + gs * 8);
    }
    return true;
  });
}

// ---- rank 0: softmax (warps 4-7, thread = query row = TMEM lane) -------------------------

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

struct RowInfo {
  bool ok;
  int t, h;
  int nsplit;
  size_t slot;
};

__device__ __forceinline__ RowInfo row_info(const DecodeParams &p, int idx, const Item &it, int piece, int r) {
  RowInfo ri;
  ri.ok = r < it.rows;
  const int R = it.row0 + (ri.ok ? r : 0);
  ri.t = R / p.H;
  ri.h = R % p.H;
  ri.nsplit = p.num_splits[idx + 1] - p.num_splits[idx];
  ri.slot = (size_t)p.num_splits[idx] + piece;
  return ri;
}

// Query row r, column blocks [kb0, kb1) of its 576 dims -> TMEM columns
// TM_Q + 32*kb.. (bf16 pairs).
__device__ __forceinline__ void load_q(const DecodeParams &p, uint32_t lane_tmem, const Item &it,
                                       const RowInfo &ri, int kb0, int kb1) {
  const uint4 *src = reinterpret_cast<const uint4 *>(p.q + (((size_t)it.b * p.T + ri.t) * p.H + ri.h) * D_QK);
  for (int kb = kb0; kb < kb1; kb++) {
    uint32_t v[32];
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const uint4 x = ri.ok ? __ldg(src + kb * 8 + j) : make_uint4(0, 0, 0, 0);
      v[4 * j] = x.x;
      v[4 * j + 1] = x.y;
      v[4 * j + 2] = x.z;
      v[4 * j + 3] = x.w;
    }
    tmem_st32(lane_tmem + TM_Q + kb * 32, v);
  }
  tmem_wait_st();
}

// Thread (q, hf) of warp w = 4 + 4*hf + q owns query row r = 32q + lane and
// tokens [32*hf, 32*hf + 32) of each tile.  Both threads of a row read all 64
// scores, so they reach the same running max and rescale decisions without
// talking to each other; each exponentiates and publishes its own 32 tokens
// and keeps its own part of the row sum.  The halves of the row sum meet in
// shared memory at the last tile of a piece.
__device__ void softmax_role(const Ctx &c, uint32_t tmem, int w, int lane) {
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  const int q = w & 3, hf = (w - 4) >> 2;
  const int r = q * 32 + lane;
  const uint32_t lt = tmem + ((uint32_t)(q * 32) << 16);
  float *lpart = reinterpret_cast<float *>(c.base + OFF_LPART);  // [2 pieces][2 halves][128]
  const float cs = p.scale_log2;
  uint32_t g = 0, pc = 0;
  for_each_piece(p, c.part, [&](int idx, const Item &it, int t0, int t1, int piece, bool empty) {
    const RowInfo ri = row_info(p, idx, it, piece, r);
    float *lse_dst = p.lse + ((size_t)it.b * p.H + ri.h) * p.T + ri.t;
    if (empty) {  // no key: LSE = -inf (rank 1 writes O = 0)
      if (ri.ok && hf == 0) *lse_dst = -INFINITY;
      return true;
    }
    load_q(p, lt, it, ri, hf ? 5 : 0, hf ? 9 : 5);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&br.q_ready));
    const int sk = clamp_seqlen(p.seqlens[it.b], p.status);
    const int my_len = (p.topk_len > 0) ? 0x7fffffff : row_kv_len(sk, p.T, ri.t, p.causal);
    float m_ref = -INFINITY;  // reference max, raw score units
    float l = 0.f;            // this half's part of the row sum
    float l_all = 0.f;
    for (int tile = t0; tile < t1; tile++, g++) {
      const uint32_t b = g & 1, u = g >> 1, mi = g % kMaskRing;
      // 1. tile validity and this row's 64 scores
      if (!wait_or_abort(c, &br.mfull[mi], (g / kMaskRing) & 1)) return false;
      uint32_t mlo = br.mask[mi][0], mhi = br.mask[mi][1];
      const int lim = my_len - tile * PAGE;
      if (lim < 64) {
        const uint64_t keep = lim <= 0 ? 0ull : ((1ull << lim) - 1ull);
        mlo &= (uint32_t)keep;
        mhi &= (uint32_t)(keep >> 32);
      }
      if (!wait_or_abort(c, &br.s_full[b], u & 1)) return false;
      tc_fence_after();
      float own[32], oth[32];  // this half's 32 scores and the partner half's
      tmem_ld32(lt + TM_S + b * 64 + hf * 32, *reinterpret_cast<uint32_t(*)[32]>(&own[0]));
      tmem_ld32(lt + TM_S + b * 64 + (hf ^ 1) * 32, *reinterpret_cast<uint32_t(*)[32]>(&oth[0]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&br.s_free[b]));
      // 2. mask (skipped for fully valid tiles) and tile max (raw units; the
      //    scale is positive), as a tree
      const uint32_t mown = hf ? mhi : mlo, moth = hf ? mlo : mhi;
      if ((mown & moth) != 0xffffffffu) {
#pragma unroll
        for (int n = 0; n < 32; n++) {
          own[n] = ((mown >> n) & 1u) ? own[n] : -INFINITY;
          oth[n] = ((moth >> n) & 1u) ? oth[n] : -INFINITY;
        }
      }
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; k++)
        mx[k] = fmaxf(fmaxf(fmaxf(own[k], own[k + 8]), fmaxf(own[k + 16], own[k + 24])),
                      fmaxf(fmaxf(oth[k], oth[k + 8]), fmaxf(oth[k + 16], oth[k + 24])));
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      // 3. conditional rescale: move the reference only when the max grew by
      //    more than 2^8 (FlashAttention-4's conditional rescaling)
      float alpha = 1.f;
      bool resc = false;
      if ((mt - m_ref) * cs > kRescaleThreshold) {
        if (m_ref != -INFINITY) {
          alpha = ex2((m_ref - mt) * cs);
          resc = true;
        }
        m_ref = mt;
        l *= alpha;
      }
      const float nb = (m_ref == -INFINITY) ? 0.f : -m_ref * cs;
      // 4. P = 2^(s*c - m_ref*c) for this half's 32 tokens -> bf16 into ring
      //    slot g % P_RING, chunk-major (chunk ch of row r at ch*2048 + r*16)
      const uint32_t gs = g % P_RING;
      if (!wait_cluster_or_abort(c, &br.gfree[gs], ((g / P_RING) & 1) ^ 1)) return false;
      uint8_t *slot = p.ws_p + ((size_t)c.part * P_RING + gs) * P_SLOT_BYTES;
      float psum = 0.f;
#pragma unroll
      for (int cc = 0; cc < 4; cc++) {
        const int ch = hf * 4 + cc;
        uint32_t wv[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const float p0 = ex2(fmaf(own[cc * 8 + 2 * e], cs, nb));
          const float p1 = ex2(fmaf(own[cc * 8 + 2 * e + 1], cs, nb));
          psum += p0 + p1;
          wv[e] = pack_bf16(p0, p1);
        }
        *reinterpret_cast<uint4 *>(slot + ch * 2048 + r * 16) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
      l += psum;
      Meta *mo = reinterpret_cast<Meta *>(slot + kPBytes);
      if (hf == 0) mo->alpha[r] = alpha;
      const bool any = __any_sync(0xffffffffu, resc);
      if (lane == 0) mo->flags[w - 4] = any ? 1u : 0u;
      if (tile == t1 - 1) {  // last tile: both halves of the row sum
        float *lp = lpart + (pc & 1) * 2 * M_TILE;
        lp[hf * M_TILE + r] = l;
        named_bar_sync(1 + q, 64);
        l_all = lp[r] + lp[M_TILE + r];
        if (hf == 0) mo->ell[r] = l_all;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&br.pwritten[gs]));
    }
    pc++;
    // LSE of this piece (final, natural log; or the split partial, base 2)
    if (ri.ok && hf == 0) {
      const float lse2 = l_all > 0.f ? m_ref * cs + __log2f(l_all) : -INFINITY;
      if (ri.nsplit <= 1)
        *lse_dst = lse2 * LN2;
      else
        p.ws_lse[ri.slot * M_TILE + r] = lse2;
    }
    return true;
  });
}

// ---- rank 0: P publisher (one thread) ---------------------------------------------------
//
// Waits until the eight softmax warps have written ring slot g % P_RING,
// makes those writes visible device-wide, and signals rank 1.  Keeping this
// off the softmax warps keeps the store round trip off their critical path.

__device__ void p_publisher(const Ctx &c) {
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  const uint32_t pfull1 = mapa(smem_u32(&br.p_full[0]), 1);
  uint32_t g = 0;
  for_each_piece(p, c.part, [&](int, const Item &, int t0, int t1, int, bool empty) {
    if (empty) return true;
    for (int tile = t0; tile < t1; tile++, g++) {
      const uint32_t gs = g % P_RING;
      if (!wait_or_abort(c, &br.pwritten[gs], (g / P_RING) & 1)) return false;
      __threadfence();
      mbar_arrive_remote(pfull1 + gs * 8);
    }
    return true;
  });
}

// ---- rank 1: O rescale and epilogue (warps 4-11) --------------------------------------------

__device__ void epilogue_role(const Ctx &c, uint32_t tmem, int w, int lane) {
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  const int q = w & 3, hf = (w - 4) >> 2;
  const int r = q * 32 + lane;
  const uint32_t lt = tmem + ((uint32_t)(q * 32) << 16) + TM_O + hf * 256;
  const Meta *rcv_m = reinterpret_cast<const Meta *>(c.base + OFF_RCV_META);
  uint32_t g = 0;
  for_each_piece(p, c.part, [&](int idx, const Item &it, int t0, int t1, int piece, bool empty) {
    const RowInfo ri = row_info(p, idx, it, piece, r);
    __nv_bfloat16 *orow = p.out + (((size_t)it.b * p.T + ri.t) * p.H + ri.h) * D_V + hf * 256;
    if (empty) {
      if (ri.ok) {
        uint4 *o4 = reinterpret_cast<uint4 *>(orow);
        for (int j = 0; j < 32; j++) o4[j] = make_uint4(0, 0, 0, 0);
      }
      return true;
    }
    float ell = 0.f;
    for (int tile = t0; tile < t1; tile++, g++) {
      const uint32_t b = g & 1, u = g >> 1;
      if (!wait_or_abort(c, &br.p_land[b], u & 1)) return false;
      const Meta &m = rcv_m[b];
      uint32_t fl = 0;
#pragma unroll
      for (int k = 0; k < kSoftmaxWarps; k++) fl |= m.flags[k];
      if (tile == t1 - 1) ell = m.ell[r];
      if (fl != 0u) {  // rare: O *= alpha after PV(g-1), before PV(g)
        const float alpha = m.alpha[r];
        if (!wait_or_abort(c, &br.o_done[(g - 1) & 1], ((g - 1) >> 1) & 1)) return false;
        tc_fence_after();
        for (int cc = 0; cc < 8; cc++) {
          uint32_t o[32];
          tmem_ld32(lt + cc * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e++) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(lt + cc * 32, o);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&br.o_ready[b]));
    }
    // O / l for the final output, or the normalised split partial (the
    // commit after the last PV covers every earlier MMA)
    if (!wait_or_abort(c, &br.o_done[(g - 1) & 1], ((g - 1) >> 1) & 1)) return false;
    tc_fence_after();
    const float inv = ell > 0.f ? 1.f / ell : 0.f;
    float *wrow = p.ws_o + (ri.slot * M_TILE + r) * D_V + hf * 256;
    for (int cc = 0; cc < 8; cc++) {
      uint32_t o[32];
      tmem_ld32(lt + cc * 32, o);
      tmem_wait_ld();
      if (!ri.ok) continue;
      if (ri.nsplit <= 1) {
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
    return true;
  });
}

// ---- kernel ---------------------------------------------------------------------

template <bool kGather>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // the shared-memory map needs a 1024-aligned base
    if (threadIdx.x == 0) atomicOr(p.status, MLA_STATUS_WAIT_TIMEOUT);
    return;
  }
  uint8_t *base = smem_raw;
  Bars &br = *reinterpret_cast<Bars *>(base + OFF_BARS);
  const uint32_t rank = cluster_ctarank();
  const Ctx c{&p, base, &br, rank, (int)cluster_id_x()};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 3; s++) {
      mbar_init(smem_u32(&br.kv_full[s]), kGather ? kGatherThreads : 1);
      mbar_init(smem_u32(&br.kv_empty[s]), 1);
    }
    for (int i = 0; i < kMaskRing; i++) mbar_init(smem_u32(&br.mfull[i]), kGather ? 2 : 1);
    for (int i = 0; i < P_RING; i++) {
      mbar_init(smem_u32(&br.gfree[i]), 1);
      mbar_init(smem_u32(&br.pwritten[i]), kSoftmaxWarps);
      mbar_init(smem_u32(&br.p_full[i]), 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(smem_u32(&br.s_full[b]), 1);
      mbar_init(smem_u32(&br.s_free[b]), kSoftmaxWarps);
      mbar_init(smem_u32(&br.p_land[b]), 1);
      mbar_init(smem_u32(&br.p_empty[b]), 1);
      mbar_init(smem_u32(&br.o_ready[b]), kSoftmaxWarps);
      mbar_init(smem_u32(&br.o_done[b]), 1);
    }
    mbar_init(smem_u32(&br.q_ready), kSoftmaxWarps);
    br.abort = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&br.tmem_base), TM_COLS);
    tmem_relinquish();
  }
  if (!kGather && threadIdx.x == 0) prefetch_tensormap(&kv_map);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote arrive or copy
  const uint32_t tmem = br.tmem_base;

  if (kGather) {
    if (warp == 0 || warp == 3) producer_gather(c, warp == 0 ? lane : 32 + lane);
  } else if (warp == 0 && lane == 0) {
    producer_tma(c, &kv_map);
  }
  if (warp == 1 && lane == 0) {
    if (rank == 0) mma_qk(c, tmem);
    else mma_pv(c, tmem);
  }
  if (warp == 2 && lane == 0) {
    if (rank == 0) p_publisher(c);
    else p_loader(c);
  }
  if (warp >= 4) {
    if (rank == 0) softmax_role(c, tmem, warp, lane);
    else epilogue_role(c, tmem, warp, lane);
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (br.abort) {  // a bounded wait gave up: let copies / MMAs in flight drain
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 2000000ull) {
    }
  }
  cluster_sync();  // the peer no longer copies into or arrives on this CTA
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
  const size_t smem = OFF_BARS + sizeof(Bars);
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
