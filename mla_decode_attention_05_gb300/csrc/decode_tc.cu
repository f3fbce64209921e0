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
//          per-row rescale factors go to rank 1, one message per tile.
//   rank 1 ("O engine"): O (+)= P V over the 512 latent dims, O resident in
//          TMEM; applies the rare O rescales; normalises and writes O.
//
// Only P crosses between the SMs, never a partial S.  P travels through L2:
// the softmax threads of rank 0 write P and the per-row rescale factors into
// a small per-worker ring in the workspace, and rank 1's epilogue warps copy
// each slot into shared memory with plain L2 loads.  P is stored chunk-major, [8 chunks of 8 tokens][128
// rows][16 bytes], so each warp store covers 512 contiguous bytes, and that
// same image is the A operand of rank 1's MMA (K-major, no swizzle: core
// matrices of 8 rows x 16 bytes, 2048 bytes apart along K, 128 along M).  The direct SM-to-SM
// path (DSMEM) is several times narrower than that per SM.
//
// Per CTA, 384 threads (480 in the gather kernel):
//   warp 0      producer: one 4-D TMA per page (rank 0: the 9 column blocks
//               into a 3-stage ring; rank 1: the 8 V blocks), or with warps
//               3, 13 and 14 the row gather / FP8 dequantisation into the
//               same layout (with warps 6, 7, 10 and 11 too when every item
//               has at most 64 query rows, since their rows are padding)
//   warp 1      TMEM allocation and the MMA warp (one elected lane issues)
//   warp 2      rank 0: publishes written P slots to rank 1; rank 1: idle
//   warp 3      the MMA warp's waiter (warp 12 in the gather kernel)
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

// 12 warps, 15 in the gather kernel, where warps 0, 3, 13 and 14 gather and
// warp 12 waits for the MMA warp
__host__ __device__ constexpr int threads_of(bool gather) { return gather ? 480 : 384; }
__host__ __device__ constexpr int waiter_warp(bool gather) { return gather ? 12 : 3; }
constexpr int kSoftmaxWarps = 8;
constexpr int kBlkBytes = PAGE * 128;             // 64 tokens x 64 dims bf16, 128-byte swizzle
constexpr int kStages0 = 3;                       // rank 0: K stages of 9 blocks (one page)
constexpr int kStage0Bytes = 9 * kBlkBytes;       // 73728
constexpr int kStages1 = 3;                       // rank 1: V stages of 8 blocks (one page)
constexpr int kStage1Bytes = 8 * kBlkBytes;       // 65536
constexpr int kPBytes = M_TILE * 128;             // P tile: 128 rows x 64 tokens bf16
constexpr int kMetaBytes = 1056;                  // alpha[128], ell[128], flags[8]
constexpr int kSlotBytes = kPBytes + kMetaBytes;  // one P message (P_SLOT_BYTES apart)
static_assert(kSlotBytes <= P_SLOT_BYTES, "P ring slot");
constexpr int kMaskRing = 8;
constexpr int kPublishBatch = 4;                  // P messages published per fence, at most
constexpr float kRescaleThreshold = 8.0f;         // log2 units

// shared memory map (byte offsets from a 1024-aligned base)
constexpr uint32_t OFF_KV = 0;
constexpr uint32_t OFF_XCHG = kStages0 * kStage0Bytes;              // rank 0, dual GEMM: S_b hand-over (8 KB)
// The row-gather kernel keeps two K / V stages and, in the memory of the
// third, a ring of two raw slots for the FP8 rows of the next tiles.
__host__ __device__ constexpr int ring_stages(bool gather) { return gather ? 2 : 3; }
constexpr uint32_t OFF_RAW0 = 2 * kStage0Bytes;                     // gather, rank 0: 2 x 64 rows x 640 bytes
constexpr uint32_t OFF_RAW1 = 2 * kStage1Bytes;                     // gather, rank 1: 2 x 64 rows x 512 bytes
constexpr uint32_t kRawSlot0 = PAGE * FP8_ROW;
constexpr uint32_t kRawSlot1 = PAGE * 512;
constexpr uint32_t OFF_RCV_P = kStages1 * kStage1Bytes;             // rank 1: 196608
constexpr uint32_t OFF_BARS = OFF_RCV_P + 2 * kPBytes;              // 229376
constexpr uint32_t kXchgBytes = 64 * 32 * 4;                         // 64 rows x 32 scores

// TMEM columns
constexpr uint32_t TM_Q = 0;      // rank 0: 288 columns (576 bf16 per row)
constexpr uint32_t TM_S = 320;    // rank 0: two S buffers of 64 columns
constexpr uint32_t TM_O = 0;      // rank 1: 512 columns
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 64, false, false);
// Dual GEMM for items of at most 64 query rows (FlashMLA issue #169, "dual
// gemm"): the QK reduction over the 512 latent dims is split in two, blocks
// 0, 2, 4, 6 in TMEM lanes 0-63 of Q and blocks 1, 3, 5, 7 in lanes 64-127,
// and one weight-stationary M = 64, N = 128 MMA whose B descriptor spans a
// block pair (block 2p in rows 0-63, block 2p + 1 in rows 64-127, 8 KB apart
// in the K-major layout) gives the two partial score tiles S_a (lanes 0-63)
// and S_b (lanes 64-127): 16 MMAs where M = 128 with padding took 32.  The
// 64 RoPE dims are 4 ordinary M = 128 MMAs with Q's RoPE values in lanes
// 0-63 and zeros in lanes 64-127.  The softmax warps of lanes 64-127 hand
// S_b to those of lanes 0-63 through an 8 KB area of shared memory, 32
// scores per row at a time (see dual_exchange), and write zero P rows.
constexpr uint32_t IDESC_QK_WS = idesc_bf16_f32(64, 128, false, false);
constexpr uint32_t TM_QROPE_DUAL = 128;           // rank 0, dual: RoPE columns of Q

constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 256, false, true);

struct Bars {
  uint64_t kv_full[3], kv_empty[3];      // rank 0: blocks 0-4 of a K stage; rank 1: V stages
  uint64_t kv_full_b[3], kv_empty_b[3];  // rank 0: blocks 5-8 of a K stage
  uint64_t raw_full[3];                  // gather kernel: the stage's raw FP8 rows landed
  uint64_t xfull[2], xempty[2];          // dual: S_b hand-over, scores 0-31 (0) and 32-63 (1)
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
  uint64_t lsum[4][2];   // rank 0: both halves of row group q wrote their row sums (piece parity)
  uint32_t mask[kMaskRing][2];
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t OFF_LPART = OFF_BARS + (sizeof(Bars) + 15) / 16 * 16;  // rank 0: float[2][2][128]
constexpr uint32_t kSmemBytes = OFF_LPART + 4 * M_TILE * 4;
static_assert(OFF_RAW0 + 2 * kRawSlot0 <= OFF_BARS, "gather raw ring, rank 0");
static_assert(OFF_RAW1 + 2 * kRawSlot1 <= OFF_RCV_P, "gather raw ring, rank 1");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(OFF_XCHG + kXchgBytes <= OFF_BARS, "rank 0 map");
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
  if (mbar_wait<false>(smem_u32(bar), parity, &c.bars->abort, c.p->wait_ns)) return true;
  atomicOr(c.p->status, MLA_STATUS_WAIT_TIMEOUT);
  c.bars->abort = 1;
  return false;
}

__device__ __forceinline__ bool wait_cluster_or_abort(const Ctx &c, uint64_t *bar, uint32_t parity) {
  if (mbar_wait<true>(smem_u32(bar), parity, &c.bars->abort, c.p->wait_ns)) return true;
  atomicOr(c.p->status, MLA_STATUS_WAIT_TIMEOUT);
  c.bars->abort = 1;
  return false;
}

// Whole-warp forms for the softmax and epilogue warps, whose lanes go on to
// warp-collective tcgen05 loads and stores: every lane returns the same
// answer (false if any lane's wait gave up), so a warp never splits between
// giving up and going on.  `need` false: this lane only votes.
__device__ __forceinline__ bool warp_wait(const Ctx &c, uint64_t *bar, uint32_t parity, bool need = true) {
  return __all_sync(0xffffffffu, !need || wait_or_abort(c, bar, parity));
}

__device__ __forceinline__ bool warp_wait_cluster(const Ctx &c, uint64_t *bar, uint32_t parity) {
  return __all_sync(0xffffffffu, wait_cluster_or_abort(c, bar, parity));
}

// Walk the pieces of this worker: f(item_index, item, t0, t1, piece, empty).
template <class F>
__device__ __forceinline__ bool for_each_piece(const DecodeParams &p, int part, F &&f) {
  const int32_t *md = p.tile_md + (size_t)part * MD_STRIDE;
  const int a = md[0], bt = md[1], z = md[2], et = md[3], fp = md[4], at_start = md[5];
  for (int i = a; i <= z; i++) {
    Item it = item_at(i, p.seqlens, p.B, p.H, p.T, p.topk_len, p.causal, p.status);
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
// rank 0's stage ring carries, per piece, the item's query rows (one stage
// per 64 rows, loaded by TMA in the K layout) before its key tiles.
__device__ __forceinline__ int q_stages(const Item &it) { return it.rows > 64 ? 2 : 1; }

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

// Validity mask of key tile `tile` of an item (bit n: key n of the tile is
// in the sequence and its page resolved), published in ring entry mi.
__device__ __forceinline__ void publish_mask(Bars &br, uint32_t mi, int page, int nvalid) {
  uint64_t m = 0;
  if (page >= 0 && nvalid > 0) m = nvalid >= 64 ? ~0ull : ((1ull << nvalid) - 1ull);
  br.mask[mi][0] = (uint32_t)m;
  br.mask[mi][1] = (uint32_t)(m >> 32);
  mbar_arrive(smem_u32(&br.mfull[mi]));
}

// ---- producer: TMA of whole pages ------------------------------------------------
//
// The page pool is viewed as a 4-D tensor [page][9 blocks][64 tokens][64
// dims] (strides 73728, 128, 1152 bytes), so one TMA box brings a whole page
// into shared memory as 9 (rank 0) or 8 (rank 1) column blocks of 64 tokens
// x 128 bytes, 128-byte swizzled: the K-major operand layout.  One
// instruction per page keeps the producer thread off the critical path.
// rank 0 also publishes each tile's validity mask.

// rank 0 loads each K page as two boxes, blocks 0-4 and 5-8, with their own
// barriers, so the first half of a stage can be refilled as soon as the QK
// MMAs that read it are done (about half a tile earlier than the whole).
__device__ void producer_tma(const Ctx &c, const CUtensorMap *map, const CUtensorMap *map_b,
                             const CUtensorMap *q_map, int lane) {
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  // rank 1 is the last reader of each page, unless the sequence has several
  // M tiles: then the worker holding the same tile range of the next M tile
  // reads the page again, at about the same time (the items are ordered
  // m-tile-major), and it should find it in L2
  const uint64_t pol = (c.rank == 0 || p.n_mt > 1) ? policy_evict_normal() : policy_evict_first();
  const uint32_t stage_bytes = c.rank == 0 ? kStage0Bytes : kStage1Bytes;
  const uint32_t kv0 = smem_u32(c.base + OFF_KV);
  const int split = p.dual ? 4 : 5;  // rank 0: first box = blocks [0, split), second = [split, 9)
  uint32_t g = 0, s = 0, ph = 1;  // stage s of tile g; parity of its previous release
  for_each_piece(p, c.part, [&](int, const Item &it, int t0, int t1, int, bool empty) {
    if (empty) return true;
    if (c.rank == 0) {
      // the item's query rows are contiguous (row0 .. row0+rows-1 of
      // sequence b): one or two boxes of 64 rows x 9 blocks
      const int qrow = it.b * p.T * p.H + it.row0;
      for (int qh = 0; qh < q_stages(it); qh++) {
        bool ok = true;
        if (lane == 0) {
          ok = wait_or_abort(c, &br.kv_empty[s], ph) && wait_or_abort(c, &br.kv_empty_b[s], ph);
          if (ok) {
            const uint32_t bar = smem_u32(&br.kv_full[s]);
            mbar_arrive_expect_tx(bar, kStage0Bytes);
            tma_load_3d(kv0 + s * kStage0Bytes, q_map, bar, 0, qrow + 64 * qh, 0, policy_evict_first());
            mbar_arrive(smem_u32(&br.kv_full_b[s]));  // the whole stage is in the first box
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
        if (++s == 3) {
          s = 0;
          ph ^= 1;
        }
      }
    }
    // The whole warp reads the block-table entries of up to 32 tiles at once
    // (a lone lane would pay a global-memory round trip per tile); lane 0
    // issues the copies.
    for (int base = t0; base < t1; base += 32) {
      const int pg = (base + lane < t1) ? page_of(p, it.b, base + lane) : -1;
      const int cnt = min(32, t1 - base);
      for (int i = 0; i < cnt; i++, g++) {
        const int page = __shfl_sync(0xffffffffu, pg, i);
        bool ok = true;
        if (lane == 0) {
          if (c.rank == 0) publish_mask(br, g % kMaskRing, page, it.kv_len - (base + i) * PAGE);
          ok = wait_or_abort(c, &br.kv_empty[s], ph);
          if (ok) {
            const uint32_t bar = smem_u32(&br.kv_full[s]);
            const uint32_t bytes = c.rank == 0 ? split * kBlkBytes : stage_bytes;
            mbar_arrive_expect_tx(bar, bytes);
            tma_load_4d(kv0 + s * stage_bytes, map, bar, 0, 0, 0, page < 0 ? 0 : page, pol);
          }
          if (ok && c.rank == 0) {
            ok = wait_or_abort(c, &br.kv_empty_b[s], ph);
            if (ok) {
              const uint32_t bar = smem_u32(&br.kv_full_b[s]);
              mbar_arrive_expect_tx(bar, (9 - split) * kBlkBytes);
              tma_load_4d(kv0 + s * stage_bytes + split * kBlkBytes, map_b, bar, 0, 0, split, page < 0 ? 0 : page, pol);
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
        if (++s == 3) {
          s = 0;
          ph ^= 1;
        }
      }
    }
    return true;
  });
}

// ---- producer: row gather / FP8 dequantisation (warps 0, 3, 13, 14) -------------------

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

// Row gather: two threads per key slot (128 threads in warps 0, 3, 13, 14),
// or four (256 threads, also warps 6, 7, 10, 11) when every item has at most
// 64 query rows (DecodeParams::help): a slot's threads split its column
// blocks into NQ parts.
__host__ __device__ constexpr int gather_threads(bool help) { return help ? 256 : 128; }
__host__ __device__ constexpr int softmax_warps(bool help) { return help ? 4 : 8; }

// Pool row of key slot pi of tile `tile` of an item: the top-k index or the
// position, through the block table, with bounds checks; -1 for none.  It
// takes two dependent loads (index, then block-table entry), so the gather
// producer runs it as a pipeline over tiles: slot_id loads tile t+2's index,
// slot_key checks tile t+1's and slot_page loads its block-table entry, and
// slot_row resolves tile t from values loaded one and two tiles earlier.

// Raw index of the slot (-2: past the item's keys).
__device__ __forceinline__ int slot_id(const DecodeParams &p, const Item &it, int t_item, int tile, int pi) {
  const int slot = tile * PAGE + pi;
  if (p.topk_len > 0)
    return slot < p.topk_len ? __ldg(p.topk + ((size_t)it.b * p.T + t_item) * p.topk_len + slot) : -2;
  return slot < it.kv_len ? slot : -2;
}

// Key index within the sequence, or -1 (an out-of-range top-k index sets
// MLA_STATUS_BAD_TOPK).
__device__ __forceinline__ int slot_key(const DecodeParams &p, int id, int sk) {
  if (id == -2) return -1;
  if (p.topk_len > 0 && (id >= sk || id < -1)) {
    atomicOr(p.status, MLA_STATUS_BAD_TOPK);
    return -1;
  }
  return id;
}

// Block-table entry of key n (loaded, not yet checked), or -1.
__device__ __forceinline__ int slot_page(const DecodeParams &p, int b, int n) {
  if (n < 0) return -1;
  if (n / PAGE >= p.max_pages) {
    atomicOr(p.status, MLA_STATUS_BAD_SEQLEN);
    return -1;
  }
  return __ldg(p.block_table + (size_t)b * p.max_pages + n / PAGE);
}

// The pool row of key n in page pg; n becomes -1 when there is none (a page
// outside the pool sets MLA_STATUS_BAD_PAGE).
__device__ __forceinline__ long long slot_row(const DecodeParams &p, int &n, int pg) {
  if (n < 0) return -1;
  if (pg < 0 || pg >= p.num_pages) {
    if (pg >= 0 || n / PAGE < p.max_pages) atomicOr(p.status, MLA_STATUS_BAD_PAGE);
    n = -1;
    return -1;
  }
  return (long long)pg * PAGE + (n % PAGE);
}

// 16-byte asynchronous copy global -> shared (cp.async); with ok false it
// writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)),
               "r"(ok ? 16 : 0)
               : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

constexpr uint32_t kGatherBar = 2;  // named barrier of the 128 gather threads

// Row pi of one tile: pool row `row` (zeros for -1) into the stage at
// shared address st, as bf16 column blocks 0-7 (+ the RoPE block 8 when
// rope), 128-byte swizzled (row pi of block kb at kb*8192 + pi*128, chunk j
// at ((j ^ (pi & 7)) << 4)).
//
// FP8 rows arrive first in a raw slot (row pi at pi * rowbytes;
// issue_raw_tile, two tiles ahead) and are then dequantised into the stage
// by the row's two threads, each half of its column blocks (fp8_row_to_stage).
// bf16 rows are copied 16 bytes at a time straight into place, the blocks
// shared between the two threads.

// Bytes of an FP8 cache row: 640 (e4m3 latent + bf16 RoPE), or 576 in the
// per-tensor format (all e4m3).
__device__ __forceinline__ uint32_t fp8_row_bytes(const DecodeParams &p) {
  return p.kv_format == MLA_KV_FP8_E4M3_TENSOR ? D_QK : FP8_ROW;
}

// Staged rows sit 640, 576 or 512 bytes apart, a multiple of 128 bytes of
// bank offset, so the same 16-byte chunk of 8 consecutive rows would fall in
// the same 4 banks (an 8-way conflict for each reading quarter-warp).  Chunk
// c of staged row pi is therefore stored at position raw_chunk(c, pi): its
// low bits XORed with the row within its group of 8 chunks (4 for the 64-byte
// tail of a 576-byte row), which spreads 8 rows over all 32 banks.
__device__ __forceinline__ uint32_t raw_chunk(int c, int pi, int tail_mask) {
  return c < 32 ? (uint32_t)((c & ~7) | ((c ^ pi) & 7)) : (uint32_t)(32 | ((c ^ pi) & tail_mask));
}

// FP8 rows of one tile into the stage's staging area, completing on raw_bar
// (one arrival per gather thread, made when its copies have landed).  Each
// gather warp copies 16 rows, one row at a time with all 32 lanes: every
// 16-byte cp.async of a warp instruction reads the same 512 contiguous bytes
// of one row (the first 512 bytes, then the RoPE bytes on rank 0), so the
// requests are coalesced and up to a whole tile of rows is in flight per SM.
// (One bulk copy per row went through the copy engine one row at a time:
// about 6 us for a tile's 64 rows.)  Lane l of the warp holds the pool row
// of key slot (gt & 32) + l; the NQ warps that hold the same 32 slots copy
// 32 / NQ of them each (part h: slots h * 32 / NQ ...).  A row of -1 is
// filled with zeros.
template <int NQ>
__device__ __forceinline__ void issue_raw_tile(const Ctx &c, long long row, uint32_t st, int gt, bool rope,
                                               uint64_t *raw_bar) {
  constexpr int kRows = 32 / NQ;  // rows copied by each warp
  const uint32_t stride = fp8_row_bytes(*c.p);
  const uint32_t rowbytes = rope ? stride : 512;
  const int lane = gt & 31, sbase = gt & 32, h = gt >> 6;
  const bool tail = rope && (uint32_t)lane * 16 + 512 < rowbytes;
  const int tm = stride == FP8_ROW ? 7 : 3;
#pragma unroll 4
  for (int k = 0; k < kRows; k++) {
    const int j = h * kRows + k, pj = sbase + j;
    const long long rj = __shfl_sync(0xffffffffu, row, j);
    const bool ok = rj >= 0;
    const uint8_t *src = c.p->kv + (ok ? rj : 0) * stride + lane * 16;
    const uint32_t dst = st + pj * rowbytes;
    cp_async16(dst + raw_chunk(lane, pj, tm) * 16, src, ok);
    if (tail) cp_async16(dst + raw_chunk(32 + lane, pj, tm) * 16, src + 512, ok);
  }
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(raw_bar)) : "memory");
}

// The four per-128 scales of an FP8 row (the one scale of a per-tensor
// cache four times; zeros for no row), loaded a tile ahead of their use.
__device__ __forceinline__ float4 row_scales(const DecodeParams &p, long long row) {
  if (row < 0) return make_float4(0, 0, 0, 0);
  if (p.kv_format == MLA_KV_FP8_E4M3_TENSOR) {
    const float k = __ldg(p.kv_scales);
    return make_float4(k, k, k, k);
  }
  return __ldg(reinterpret_cast<const float4 *>(p.kv_scales + row * 4));
}

// A bf16 row (top-k over a bf16 cache): 16-byte cp.async straight into the
// K layout, the blocks shared among the slot's NQ threads.
template <int NQ>
__device__ __forceinline__ void bf16_row_to_stage(const DecodeParams &p, long long row, uint32_t st, int pi, int part,
                                                  bool rope) {
  const bool ok = row >= 0;
  const int sw = pi & 7;
  const uint8_t *src = p.kv + (ok ? row : 0) * (D_QK * 2);
  const int nb = rope ? 9 : 8;
  for (int kb = part; kb < nb; kb += NQ)
#pragma unroll
    for (int j = 0; j < 8; j++) cp_async16(st + kb * kBlkBytes + pi * 128 + ((j ^ sw) << 4), src + kb * 128 + j * 16, ok);
  cp_async_wait_all();
}

// An FP8 row from its raw slot (row pi at raw, chunks placed by raw_chunk)
// into the stage as bf16 column blocks: part h of NQ takes latent blocks
// h * 8 / NQ ... (scale tile kb / 2 for block kb) and part 0, on rank 0, the
// RoPE block too.
template <int NQ>
__device__ __forceinline__ void fp8_row_to_stage(const DecodeParams &p, uint32_t raw, uint32_t st, int pi, int part,
                                                 bool rope, float4 sc) {
  constexpr int kBlocks = 8 / NQ;
  const int tm = fp8_row_bytes(p) == FP8_ROW ? 7 : 3;
  const int sw = pi & 7;
#pragma unroll
  for (int k = 0; k < kBlocks; k++) {
    const int kb = part * kBlocks + k;
    const int t = kb >> 1;
    const float scl = t == 0 ? sc.x : t == 1 ? sc.y : t == 2 ? sc.z : sc.w;
#pragma unroll
    for (int u = 0; u < 4; u++) {
      uint4 lo, hi;
      dequant16(ld_shared_v4(raw + raw_chunk(kb * 4 + u, pi, tm) * 16), scl, lo, hi);
      st_shared_v4(st + kb * kBlkBytes + pi * 128 + (((2 * u) ^ sw) << 4), lo);
      st_shared_v4(st + kb * kBlkBytes + pi * 128 + (((2 * u + 1) ^ sw) << 4), hi);
    }
  }
  if (rope && part == 0) {
    if (p.kv_format == MLA_KV_FP8_E4M3_TENSOR) {  // 64 e4m3 RoPE values x the scale
#pragma unroll
      for (int u = 0; u < 4; u++) {
        uint4 lo, hi;
        dequant16(ld_shared_v4(raw + raw_chunk(32 + u, pi, tm) * 16), sc.x, lo, hi);
        st_shared_v4(st + 8 * kBlkBytes + pi * 128 + (((2 * u) ^ sw) << 4), lo);
        st_shared_v4(st + 8 * kBlkBytes + pi * 128 + (((2 * u + 1) ^ sw) << 4), hi);
      }
    } else {  // 64 bf16 RoPE values, copied
#pragma unroll
      for (int j = 0; j < 8; j++)
        st_shared_v4(st + 8 * kBlkBytes + pi * 128 + ((j ^ sw) << 4), ld_shared_v4(raw + raw_chunk(32 + j, pi, tm) * 16));
    }
  }
}

// Threads gt, gt + 64, ... (gt < 64) of the gather warps own key slot
// pi = gt of every tile: each resolves the row and writes its part of it,
// dequantised to bf16, into row pi of the column blocks of the stage (9
// blocks on rank 0, 8 on rank 1).  On rank 0 the first thread of the slot
// also publishes the tile's validity mask and the gathered-index record.
//
// FP8 rows go through a ring of two raw slots of their own (in the memory of
// the kernel's third stage): the rows of tile t + 2 are fetched into tile
// t's slot as soon as every gather thread has read it, so a fetch has about
// two tiles' time to land, and a K / V stage is held only from its tile's
// dequantisation to the MMA that reads it.
template <int NQ>
__device__ void producer_gather(const Ctx &c, const CUtensorMap *q_map, int gt) {
  constexpr uint32_t NS = ring_stages(true);
  constexpr int kThreads = 64 * NQ;
  const int pi = gt & 63, part = gt >> 6;
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  const bool fp8 = p.kv_format != MLA_KV_BF16;
  const bool rope = c.rank == 0;
  const uint32_t stage_bytes = c.rank == 0 ? kStage0Bytes : kStage1Bytes;
  const uint32_t kv0 = smem_u32(c.base + OFF_KV);
  const uint32_t raw0 = smem_u32(c.base + (c.rank == 0 ? OFF_RAW0 : OFF_RAW1));
  const uint32_t raw_slot = c.rank == 0 ? kRawSlot0 : kRawSlot1;
  const uint32_t rowbytes = rope ? fp8_row_bytes(p) : 512;
  uint32_t g = 0, sq = 0, rt = 0;  // tiles; stages of the ring (rank 0: query stages too); raw-slot uses
  for_each_piece(p, c.part, [&](int idx, const Item &it, int t0, int t1, int, bool empty) {
    if (empty) return true;
    const int t_item = (p.topk_len > 0) ? (idx % p.T) : 0;
    const int sk = clamp_seqlen(p.seqlens[it.b], p.status);
    if (c.rank == 0) {  // the query rows, by TMA (thread 0 issues, all 64 arrive)
      const int qrow = it.b * p.T * p.H + it.row0;
      for (int qh = 0; qh < q_stages(it); qh++, sq++) {
        const uint32_t s = sq % NS;
        bool ok = wait_or_abort(c, &br.kv_empty[s], ((sq / NS) & 1) ^ 1);
        if (ok) ok = wait_or_abort(c, &br.kv_empty_b[s], ((sq / NS) & 1) ^ 1);
        if (bar_red_or(kGatherBar, kThreads, !ok)) return false;  // all gather threads give up together
        const uint32_t bar = smem_u32(&br.kv_full[s]);
        if (gt == 0) {
          mbar_arrive_expect_tx(bar, kStage0Bytes);
          tma_load_3d(kv0 + s * kStage0Bytes, q_map, bar, 0, qrow + 64 * qh, 0, policy_evict_first());
        } else {
          mbar_arrive(bar);
        }
        mbar_arrive(smem_u32(&br.kv_full_b[s]));
      }
    }
    // row pipeline (see slot_id): n0 / pg0 and n1 / pg1 = key and
    // block-table entry of this tile and the next, id2 = raw index of the one
    // after; each iteration loads the index three tiles ahead and the
    // block-table entry two ahead
    int n0 = t0 < t1 ? slot_key(p, slot_id(p, it, t_item, t0, pi), sk) : -1;
    int pg0 = slot_page(p, it.b, n0);
    int n1 = t0 + 1 < t1 ? slot_key(p, slot_id(p, it, t_item, t0 + 1, pi), sk) : -1;
    int pg1 = slot_page(p, it.b, n1);
    int id2 = t0 + 2 < t1 ? slot_id(p, it, t_item, t0 + 2, pi) : -2;
    // FP8: the raw rows and scales of the piece's first two tiles
    float4 sc0 = make_float4(0, 0, 0, 0), sc1 = make_float4(0, 0, 0, 0);
    if (fp8) {
      for (int k = 0; k < 2 && t0 + k < t1; k++) {
        int n = k ? n1 : n0;
        const long long r = slot_row(p, n, k ? pg1 : pg0);
        if (k) sc1 = row_scales(p, r);
        else sc0 = row_scales(p, r);
        issue_raw_tile<NQ>(c, r, raw0 + ((rt + k) % 2) * raw_slot, gt, rope, &br.raw_full[(rt + k) % 2]);
      }
    }
    for (int tile = t0; tile < t1; tile++, g++, sq++) {
      const uint32_t s = sq % NS;
      const int id3 = tile + 3 < t1 ? slot_id(p, it, t_item, tile + 3, pi) : -2;
      const int n2 = slot_key(p, id2, sk);
      const int pg2 = slot_page(p, it.b, n2);
      int n = n0;
      const long long row = slot_row(p, n, pg0);
      n0 = n1;
      pg0 = pg1;
      n1 = n2;  // n1 / pg1: tile + 2 from here on
      pg1 = pg2;
      id2 = id3;
      if (c.rank == 0 && part == 0) {
        const uint32_t bits = __ballot_sync(0xffffffffu, row >= 0);
        const uint32_t mi = g % kMaskRing;
        if ((pi & 31) == 0) br.mask[mi][pi >> 5] = bits;
        if (p.gathered != nullptr && p.topk_len > 0) {
          const int slot = tile * PAGE + pi;
          if (slot < p.topk_len) p.gathered[((size_t)it.b * p.T + t_item) * p.topk_len + slot] = n;
        }
        __syncwarp();
        if ((pi & 31) == 0) mbar_arrive(smem_u32(&br.mfull[mi]));
      }
      // The tile's stage is free once its previous tile's MMAs are done.
      // Each gather thread waits for that itself and writes its part; a
      // thread whose wait gives up skips the work but still meets the other
      // gather threads at the barrier below, so all of them leave together.
      bool ok = wait_or_abort(c, &br.kv_empty[s], ((sq / NS) & 1) ^ 1);
      if (ok && c.rank == 0) ok = wait_or_abort(c, &br.kv_empty_b[s], ((sq / NS) & 1) ^ 1);
      if (fp8) {
        const uint32_t slot = rt % 2;
        const uint32_t rs = raw0 + slot * raw_slot;
        const bool landed = ok && wait_or_abort(c, &br.raw_full[slot], (rt / 2) & 1);
        if (landed) fp8_row_to_stage<NQ>(p, rs + pi * rowbytes, kv0 + s * stage_bytes, pi, part, rope, sc0);
        // this thread's part of the stage is written: it is handed to the
        // MMA before the next raw fetch goes out, since the proxy fence waits
        // for the thread's copies in flight
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&br.kv_full[s]));
        if (c.rank == 0) mbar_arrive(smem_u32(&br.kv_full_b[s]));
        if (bar_red_or(kGatherBar, kThreads, !landed)) return false;  // the slot has been read
        sc0 = sc1;
        if (tile + 2 < t1) {  // the slot takes the rows of tile + 2
          int nn = n1;
          const long long r2 = slot_row(p, nn, pg1);
          sc1 = row_scales(p, r2);
          issue_raw_tile<NQ>(c, r2, rs, gt, rope, &br.raw_full[slot]);
        }
        rt++;
      } else {
        if (ok) bf16_row_to_stage<NQ>(p, row, kv0 + s * stage_bytes, pi, part, rope);
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&br.kv_full[s]));
        if (c.rank == 0) mbar_arrive(smem_u32(&br.kv_full_b[s]));
        if (bar_red_or(kGatherBar, kThreads, !ok)) return false;
      }
    }
    return true;
  });
}

// ---- MMA warps and their waiters ------------------------------------------------------
//
// An mbarrier wait (or any shared-memory load) by the warp that issues
// tcgen05.mma waits for that warp's MMAs in flight, which would drain the
// tensor pipe at every wait.  So each MMA warp has a waiter warp: the waiter
// does every mbarrier wait the MMAs depend on and then meets the MMA warp at
// named barrier kMmaBar (bar.red, which also carries an abort flag); the MMA
// warp only computes descriptors, issues MMAs and commits.

constexpr uint32_t kMmaBar = 1;
constexpr uint32_t kMmaBarThreads = 64;

// Lane 0 of a waiter warp has done its waits (ok = all completed); the whole
// warp meets the MMA warp.  True if either side gives up.
__device__ __forceinline__ bool waiter_meet(bool ok) {
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return bar_red_or(kMmaBar, kMmaBarThreads, !ok);
}

// ---- rank 0: QK MMA issuer ----------------------------------------------------------
//
// Per tile g: S[g&1] = Q . K^T (M = 128, N = 64 tokens, K = 576 in 36 steps
// of 16; A = Q from TMEM, B = the K-major swizzled key blocks of the stage),
// commit -> kv_empty, s_full.  S is double-buffered, so QK(g+1) overlaps the
// softmax of g.  The waiter meets the MMA warp once per piece (Q is in
// TMEM) and once per tile (stage full and S[g&1] free).

template <bool kGather>
__device__ void qk_waiter(const Ctx &c, int lane) {
  constexpr uint32_t NS = ring_stages(kGather);
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  uint32_t g = 0, qn = 0, sq = 0;  // tiles, pieces, ring stages
  for_each_piece(p, c.part, [&](int, const Item &it, int t0, int t1, int, bool empty) {
    if (empty) return true;
    bool ok = true;
    if (lane == 0) ok = wait_or_abort(c, &br.q_ready, qn & 1);
    qn++;
    sq += q_stages(it);  // the query stages, read by the softmax warps
    if (waiter_meet(ok)) return false;
    for (int tile = t0; tile < t1; tile++, g++, sq++) {
      if (lane == 0) {
        ok = wait_or_abort(c, &br.s_free[g & 1], ((g >> 1) & 1) ^ 1);
        if (ok) ok = wait_or_abort(c, &br.kv_full[sq % NS], (sq / NS) & 1);
      }
      if (waiter_meet(ok)) return false;  // blocks 0-4 of the stage, S free
      if (lane == 0) ok = wait_or_abort(c, &br.kv_full_b[sq % NS], (sq / NS) & 1);
      if (waiter_meet(ok)) return false;  // blocks 5-8
    }
    return true;
  });
}

template <bool kGather, bool kDual>
__device__ void mma_qk(const Ctx &c, uint32_t tmem) {
  constexpr uint32_t NS = ring_stages(kGather);
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  const uint32_t kv0 = smem_u32(c.base + OFF_KV);
  const uint32_t kv_empty0 = smem_u32(&br.kv_empty[0]), s_full0 = smem_u32(&br.s_full[0]);
  const uint32_t kv_empty_b0 = smem_u32(&br.kv_empty_b[0]);
  uint32_t g = 0, sq = 0;  // tiles, ring stages
  for_each_piece(p, c.part, [&](int, const Item &it, int t0, int t1, int, bool empty) {
    if (empty) return true;
    if (bar_red_or(kMmaBar, kMmaBarThreads, false)) return false;  // Q is in TMEM
    tc_fence_after();
    // the softmax warps have copied the query stages into TMEM: release them
    // (the commit arrives once the MMAs issued so far are done)
    if (elect_one())
      for (int qh = 0; qh < q_stages(it); qh++) {
        mma_commit(kv_empty0 + ((sq + qh) % NS) * 8);
        mma_commit(kv_empty_b0 + ((sq + qh) % NS) * 8);
      }
    __syncwarp();
    sq += q_stages(it);
    for (int tile = t0; tile < t1; tile++, g++, sq++) {
      const uint32_t s = sq % NS, b = g & 1;
      if (bar_red_or(kMmaBar, kMmaBarThreads, false)) return false;  // blocks 0-4 in, S free
      tc_fence_after();
      // one base descriptor per tile; block kb / step kk only move its
      // start-address field (16-byte units: 512 per 8 KB block, 2 per 32 B)
      const uint64_t kd0 = smem_desc_sw128(kv0 + s * kStage0Bytes, 16, 1024);
      const uint32_t d = tmem + TM_S + b * 64;
      if (elect_one()) {
        if (kDual) {  // block pairs (0, 1), (2, 3)
#pragma unroll
          for (int i = 0; i < 8; i++) {
            const int pr = i >> 2, kk = i & 3;
            mma_ws_ts(d, tmem + TM_Q + pr * 32 + kk * 8, kd0 + (uint64_t)(pr * 1024 + kk * 2), IDESC_QK_WS,
                      i ? 1u : 0u);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 20; i++) {
            const int kb = i >> 2, kk = i & 3;
            mma_ts(d, tmem + TM_Q + kb * 32 + kk * 8, kd0 + (uint64_t)(kb * 512 + kk * 2), IDESC_QK, i ? 1u : 0u);
          }
        }
        mma_commit(kv_empty0 + s * 8);
      }
      __syncwarp();
      if (bar_red_or(kMmaBar, kMmaBarThreads, false)) return false;  // blocks 5-8 in
      tc_fence_after();
      if (elect_one()) {
        if (kDual) {  // block pairs (4, 5), (6, 7), then the RoPE block with zeros in lanes 64-127
#pragma unroll
          for (int i = 0; i < 8; i++) {
            const int pr = 2 + (i >> 2), kk = i & 3;
            mma_ws_ts(d, tmem + TM_Q + pr * 32 + kk * 8, kd0 + (uint64_t)(pr * 1024 + kk * 2), IDESC_QK_WS, 1u);
          }
#pragma unroll
          for (int kk = 0; kk < 4; kk++)
            mma_ts(d, tmem + TM_QROPE_DUAL + kk * 8, kd0 + (uint64_t)(8 * 512 + kk * 2), IDESC_QK, 1u);
        } else {
#pragma unroll
          for (int i = 20; i < 36; i++) {
            const int kb = i >> 2, kk = i & 3;
            mma_ts(d, tmem + TM_Q + kb * 32 + kk * 8, kd0 + (uint64_t)(kb * 512 + kk * 2), IDESC_QK, 1u);
          }
        }
        mma_commit(kv_empty_b0 + s * 8);
        mma_commit(s_full0 + b * 8);
      }
      __syncwarp();
    }
    return true;
  });
}

// ---- rank 1: PV MMA issuer ----------------------------------------------------------
//
// Per tile g: O[:, 0:256) and O[:, 256:512) (+)= P(g) . V(g) (M=128, N=256,
// K=64 tokens in 4 steps; A = P from shared memory, K-major; B = the V
// blocks of the stage read MN-major).  The first tile of a piece overwrites
// O.  The waiter meets the MMA warp once per tile, after the V stage is full,
// P is in shared memory and the epilogue warps have applied any rescale
// (o_ready).

template <bool kGather>
__device__ void pv_waiter(const Ctx &c, int lane) {
  constexpr uint32_t NS = ring_stages(kGather);
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  uint32_t g = 0;
  for_each_piece(p, c.part, [&](int, const Item &, int t0, int t1, int, bool empty) {
    if (empty) return true;
    for (int tile = t0; tile < t1; tile++, g++) {
      const uint32_t b = g & 1, u = g >> 1;
      bool ok = true;
      if (lane == 0) {
        ok = wait_or_abort(c, &br.kv_full[g % NS], (g / NS) & 1);
        if (ok) ok = wait_or_abort(c, &br.p_land[b], u & 1);
        if (ok) ok = wait_or_abort(c, &br.o_ready[b], u & 1);
      }
      if (waiter_meet(ok)) return false;
    }
    return true;
  });
}

template <bool kGather>
__device__ void mma_pv(const Ctx &c, uint32_t tmem) {
  constexpr uint32_t NS = ring_stages(kGather);
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  const uint32_t kv0 = smem_u32(c.base + OFF_KV);
  const uint32_t pbuf = smem_u32(c.base + OFF_RCV_P);
  const uint32_t kv_empty0 = smem_u32(&br.kv_empty[0]), p_empty0 = smem_u32(&br.p_empty[0]);
  const uint32_t o_done0 = smem_u32(&br.o_done[0]);
  uint32_t g = 0;
  for_each_piece(p, c.part, [&](int, const Item &, int t0, int t1, int, bool empty) {
    if (empty) return true;
    const uint32_t gfirst = g;
    for (int tile = t0; tile < t1; tile++, g++) {
      const uint32_t s = g % NS, b = g & 1;
      if (bar_red_or(kMmaBar, kMmaBarThreads, false)) return false;
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 4; kk++) {
          const uint64_t a = smem_desc_noswz(pbuf + b * kPBytes + kk * 2 * 2048, 2048, 128);
#pragma unroll
          for (int nh = 0; nh < 2; nh++) {
            const uint64_t v = smem_desc_sw128(kv0 + s * kStage1Bytes + nh * 4 * kBlkBytes + kk * 2048, kBlkBytes, 1024);
            mma_ss(tmem + TM_O + nh * 256, a, v, IDESC_PV, (g == gfirst && kk == 0) ? 0u : 1u);
          }
        }
        mma_commit(kv_empty0 + s * 8);
        mma_commit(p_empty0 + b * 8);
        mma_commit(o_done0 + b * 8);
      }
      __syncwarp();
    }
    return true;
  });
}

__device__ __forceinline__ const uint8_t *ring_slot(const DecodeParams &p, int part, uint32_t g) {
  return p.ws_p + ((size_t)part * P_RING + (g % P_RING)) * P_SLOT_BYTES;
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

// Query row r of the item, column blocks [kb0, kb1) of its 576 dims ->
// TMEM columns TM_Q + 32*kb.. as bf16 pairs, from the ring stage that holds
// the item's rows 64*(r/64) .. (K-major 128-byte swizzled layout: row rr of
// block kb at kb*8192 + rr*128, 16-byte chunk j at (j ^ (rr & 7)) * 16).
// Rows past the item get zeros.  Not inlined: it runs once per piece, and
// inlined its registers would crowd the softmax loop.
__device__ __noinline__ void load_q(uint32_t lane_tmem, uint32_t stage, int rr, bool ok, int kb0, int kb1) {
  for (int kb = kb0; kb < kb1; kb++) {
    uint32_t v[32];
#pragma unroll
    for (int j = 0; j < 8; j++) {
      uint4 x = make_uint4(0, 0, 0, 0);
      if (ok)
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
                     : "r"(stage + kb * kBlkBytes + rr * 128 + ((j ^ (rr & 7)) << 4)));
      v[4 * j] = x.x;
      v[4 * j + 1] = x.y;
      v[4 * j + 2] = x.z;
      v[4 * j + 3] = x.w;
    }
    tmem_st32(lane_tmem + TM_Q + kb * 32, v);
  }
  tmem_wait_st();
}

// Dual GEMM: the query row's blocks for lanes 0-63 (`upper` false: blocks
// 0, 2, 4, 6 at columns 0, 32, 64, 96, and the RoPE block 8 at column 128)
// or for lanes 64-127 (`upper`: blocks 1, 3, 5, 7, and zeros at 128-159);
// hf 0 takes the first two of them and the RoPE columns, hf 1 the last two.
__device__ __noinline__ void load_q_dual(uint32_t lane_tmem, uint32_t stage, int rr, bool ok, bool upper, int hf) {
  for (int i = 0; i < 3; i++) {
    if (hf == 1 && i == 2) break;
    const int pr = 2 * hf + i;           // pair index (i < 2)
    const bool rope = i == 2;
    const int kb = rope ? 8 : 2 * pr + (upper ? 1 : 0);
    const uint32_t col = rope ? TM_QROPE_DUAL : (uint32_t)pr * 32;
    const bool live = ok && !(rope && upper);
    uint32_t v[32];
#pragma unroll
    for (int j = 0; j < 8; j++) {
      uint4 x = make_uint4(0, 0, 0, 0);
      if (live)
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
                     : "r"(stage + kb * kBlkBytes + rr * 128 + ((j ^ (rr & 7)) << 4)));
      v[4 * j] = x.x;
      v[4 * j + 1] = x.y;
      v[4 * j + 2] = x.z;
      v[4 * j + 3] = x.w;
    }
    tmem_st32(lane_tmem + col, v);
  }
  tmem_wait_st();
}

// Dual GEMM: S_b hand-over from the softmax warps of lanes 64-127 to those of
// lanes 0-63, in two rounds through one 8 KB area (64 rows x 32 scores, row
// R at R * 128, 16-byte chunk j at position j ^ (R & 7) so that 8 consecutive
// rows' chunks fall in different banks): round h carries scores 32h..32h+31,
// written by the two warps (q = 2, 3) of half h, which hold them as `own`,
// and added by the four warps of lanes 0-63 (to `own` for hf == h, else to
// `oth`).  The writers of round 0 wait for the previous tile's round-1 reads,
// those of round 1 for this tile's round-0 reads; every wait is bounded.
__device__ __forceinline__ uint32_t xchg_addr(uint32_t xb, int R, int j) {
  return xb + R * 128 + ((j ^ (R & 7)) << 4);
}

__device__ __forceinline__ bool dual_exchange(const Ctx &c, float (&own)[32], float (&oth)[32], int q, int hf, int R,
                                              uint32_t g) {
  Bars &br = *c.bars;
  const uint32_t xb = smem_u32(c.base + OFF_XCHG);
  const int lane = threadIdx.x & 31;
  const uint32_t ph = g & 1;
  for (int h = 0; h < 2; h++) {
    if (q >= 2) {
      if (hf != h) continue;
      // the area is free: round 1 of the previous tile (h = 0) or round 0 of
      // this tile (h = 1) has been read
      const bool ok = h == 0 ? warp_wait(c, &br.xempty[1], ph ^ 1) : warp_wait(c, &br.xempty[0], ph);
      if (!ok) return false;
#pragma unroll
      for (int j = 0; j < 8; j++)
        st_shared_v4(xchg_addr(xb, R, j), make_uint4(__float_as_uint(own[4 * j]), __float_as_uint(own[4 * j + 1]),
                                                     __float_as_uint(own[4 * j + 2]), __float_as_uint(own[4 * j + 3])));
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&br.xfull[h]));
    } else {
      if (!warp_wait(c, &br.xfull[h], ph)) return false;
      float(&dst)[32] = hf == h ? own : oth;
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const uint4 a = ld_shared_v4(xchg_addr(xb, R, j));
        dst[4 * j] += __uint_as_float(a.x);
        dst[4 * j + 1] += __uint_as_float(a.y);
        dst[4 * j + 2] += __uint_as_float(a.z);
        dst[4 * j + 3] += __uint_as_float(a.w);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&br.xempty[h]));
    }
  }
  return true;
}

__device__ __forceinline__ float max32(const float (&v)[32]) {
  float mx[8];
#pragma unroll
  for (int k = 0; k < 8; k++) mx[k] = fmaxf(fmaxf(v[k], v[k + 8]), fmaxf(v[k + 16], v[k + 24]));
  return fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
}

// Masked-out scores become -inf (skipped when all 32 are valid).
__device__ __forceinline__ void mask32(float (&v)[32], uint32_t m) {
  if (m != 0xffffffffu) {
#pragma unroll
    for (int n = 0; n < 32; n++) v[n] = ((m >> n) & 1u) ? v[n] : -INFINITY;
  }
}

// Thread (q, hf) of warp w = 4 + 4*hf + q owns query row r = 32q + lane and
// tokens [32*hf, 32*hf + 32) of each tile.  Both threads of a row read all 64
// scores, so they reach the same running max and rescale decisions without
// talking to each other; each exponentiates and writes its own 32 tokens of
// the tile's P message and keeps its own part of the row sum.  The halves of
// the row sum meet in shared memory at the last tile of a piece.
template <bool kGather, bool kDual>
__device__ void softmax_role(const Ctx &c, uint32_t tmem, int w, int lane) {
  constexpr uint32_t NS = ring_stages(kGather);
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  const int q = w & 3, hf = (w - 4) >> 2;
  const int r = q * 32 + lane;
  const uint32_t lt = tmem + ((uint32_t)(q * 32) << 16);
  float *lpart = reinterpret_cast<float *>(c.base + OFF_LPART);  // [2 pieces][2 halves][128]
  const float cs = p.scale_log2;
  const uint32_t kv0 = smem_u32(c.base + OFF_KV);
  uint32_t g = 0, pc = 0, sq = 0;  // tiles, pieces, ring stages
  for_each_piece(p, c.part, [&](int idx, const Item &it, int t0, int t1, int piece, bool empty) {
    const RowInfo ri = row_info(p, idx, it, piece, r);
    float *lse_dst = p.lse + ((size_t)it.b * p.H + ri.h) * p.T + ri.t;
    if (empty) {  // no key: LSE = -inf (rank 1 writes O = 0)
      if (ri.ok && hf == 0) *lse_dst = -INFINITY;
      return true;
    }
    {  // the query rows, from the stage ring into TMEM
      // (dual: lanes 64-127 hold rows 0-63 too, in the item's single stage)
      const int qr = kDual ? (r & 63) : r;
      const bool qok = qr < it.rows;  // rows past the item read nothing
      const uint32_t qs = sq + (qr >> 6);
      if (!warp_wait(c, &br.kv_full[qs % NS], (qs / NS) & 1, qok)) return false;
      if (kDual)
        load_q_dual(lt, kv0 + (qs % NS) * kStage0Bytes, qr & 63, qok, q >= 2, hf);
      else
        load_q(lt, kv0 + (qs % NS) * kStage0Bytes, r & 63, qok, hf ? 5 : 0, hf ? 9 : 5);
      sq += q_stages(it) + (t1 - t0);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&br.q_ready));
    }
    const int sk = clamp_seqlen(p.seqlens[it.b], p.status);
    const int my_len = (p.topk_len > 0) ? 0x7fffffff : row_kv_len(sk, p.T, ri.t, p.causal);
    float m_ref = -INFINITY;  // reference max, raw score units
    float l = 0.f;            // this half's part of the row sum
    float l_all = 0.f;
    for (int tile = t0; tile < t1; tile++, g++) {
      const uint32_t b = g & 1, u = g >> 1, mi = g % kMaskRing;
      // 1. tile validity and this row's 64 scores
      if (!warp_wait(c, &br.mfull[mi], (g / kMaskRing) & 1)) return false;
      uint32_t mlo = br.mask[mi][0], mhi = br.mask[mi][1];
      const int lim = my_len - tile * PAGE;
      if (lim < 64) {
        const uint64_t keep = lim <= 0 ? 0ull : ((1ull << lim) - 1ull);
        mlo &= (uint32_t)keep;
        mhi &= (uint32_t)(keep >> 32);
      }
      if (!warp_wait(c, &br.s_full[b], u & 1)) return false;
      tc_fence_after();
      float own[32], oth[32];  // this half's 32 scores and the partner half's
      tmem_ld32(lt + TM_S + b * 64 + hf * 32, *reinterpret_cast<uint32_t(*)[32]>(&own[0]));
      tmem_ld32(lt + TM_S + b * 64 + (hf ^ 1) * 32, *reinterpret_cast<uint32_t(*)[32]>(&oth[0]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&br.s_free[b]));
      if (kDual) {  // S = S_a (lanes 0-63) + S_b (lanes 64-127)
        if (!dual_exchange(c, own, oth, q, hf, r & 63, g)) return false;
        if (q >= 2) {  // lanes 64-127 hold no row of their own: a fully masked row, P = 0
          mlo = 0u;
          mhi = 0u;
        }
      }
      // 2. mask (skipped for fully valid tiles) and tile max (raw units; the
      //    scale is positive)
      mask32(own, hf ? mhi : mlo);
      mask32(oth, hf ? mlo : mhi);
      const float mt = fmaxf(max32(own), max32(oth));
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
      if (!warp_wait_cluster(c, &br.gfree[gs], ((g / P_RING) & 1) ^ 1)) return false;
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
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&br.lsum[q][pc & 1]));
        if (!warp_wait(c, &br.lsum[q][pc & 1], (pc >> 1) & 1)) return false;
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
// takes along every following message that is already written (up to
// kPublishBatch), makes them visible to rank 1 with one fence and signals
// each with a relaxed remote arrive (fence + relaxed arrive is a release).
// A fence waits for the stores to reach L2, about 2000 cycles under load;
// keeping it off the softmax warps and sharing it among messages keeps it
// off the critical path.

__device__ void p_publisher(const Ctx &c) {
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  const uint32_t pfull1 = mapa(smem_u32(&br.p_full[0]), 1);
  uint32_t total = 0;
  for_each_piece(p, c.part, [&](int, const Item &, int t0, int t1, int, bool empty) {
    if (!empty) total += (uint32_t)(t1 - t0);
    return true;
  });
  for (uint32_t g = 0; g < total;) {
    if (!wait_or_abort(c, &br.pwritten[g % P_RING], (g / P_RING) & 1)) return;
    uint32_t n = 1;
    while (n < kPublishBatch && g + n < total &&
           mbar_test_wait(smem_u32(&br.pwritten[(g + n) % P_RING]), ((g + n) / P_RING) & 1))
      n++;
    fence_acq_rel_cluster();
    for (uint32_t i = 0; i < n; i++) mbar_arrive_remote_relaxed(pfull1 + ((g + i) % P_RING) * 8);
    g += n;
  }
}

// ---- rank 1: O rescale and epilogue (warps 4-11) --------------------------------------------

__device__ void epilogue_role(const Ctx &c, uint32_t tmem, int w, int lane) {
  const DecodeParams &p = *c.p;
  Bars &br = *c.bars;
  const int q = w & 3, hf = (w - 4) >> 2;
  const int r = q * 32 + lane;
  // the thread's 16-byte units of the 16 KB P image (unit ch * 128 + r: key
  // chunk ch, row r): e, e + 256, e + 512, e + 768; with `help` only the
  // four warps of rows 0-63 run here and copy those rows' 512 units
  const bool help = p.help;
  const int e = help ? ((w - 4) >> 2) * 64 + (w & 3) * 32 + lane : (w - 4) * 32 + lane;
  auto unit = [&](int k) { return help ? (2 * k + (e >> 6)) * 128 + (e & 63) : e + 256 * k; };
  const uint32_t lt = tmem + ((uint32_t)(q * 32) << 16) + TM_O + hf * 256;
  const uint32_t pbuf = smem_u32(c.base + OFF_RCV_P);
  const uint32_t gfree0 = mapa(smem_u32(&br.gfree[0]), 0);
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
      const uint32_t b = g & 1, u = g >> 1, gs = g % P_RING;
      // 1. the message is published: load it (P is the 16 KB MMA operand
      //    image) with plain L2 loads, before waiting for the shared buffer,
      //    so the L2 latency overlaps PV(g-2).  The bulk-copy engine would
      //    queue it behind this SM's V loads.  .cg: the slot was rewritten by
      //    another SM since this SM last read it.
      if (!warp_wait_cluster(c, &br.p_full[gs], (g / P_RING) & 1)) return false;
      const uint8_t *slot = ring_slot(p, c.part, g);
      const uint4 *src = reinterpret_cast<const uint4 *>(slot);
      uint4 v[4];
#pragma unroll
      for (int k = 0; k < 4; k++) v[k] = __ldcg(src + unit(k));
      const Meta *m = reinterpret_cast<const Meta *>(slot + kPBytes);
      const uint4 f0 = __ldcg(reinterpret_cast<const uint4 *>(m->flags));
      const uint4 f1 = __ldcg(reinterpret_cast<const uint4 *>(m->flags) + 1);
      const float alpha = __ldcg(&m->alpha[r]);
      if (tile == t1 - 1) ell = __ldcg(&m->ell[r]);
      // 2. shared buffer b is free once PV(g-2) is done
      if (!warp_wait(c, &br.p_empty[b], (u & 1) ^ 1)) return false;
#pragma unroll
      for (int k = 0; k < 4; k++) st_shared_v4(pbuf + b * kPBytes + unit(k) * 16, v[k]);
      // The slot goes back to rank 0 once this warp's loads are done: the P
      // chunks are consumed by the stores above, and this instruction
      // consumes the meta values, so no load is in flight at the arrive.  A
      // release arrive would also wait for the shared-memory stores and
      // costs far more.
      {
        uint32_t dep;
        asm volatile("add.u32 %0, %1, %2;" : "=r"(dep) : "r"(__float_as_uint(alpha)), "r"(__float_as_uint(ell)));
        asm volatile("" ::"r"(dep), "r"(f0.x), "r"(f1.w));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&br.p_land[b]));
        mbar_arrive_remote_relaxed(gfree0 + gs * 8);
      }
      // (with `help` only the flags of softmax warps 4, 5, 8 and 9)
      const uint32_t fl = help ? f0.x | f0.y | f1.x | f1.y : f0.x | f0.y | f0.z | f0.w | f1.x | f1.y | f1.z | f1.w;
      if (fl != 0u) {  // rare: O *= alpha after PV(g-1), before PV(g)
        if (!warp_wait(c, &br.o_done[(g - 1) & 1], ((g - 1) >> 1) & 1)) return false;
        tc_fence_after();
        for (int cc = 0; cc < 8; cc++) {
          uint32_t o[32];
          tmem_ld32(lt + cc * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; j++) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
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
    if (!warp_wait(c, &br.o_done[(g - 1) & 1], ((g - 1) >> 1) & 1)) return false;
    tc_fence_after();
    const float inv = ell > 0.f ? 1.f / ell : 0.f;
    // Split partials are stored chunk-major, [slot][64 chunks of 8 columns]
    // [128 rows][8 floats]: the 32 lanes of a warp (32 consecutive rows)
    // store one chunk as 1 KB of contiguous memory.  The TMEM load of the
    // next 32 columns is in flight while this thread stores the current ones.
    float *wbase = p.ws_o + ((size_t)ri.slot * 64 + hf * 32) * (M_TILE * 8) + (size_t)r * 8;
    uint32_t o[2][32];
    tmem_ld32(lt, o[0]);
#pragma unroll
    for (int cc = 0; cc < 8; cc++) {
      tmem_wait_ld();
      if (cc + 1 < 8) tmem_ld32(lt + (cc + 1) * 32, o[(cc + 1) & 1]);
      uint32_t(&v)[32] = o[cc & 1];
      if (!ri.ok) continue;
      if (ri.nsplit <= 1) {
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; j++) w[j] = pack_bf16(__uint_as_float(v[2 * j]) * inv, __uint_as_float(v[2 * j + 1]) * inv);
        __nv_bfloat16 *dst = orow + cc * 32;
        if (p.out_v8) {  // 32-byte stores: whole L2 sectors of the row
          st_global_v8(dst, *reinterpret_cast<const uint32_t(*)[8]>(&w[0]));
          st_global_v8(dst + 16, *reinterpret_cast<const uint32_t(*)[8]>(&w[8]));
        } else {
          uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
          for (int j = 0; j < 4; j++) d4[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; j++) v[j] = __float_as_uint(__uint_as_float(v[j]) * inv);
#pragma unroll
        for (int j = 0; j < 4; j++)
          st_global_v8(wbase + (size_t)(cc * 4 + j) * (M_TILE * 8), *reinterpret_cast<const uint32_t(*)[8]>(&v[8 * j]));
      }
    }
    return true;
  });
}

// ---- kernel ---------------------------------------------------------------------

template <bool kGather, bool kDual>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(threads_of(kGather), 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap kb_map,
                     const __grid_constant__ CUtensorMap v_map, const __grid_constant__ CUtensorMap q_map,
                     const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // the shared-memory map needs a 1024-aligned base
    if (threadIdx.x == 0) atomicOr(p.status, MLA_STATUS_SMEM_ALIGN);
    return;
  }
  uint8_t *base = smem_raw;
  Bars &br = *reinterpret_cast<Bars *>(base + OFF_BARS);
  const uint32_t rank = cluster_ctarank();
  const Ctx c{&p, base, &br, rank, (int)cluster_id_x()};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // with `help`, four warps of rows 64-127 (all padding) gather instead of
  // running the softmax (rank 0) or the O epilogue (rank 1)
  const bool help = kGather && p.help;
  const uint32_t n_gather = gather_threads(help), n_soft = softmax_warps(help);
  if (threadIdx.x == 0) {
    for (int s = 0; s < 3; s++) {
      mbar_init(smem_u32(&br.kv_full[s]), kGather ? n_gather : 1);
      mbar_init(smem_u32(&br.kv_empty[s]), 1);
      mbar_init(smem_u32(&br.kv_full_b[s]), kGather ? n_gather : 1);
      mbar_init(smem_u32(&br.kv_empty_b[s]), 1);
      mbar_init(smem_u32(&br.raw_full[s]), n_gather);
    }
    for (int i = 0; i < kMaskRing; i++) mbar_init(smem_u32(&br.mfull[i]), kGather ? 2 : 1);
    for (int i = 0; i < P_RING; i++) {
      mbar_init(smem_u32(&br.gfree[i]), n_soft);
      mbar_init(smem_u32(&br.pwritten[i]), n_soft);
      mbar_init(smem_u32(&br.p_full[i]), 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(smem_u32(&br.s_full[b]), 1);
      mbar_init(smem_u32(&br.s_free[b]), n_soft);
      mbar_init(smem_u32(&br.p_land[b]), n_soft);
      mbar_init(smem_u32(&br.p_empty[b]), 1);
      mbar_init(smem_u32(&br.o_ready[b]), n_soft);
      mbar_init(smem_u32(&br.o_done[b]), 1);
    }
    mbar_init(smem_u32(&br.q_ready), n_soft);
    for (int h = 0; h < 2; h++) {
      mbar_init(smem_u32(&br.xfull[h]), 2);   // the two writer warps of the round
      mbar_init(smem_u32(&br.xempty[h]), 4);  // the four reader warps
    }
    for (int q = 0; q < 4; q++)
      for (int b = 0; b < 2; b++) mbar_init(smem_u32(&br.lsum[q][b]), 2);
    br.abort = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&br.tmem_base), TM_COLS);
    tmem_relinquish();
  }
  if (!kGather && threadIdx.x == 0) prefetch_tensormap(rank == 0 ? (const void *)&k_map : (const void *)&v_map);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote arrive or copy
  const uint32_t tmem = br.tmem_base;
  // Everything above overlaps the kernel before this one (the schedule);
  // no input is read before this point.  The combine kernel may launch once
  // every CTA has finished its pieces (grid_dep_trigger below): launched
  // earlier, its blocks would only sit beside these CTAs waiting.
  grid_dep_wait();

  // (warps 6, 7, 10, 11: bit 1 of the warp index set among the softmax warps)
  const bool soft_helper = help && warp >= 4 && warp < 4 + kSoftmaxWarps && (warp & 2);
  if (kGather) {
    int gt = -1;
    if (warp == 0 || warp == 3 || warp == 13 || warp == 14)
      gt = (warp == 0 ? 0 : warp == 3 ? 32 : warp == 13 ? 64 : 96) + lane;
    else if (soft_helper)
      gt = 128 + (warp == 6 ? 0 : warp == 7 ? 32 : warp == 10 ? 64 : 96) + lane;
    if (gt >= 0) {
      if (help) producer_gather<4>(c, &q_map, gt);
      else producer_gather<2>(c, &q_map, gt);
    }
  } else if (warp == 0) {
    producer_tma(c, rank == 0 ? &k_map : &v_map, &kb_map, &q_map, lane);
  }
  if (warp == 1) {
    if (rank == 0) mma_qk<kGather, kDual>(c, tmem);
    else mma_pv<kGather>(c, tmem);
  }
  if (warp == waiter_warp(kGather)) {
    if (rank == 0) qk_waiter<kGather>(c, lane);
    else pv_waiter<kGather>(c, lane);
  }
  if (warp == 2 && lane == 0 && rank == 0) p_publisher(c);
  if (warp >= 4 && warp < 4 + kSoftmaxWarps && !soft_helper) {
    if (rank == 0) softmax_role<kGather, kDual>(c, tmem, warp, lane);
    else epilogue_role(c, tmem, warp, lane);
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  grid_dep_trigger();
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

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (a function-local static: initialised exactly once even when several
// threads make their first call together).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    cudaDriverEntryPointQueryResult q;
    void *f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, cudaStream_t stream, cudaEvent_t ev_before,
                          cudaEvent_t ev_after) {
  const bool gather = p.kv_format != MLA_KV_BF16 || p.topk_len > 0;
  CUtensorMap maps[4];
  memset(maps, 0, sizeof maps);
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint32_t estr[4] = {1, 1, 1, 1};
  if (!gather) {
    // The page pool as a 4-D tensor [page][9 blocks][64 tokens][64 dims] of
    // bf16 (strides 73728, 128 and 1152 bytes); a box = column blocks 0-4 or
    // 5-8 of a page (K, rank 0) or blocks 0-7 (V, rank 1), 128-byte swizzle.
    cuuint64_t dims[4] = {64, (cuuint64_t)PAGE, 9, (cuuint64_t)p.num_pages};
    cuuint64_t strides[3] = {(cuuint64_t)D_QK * 2, 128, (cuuint64_t)D_QK * 2 * PAGE};
    // K blocks [0, split) and [split, 9) (split = 4 for the dual GEMM, else 5), V
    const cuuint32_t nblk[3] = {p.dual ? 4u : 5u, p.dual ? 5u : 4u, 8u};
    for (int m = 0; m < 3; m++) {
      cuuint32_t box[4] = {64, (cuuint32_t)PAGE, nblk[m], 1};
      CUresult r = fn(&maps[m], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint8_t *>(p.kv), dims, strides,
                      box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
  }
  {
    // The queries as a 3-D tensor [9 blocks][B*T*H rows][64 dims] (strides
    // 128 and 1152 bytes); one box = 64 query rows in the K layout.  Rows
    // past the end read as zeros.
    cuuint64_t dims[3] = {64, (cuuint64_t)p.B * p.T * p.H, 9};
    cuuint64_t strides[2] = {(cuuint64_t)D_QK * 2, 128};
    cuuint32_t box[3] = {64, 64, 9};
    CUresult r = fn(&maps[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16 *>(p.q), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  const size_t smem = kSmemBytes;
  // (the dual GEMM's exchange area lies in the gather kernel's raw ring: the
  // host selects it for the page path only)
  auto kern = gather ? decode_tc_kernel<true, false>
                     : (p.dual ? decode_tc_kernel<false, true> : decode_tc_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (ev_before) cudaEventRecord(ev_before, stream);
  // A programmatic dependent of the previous kernel of the stream (normally
  // the schedule): set-up runs while that kernel finishes, inputs are read
  // after grid_dep_wait().
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.num_parts);
  cfg.blockDim = dim3(threads_of(gather));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], p);
  if (ev_after) cudaEventRecord(ev_after, stream);
  return e;
}

}  // namespace mla
