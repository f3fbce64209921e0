// Shared definitions of the MLA decode kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_decode.h"

namespace mla {

constexpr int D_QK = 576;    // latent (512) + RoPE (64)
constexpr int D_V = 512;     // V = first 512 values of the latent row
constexpr int D_ROPE = 64;
constexpr int PAGE = 64;     // tokens per cache page = keys per tile
constexpr int M_TILE = 128;  // query rows per work item
constexpr int FIXED_COST = 4;
constexpr int MD_STRIDE = 8; // ints per tile_md entry
constexpr int FP8_ROW = 640; // 512 e4m3 + 64 bf16 RoPE bytes
// P messages from the S engine to the O engine of a worker pass through a
// small ring in the workspace (L2-resident): P_RING slots of P_SLOT_BYTES.
constexpr int P_RING = 8;
constexpr int P_SLOT_BYTES = 17920;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// Everything a decode / combine kernel needs, by value.
struct DecodeParams {
  const __nv_bfloat16 *q;
  const uint8_t *kv;  // raw rows
  const float *kv_scales;
  const int32_t *block_table;
  const int32_t *seqlens;
  const int32_t *topk;
  int32_t *gathered;
  const int32_t *tile_md;
  const int32_t *num_splits;
  float *ws_lse;  // [slots][128] (log2 domain)
  float *ws_o;    // [slots][128][512]
  uint8_t *ws_p;  // [num_parts][P_RING][P_SLOT_BYTES]
  __nv_bfloat16 *out;
  float *lse;
  unsigned int *status;
  int kv_format;
  int num_pages;
  int max_pages;
  int topk_len;
  int causal;
  int B, T, H;
  int n_mt;     // M tiles per sequence (dense / causal)
  int n_items;
  int num_parts;
  int out_v8;        // out is 32-byte aligned: 32-byte stores
  float scale_log2;  // softmax_scale * log2(e)
  unsigned long long wait_ns;  // limit of every bounded device wait
  int dual;                    // every item has at most 64 query rows: QK as a dual GEMM (M = 64, .ws)
  int help;                    // row gather, every item has at most 64 query rows: the four
                               // softmax / epilogue warps of rows 64-127 gather instead
};

// Default limit of the decode kernel's bounded waits.
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s

// Geometry of one work item.
struct Item {
  int b;       // sequence
  int row0;    // first query row (row = t*H + h) of the item
  int rows;    // rows in the item (<= 128)
  int ntiles;  // 64-key tiles
  int kv_len;  // keys of the item's last row (dense/causal); topk length
};

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ inline int clamp_seqlen(int sk, unsigned int *status) {
  if (sk < 0) {
    atomicOr(status, MLA_STATUS_BAD_SEQLEN);
    return 0;
  }
  return sk;
}

// Item i: with top-k, query token i % T of sequence i / T; otherwise M tile
// i / B of sequence i % B (m-tile-major: a sequence's M tiles share its
// keys, and in this order the workers holding the same tile range of them
// run at the same time, so each page is read from HBM once).
__device__ inline Item item_at(int i, const int32_t *seqlens, int B, int H, int T,
                               int topk, int causal, unsigned int *status) {
  Item it;
  if (topk > 0) {
    it.b = i / T;
    int t = i % T;
    it.row0 = t * H;
    it.rows = H;
    it.kv_len = topk;
    it.ntiles = ceil_div(topk, PAGE);
    return it;
  }
  it.b = i % B;
  int mt = i / B;
  int sk = clamp_seqlen(seqlens[it.b], status);
  it.row0 = mt * M_TILE;
  int total = T * H;
  it.rows = min(M_TILE, total - it.row0);
  int k = sk;
  if (causal) {
    int t_last = (it.row0 + it.rows - 1) / H;
    k = min(max(sk - T + t_last + 1, 0), sk);
  }
  it.kv_len = k;
  it.ntiles = ceil_div(k, PAGE);
  return it;
}

// Keys visible to query token t (dense / causal).
__device__ inline int row_kv_len(int sk, int T, int t, int causal) {
  if (!causal) return sk;
  return min(max(sk - T + t + 1, 0), sk);
}

__device__ inline float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

// OCP FP8 E4M3 -> float (exact), written from the format: bias 7,
// subnormals at exponent 0, S.1111.111 is NaN.
__device__ inline float e4m3_to_float(uint32_t c) {
  uint32_t s = (c & 0x80u) << 24;
  uint32_t e = (c >> 3) & 0xFu;
  uint32_t m = c & 0x7u;
  float v;
  if (e == 0) {
    v = (float)m * 0.001953125f;  // m/8 * 2^-6
  } else {
    v = __uint_as_float(((e + 120u) << 23) | (m << 20));
    if (e == 0xFu && m == 0x7u) v = __uint_as_float(0x7FC00000u);
  }
  return __uint_as_float(__float_as_uint(v) | s);
}

// Programmatic dependent launch (griddepcontrol): a kernel launched with the
// programmatic-serialization attribute may begin while the kernel before it
// in the stream is still running.  grid_dep_wait() blocks until that kernel
// has completed and its memory operations are visible (a no-op for a kernel
// launched without the attribute), so it comes before the first read of any
// input; grid_dep_trigger() lets the next such kernel begin launching.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace mla

// Host-side launchers (one per translation unit).
namespace mla {
cudaError_t launch_metadata(const int32_t *seqlens, int B, int H, int T,
                            int topk, int causal, int num_parts, int n_mt,
                            int n_items, int32_t *tile_md, int32_t *num_splits,
                            unsigned int *status, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams &p, cudaStream_t stream,
                          cudaEvent_t ev_before, cudaEvent_t ev_after);
cudaError_t launch_combine(const DecodeParams &p, cudaStream_t stream);

// One KV insert call (mla_kv_insert), by value.
struct KvInsertParams {
  const __nv_bfloat16 *kv_c;  // latent rows, stride ld_kv elements
  const __nv_bfloat16 *k_pe;  // RoPE rows, stride ld_pe elements
  const __nv_bfloat16 *w_kva;
  const int64_t *slots;
  uint8_t *cache;
  float *kv_scales;
  const float *k_scale_inv;
  unsigned int *status;
  long long n_slots;  // num_pages * page_size
  int ld_kv, ld_pe;
  int N;
  int kv_format;
  float eps;
};
cudaError_t launch_kv_insert(const KvInsertParams &p, cudaStream_t stream);
void set_last_error(const char *msg);
int status_word(unsigned int **out);
}  // namespace mla
