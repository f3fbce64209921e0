// Split-KV scheduling metadata (one CTA on the caller's stream).
//
// STAGE_D2.md, "Grid vs. Persistent Tile Scheduler": a static grid is enough
// for fixed-length decode, variable sequence lengths want a persistent
// scheduler over a fixed set of workers.  The rule (stated in mla_decode.h):
// item i costs n_i + FIXED_COST on a line, the line is cut into num_parts
// segments of L = ceil(total / num_parts), and a key tile belongs to the
// segment holding its coordinate C_i + FIXED_COST + k.
#include "common.cuh"

namespace mla {
namespace {

constexpr int kThreads = 1024;

__device__ inline int block_inclusive_scan(int v, int *warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) warp_sums[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += u;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  if (warp > 0) v += warp_sums[warp - 1];
  return v;
}

// largest i in [0, n] with C[i] <= x  (C nondecreasing, C[0] = 0 <= x)
__device__ inline int last_le(const int *C, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (C[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kThreads)
metadata_kernel(const int32_t *seqlens, int H, int T, int topk, int causal,
                int num_parts, int n_mt, int n_items, int32_t *tile_md,
                int32_t *num_splits, unsigned int *status) {
  __shared__ int C[MLA_MAX_ITEMS + 1];
  __shared__ int warp_sums[32];
  __shared__ int carry;
  const int tid = threadIdx.x;
  grid_dep_trigger();  // the decode kernel may set itself up meanwhile
  if (tid == 0) { carry = 0; C[0] = 0; }
  __syncthreads();
  // 1. cost line: C[i+1] = C[i] + FIXED_COST + n_i
  for (int base = 0; base < n_items; base += kThreads) {
    int i = base + tid;
    int w = 0;
    if (i < n_items)
      w = FIXED_COST + item_at(i, seqlens, n_items / (topk > 0 ? T : n_mt), H, T, topk, causal, status).ntiles;
    int incl = block_inclusive_scan(w, warp_sums);
    if (i < n_items) C[i + 1] = carry + incl;
    __syncthreads();
    if (tid == kThreads - 1) carry += incl;
    __syncthreads();
  }
  const int W = C[n_items];
  const int L = ceil_div(W, num_parts);
  // 2. one entry per part
  for (int p = tid; p < num_parts; p += kThreads) {
    int32_t *md = tile_md + (size_t)p * MD_STRIDE;
    long long lo_ll = (long long)p * L;
    if (lo_ll >= W) {
      md[0] = n_items; md[1] = 0; md[2] = n_items - 1; md[3] = 0;
      md[4] = 0; md[5] = 0; md[6] = 0; md[7] = 0;
      continue;
    }
    int lo = (int)lo_ll;
    int hi = min(lo + L, W);
    int a = last_le(C, n_items, lo);
    int z = last_le(C, n_items, hi - 1);
    int na = C[a + 1] - C[a] - FIXED_COST;
    int nz = C[z + 1] - C[z] - FIXED_COST;
    int bt = min(max(lo - C[a] - FIXED_COST, 0), na);
    int et = min(max(hi - C[z] - FIXED_COST, 0), nz);
    int fp = 0;
    if (na > 0) fp = max(p - (C[a] + FIXED_COST) / L, 0);
    md[0] = a; md[1] = bt; md[2] = z; md[3] = et;
    md[4] = fp; md[5] = (C[a] == lo) ? 1 : 0; md[6] = 0; md[7] = 0;
  }
  // 3. exclusive prefix of workers per item
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < n_items; base += kThreads) {
    int i = base + tid;
    int ns = 0;
    if (i < n_items) {
      int n = C[i + 1] - C[i] - FIXED_COST;
      if (n == 0) {
        ns = 1;
      } else {
        int first = C[i] + FIXED_COST;
        ns = (first + n - 1) / L - first / L + 1;
      }
    }
    int incl = block_inclusive_scan(ns, warp_sums);
    if (i < n_items) num_splits[i + 1] = carry + incl;
    __syncthreads();
    if (tid == kThreads - 1) carry += incl;
    __syncthreads();
  }
  if (tid == 0) num_splits[0] = 0;
}

}  // namespace

cudaError_t launch_metadata(const int32_t *seqlens, int B, int H, int T,
                            int topk, int causal, int num_parts, int n_mt,
                            int n_items, int32_t *tile_md, int32_t *num_splits,
                            unsigned int *status, cudaStream_t stream) {
  (void)B;
  metadata_kernel<<<1, kThreads, 0, stream>>>(seqlens, H, T, topk, causal,
                                              num_parts, n_mt, n_items,
                                              tile_md, num_splits, status);
  return cudaGetLastError();
}

}  // namespace mla
