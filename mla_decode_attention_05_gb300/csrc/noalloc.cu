// MLA decode for callers that cannot allocate device memory.
//
// mla_decode needs two small schedule arrays and a workspace that the caller
// allocates.  Some callers cannot do that: a host program may own every byte
// of device memory (a runtime that plans its memory up front, or a plugin
// contract that forbids the plugin from allocating), or the caller may reach
// this library through a foreign-function layer with no device allocator at
// hand.  This entry point takes only the inputs and outputs and keeps all of
// its scratch in one fixed array that lives in the library's own device
// memory: every GPU that loads the library holds MLA_NOALLOC_SCRATCH_BYTES of
// it until the process exits.  It runs the same three kernels as
// mla_decode_metadata + mla_decode, on the same number of workers.
#include <cstdio>
#include <mutex>

#include "common.cuh"

// The scratch.  In host code this name is only a host-side stand-in; the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint8_t *g_scratch_ptr[kMaxDevices] = {};

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

int fail(int code, const char *msg) {
  mla::set_last_error(msg);
  return code;
}

// Device address of the scratch on the current device, looked up on the
// first call made with that device current.
int scratch_ptr(uint8_t **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(MLA_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return fail(MLA_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[256];
      snprintf(msg, sizeof msg, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
      return fail(MLA_ERR_CUDA, msg);
    }
    g_scratch_ptr[dev] = static_cast<uint8_t *>(p);
  }
  *out = g_scratch_ptr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_noalloc(const void *q, const void *kv_cache, int kv_format,
                                  int num_pages, int page_size, const int32_t *block_table,
                                  int max_pages, const int32_t *cache_seqlens,
                                  const int32_t *topk_indices, int topk,
                                  const float *kv_scales, float softmax_scale, int causal,
                                  void *out, float *lse, int B, int T, int H,
                                  mla_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(MLA_ERR_CUDA, "cudaGetDevice failed");
  const int num_parts = mla_default_num_parts(dev);
  if (num_parts <= 0) return num_parts < 0 ? num_parts : fail(MLA_ERR_CUDA, "no workers");
  size_t md_elems = 0, ns_elems = 0;
  int rc = mla_decode_metadata_sizes(B, H, T, topk, num_parts, &md_elems, &ns_elems);
  if (rc != MLA_OK) return rc;
  const size_t md_bytes = round256(md_elems * sizeof(int32_t));
  const size_t ns_bytes = round256(ns_elems * sizeof(int32_t));
  const size_t ws_bytes = mla_decode_workspace_bytes(B, H, T, topk, num_parts);
  if (ws_bytes == 0) return fail(MLA_ERR_INVALID_ARG, "bad sizes");
  const size_t need = md_bytes + ns_bytes + ws_bytes;
  if (need > (size_t)MLA_NOALLOC_SCRATCH_BYTES) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "request needs %zu bytes of scratch, more than the fixed %zu of mla_decode_noalloc; "
             "use mla_decode with a caller-allocated workspace",
             need, (size_t)MLA_NOALLOC_SCRATCH_BYTES);
    return fail(MLA_ERR_WORKSPACE, msg);
  }
  uint8_t *scratch = nullptr;
  if ((rc = scratch_ptr(&scratch)) != MLA_OK) return rc;
  int32_t *tile_md = reinterpret_cast<int32_t *>(scratch);
  int32_t *num_splits = reinterpret_cast<int32_t *>(scratch + md_bytes);
  void *workspace = scratch + md_bytes + ns_bytes;
  // Check every argument before anything is enqueued: with no workspace,
  // mla_decode reports MLA_ERR_WORKSPACE exactly when all other arguments
  // are valid, and launches nothing.
  rc = mla_decode(q, kv_cache, kv_format, num_pages, page_size, block_table, max_pages,
                  cache_seqlens, topk_indices, topk, nullptr, kv_scales, softmax_scale, causal,
                  tile_md, num_splits, num_parts, nullptr, 0, out, lse, B, T, H, stream);
  if (rc != MLA_ERR_WORKSPACE) return rc == MLA_OK ? fail(MLA_ERR_CUDA, "unexpected validation result") : rc;
  // Nothing in the scratch has to start at zero: the metadata kernel writes
  // both schedule arrays and the decode kernel writes every workspace byte it
  // later reads, in stream order.
  rc = mla_decode_metadata(cache_seqlens, B, H, T, topk, causal, num_parts, tile_md, num_splits, stream);
  if (rc != MLA_OK) return rc;
  return mla_decode(q, kv_cache, kv_format, num_pages, page_size, block_table, max_pages,
                    cache_seqlens, topk_indices, topk, nullptr, kv_scales, softmax_scale, causal,
                    tile_md, num_splits, num_parts, workspace, ws_bytes, out, lse, B, T, H, stream);
}
