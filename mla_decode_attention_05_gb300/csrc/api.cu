// C ABI of the MLA decode library: argument checks, workspace layout and
// kernel launches.  Nothing here computes attention; every step runs in the
// device kernels of this directory.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"

// Device status word (MLA_STATUS_* bits), one per device that loads the
// library.  Kernels receive its address as a parameter.
__device__ unsigned int g_mla_status;

namespace {

thread_local char g_err[512] = "";
thread_local cudaEvent_t g_ev_before = nullptr;
thread_local cudaEvent_t g_ev_after = nullptr;
thread_local unsigned long long g_wait_ns = mla::kDefaultWaitNs;
thread_local int g_dual_gemm = 0;

int fail(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_err[0] = '\0';
  return MLA_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int kMaxDevices = 64;
std::mutex g_status_mu;
unsigned int *g_status_ptr[kMaxDevices] = {};

// Address of the status word on the current device (looked up once per
// device with that device current).
int status_ptr(unsigned int **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(MLA_ERR_UNSUPPORTED, "device %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (g_status_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_mla_status);
    if (e != cudaSuccess)
      return fail(MLA_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
    g_status_ptr[dev] = static_cast<unsigned int *>(p);
  }
  *out = g_status_ptr[dev];
  return MLA_OK;
}

int n_mt_of(int H, int T) { return mla::ceil_div(T * H, mla::M_TILE); }

int check_shape(int B, int H, int T, int topk) {
  if (B < 1) return fail(MLA_ERR_INVALID_ARG, "B = %d must be >= 1", B);
  if (H < 1 || H > MLA_MAX_HEADS) return fail(MLA_ERR_INVALID_ARG, "H = %d not in [1, %d]", H, MLA_MAX_HEADS);
  if (T < 1 || T > MLA_MAX_QUERY_TOKENS)
    return fail(MLA_ERR_INVALID_ARG, "T = %d not in [1, %d]", T, MLA_MAX_QUERY_TOKENS);
  if (topk < 0) return fail(MLA_ERR_INVALID_ARG, "topk = %d must be >= 0", topk);
  long long items = topk > 0 ? (long long)B * T : (long long)B * n_mt_of(H, T);
  if (items > MLA_MAX_ITEMS)
    return fail(MLA_ERR_UNSUPPORTED, "%lld work items exceed the limit %d", items, MLA_MAX_ITEMS);
  return MLA_OK;
}

int items_of(int B, int H, int T, int topk) { return topk > 0 ? B * T : B * n_mt_of(H, T); }

struct WsLayout {
  size_t lse_off, o_off, p_off, total;
};

WsLayout ws_layout(int n_items, int num_parts) {
  size_t slots = (size_t)n_items + (size_t)num_parts;
  WsLayout l;
  l.lse_off = 0;
  size_t lse_bytes = slots * mla::M_TILE * sizeof(float);
  l.o_off = (lse_bytes + 255) / 256 * 256;
  size_t o_bytes = slots * mla::M_TILE * mla::D_V * sizeof(float);
  l.p_off = (l.o_off + o_bytes + 255) / 256 * 256;
  size_t p_bytes = (size_t)num_parts * mla::P_RING * mla::P_SLOT_BYTES;
  l.total = (l.p_off + p_bytes + 255) / 256 * 256;
  return l;
}

}  // namespace

namespace mla {
// Records the text of an error for mla_last_error_string() (used by the
// entry points of other translation units).
void set_last_error(const char *msg) {
  snprintf(g_err, sizeof g_err, "%s", msg);
}
// Address of the device status word on the current device (for the entry
// points of other translation units).
int status_word(unsigned int **out) { return status_ptr(out); }
}  // namespace mla

extern "C" {

int mla_default_num_parts(int device) {
  int sms = 0;
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "SM count: %s", cudaGetErrorString(e));
  ok();
  return sms / 2 > 0 ? sms / 2 : 1;
}

int mla_decode_num_items(int B, int H, int T, int topk) {
  int rc = check_shape(B, H, T, topk);
  if (rc != MLA_OK) return rc;
  ok();
  return items_of(B, H, T, topk);
}

int mla_decode_metadata_sizes(int B, int H, int T, int topk, int num_parts,
                              size_t *tile_md_elems, size_t *num_splits_elems) {
  int rc = check_shape(B, H, T, topk);
  if (rc != MLA_OK) return rc;
  if (num_parts < 1) return fail(MLA_ERR_INVALID_ARG, "num_parts = %d must be >= 1", num_parts);
  if (!tile_md_elems || !num_splits_elems) return fail(MLA_ERR_INVALID_ARG, "null output pointer");
  *tile_md_elems = (size_t)num_parts * mla::MD_STRIDE;
  *num_splits_elems = (size_t)items_of(B, H, T, topk) + 1;
  return ok();
}

int mla_decode_metadata(const int32_t *cache_seqlens, int B, int H, int T,
                        int topk, int causal, int num_parts, int32_t *tile_md,
                        int32_t *num_splits, mla_stream_t stream) {
  int rc = check_shape(B, H, T, topk);
  if (rc != MLA_OK) return rc;
  if (!cache_seqlens || !tile_md || !num_splits) return fail(MLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(cache_seqlens, 4) || !aligned(tile_md, 4) || !aligned(num_splits, 4))
    return fail(MLA_ERR_INVALID_ARG, "int32 arrays must be 4-byte aligned");
  if (causal != 0 && causal != 1) return fail(MLA_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (causal && topk > 0) return fail(MLA_ERR_INVALID_ARG, "causal with top-k is not defined");
  if (num_parts < 1 || num_parts > 65535) return fail(MLA_ERR_INVALID_ARG, "num_parts = %d", num_parts);
  unsigned int *st = nullptr;
  if ((rc = status_ptr(&st)) != MLA_OK) return rc;
  cudaError_t e = mla::launch_metadata(cache_seqlens, B, H, T, topk, causal, num_parts,
                                       n_mt_of(H, T), items_of(B, H, T, topk), tile_md,
                                       num_splits, st, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "metadata launch: %s", cudaGetErrorString(e));
  return ok();
}

size_t mla_decode_workspace_bytes(int B, int H, int T, int topk, int num_parts) {
  if (check_shape(B, H, T, topk) != MLA_OK || num_parts < 1) return 0;
  return ws_layout(items_of(B, H, T, topk), num_parts).total;
}

int mla_decode(const void *q, const void *kv_cache, int kv_format,
               int num_pages, int page_size, const int32_t *block_table,
               int max_pages, const int32_t *cache_seqlens,
               const int32_t *topk_indices, int topk, int32_t *gathered,
               const float *kv_scales, float softmax_scale, int causal,
               const int32_t *tile_md, const int32_t *num_splits,
               int num_parts, void *workspace, size_t workspace_bytes,
               void *out, float *lse, int B, int T, int H,
               mla_stream_t stream) {
  int rc = check_shape(B, H, T, topk);
  if (rc != MLA_OK) return rc;
  if (!q || !kv_cache || !block_table || !cache_seqlens || !tile_md || !num_splits || !out || !lse)
    return fail(MLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16))
    return fail(MLA_ERR_INVALID_ARG, "q, kv_cache and out must be 16-byte aligned");
  if (!aligned(block_table, 4) || !aligned(cache_seqlens, 4) || !aligned(lse, 4) ||
      !aligned(tile_md, 4) || !aligned(num_splits, 4))
    return fail(MLA_ERR_INVALID_ARG, "int32/fp32 arrays must be 4-byte aligned");
  if (kv_format != MLA_KV_BF16 && kv_format != MLA_KV_FP8_E4M3 && kv_format != MLA_KV_FP8_E4M3_TENSOR)
    return fail(MLA_ERR_INVALID_ARG, "kv_format = %d", kv_format);
  if (kv_format == MLA_KV_FP8_E4M3 && (!kv_scales || !aligned(kv_scales, 16)))
    return fail(MLA_ERR_INVALID_ARG, "FP8 cache needs 16-byte aligned kv_scales");
  if (kv_format == MLA_KV_FP8_E4M3_TENSOR && (!kv_scales || !aligned(kv_scales, 4)))
    return fail(MLA_ERR_INVALID_ARG, "per-tensor FP8 cache needs kv_scales (one fp32 scale)");
  if (page_size != MLA_PAGE_SIZE) return fail(MLA_ERR_UNSUPPORTED, "page_size = %d (only 64)", page_size);
  if (num_pages < 1 || max_pages < 1) return fail(MLA_ERR_INVALID_ARG, "num_pages/max_pages < 1");
  if ((topk > 0) != (topk_indices != nullptr))
    return fail(MLA_ERR_INVALID_ARG, "topk_indices and topk > 0 go together");
  if (topk_indices && !aligned(topk_indices, 4)) return fail(MLA_ERR_INVALID_ARG, "topk_indices alignment");
  if (gathered && (topk == 0 || !aligned(gathered, 4)))
    return fail(MLA_ERR_INVALID_ARG, "gathered needs top-k and 4-byte alignment");
  if (causal != 0 && causal != 1) return fail(MLA_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (causal && topk > 0) return fail(MLA_ERR_INVALID_ARG, "causal with top-k is not defined");
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    return fail(MLA_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
  if (num_parts < 1 || num_parts > 65535) return fail(MLA_ERR_INVALID_ARG, "num_parts = %d", num_parts);
  const int n_items = items_of(B, H, T, topk);
  WsLayout wl = ws_layout(n_items, num_parts);
  if (!workspace || workspace_bytes < wl.total)
    return fail(MLA_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", wl.total, workspace_bytes);
  if (!aligned(workspace, 256)) return fail(MLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");

  unsigned int *st = nullptr;
  if ((rc = status_ptr(&st)) != MLA_OK) return rc;
  mla::DecodeParams p;
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.kv = static_cast<const uint8_t *>(kv_cache);
  p.kv_scales = kv_scales;
  p.block_table = block_table;
  p.seqlens = cache_seqlens;
  p.topk = topk_indices;
  p.gathered = gathered;
  p.tile_md = tile_md;
  p.num_splits = num_splits;
  p.ws_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + wl.lse_off);
  p.ws_o = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + wl.o_off);
  p.ws_p = static_cast<uint8_t *>(workspace) + wl.p_off;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.lse = lse;
  p.status = st;
  p.kv_format = kv_format;
  p.num_pages = num_pages;
  p.max_pages = max_pages;
  p.topk_len = topk;
  p.causal = causal;
  p.B = B;
  p.T = T;
  p.H = H;
  p.n_mt = n_mt_of(H, T);
  p.n_items = n_items;
  p.num_parts = num_parts;
  p.out_v8 = aligned(out, 32) ? 1 : 0;
  p.scale_log2 = softmax_scale * mla::LOG2E;
  p.wait_ns = g_wait_ns;
  // the M = 64 dual GEMM for QK, when selected, on the page path, when every
  // item has at most 64 query rows (the row-gather kernel's shared memory
  // holds its raw ring where the dual GEMM would hand over its scores)
  p.dual = (g_dual_gemm && kv_format == MLA_KV_BF16 && topk == 0 && T * H <= 64) ? 1 : 0;
  // the row-gather kernel, every item at most 64 query rows: rows 64-127 of
  // the M = 128 tile are padding, so their four softmax (rank 0) and
  // epilogue (rank 1) warps join the row gather instead
  p.help = ((kv_format != MLA_KV_BF16 || topk > 0) && (topk > 0 ? H : T * H) <= 64) ? 1 : 0;

  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = mla::launch_decode(p, s, g_ev_before, g_ev_after);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  e = mla::launch_combine(p, s);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "combine launch: %s", cudaGetErrorString(e));
  return ok();
}

int mla_kv_insert(const void *kv_c, int ld_kv, const void *k_pe, int ld_pe, const void *w_kva, float eps,
                  const int64_t *slots, int N, void *kv_cache, int kv_format, int num_pages, int page_size,
                  float *kv_scales, const float *k_scale_inv, mla_stream_t stream) {
  if (N < 0) return fail(MLA_ERR_INVALID_ARG, "N = %d must be >= 0", N);
  if (kv_format != MLA_KV_BF16 && kv_format != MLA_KV_FP8_E4M3 && kv_format != MLA_KV_FP8_E4M3_TENSOR)
    return fail(MLA_ERR_INVALID_ARG, "kv_format %d unknown", kv_format);
  if (num_pages < 1 || page_size < 1)
    return fail(MLA_ERR_INVALID_ARG, "num_pages = %d, page_size = %d must be >= 1", num_pages, page_size);
  if (ld_kv < mla::D_V || ld_kv % 8) return fail(MLA_ERR_INVALID_ARG, "ld_kv = %d: need >= 512, multiple of 8", ld_kv);
  if (ld_pe < mla::D_ROPE || ld_pe % 8)
    return fail(MLA_ERR_INVALID_ARG, "ld_pe = %d: need >= 64, multiple of 8", ld_pe);
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(MLA_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (N == 0) return ok();
  if (!kv_c || !k_pe || !w_kva || !slots || !kv_cache) return fail(MLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(kv_c, 16) || !aligned(k_pe, 16) || !aligned(w_kva, 16) || !aligned(kv_cache, 16) ||
      !aligned(slots, 8))
    return fail(MLA_ERR_INVALID_ARG, "kv_c, k_pe, w_kva, kv_cache must be 16-byte aligned, slots 8");
  if (kv_format == MLA_KV_FP8_E4M3 && (!kv_scales || !aligned(kv_scales, 16)))
    return fail(MLA_ERR_INVALID_ARG, "kv_scales must be a 16-byte aligned pointer for MLA_KV_FP8_E4M3");
  if (kv_format == MLA_KV_FP8_E4M3_TENSOR && (!k_scale_inv || !aligned(k_scale_inv, 4)))
    return fail(MLA_ERR_INVALID_ARG, "k_scale_inv must be a 4-byte aligned pointer for MLA_KV_FP8_E4M3_TENSOR");
  unsigned int *st = nullptr;
  int rc;
  if ((rc = status_ptr(&st)) != MLA_OK) return rc;
  mla::KvInsertParams p{};
  p.kv_c = static_cast<const __nv_bfloat16 *>(kv_c);
  p.k_pe = static_cast<const __nv_bfloat16 *>(k_pe);
  p.w_kva = static_cast<const __nv_bfloat16 *>(w_kva);
  p.slots = slots;
  p.cache = static_cast<uint8_t *>(kv_cache);
  p.kv_scales = kv_scales;
  p.k_scale_inv = k_scale_inv;
  p.status = st;
  p.n_slots = (long long)num_pages * page_size;
  p.ld_kv = ld_kv;
  p.ld_pe = ld_pe;
  p.N = N;
  p.kv_format = kv_format;
  p.eps = eps;
  cudaError_t e = mla::launch_kv_insert(p, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "kv insert launch: %s", cudaGetErrorString(e));
  return ok();
}

const char *mla_last_error_string(void) { return g_err; }

int mla_device_status(uint32_t *status) {
  if (!status) return fail(MLA_ERR_INVALID_ARG, "null status pointer");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "synchronize: %s", cudaGetErrorString(e));
  unsigned int v = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&v, g_mla_status, sizeof v);
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_mla_status, &zero, sizeof zero);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  *status = v;
  return ok();
}

int mla_set_dual_gemm(int enable) {
  g_dual_gemm = enable ? 1 : 0;
  return ok();
}

int mla_set_wait_limit_ns(uint64_t ns) {
  g_wait_ns = ns == 0 ? mla::kDefaultWaitNs : (unsigned long long)ns;
  return ok();
}

int mla_profile_events(void *before, void *after) {
  if (before && after) {
    g_ev_before = static_cast<cudaEvent_t>(before);
    g_ev_after = static_cast<cudaEvent_t>(after);
  } else {
    g_ev_before = nullptr;
    g_ev_after = nullptr;
  }
  return ok();
}

}  // extern "C"
