/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) MLA decode library.
 *
 * Multi-head latent attention decode: every query head of a sequence attends
 * to one shared latent KV row per cached token (STAGE_D2.md, "DSV4 is MQA":
 * Q is per head, K/V has a single head shared by all query heads).  A row
 * holds 576 values, a 512-wide no-RoPE latent followed by 64 RoPE values; the
 * RoPE part is simply one more block of the QK reduction and V is the first
 * 512 values (FlashMLA issue #169 "dual gemm": RoPE behaves like an extra
 * block of size 64; the D_ROPE / D_NOPE split of the quoted kernel).  For
 * query row (b, t, h):
 *
 *   s_n = softmax_scale * sum_{d<576} q[b,t,h,d] * K_n[d]      n in N(b,t)
 *   lse = ln sum_n exp(s_n)                  (natural log; -inf if N empty)
 *   out = sum_n exp(s_n - lse) * K_n[0:512]  (0 if N empty)
 *
 * where N(b,t) = {n < s_k}                       dense
 *               {n < s_k - T + t + 1}           causal (query token t of T)
 *               {topk[b,t,j] : j, != -1}        sparse top-k (distinct)
 * and K_n is the cache row of logical token n of sequence b, found at page
 * block_table[b][n / 64], slot n % 64 (vLLM MlaQuery.insert: page, offset =
 * slot // page_size, slot % page_size).
 *
 * Ownership: the caller owns every buffer.  The library allocates no device
 * memory of its own, with one exception: mla_decode_noalloc keeps one fixed
 * scratch array per device.  TMA tensor maps are encoded on the host at each call and passed as
 * kernel parameters.  Every call is asynchronous on `stream` and never
 * synchronises the host, except mla_device_status().
 *
 * CUDA graphs: mla_decode_metadata, mla_decode, mla_kv_insert and
 * mla_query_absorb can be captured into a CUDA graph on `stream` once the
 * calling thread has made the same kind of call outside capture (the first
 * call does one-time host set-up).  A replay uses the buffers seen at
 * capture and reads their contents at replay time; the split-KV schedule is
 * a device kernel, so it follows the sequence lengths of each replay.
 *
 * Errors: each call returns MLA_OK (0) or a negative code; the text of the
 * last error of the calling thread is kept for mla_last_error_string().
 * Argument checks happen on the host before anything is launched: a call that
 * returns an error has enqueued nothing.  Values that only the device can see
 * (a page id outside the pool, a top-k index at or beyond s_k, a negative
 * s_k) never fault or trap: the row is skipped (treated as -1 / length 0) and
 * a bit is set in a device status word that mla_device_status() reads.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_OK 0
#define MLA_ERR_INVALID_ARG (-1) /* null/misaligned pointer, bad size or flag */
#define MLA_ERR_UNSUPPORTED (-2) /* valid request this library does not serve */
#define MLA_ERR_WORKSPACE (-3)   /* workspace null or smaller than required   */
#define MLA_ERR_CUDA (-4)        /* a CUDA runtime/driver call failed         */

#define MLA_KV_BF16 0     /* row = 576 bf16 (1152 bytes)                        */
#define MLA_KV_FP8_E4M3 1 /* row = 512 e4m3 bytes + 64 bf16 RoPE (640 bytes),
                             plus 4 fp32 scales per row in kv_scales            */
#define MLA_KV_FP8_E4M3_TENSOR 2 /* row = 576 e4m3 bytes, RoPE included (576 bytes),
                                  one fp32 scale for the whole cache */

/* Device status bits (mla_device_status). */
#define MLA_STATUS_BAD_PAGE 1u      /* block_table entry outside [0, num_pages) */
#define MLA_STATUS_BAD_TOPK 2u      /* top-k index >= s_k or < -1               */
#define MLA_STATUS_BAD_SEQLEN 4u    /* negative s_k, or more pages than max_pages */
#define MLA_STATUS_WAIT_TIMEOUT 8u  /* a bounded device wait gave up            */
#define MLA_STATUS_SMEM_ALIGN 16u   /* dynamic shared memory not 1024-byte aligned:
                                       the decode kernel did nothing */

/* Limits of this library. */
#define MLA_PAGE_SIZE 64
#define MLA_MAX_HEADS 128
#define MLA_MAX_QUERY_TOKENS 16
#define MLA_MAX_ITEMS 8192 /* work items = B * ceil(T*H/128), or B*T with top-k */

/* cudaStream_t-compatible handle (a CUstream). NULL = the legacy stream. */
typedef struct CUstream_st *mla_stream_t;

/*
 * Number of workers the split-KV partition should target on `device`: the
 * decode kernel runs one persistent cluster of two CTAs per worker, so this
 * is the SM count / 2 (76 on a 152-SM GB300).  Returns <= 0 on error.
 */
int mla_default_num_parts(int device);

/* Work items of a request (see mla_decode_metadata), or a negative code. */
int mla_decode_num_items(int B, int H, int T, int topk);

/*
 * Element counts of the two metadata arrays for a request:
 *   tile_md     int32 [num_parts][8]
 *   num_splits  int32 [num_items + 1]
 */
int mla_decode_metadata_sizes(int B, int H, int T, int topk, int num_parts,
                              size_t *tile_md_elems, size_t *num_splits_elems);

/*
 * Split-KV scheduling (STAGE_D2.md, "Grid vs. Persistent Tile Scheduler": a
 * persistent scheduler balances variable sequence lengths over a fixed set
 * of workers).  One small device kernel on `stream` reads cache_seqlens and
 * writes the partition of all key tiles over num_parts workers.
 *
 *   cache_seqlens  device int32 [B]            s_k per sequence (>= 0)
 *   B, H, T        batch, query heads (1..128), query tokens (1..16)
 *   topk           0 = dense/causal; > 0 = top-k length (keys per query token)
 *   causal         0/1; must be 0 when topk > 0
 *   num_parts      workers (>= 1); pass mla_default_num_parts(device)
 *   tile_md        device int32 [num_parts][8], written
 *   num_splits     device int32 [num_items + 1], written
 *
 * Rule (identical on host and device; one 64-key tile per cache page):
 * items are M tiles of up to 128 query rows (row = t*H + h) per sequence,
 * item mt * B + b for M tile mt of sequence b (m-tile-major: the workers that
 * hold the same tile range of a sequence's M tiles then run at the same time
 * and share its pages through L2), or one query token per item with top-k
 * (item b * T + t); item i has n_i key tiles (ceil(s_k/64);
 * causal: ceil(min(s_k, s_k - T + t_last + 1)/64); top-k: ceil(topk/64)) and
 * costs n_i + 4 on a line; the line is cut into num_parts equal segments of
 * L = ceil(total / num_parts) and each tile belongs to the segment holding
 * its coordinate.  tile_md[p] = {begin_item, begin_tile, last_item,
 * end_tile (exclusive), first_piece, begin_at_item_start, 0, 0}; num_splits
 * is the exclusive prefix over items of the number of workers per item.
 * The arrays are only meaningful to mla_decode with the same B, H, T, topk,
 * causal, num_parts and cache_seqlens.
 */
int mla_decode_metadata(const int32_t *cache_seqlens, int B, int H, int T,
                        int topk, int causal, int num_parts, int32_t *tile_md,
                        int32_t *num_splits, mla_stream_t stream);

/*
 * Bytes of workspace mla_decode needs: fp32 partial outputs and partial LSEs
 * of the split items, (num_items + num_parts) x 128 rows x (512 + 1) floats,
 * plus a ring of 8 x 17.5 KB per worker through which the two SMs of a
 * worker pass the softmax probabilities, each part rounded up to 256 bytes.
 * The workspace needs no initialisation and may be reused by later calls on
 * the same stream (calls that overlap on the GPU need separate workspaces).
 */
size_t mla_decode_workspace_bytes(int B, int H, int T, int topk, int num_parts);

/*
 * MLA decode attention (the formula at the top of this file).
 *
 *   q              device bf16 [B][T][H][576]   (row-major, 16-byte aligned)
 *   kv_cache       device, MLA_KV_BF16: bf16 [num_pages][64][576];
 *                  MLA_KV_FP8_E4M3: bytes [num_pages][64][640];
 *                  MLA_KV_FP8_E4M3_TENSOR: bytes [num_pages][64][576]
 *                  (16-byte aligned)
 *   kv_format      MLA_KV_BF16, MLA_KV_FP8_E4M3 or MLA_KV_FP8_E4M3_TENSOR
 *   num_pages      pages in the pool; page_size must be 64
 *   block_table    device int32 [B][max_pages]: page of the j-th 64 tokens
 *   cache_seqlens  device int32 [B]: s_k per sequence
 *   topk_indices   device int32 [B][T][topk] or NULL: token positions within
 *                  the sequence, -1 = unused slot; requires causal == 0.
 *                  The positions of one (b, t) list must be distinct (a
 *                  top-k selection names each cache token at most once;
 *                  -1 may repeat).  This is a precondition, not checked: a
 *                  position listed twice would be loaded and weighted twice,
 *                  which is not the attention defined above.
 *   gathered       device int32 [B][T][topk] or NULL (top-k only): if given,
 *                  the kernel writes, per slot, the token position whose row
 *                  it loaded, or -1 for a slot it skipped
 *   kv_scales      device fp32 [num_pages][64][4] for MLA_KV_FP8_E4M3
 *                  (value = e4m3(byte) * kv_scales[page][slot][d / 128]);
 *                  one device fp32 for MLA_KV_FP8_E4M3_TENSOR (value =
 *                  e4m3(byte) * kv_scales[0] for all 576 values: the
 *                  reciprocal of the k_scale_inv mla_kv_insert used); else
 *                  NULL
 *   softmax_scale  > 0 (1/sqrt(192) for the 128 no-PE + 64 RoPE query dims)
 *   causal         0/1
 *   tile_md, num_splits, num_parts   from mla_decode_metadata
 *   workspace      device, >= mla_decode_workspace_bytes(...), 256-aligned
 *   out            device bf16 [B][T][H][512], written
 *   lse            device fp32 [B][H][T], written (natural log)
 *
 * Launches the decode kernel and the LSE combine kernel (which merges the
 * items split over several workers) on `stream`, both as programmatic
 * dependents of the kernel before them: the decode kernel sets itself up
 * while the previous kernel of the stream (normally mla_decode_metadata's)
 * finishes and reads no input before that kernel has completed; the
 * combine kernel launches as the decode kernel's CTAs finish.  Cache rows past s_k in
 * a sequence's last page are read but carry zero weight; they must hold
 * finite values (a NaN there would reach `out` through 0 * NaN).
 */
int mla_decode(const void *q, const void *kv_cache, int kv_format,
               int num_pages, int page_size, const int32_t *block_table,
               int max_pages, const int32_t *cache_seqlens,
               const int32_t *topk_indices, int topk, int32_t *gathered,
               const float *kv_scales, float softmax_scale, int causal,
               const int32_t *tile_md, const int32_t *num_splits,
               int num_parts, void *workspace, size_t workspace_bytes,
               void *out, float *lse, int B, int T, int H,
               mla_stream_t stream);

/*
 * Size of the fixed device scratch of mla_decode_noalloc (64 MiB per device).
 */
#define MLA_NOALLOC_SCRATCH_BYTES (64u << 20)

/*
 * MLA decode for callers that cannot allocate device memory.  (No counterpart
 * on the source pages: this is a convenience of this library.)
 *
 * Some callers cannot provide the schedule arrays and the workspace that
 * mla_decode_metadata / mla_decode take: the host program may own every byte
 * of device memory (a runtime that plans all of its memory up front, or a
 * plugin contract that forbids the plugin from allocating), or the call may
 * come through a foreign-function layer with no device allocator at hand.
 * This entry point takes the same inputs and outputs as mla_decode (no
 * `gathered` record) and keeps its scratch in one array of
 * MLA_NOALLOC_SCRATCH_BYTES inside the library's device memory, which every
 * GPU that loads the library holds until the process exits.  It runs the same
 * metadata, decode and combine kernels, with mla_default_num_parts(device)
 * workers, and allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library call.
 *
 *   Limits: a request fits when its schedule (num_parts * 32 bytes and
 *   (num_items + 1) * 4 bytes, each rounded up to 256) plus
 *   mla_decode_workspace_bytes(B, H, T, topk, num_parts) is at most
 *   MLA_NOALLOC_SCRATCH_BYTES, with num_parts = mla_default_num_parts(device).
 *   On a 152-SM GB300 (76 workers) that is at most 138 work items: B <= 138
 *   at T * H <= 128, B <= 69 at T * H = 256.  Larger requests return
 *   MLA_ERR_WORKSPACE, with the byte counts in mla_last_error_string(), and
 *   enqueue nothing; use mla_decode for those.
 *   Set-up: the first call on a device, with that device current, looks up
 *   the scratch's device address (cudaGetSymbolAddress); make that first call
 *   before any stream capture.
 *   Sharing: all calls on a device share the one scratch, which keeps the last
 *   call's contents (nothing in it needs to start at zero).  Calls whose
 *   kernels overlap on the GPU (different streams, or threads without
 *   ordering) race on it; issue them in order on one stream.
 *   Errors: as mla_decode; an argument error is reported before anything is
 *   enqueued.
 */
int mla_decode_noalloc(const void *q, const void *kv_cache, int kv_format,
                       int num_pages, int page_size, const int32_t *block_table,
                       int max_pages, const int32_t *cache_seqlens,
                       const int32_t *topk_indices, int topk,
                       const float *kv_scales, float softmax_scale, int causal,
                       void *out, float *lse, int B, int T, int H,
                       mla_stream_t stream);

/*
 * KV insert: the producer of the cache this library reads (vLLM kimi_k3
 * specialized-decode "mla.query" page, MlaQuery.insert: RMSNorm of the
 * latent KV row, then the write of that row and k_pe into its cache slot).
 * For each new token j with slot = slots[j] >= 0 (slot = page * page_size +
 * offset; -1 = skip):
 *   x      = the 512 latent values of row j (bf16, at kv_c + j * ld_kv)
 *   S      = sum(x_i^2), exact, rounded once to fp32
 *   mean   = fp32(fp32(S / 512) + eps)
 *   r      = fp32(1 / fp32(sqrt(mean)))  (0 if mean == 0)
 *   n_i    = bf16(fp32(fp32(x_i * w_kva[i]) * r))
 *            (fp32 steps and the bf16 rounding: IEEE, to nearest even)
 *   pe     = the 64 RoPE'd key values of row j (bf16, at k_pe + j * ld_pe)
 * and writes the cache row cache[page][offset] as
 *   MLA_KV_BF16:             n_0..n_511, pe_0..pe_63 (bf16, 1152 bytes)
 *   MLA_KV_FP8_E4M3:         per 128-value tile t: s_t = fp32(max|n| / 448),
 *                            at least 2^-126 (1 when the tile is all zeros), into
 *                            kv_scales[page][offset][t],
 *                            e4m3(fp32(n_i * fp32(1 / s_t)));
 *                            then pe as bf16 (640 bytes: the decode's FP8
 *                            rows, value = e4m3 * scale)
 *   MLA_KV_FP8_E4M3_TENSOR:  e4m3(fp32(n_i * k_scale_inv)), e4m3(fp32(pe_i *
 *                            k_scale_inv)) (576 bytes; the per-tensor
 *                            FP8 layout; mla_decode reads it with the one
 *                            scale 1 / k_scale_inv)
 * e4m3 = OCP FP8 E4M3, round to nearest even, saturated to +-448.  The sum
 * of squares is taken as integers (a bf16 square is an 8-bit integer squared
 * times a power of two), so the written bytes are a function of the inputs
 * alone, independent of the order of additions.  Inputs must be finite.
 * Slots must be distinct (two tokens writing one slot race).
 *
 *   kv_c, ld_kv   device bf16 rows, latent at columns 0..511, row stride ld_kv
 *                 elements (>= 512, multiple of 8; e.g. a fused qkv row with
 *                 kv_c = qkv + 1536 and ld_kv = 2112)
 *   k_pe, ld_pe   device bf16 rows, RoPE'd key at columns 0..63 (ld_pe >= 64,
 *                 multiple of 8)
 *   w_kva         device bf16 [512] RMSNorm weight;  eps >= 0
 *   slots         device int64 [N]
 *   kv_cache      device [num_pages][page_size][row bytes] of the format
 *   kv_scales     MLA_KV_FP8_E4M3: device fp32 [num_pages][page_size][4]
 *                 (written); otherwise unused
 *   k_scale_inv   MLA_KV_FP8_E4M3_TENSOR: device fp32 scalar; otherwise unused
 * All pointers 16-byte aligned (slots 8).  Asynchronous on stream.  A slot
 * outside [0, num_pages * page_size) other than -1 is skipped and sets
 * MLA_STATUS_BAD_PAGE.  Returns MLA_OK or a negative MLA_ERR_* code.
 */
int mla_kv_insert(const void *kv_c, int ld_kv, const void *k_pe, int ld_pe, const void *w_kva, float eps,
                  const int64_t *slots, int N, void *kv_cache, int kv_format, int num_pages, int page_size,
                  float *kv_scales, const float *k_scale_inv, mla_stream_t stream);

/*
 * Query absorption: the query rows `q` that mla_decode reads, from the query
 * part of the fused projection output (vLLM kimi_k3 specialized-decode
 * "mla.query" page, MlaQuery.kernel: q_a RMSNorm, Q_B, W_UK).  For each of
 * the N tokens (N = B * T; token n = b * T + t):
 *   x     = the 1536 q_a values of row n (bf16, at q_a + n * ld_qa)
 *   S     = sum(x_i^2), exact, rounded once to fp32
 *   mean  = fp32(fp32(S / 1536) + eps);  r = fp32(1 / fp32(sqrt(mean))) (0 if mean == 0)
 *   xq_i  = bf16(fp32(fp32(x_i * w_qa[i]) * r))
 *   qb[h][p] = bf16(sum_k w_qb[h * 192 + p][k] * xq_k)     p < 192
 *   q[n][h][l]       = bf16(sum_{p<128} qb[h][p] * w_uk[h][p][l])   l < 512
 *   q[n][h][512 + i] = qb[h][128 + i]                               i < 64
 * The sums of products accumulate in fp32 in tensor memory (Q_B and W_UK
 * are this library's tcgen05 GEMMs); the RMSNorm is exact as stated.  The
 * three kernels are chained by programmatic dependent launch.  A wait that
 * gives up sets MLA_STATUS_WAIT_TIMEOUT in the device status word.
 *
 *   q_a, ld_qa  device bf16 rows, q_a values at columns 0..1535, row stride
 *               ld_qa elements (>= 1536, multiple of 8; the fused row:
 *               ld_qa = 2112)
 *   w_qa        device bf16 [1536];  eps >= 0
 *   w_qb        device bf16 [H * 192][1536] (row h * 192 + p: head h, row p;
 *               rows 0..127 no-PE, 128..191 RoPE)
 *   w_uk        device bf16 [H][128][512]
 *   q           device bf16 [N][H][576], written
 *   workspace   device, >= mla_query_absorb_workspace_bytes(N, H), 256-byte
 *               aligned: xq bf16 [N][1536] at 0, then qb bf16 [N][H * 192] at
 *               the next multiple of 256 bytes (both left there)
 * All other pointers 16-byte aligned.  Asynchronous on `stream`.  Returns
 * MLA_OK or a negative MLA_ERR_* code.
 */
size_t mla_query_absorb_workspace_bytes(int N, int H);
int mla_query_absorb(const void *q_a, int ld_qa, const void *w_qa, float eps, const void *w_qb,
                     const void *w_uk, int N, int H, void *q, void *workspace, size_t workspace_bytes,
                     mla_stream_t stream);

/* Text of the calling thread's last error ("" if none). */
const char *mla_last_error_string(void);

/*
 * Reads and clears the device status word of the current device (an OR of
 * MLA_STATUS_* bits set by earlier kernels).  Synchronous: waits for all
 * work on the device.  Returns MLA_OK or MLA_ERR_CUDA.
 */
int mla_device_status(uint32_t *status);

/*
 * Profiling hook: when both are non-NULL cudaEvent_t handles, every later
 * mla_decode call on this thread records `before` on its stream right before
 * the decode kernel launch and `after` right after it (an event between
 * kernels keeps the next one from starting early; the combine kernel
 * is outside).  Pass NULL, NULL to stop.  Returns MLA_OK.
 */
int mla_profile_events(void *before, void *after);

/*
 * Selects, for later mla_decode and mla_decode_noalloc calls made on the
 * calling thread, how QK^T is computed for requests on a bf16 cache without
 * top-k whose items have at most 64 query rows (T * H <= 64):
 *   0 (default): as for larger items, M = 128 MMAs with the rows past the
 *     item zero;
 *   1: the dual GEMM of FlashMLA issue #169 ("dual gemm": a weight-stationary
 *     M = 64 MMA that computes two halves of the reduction in the two lane
 *     halves of tensor memory, the halves of the scores then added by the
 *     softmax warps): half the QK MMAs per key tile.
 * Both give the attention defined at the top of this file.  On GB300 the
 * dual GEMM measured slower on every H = 64 workload tried (e.g. 45 -> 51 us
 * for B = 16, H = 64, s_k = 4096): those workloads are bound by HBM or by the
 * row gather, not by the tensor pipe, and handing the partial scores between
 * the softmax warps lengthens each tile's path to P.  Returns MLA_OK.
 */
int mla_set_dual_gemm(int enable);

/*
 * Test hook for the failure path: the time limit, in nanoseconds, of every
 * bounded wait inside the decode kernel of later mla_decode and
 * mla_decode_noalloc calls made on the calling thread (0 restores the
 * default of 2 s).  A wait that runs out sets MLA_STATUS_WAIT_TIMEOUT; every
 * role of the kernel then gives up at its next wait, the kernel waits for
 * its own copies and MMAs in flight, frees its tensor memory and returns, and
 * the context stays usable.  The out and lse of such a call are undefined.
 * With a limit of a few microseconds, real waits of an ordinary call run
 * out, so a test can exercise this path without faulting or hanging the GPU.
 * Not meant for production calls.  Returns MLA_OK.
 */
int mla_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H */
