/*
 * pkv.h — C ABI of the paged KV-cache decode library (GB300, sm_103a).
 *
 * The library implements single-token decode attention over a paged KV cache,
 * with GQA head grouping, fp16/bf16 or INT8 (per-token or per-64-token-group
 * scale/zero-point) keys and values dequantised inside the kernels, and a
 * query-aware sparse mode that scores pages by a per-page channel bounding box
 * and attends only over the top-K pages.
 *
 * Sources, cited by short name and section:
 *   [Gemini page]      "GPU显存占用直降63%！Gemini KV Cache优化实战：FlashAttention-3适配全链路拆解"
 *   [KV-practice page] "LLM推理中的KV Cache优化与显存管理实践"
 *   [HBM-layout page]  "Transformer 推理的内存布局优化：从 HBM 带宽利用率的视角重新设计 KV Cache"
 *   [TinyServe page]   "LLM推理中的KV缓存优化技术与TinyServe实践"
 *
 * Conventions (every call):
 *   - Pointers named *_pages, q, out, k_new, v_new, block_table, seq_lens,
 *     positions, new_lens, sel_*, scores_out, workspace, dev_status and the
 *     pointer members of pkv_cache are DEVICE pointers owned by the caller.
 *     The library allocates no device memory and keeps no pointer after a call
 *     returns. `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *   - Calls are asynchronous on `stream`. A host-detectable error (null or
 *     misaligned pointer, unsupported shape or dtype, short workspace) is
 *     returned before anything is launched. Device pools, q and out must be
 *     16-byte aligned.
 *   - Device-detectable errors never trap: the kernel ORs a PKV_DEV_* bit into
 *     *dev_status (a caller-owned int32 the caller zeroes; may be NULL only if
 *     the caller accepts losing the report), skips the offending page or token,
 *     and finishes. Read *dev_status after synchronising the stream.
 *   - All calls are stateless and re-entrant; two calls that share a workspace
 *     must not run concurrently.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_ABI_VERSION 6

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or shape */
  PKV_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head_dim 96) */
  PKV_ERR_OUT_OF_PAGES = 3,  /* host allocator: not enough free pages */
  PKV_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  PKV_ERR_WORKSPACE = 5      /* workspace too small */
} pkv_status;

/* Bits ORed into *dev_status by the kernels. */
#define PKV_DEV_BAD_PAGE 1      /* block-table entry outside [0, num_pages) */
#define PKV_DEV_BAD_SELECTED 2  /* selected logical page outside the sequence */
#define PKV_DEV_BAD_POSITION 4  /* append slot beyond the block table / bad length */
#define PKV_DEV_TIMEOUT 8       /* a bounded wait inside a kernel gave up */
#define PKV_DEV_BAD_CONFIG 16   /* launch parameters a kernel refuses to run with */

/* PKV_U4: unsigned 4-bit codes, two per byte (the even channel in the low
 * nibble), for KV pools only. */
typedef enum { PKV_F16 = 0, PKV_BF16 = 1, PKV_F32 = 2, PKV_I8 = 3, PKV_U4 = 4 } pkv_dtype;

/* Who selects pages in pkv_page_score_topk. The pages score one query per page;
 * the group modes are this library's readings for query-head groups (GQA). */
typedef enum {
  PKV_SELECT_PER_HEAD = 0,   /* every query head selects its own pages */
  PKV_SELECT_GROUP_SUM = 1,  /* one list per kv head: the sum of its G heads' scores */
  PKV_SELECT_GROUP_MAX = 2   /* one list per kv head: the max of its G heads' scores */
} pkv_select_mode;

typedef enum {
  PKV_QUANT_NONE = 0,       /* kv_dtype F16 or BF16: values stored as is */
  PKV_QUANT_PER_TOKEN = 1,  /* kv_dtype I8 or U4: one (scale, zero) per token and kv head
                               [HBM-layout page, section 二; 4-bit: KV-practice page,
                               section 3.2] */
  PKV_QUANT_PER_GROUP64 = 2 /* kv_dtype I8: one (scale, zero) per 64 tokens and kv head
                               [Gemini page, 第一章] */
} pkv_quant;

/*
 * A paged KV cache (one layer). Fixed-size pages are allocated on demand and
 * need not be contiguous; a per-sequence block table maps logical page i to a
 * physical page id [HBM-layout page, sections 二 (layout C) and 三].
 *
 * Layouts (all row-major, device memory, caller-owned):
 *   k_pages, v_pages : [num_pages][num_kv_heads][page_size][head_dim] of kv_dtype
 *                      (I8: unsigned bytes u = code + 128; U4: [..][head_dim / 2]
 *                      bytes, channel 2i in the low nibble of byte i). Token
 *                      slot s of logical page i of a sequence holds its token
 *                      i * page_size + s.
 *   kv_sz            : I8 and U4 only, fp32 [num_pages][num_kv_heads][page_size / gran][4]
 *                      with gran = 1 (per token) or 64 (per group, I8 only); the
 *                      4 floats are (k_scale, k_zero, v_scale, v_zero).
 *                      Restoration: x = u * scale + zero, u the stored byte
 *                      (I8: u = code + 128 in [0, 255]; U4: u in [0, 15]).
 *   tail             : PER_GROUP64 only, fp32
 *                      [tail_rows][num_kv_heads][2 (K, V)][2 (group parity)][64][head_dim]:
 *                      original values of each sequence's open (partially filled)
 *                      64-token group, kept so that every append re-quantises
 *                      the open group from its members. Row b belongs to batch
 *                      row b of kv_append. Contents are managed by kv_append.
 *   page_meta        : optional (NULL = no sparse metadata), fp32
 *                      [num_pages][num_kv_heads][2][head_dim]: per channel, the
 *                      minimum (row 0) and maximum (row 1) of the page's valid
 *                      keys [TinyServe page, section 2.1]; kept in fp32
 *                      [TinyServe page, section 5.2]. For INT8 keys the box is
 *                      built from fl32(fl32((c + 128) * s) + z), for 4-bit keys
 *                      from fl32(fl32(u * s) + z).
 */
typedef struct {
  int32_t num_pages;
  int32_t page_size;     /* multiple of 16; multiple of 64 for PER_GROUP64 */
  int32_t num_kv_heads;
  int32_t head_dim;      /* 64 or 128 */
  pkv_dtype kv_dtype;    /* F16, BF16 (with QUANT_NONE), I8, or U4 (with QUANT_PER_TOKEN) */
  pkv_quant quant;
  void* k_pages;
  void* v_pages;
  float* kv_sz;
  float* tail;
  int32_t tail_rows;
  float* page_meta;
} pkv_cache;

/* Status text for a pkv_status value (static string). */
const char* pkv_status_string(pkv_status s);

/* PKV_ABI_VERSION of the loaded library. */
int32_t pkv_abi_version(void);

/*
 * Re-read the tuning variables PKV_ATTN_MMA, PKV_ATTN_RING_KB, PKV_ATTN_STAGES,
 * PKV_ATTN_CTAS_PER_SM and PKV_ATTN_COMB_RG from the environment. They only
 * choose among equivalent launch shapes (results never depend on them) and are
 * read once, by the first call that plans an attention launch; a process that
 * changes them later calls this. Not part of the pages' problem statement.
 */
void pkv_tuning_reload(void);

/*
 * kv_append — write new tokens' K and V into their pages.
 * [HBM-layout page, section 三 append_kv]: token position pos goes to logical
 * page pos / page_size, slot pos % page_size, through the block table.
 *   k_new, v_new : [batch][t_new][num_kv_heads][head_dim] of src_dtype (F16/BF16).
 *   block_table  : int32 [batch][max_pages] physical page ids (pages must
 *                  already be allocated for every written position).
 *   positions    : int32 [batch], position of the first new token of row b
 *                  (its current length).
 *   new_lens     : int32 [batch] tokens to write for row b (<= t_new), or NULL
 *                  for t_new each. The caller updates its seq_lens afterwards.
 * F16/BF16 caches store the values (converted to kv_dtype). INT8 caches
 * quantise: per token over head_dim values; per group over the group's
 * members, re-quantising the open group from the originals kept in `tail`
 * (closed groups never change). If page_meta is set, the bounding box of every
 * page the append touched is recomputed from the stored keys.
 * Quantiser (bit-exact definition, fp32 ops, ties to even):
 *   I8: s = (max - min) / 255; z = min; code = clamp(rint((x - z) / s), 0, 255) - 128,
 *       stored as the byte u = code + 128; a constant block stores s = 0 and
 *       codes -128 (bytes 0).
 *   U4: s = (max - min) / 15; z = min; u = clamp(rint((x - z) / s), 0, 15);
 *       a constant row stores s = 0 and codes 0.
 * Device errors: PKV_DEV_BAD_POSITION (slot beyond max_pages * page_size or
 * negative position / length), PKV_DEV_BAD_PAGE; the token is skipped.
 */
pkv_status pkv_kv_append(const pkv_cache* cache, int32_t batch, int32_t t_new,
                         const void* k_new, const void* v_new, pkv_dtype src_dtype,
                         const int32_t* block_table, int32_t max_pages,
                         const int32_t* positions, const int32_t* new_lens,
                         int32_t* dev_status, void* stream);

/*
 * page_score_topk — relevance of every page of every sequence to each query
 * head, and the top-K pages [TinyServe page, sections 2.1 and 3.1 phases 1-2]:
 *   r(q, page) = sum_i (q_i >= 0 ? q_i * max_i : q_i * min_i)      (fp32)
 * Query head h uses kv head h / G (G = num_q_heads / num_kv_heads). A "row" is
 * what selects: each query head (group_mode PKV_SELECT_PER_HEAD, R = num_q_heads
 * rows per sequence), or each kv head with the sum or the max of its G heads'
 * scores (PKV_SELECT_GROUP_SUM / _MAX, R = num_kv_heads), so that the group
 * reads one page list. K = min(top_k, pages of the sequence); ties go to the
 * lower logical page index; the kept pages are written in ascending order.
 *   q          : [batch][num_q_heads][head_dim] of q_dtype (F16/BF16/F32).
 *   seq_lens   : int32 [batch]; sequence b has ceil(seq_lens[b] / page_size) pages.
 *   sel_pages  : int32 [batch][R][top_k] (entries past sel_count are -1).
 *   sel_count  : int32 [batch][R].
 *   scores_out : fp32 [batch][R][max_pages] or NULL (the row's scores); entries
 *                past the sequence's pages are -inf.
 *   early_start: 0, or 1: a promise that the work launched just before this
 *                call on `stream` (one kernel, or both kernels of a preceding
 *                attention call) writes nothing this call reads: q, the block
 *                table, the lengths and the page boxes. The call then reads and
 *                scores at once and waits for that work only before its first
 *                write (sel_pages, sel_count, scores_out, which may be shared
 *                with that work); only dev_status flags can be raised before
 *                the wait. Not after an append that refreshed the boxes (pass
 *                0 there). A false promise gives wrong results, not a fault.
 * Needs cache->page_meta. Pages per sequence are limited to 16384.
 * Device errors: PKV_DEV_BAD_PAGE (that page scores -inf).
 */
pkv_status pkv_page_score_topk(const pkv_cache* cache, int32_t batch, int32_t num_q_heads,
                               const void* q, pkv_dtype q_dtype,
                               const int32_t* block_table, int32_t max_pages,
                               const int32_t* seq_lens, int32_t top_k, int32_t group_mode,
                               int32_t early_start, int32_t* sel_pages, int32_t* sel_count,
                               float* scores_out, int32_t* dev_status, void* stream);

/*
 * Workspace bytes needed by pkv_paged_decode_attention for these shapes.
 * sparse: 0 dense, 1 page lists per query head, 2 page lists shared by each
 * kv head's group (sel_shared). num_splits as in the call (0 = automatic,
 * which queries the current device). Returns 0 on bad input.
 */
size_t pkv_attention_workspace_bytes(const pkv_cache* cache, int32_t batch, int32_t num_q_heads,
                                     int32_t sparse, int32_t num_splits);

/*
 * paged_decode_attention — out[b][h] = softmax(sm_scale * q[b][h] . K^T) V over
 * the tokens of sequence b [KV-practice page, section 2.1], K and V of kv head
 * h / G (G = num_q_heads / num_kv_heads), read through the block table and
 * dequantised in the kernel. Dense mode attends over tokens [0, seq_lens[b]).
 * Sparse mode (sel_pages != NULL) attends over the tokens of the logical pages
 * sel_pages[b][r][0 .. sel_count[b][r]) of row r, softmax renormalised over
 * them [TinyServe page, section 3.1 phase 3], in any order. With sel_shared = 0
 * a row is a query head (r = h, lists from PKV_SELECT_PER_HEAD); with
 * sel_shared = 1 a row is a kv head whose G query heads share its list (r =
 * h / G, lists from a group mode), and the group's K/V are read once.
 *   q           : [batch][num_q_heads][head_dim] of q_dtype (F16/BF16/F32).
 *   sel_stride  : row length of sel_pages (its top_k); ignored in dense mode.
 *   sel_shared  : 0 or 1, as above; ignored in dense mode.
 *   out         : [batch][num_q_heads][head_dim] of out_dtype (F32/F16/BF16).
 *   num_splits  : number of cooperating thread blocks that share the work
 *                 (split-K over the whole batch's pages, each block taking an
 *                 equal share); 0 = automatic: one full wave of the device,
 *                 or, for a call whose block-table width (dense) or page-list
 *                 stride (sparse) bounds it below 4 chunks of 16 tokens per
 *                 block of that wave, max(SMs, bound / 4) blocks.
 *   fresh_rows  : -1, or a promise that lets the call start before the
 *                 work launched just before it on `stream` (one kernel, or
 *                 both kernels of a preceding attention call) has finished:
 *                 that work writes nothing this call reads except the K/V
 *                 rows (and scales) that a pkv_kv_append of the last
 *                 fresh_rows tokens of each sequence writes, i.e. positions
 *                 >= seq_lens[b] - fresh_rows (per-group INT8: from the
 *                 start of the 64-token group holding that position, which
 *                 the append re-quantises), and, in sparse mode, the page
 *                 lists sel_pages / sel_count. Typical use: the call right
 *                 after this step's pkv_kv_append (fresh_rows = its t_new),
 *                 right after another attention call (fresh_rows = 0), or a
 *                 sparse call right after the pkv_page_score_topk that wrote
 *                 its lists (fresh_rows = 0). A sparse call that starts early
 *                 plans its work from the lengths alone (every row of
 *                 sequence b is given min(sel_stride, pages of b) pages) and
 *                 reads at most that many entries of a list. The
 *                 call then reads q, the tables, the lengths and all older
 *                 rows at once, and waits for that kernel before copying a
 *                 chunk with fresh rows and before its first write to out or
 *                 the workspace (so both may be shared with that kernel);
 *                 only dev_status flags can be raised before the wait. A
 *                 false promise gives wrong results, not a fault. -1 (no
 *                 promise) waits before the first global access.
 *   workspace   : >= pkv_attention_workspace_bytes(...) bytes, 256-byte
 *                 aligned, any contents (it holds the per-block partial states
 *                 of one call; no initialisation is needed).
 * Two launches: the attention kernel, and a combine kernel that merges, for each (sequence, kv head) shared by several blocks,
 * the blocks' partial (running max, sum, accumulator) states. Both are
 * launched with programmatic stream serialization. Every kernel of this
 * library waits for the preceding kernel on the stream before its first
 * global memory access (the attention kernel with fresh_rows >= 0: before
 * its first access to anything outside the promise above) and before it
 * completes, so stream order is kept. The attention kernel and the
 * single-launch calls let their dependents start only after that wait; the
 * combine kernel lets them start at once, so the next call's kernel can
 * overlap this call's tail (its own wait still covers this whole call).
 * A sequence with no tokens (or no selected pages) yields zeros.
 * Device errors: PKV_DEV_BAD_PAGE, PKV_DEV_BAD_SELECTED (chunk skipped),
 * PKV_DEV_TIMEOUT.
 */
pkv_status pkv_paged_decode_attention(const pkv_cache* cache, int32_t batch, int32_t num_q_heads,
                                      const void* q, pkv_dtype q_dtype, float sm_scale,
                                      const int32_t* block_table, int32_t max_pages,
                                      const int32_t* seq_lens,
                                      const int32_t* sel_pages, const int32_t* sel_count,
                                      int32_t sel_stride, int32_t sel_shared,
                                      void* out, pkv_dtype out_dtype, int32_t num_splits,
                                      int32_t fresh_rows, void* workspace, size_t workspace_bytes,
                                      int32_t* dev_status, void* stream);

/*
 * append_decode_attention — one decode step of a layer in one call: write each
 * sequence's new token (K and V of every kv head) at position seq_lens[b] - 1,
 * as pkv_kv_append with t_new = 1 would [HBM-layout page, section 三; per-token
 * INT8: section 二], then dense paged_decode_attention over [0, seq_lens[b]).
 * The block that streams the sequence's last chunk writes the row itself and
 * copies the chunk after it, so the step needs no separate append launch and
 * no wait between the two. The pages have no counterpart; this is a packaging
 * choice of the library.
 *   k_new, v_new : [batch][num_kv_heads][head_dim] of src_dtype (F16/BF16),
 *                  16-byte aligned; for fp16/bf16 caches src_dtype must be the
 *                  cache dtype.
 *   Other arguments as pkv_paged_decode_attention in dense mode; with
 *   fresh_rows >= 0 the work before the call must also leave the new rows
 *   alone (the kernel writes them before it waits for that work).
 * Caches: fp16/bf16, per-token INT8 and 4-bit without page metadata take the
 * single launch above. Per-group INT8 caches (the append re-quantises the whole
 * open group of up to 64 rows, which the attention's streaming does not hold)
 * and caches with page boxes take two launches: the kv_append of the new token,
 * which waits for all earlier work, then the attention, which starts under it
 * (as with fresh_rows = 1 after that append); the caller's fresh_rows is then
 * not needed, and the results equal those of pkv_kv_append followed by
 * pkv_paged_decode_attention. For those caches the arguments of both calls are
 * checked before either is launched.
 * Sequences with seq_lens[b] = 0 get no token.
 */
pkv_status pkv_append_decode_attention(const pkv_cache* cache, int32_t batch, int32_t num_q_heads,
                                       const void* k_new, const void* v_new, pkv_dtype src_dtype,
                                       const void* q, pkv_dtype q_dtype, float sm_scale,
                                       const int32_t* block_table, int32_t max_pages,
                                       const int32_t* seq_lens, void* out, pkv_dtype out_dtype,
                                       int32_t num_splits, int32_t fresh_rows, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * paged_decode_attention_noalloc — the same computation and arguments as
 * pkv_paged_decode_attention with fresh_rows = -1, minus the workspace, for callers that cannot
 * allocate device memory: a program that reserves all device memory at start-up
 * and allows no later cudaMalloc (which can stall every stream on the device),
 * or a plugin that only receives its input and output buffers. The pages have
 * no counterpart; this is a packaging choice of the library.
 *   Scratch: a fixed 8 MiB array inside the library's device image. CUDA loads
 *   the module holding it lazily by default, so the array's memory is taken
 *   on a device by the first call made with that device current (or when the
 *   context is created, if the process runs with CUDA_MODULE_LOADING=EAGER),
 *   and held until the process exits: make that first call (it may be a
 *   warm-up call) before reserving the rest of device memory, and before any
 *   stream capture on that device. Later calls take no device memory.
 *   A call whose workspace (its own plan's, as pkv_attention_workspace_bytes
 *   gives for a full-wave split count) exceeds 8 MiB returns PKV_ERR_WORKSPACE
 *   and launches nothing.
 *   Set-up: the first call with a given device current looks up the array's
 *   device address (cudaGetSymbolAddress) and keeps it for that device; after
 *   cudaDeviceReset on a device that address is stale, so no call may follow
 *   a reset.
 *   Sharing: every call uses the same array, and its contents are whatever the
 *   last call left (nothing needs to start at zero). Calls that may run at the
 *   same time on the GPU (other streams, other host threads) race: issue them
 *   one after another on one stream.
 *   Allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 */
pkv_status pkv_paged_decode_attention_noalloc(const pkv_cache* cache, int32_t batch,
                                              int32_t num_q_heads, const void* q, pkv_dtype q_dtype,
                                              float sm_scale, const int32_t* block_table,
                                              int32_t max_pages, const int32_t* seq_lens,
                                              const int32_t* sel_pages, const int32_t* sel_count,
                                              int32_t sel_stride, int32_t sel_shared, void* out,
                                              pkv_dtype out_dtype, int32_t num_splits,
                                              int32_t* dev_status, void* stream);

/*
 * Host page allocator [HBM-layout page, section 三 allocate_blocks /
 * free_sequence]: a free list of physical page ids; a sequence needs
 * ceil(tokens / page_size) pages; an allocation that cannot be met fails
 * without taking any page. Host memory only; not thread-safe.
 */
typedef struct pkv_allocator pkv_allocator;

pkv_status pkv_alloc_create(int32_t num_pages, pkv_allocator** out);
void pkv_alloc_destroy(pkv_allocator* a);
/* Grow sequence seq_id so it holds total_tokens tokens; writes all its page ids
 * into block_table_row[0 .. pages) (host memory, max_pages entries) and -1 past
 * them. PKV_ERR_OUT_OF_PAGES leaves the allocator unchanged. */
pkv_status pkv_alloc_reserve(pkv_allocator* a, int64_t seq_id, int32_t total_tokens,
                             int32_t page_size, int32_t* block_table_row, int32_t max_pages);
/* Return every page of seq_id to the free list. */
pkv_status pkv_alloc_free(pkv_allocator* a, int64_t seq_id);
int32_t pkv_alloc_num_free(const pkv_allocator* a);
/* Pages of seq_id (0 if unknown). */
int32_t pkv_alloc_seq_pages(const pkv_allocator* a, int64_t seq_id);
/* Consistency check: pages that are neither free nor owned by exactly one
 * sequence (leaked or double-owned) [Gemini page, section 2.3]. */
int32_t pkv_alloc_check(const pkv_allocator* a);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
