/*
 * pa.h -- C ABI of the paged decode attention library (libpa.so).
 *
 * One decode step of a transformer layer whose KV cache is paged: each
 * sequence's keys and values live in fixed-size blocks of 16 or 32 tokens
 * scattered through two global pools (one for K, one for V), and a
 * per-sequence block table maps logical block i to its physical block.
 * ("PagedAttention: The Cache Was Storing Nothing" §2.2; "Paged Attention
 * Meets FlexAttention" review, "What carries the argument": two global page
 * buffers and one block table per sequence.)
 *
 * Layouts (all row-major, contiguous, device memory unless stated):
 *   K pool, V pool   [num_blocks][Hkv][block_size][D]   kv_dtype elements
 *   block_tables     int32 [B][max_blocks]; entry i of row b is the physical
 *                    block of logical block i; entries at or past
 *                    ceil(len_b / block_size) are never read
 *   q                [B][Hq][D]  kv_dtype elements
 *   k_new, v_new     [B][Hkv][D] kv_dtype elements
 *   out              [B][Hq][D]  out_dtype elements
 * Query head h reads kv head h / (Hq / Hkv) (consecutive groups;
 * "PagedAttention: The Cache Was Storing Nothing" §3.1).
 *
 * Ownership: the caller owns every tensor. The library owns only the plan
 * object returned through pa_decode's plan_inout and the device workspace
 * inside it, both released by pa_free.
 *
 * Streams and errors: every call is asynchronous on the given stream (NULL =
 * the legacy default stream); no call synchronises the host. Argument errors
 * are detected on the host before anything is launched and return a status
 * other than PA_OK. A CUDA launch or allocation failure returns PA_ERR_CUDA.
 * Data errors that only the device can see (a length outside its range, a
 * table entry outside the pool) never fault: the kernels skip the access,
 * write zeros for the affected outputs and raise a bit in a device error word
 * that pa_last_device_error reads back.
 *
 * Supported shapes: kv_dtype PA_BF16 or PA_F32, D in {64, 128}, block_size in
 * {16, 32}, Hq a multiple of Hkv, at most 2^30 output rows (B * Hq, or
 * num_queries * Hq for the multi-query calls). Pools, q, k_new, v_new and out
 * must be 16-byte aligned.
 */
#ifndef PA_H
#define PA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is struct CUstream_st* */
struct CUevent_st;  /* cudaEvent_t is struct CUevent_st* */

typedef enum {
    PA_OK = 0,
    PA_ERR_NULL = 1,        /* a required pointer is NULL */
    PA_ERR_SHAPE = 2,       /* sizes out of range or inconsistent */
    PA_ERR_DTYPE = 3,       /* unsupported element type */
    PA_ERR_BLOCK_SIZE = 4,  /* block_size not 16 or 32 */
    PA_ERR_WORKSPACE = 5,   /* workspace too small for the request */
    PA_ERR_CUDA = 6,        /* a CUDA call failed */
    PA_ERR_BOUNDS = 7,      /* the device saw a length or table entry out of range */
    PA_ERR_ALIGN = 8,       /* a tensor is not 16-byte aligned */
    PA_ERR_NO_BLOCKS = 9    /* the block pool has too few free blocks */
} pa_status;

typedef enum { PA_F32 = 0, PA_BF16 = 1 } pa_dtype;

/* Bits of the device error word (pa_last_device_error). */
enum {
    PA_DEVERR_SEQ_LEN = 1,      /* decode: seq_len < 1 or > min(max_seq_len, max_blocks*bs) */
    PA_DEVERR_TABLE = 2,        /* a table entry outside [0, num_blocks) */
    PA_DEVERR_TIMEOUT = 4,      /* a pipeline wait gave up (the kernel returned early) */
    PA_DEVERR_CACHE_LEN = 8,    /* append: cache_len < 0 or >= max_blocks*bs */
    PA_DEVERR_COPY = 16         /* block copy: an id outside [0, num_blocks) */
};

/* Kernel selection for pa_decode (pa_plan_set_path). */
enum {
    PA_PATH_AUTO = 0,    /* bf16: tensor-core path (any g); f32: simple */
    PA_PATH_SIMPLE = 1,  /* one warp per (sequence, q head), plain loads, no split;
                            max_seq_len <= PA_SIMPLE_MAX_SEQ_LEN */
    PA_PATH_FMA = 2,     /* bf16 only: bulk-staged pages, CUDA-core dot products */
    PA_PATH_MMA = 3,     /* bf16 only: bulk-staged pages, a kv head's query heads (any g) through bf16 mma tiles */
    PA_PATH_PREFILL = 4  /* reported by pa_plan_info only: pa_decode_multi ran the prefill kernel */
};

/* Longest max_seq_len the unsplit kernel (float32 pools, or PA_PATH_SIMPLE)
 * accepts: each (sequence, q head) row is one warp walking every token, so a
 * longer row would serialise; longer calls return PA_ERR_SHAPE. */
#define PA_SIMPLE_MAX_SEQ_LEN 8192

/* Opaque: split plan, device workspace and device error word. */
typedef struct pa_plan pa_plan;

/*
 * pa_append_kv -- write one new token per sequence into its tail block.
 *
 * The cache grows by one token per generated token and only the last block
 * of a sequence is partly full ("PagedAttention: The Cache Was Storing
 * Nothing" §1 and §2.2). For every sequence b and kv head j, with
 * pos = cache_lens[b]:
 *     K[block_tables[b][pos / block_size]][j][pos % block_size][:] = k_new[b][j][:]
 * and the same for V. The copy is bit-exact (NaN payloads included).
 *
 *   k_new, v_new   device, [B][Hkv][D] kv_dtype, read only
 *   k_pool, v_pool device, [num_blocks][Hkv][block_size][D], written in place
 *   block_tables   device, int32 [B][max_blocks]
 *   cache_lens     device, int32 [B]: tokens already cached = write position
 *
 * Precondition: the written block is private to its sequence (reference
 * count 1). Shared blocks must be copied by the caller before a sequence
 * writes into them (copy on write, same page §2.3). A cache_len outside
 * [0, max_blocks*block_size) or a table entry outside [0, num_blocks) skips
 * that sequence and raises PA_DEVERR_CACHE_LEN / PA_DEVERR_TABLE in the
 * library-wide append error word (pa_last_device_error with plan = NULL).
 * B = 0 is a no-op.
 */
pa_status pa_append_kv(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                       const int32_t* block_tables, int max_blocks, const int32_t* cache_lens,
                       int B, int Hkv, int D, int block_size, int num_blocks, pa_dtype kv_dtype,
                       struct CUstream_st* stream);

/*
 * pa_decode -- paged decode attention for one new query per (sequence, head).
 *
 * out[b][h][:] = sum_t w_t v_t with w = softmax_t(scale * q[b][h] . k_t) over
 * the logical tokens t < seq_lens[b] of sequence b, k_t and v_t read through
 * the block table: exactly ordinary attention with one indirection per block
 * ("39 · PagedAttention" §1-§2; scale = 1/sqrt(D) in "FlashAttention vs
 * PagedAttention"). The sequence is split across warps; partial results
 * (m, l, acc) are merged with m = max(m1, m2), l = l1 e^(m1-m) + l2 e^(m2-m)
 * ("39 · PagedAttention" §3), by a second small kernel where a sequence
 * spans more than one warp.
 *
 *   q             device, [B][Hq][D] kv_dtype
 *   k_pool/v_pool device, [num_blocks][Hkv][block_size][D] kv_dtype, read only
 *   block_tables  device, int32 [B][max_blocks]
 *   seq_lens      device, int32 [B]: tokens attended, >= 1 (includes the token
 *                 appended this step); must be <= max_seq_len
 *   max_seq_len   host bound on every seq_lens[b]; sizes the launch. With
 *                 float32 pools (which run on the unsplit one-warp-per-row
 *                 kernel) it must be <= PA_SIMPLE_MAX_SEQ_LEN: longer returns
 *                 PA_ERR_SHAPE
 *   scale         score scale (normally 1/sqrt(D))
 *   out           device, [B][Hq][D] out_dtype (bf16 rounded to nearest even)
 *   plan_inout    in/out: *plan_inout == NULL makes the library create a plan
 *                 (device workspace allocation, the only allocation); a plan
 *                 is reused by later calls and grows its workspace only when
 *                 a call needs more. Release it with pa_free. A call that
 *                 returns an argument error (PA_ERR_NULL, _SHAPE, _DTYPE,
 *                 _BLOCK_SIZE, _ALIGN) creates no plan and launches nothing.
 *
 * Device-side violations (seq_len out of range, table entry outside the pool)
 * write zeros for the affected (b, h) rows and raise bits in the plan's error
 * word. B = 0 is a no-op (no plan is created).
 */
pa_status pa_decode(const void* q, const void* k_pool, const void* v_pool,
                    const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, int B,
                    int Hq, int Hkv, int D, int block_size, int num_blocks, int max_seq_len,
                    float scale, pa_dtype kv_dtype, void* out, pa_dtype out_dtype,
                    pa_plan** plan_inout, struct CUstream_st* stream);

/*
 * pa_append_decode -- one decode step in one call: pa_append_kv of the step's
 * new token at position seq_lens[b] - 1, then pa_decode over seq_lens[b]
 * tokens (the cache grows by the token the step attends with, "PagedAttention:
 * The Cache Was Storing Nothing" §1-§2.2; attention as in pa_decode).
 *
 *   k_new, v_new  device, [B][Hkv][D] kv_dtype, read only, 16-byte aligned
 *   k_pool/v_pool device, written in place at the new token's slot
 *   other arguments as for pa_decode
 *
 * Results and pool contents equal pa_append_kv (with cache_lens = seq_lens - 1)
 * followed by pa_decode, bit for bit. On bf16 pools with the tensor-core
 * path, up to 8 query heads per kv head and the merge kernel (the automatic
 * choices), the append runs inside the decode kernel: the warp that reads a
 * sequence's last page writes the new row into its staged copy and into the
 * pool, which saves the append's launch and its round trips. Otherwise
 * (float32 pools, a forced CUDA-core path, 9-16 query heads per kv head, the
 * fused merge) the append runs as its own kernel first, and its PA_DEVERR_*
 * bits go to the library-wide append word as for pa_append_kv.
 * Precondition as for pa_append_kv: the written block is private to its
 * sequence. A sequence whose length is out of range gets no append and zero
 * rows (PA_DEVERR_SEQ_LEN); a table entry outside the pool skips the append
 * and zeroes the affected rows (PA_DEVERR_TABLE). NULL k_new or v_new returns
 * PA_ERR_NULL.
 */
pa_status pa_append_decode(const void* q, const void* k_new, const void* v_new, void* k_pool,
                           void* v_pool, const int32_t* block_tables, int max_blocks,
                           const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int block_size,
                           int num_blocks, int max_seq_len, float scale, pa_dtype kv_dtype,
                           void* out, pa_dtype out_dtype, pa_plan** plan_inout,
                           struct CUstream_st* stream);

/* Release a plan and its device workspace. NULL is a no-op. The caller must
 * make sure no work using the plan is still running (e.g. sync its stream). */
pa_status pa_free(pa_plan* plan);

/* Static English text for a status code. Never NULL. */
const char* pa_status_str(pa_status status);

/*
 * pa_last_device_error -- read and clear a device error word (synchronous:
 * waits for the device). plan != NULL reads the plan's decode word;
 * plan == NULL reads the library-wide word of pa_append_kv and
 * pa_copy_blocks on the current device.
 * *err receives a bit set of PA_DEVERR_*; 0 means no error seen.
 */
pa_status pa_last_device_error(pa_plan* plan, int* err);

/* Force a kernel path for later pa_decode and pa_append_decode calls on this
 * plan (PA_PATH_*; pa_append_decode then appends with its own kernel first on
 * any path but PA_PATH_MMA). A forced path that does not support a call's
 * shape makes that call return PA_ERR_DTYPE. */
pa_status pa_plan_set_path(pa_plan* plan, int path);

/* Test hook for the failure handling. While enable != 0, every kernel this
 * library launches (decode, one-call append and decode, multi-query decode,
 * no-alloc decode, prefill, page scores) makes its first pipeline wait on an mbarrier that nothing
 * completes, bounded by 20 us, so that the wait expires: the kernel raises
 * PA_DEVERR_TIMEOUT, waits (bounded) for its own copies and tensor-core
 * products in flight, frees its tensor memory and returns. The outputs of
 * such calls are unspecified; the device stays usable and the next call with
 * the hook off computes normally. Off by default; process-wide (it is read
 * when a call launches its kernels). Nothing ever waits without a bound. */
pa_status pa_debug_set_wait_probe(int enable);

/* Test hook: which tensor-core kernel pa_prefill (and pa_decode_multi above
 * 16 columns) runs. PA_PREFILL_AUTO (the default) chooses from the shape, as
 * described at pa_prefill; PA_PREFILL_ONE_TILE and PA_PREFILL_TWO_TILE pin
 * one kernel for every call, so that tests can check both on any shape (the
 * key split of small pa_decode_multi calls belongs to the one-tile kernel
 * and is skipped under PA_PREFILL_TWO_TILE). Process-wide, read when a call
 * launches; PA_ERR_SHAPE for any other value. */
enum { PA_PREFILL_AUTO = 0, PA_PREFILL_ONE_TILE = 1, PA_PREFILL_TWO_TILE = 2 };
pa_status pa_debug_set_prefill_kernel(int which);

/* How pa_decode combines the partials of a sequence split across warps
 * (pa_plan_set_merge). */
enum {
    PA_MERGE_AUTO = 0,   /* the measured best for the shape (a second kernel) */
    PA_MERGE_KERNEL = 1, /* a second, small merge kernel over all split rows */
    PA_MERGE_FUSED = 2   /* the warp that writes a segment's last partial folds them
                            (atomic counter per segment, no waiting, no second kernel);
                            one query per sequence, up to 8 query heads per kv head */
};

/* Choose the merge of later pa_decode and pa_append_decode calls on this plan
 * (PA_MERGE_*; with PA_MERGE_FUSED, pa_append_decode appends with its own
 * kernel first). A
 * call whose shape the fused merge does not serve returns PA_ERR_SHAPE while
 * PA_MERGE_FUSED is set. A test and benchmark hook beside pa_plan_set_path. */
pa_status pa_plan_set_merge(pa_plan* plan, int mode);

/* Force the dynamic tail of later pa_decode / pa_decode_multi calls on this
 * plan: the last dyn_permille / 1000 of the page stream (0..500) is handed
 * out in pieces of dyn_pages pages (1..4096) to whichever warp is free, for
 * any tile; dyn_permille = 0 runs static ranges only. dyn_permille < 0
 * restores the automatic choice. A test and benchmark hook: the automatic
 * choice is the measured best for the shapes it was measured on. */
pa_status pa_plan_set_schedule(pa_plan* plan, int dyn_permille, int dyn_pages);

/* The path the last pa_decode call on this plan launched (PA_PATH_*), the
 * number of thread blocks and warps of its split kernel. Any output pointer
 * may be NULL. */
pa_status pa_plan_info(const pa_plan* plan, int* path, int* blocks, int* warps);

/* Timing hook: when both events are non-NULL, later pa_decode calls on this
 * plan record `start` right before the split-attention kernel and `stop`
 * right after it, on the call's stream. Pass NULLs to stop recording. */
pa_status pa_plan_set_split_events(pa_plan* plan, struct CUevent_st* start,
                                   struct CUevent_st* stop);

/*
 * pa_prefill -- causal paged multi-query attention (chunked prefill,
 * speculative verification) on the tensor cores.
 *
 * The newest n_b = q_start[b+1] - q_start[b] tokens of sequence b are
 * queries at once: query i sits at position L_b - n_b + i (L_b = seq_lens[b])
 * and attends to the tokens t <= its position read through the block table
 * ("FlashAttention vs PagedAttention", "How prefill and decode change the
 * diagnosis"; each row is exactly the decode attention over its prefix). The
 * K/V of the new tokens must already be in the pools.
 *
 *   q         device bf16 [num_queries][Hq][D], rows of sequence b at
 *             q_start[b] .. q_start[b+1]-1
 *   q_start   device int32 [B + 1], nondecreasing, q_start[0] = 0
 *   num_queries  host: rows of q and out (q_start[B]); a sequence whose rows
 *             fall outside them is refused on the device
 *   max_q     host bound on every n_b (sizes the launch)
 *   out       device [q_start[B]][Hq][D] out_dtype
 *   device_error  device int or NULL (NULL = the library-wide word read by
 *             pa_last_device_error(NULL, ...)): PA_DEVERR_* bits
 *
 * Supported: bf16 pools, D = 128, block_size 16 or 32, Hq / Hkv dividing 128,
 * max_blocks <= 16384, B and Hkv at most 65535 (PA_ERR_SHAPE otherwise).
 * The launch is sized by min(max_q, num_queries). A query tile holds 128 /
 * (Hq / Hkv) queries of one sequence. When every sequence fits one tile, or
 * the call has at most three waves of tiles (tiles x Hkv x B <= 3 x SMs),
 * it runs a one-tile kernel that overlaps a tile's softmax with its own
 * next score products; otherwise a kernel that alternates two tiles per
 * block (half the K/V intake per row). pa_prefill holds no workspace, so a
 * call with fewer one-tile blocks than SMs (a few sequences) streams each
 * sequence's whole key range in one block; pa_decode_multi computes the
 * same rows with a plan whose workspace lets such calls split the key range
 * over several blocks. With a few queries (max_q * Hq / Hkv <= 16, e.g. speculative
 * verification) pa_decode_multi computes the same rows at the decode's
 * bandwidth. n_b < 1, n_b > max_q, n_b > L_b,
 * L_b out of range or rows outside [0, num_queries) raise PA_DEVERR_SEQ_LEN
 * and leave that sequence's rows untouched; a table entry outside the pool
 * raises PA_DEVERR_TABLE and zeroes the affected rows.
 */
pa_status pa_prefill(const void* q, const int32_t* q_start, int num_queries, const void* k_pool,
                     const void* v_pool,
                     const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, int B,
                     int Hq, int Hkv, int D, int block_size, int num_blocks, int max_q,
                     int max_seq_len, float scale, pa_dtype kv_dtype, void* out, pa_dtype out_dtype,
                     int* device_error, struct CUstream_st* stream);

/*
 * pa_decode_multi -- paged decode attention for a few new queries per
 * sequence (speculative verification of drafted tokens).
 *
 * Computes what pa_prefill computes -- the newest n_b = q_start[b+1] -
 * q_start[b] tokens of sequence b are queries, query i at position
 * L_b - n_b + i attends to the tokens up to its position ("FlashAttention vs
 * PagedAttention", "How prefill and decode change the diagnosis") -- on the
 * split decode kernels of pa_decode: the (query, head) pairs of a kv head
 * share one tensor-core tile and the pages are streamed once for all of
 * them, so a step with few queries runs at the decode's bandwidth. Partials
 * across the split are combined as in pa_decode ("39 · PagedAttention" §3).
 *
 *   q, q_start, out   as for pa_prefill; num_queries = q_start[B] (host)
 *   max_q     host bound on every n_b
 *   plan_inout  as for pa_decode (the plan's forced path does not apply)
 *   other arguments   as for pa_decode
 *
 * The call picks the kernel from the shape: with max_q * (Hq / Hkv) <= 16
 * (query, head) columns per kv head it runs the split decode's tiles above;
 * with more it runs pa_prefill's tcgen05 kernels on the same arguments
 * (pa_plan_info then reports PA_PATH_PREFILL). On a small call (fewer
 * one-tile blocks than SMs) the one-tile kernel then splits every tile's key
 * range over several blocks, whose partials go to the plan's workspace
 * (grown on demand, like the split decode's) and are merged by a second
 * kernel. Those 128-row query tiles
 * need D = 128, Hq / Hkv dividing 128, max_blocks <= 16384 and Hkv <= 65535
 * (PA_ERR_SHAPE otherwise); its device errors then go to the plan's error
 * word.
 *
 * Supported: bf16 pools (PA_ERR_DTYPE otherwise), D in {64, 128} (128 above
 * 16 columns), block_size 16 or 32.
 * A sequence with n_b < 1, n_b > max_q, n_b > L_b, rows outside
 * [0, num_queries) or L_b out of range raises PA_DEVERR_SEQ_LEN in the plan's
 * error word and gets zero rows (q_start must still be nondecreasing); a table
 * entry outside the pool raises PA_DEVERR_TABLE and zeroes that sequence's
 * rows of the affected kv head. num_queries = 0 or B = 0 is a no-op.
 */
pa_status pa_decode_multi(const void* q, const int32_t* q_start, int num_queries, int max_q,
                          const void* k_pool, const void* v_pool, const int32_t* block_tables,
                          int max_blocks, const int32_t* seq_lens, int B, int Hq, int Hkv, int D,
                          int block_size, int num_blocks, int max_seq_len, float scale,
                          pa_dtype kv_dtype, void* out, pa_dtype out_dtype, pa_plan** plan_inout,
                          struct CUstream_st* stream);

/* ------------------------------------------------------------------------
 * Block management: free list, sharing and copy on write.
 *
 * "PagedAttention: The Cache Was Storing Nothing" §2.2-§2.3: every free block
 * fits any request; tables of several sequences may name the same physical
 * block (shared prefixes, beam candidates); a shared block is copied only when
 * a sequence diverges and writes into it. The manager lives on the host: an
 * O(1) free list (a stack of block ids) and one reference count per block
 * (the number of tables naming it). All pa_bm_* calls are thread-safe (one
 * mutex per manager) and take host pointers.
 * ---------------------------------------------------------------------- */
typedef struct pa_block_manager pa_block_manager;

/* A manager of num_blocks blocks, all free; freed with pa_bm_destroy. */
pa_status pa_bm_create(int num_blocks, pa_block_manager** out);
pa_status pa_bm_destroy(pa_block_manager* bm);
/* Take n free blocks (reference count 1 each) into ids[0..n); PA_ERR_NO_BLOCKS
 * (and no change) when fewer than n are free. */
pa_status pa_bm_alloc(pa_block_manager* bm, int n, int32_t* ids);
/* Add one reference to each of ids[0..n) (a forked table now names them too);
 * PA_ERR_BOUNDS (no change) if an id is outside the pool or not allocated. */
pa_status pa_bm_fork(pa_block_manager* bm, const int32_t* ids, int n);
/* Drop one reference from each of ids[0..n); a block whose count reaches 0
 * returns to the free list. PA_ERR_BOUNDS (no change) on an id that is not
 * held that many times. */
pa_status pa_bm_release(pa_block_manager* bm, const int32_t* ids, int n);
pa_status pa_bm_refcount(const pa_block_manager* bm, int32_t id, int* count);
pa_status pa_bm_num_free(const pa_block_manager* bm, int* n);

/*
 * pa_bm_prepare_append -- make every sequence's append target writable.
 *
 * For each b, the block of logical index cache_lens[b] / block_size in host
 * table row b (tables: host int32 [B][max_blocks]) becomes private: a missing
 * entry (< 0) gets a fresh block; a block with reference count > 1 is
 * replaced in the table by a fresh block and the pair (old, fresh) is
 * appended to copy_src / copy_dst (host arrays of capacity B), the old block
 * losing this table's reference. *n_copies receives the number of pairs; run
 * pa_copy_blocks on them (and upload the changed table rows) before
 * pa_append_kv. On any error nothing changes: PA_ERR_BOUNDS for a position
 * or id out of range, PA_ERR_NO_BLOCKS when the free list is too short.
 */
pa_status pa_bm_prepare_append(pa_block_manager* bm, int32_t* tables, int B, int max_blocks,
                               const int32_t* cache_lens, int block_size, int32_t* copy_src,
                               int32_t* copy_dst, int* n_copies);

/*
 * pa_copy_blocks -- batched whole-block copies on the device (copy on write).
 *
 * For i < n: block copy_dst[i] of both pools becomes a bit-exact copy of block
 * copy_src[i] (every kv head and slot). copy_src / copy_dst are device int32
 * arrays. The copies run in parallel: the destinations must be distinct and
 * no destination may be a source. An id outside [0, num_blocks) skips that
 * pair and raises PA_DEVERR_COPY in the library-wide word that
 * pa_last_device_error(NULL, ...) reads. n = 0 is a no-op; n <= 2^24.
 */
pa_status pa_copy_blocks(void* k_pool, void* v_pool, const int32_t* copy_src,
                         const int32_t* copy_dst, int n, int Hkv, int D, int block_size,
                         int num_blocks, pa_dtype kv_dtype, struct CUstream_st* stream);

/*
 * pa_page_scores -- PagedEviction page scores and the page to evict.
 *
 * Pith review of arXiv 2509.04377 (PagedEviction), "Core claim": a token's
 * importance is ||V||_2 / ||K||_2 of its cached value and key, a page's is the
 * mean over its tokens, and when a sequence's newest page has just filled
 * (seq_len % block_size == 0) its lowest-scoring page is evicted. K and V of a
 * token are taken over all kv heads together; ||K|| = 0 scores +inf; every
 * full page is a candidate; ties go to the lowest logical page.
 *
 *   k_pool, v_pool, block_tables, seq_lens  as for pa_decode (device, read only)
 *   scores    device float [B][max_blocks]: entry p < ceil(L_b / block_size)
 *             receives page p's mean (over its valid tokens); others untouched
 *   victims   device int32 [B]: the logical page to evict, or -1 (no full
 *             newest page this step, or a bad table entry in the sequence);
 *             until the victims are written, victims[0] is the score
 *             kernel's work counter (stream-ordered, so the caller sees only
 *             the results)
 *   device_error  device int or NULL: receives PA_DEVERR_SEQ_LEN /
 *             PA_DEVERR_TABLE bits (the caller clears it)
 *
 * Reads every attended K and V element once (HBM-bound). fp32 arithmetic.
 */
pa_status pa_page_scores(const void* k_pool, const void* v_pool, const int32_t* block_tables,
                         int max_blocks, const int32_t* seq_lens, int B, int Hkv, int D,
                         int block_size, int num_blocks, int max_seq_len, pa_dtype kv_dtype,
                         float* scores, int32_t* victims, int* device_error,
                         struct CUstream_st* stream);

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot let a library
 * allocate device memory. The pages have no counterpart of this call; it is
 * a deployment variant of the same computation.
 *
 * Who needs it: callers that own all device memory themselves, such as a
 * serving engine that has reserved the free HBM as its KV block pool and
 * budgets it exactly, or a plugin host that hands a kernel only its tensors.
 * A cudaMalloc inside their call would take memory outside that budget, and
 * cudaMalloc / cudaFree synchronise the device, stalling other streams.
 *
 * Arguments and result are those of pa_decode for bf16 pools (kv_dtype must
 * be PA_BF16; the kernel choice is pa_decode's automatic one), without a plan:
 * the split partials live in one 16 MiB device array inside the library, which
 * every GPU that loads the library holds until the process exits. No
 * cudaMalloc, cudaFree or other allocating call is made.
 *
 *   device_error  device pointer to an int that receives PA_DEVERR_* bits
 *                 (the caller clears it); NULL = errors are not reported.
 *
 * Limits and rules:
 *   - when the partials of pa_decode's dynamic tail would not fit in the
 *     array, the call runs on static ranges alone (one partial pair per
 *     warp, about 2 x query heads per kv unit x D x 4 bytes); when those do
 *     not fit either (16 query heads per kv head at D = 128 need more than
 *     about 1000 warps' worth), on fewer blocks, as many as the array holds
 *     partials for. PA_ERR_WORKSPACE (nothing launched) remains for a call
 *     whose partials would not fit for a single block, which no shape within
 *     the limits above reaches;
 *   - every call shares the array and it keeps the last call's contents;
 *     calls whose work overlaps on the GPU (unordered streams) race on it and
 *     must be serialised by the caller;
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; a failed lookup (for
 *     example inside a stream capture) returns PA_ERR_CUDA and is retried by
 *     the next call;
 *   - the array is reserved on a device when the library's device code is
 *     loaded there; with lazy module loading (the CUDA default) that can be
 *     the first call, which then takes the 16 MiB and may synchronise. Make
 *     one warm-up call on each device at start-up, before sizing the KV pool
 *     from the free memory and before any stream capture; later calls
 *     allocate nothing.
 */
pa_status pa_decode_noalloc(const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                            int B, int Hq, int Hkv, int D, int block_size, int num_blocks,
                            int max_seq_len, float scale, pa_dtype kv_dtype, void* out,
                            pa_dtype out_dtype, int* device_error, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
