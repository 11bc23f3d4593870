// Internal declarations shared by the host entry points and the kernel files.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {

// Workspace metadata written by block 0 of the split kernel and read by the
// merge kernel: [0] total pages P, [1] pages per static range, [2] warps NW,
// [3] dynamic-piece counter (zero between calls; the merge kernel resets it,
// or with the fused merge the last warp to leave the split kernel), [4] end A
// of the static part of the page stream, [5] pages per dynamic piece, [6]
// dynamic pieces, [7] warps that have left the split kernel (fused merge;
// zero between calls), [8] set when a warp gave up (fused merge: the last
// warp to leave then clears the segment counters), [9] unused, then the page
// prefix sums pre[0..B] (pre[b] = pages of sequences < b).
constexpr int kMetaHeader = 10;

// Bits of the device error word (mirrors PA_DEVERR_* in pa.h).
constexpr int kErrSeqLen = 1;
constexpr int kErrTable = 2;
constexpr int kErrTimeout = 4;
constexpr int kErrCacheLen = 8;
constexpr int kErrCopy = 16;

// Wall-clock limit of any single pipeline wait inside a kernel.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Wait-expiry probe (pa_debug_set_wait_probe): while it is on, kernels make
// their first pipeline wait on an mbarrier that nothing completes, bounded by
// this limit, so that the wait expires and the kernel takes its give-up path.
constexpr uint64_t kProbeLimitNs = 20000;  // 20 us
// 1 while the probe is on (read at launch time by every launch site).
int wait_probe();
// The prefill kernel a test has forced (PA_PREFILL_*; PA_PREFILL_AUTO: none).
int prefill_kernel_choice();

enum SplitKind { kSplitFma = 0, kSplitMma = 1 };

// Tokens per pipeline stage of the split kernels: two 16-token pages or one
// 32-token page of the same (sequence, kv unit) segment.
constexpr int kChunkTokens = 32;

// Row pitch (bytes) of the query rows in a stage of the multi-query kernel,
// which reads its query fragments from shared memory at every chunk: 16
// bytes past a row of D bf16 values, so that the 8 rows of a fragment load
// fall in different banks.
__host__ __device__ constexpr int mq_q_pitch(int D) { return D * 2 + 16; }

// Arguments of the split-attention kernels (bf16 KV).
struct SplitArgs {
    const uint16_t* q;         // [B][Hq][D] bf16 bits
    const int32_t* tables;     // [B][max_blocks]
    const int32_t* seq_lens;   // [B]
    void* out;                 // [B][Hq][D], bf16 or f32
    float* ws_acc;             // [2 * warps][GS][D]  partial value sums
    float* ws_ml;              // [2 * warps][GS][2]  partial (max, sum)
    int* ws_meta;              // kMetaHeader + B + 1 ints
    int* err;                  // device error word
    int B, Hq, Hkv, g;         // g = Hq / Hkv
    int GS, nslices, U;        // q heads per slice, slices per kv head, U = Hkv * nslices
    int max_blocks, num_blocks, max_seq_len;
    float scale_log2;          // scale * log2(e)
    int out_bf16;
    int stages;                // pipeline stages per warp
    int stage_bytes;           // bytes per stage (multiple of 1024)
    int lens_bytes;            // bytes of the per-sequence arrays at the front of shared memory
    int q_bytes;               // per warp: query-row region after the rings (0: rows in the stage)
    int dyn_permille;          // fraction of the page stream handed out dynamically (1/1000)
    int dyn_pages;             // pages per dynamic piece
    // Several queries per sequence (speculative verification): q and out are
    // [T][Hq][D] with sequence b's queries at rows q_start[b] .. q_start[b+1)
    // (at most nq), the newest tokens of the sequence; null for one query.
    const int32_t* q_start;
    int nq;
    int num_q;                 // T: rows of q and out
    int probe_wait;            // 1: the first pipeline wait of each warp expires (a test hook)
    // Fused merge (one query per sequence, one n-tile): ws_cnt[b * U + u]
    // counts the partials of segment (b, u) written so far (zero between
    // calls); the warp that writes the last one folds them into the output.
    int* ws_cnt;
    // Fused append (pa_append_decode): the step's new rows [B][Hkv][D] go to
    // position seq_lens[b] - 1 of the pools (bf16 bits), written in place.
    const uint16_t* k_new;
    const uint16_t* v_new;
    uint16_t* kpool_w;
    uint16_t* vpool_w;
};

struct SplitLaunch {
    int kind;      // SplitKind
    int D, BS, NT; // head dim, block size, n-tiles of 8 q heads (MMA)
    int warps;     // warps per block
    int blocks;    // grid size
    size_t smem;   // dynamic shared memory bytes
    int mq = 0;    // 1: several queries per sequence (tensor-core path only)
    int fused = 0; // 1: the split kernel merges its own partials (no merge kernel)
    int append = 0; // 1: the split kernel also appends the step's new K/V rows
};

// Returns the resident blocks per SM of a split-kernel variant at the given
// block size and dynamic shared memory, or 0 (and sets *status) on error.
int split_blocks_per_sm(const SplitLaunch& L, cudaError_t* status);
cudaError_t launch_split(const SplitLaunch& L, const CUtensorMap& kmap, const CUtensorMap& vmap,
                         const SplitArgs& a, cudaStream_t stream);

// Host-side planning of a split launch, shared by pa_decode,
// pa_decode_multi and pa_decode_noalloc.
constexpr size_t kSmemLimit = 232448;  // opt-in dynamic shared memory per block on sm_10x
constexpr int kMaxBatch = 8192;        // per-sequence arrays live in shared memory
constexpr int64_t kMaxRows = int64_t(1) << 30;  // output rows (rows x heads), counted in int
constexpr int kMaxGridYZ = 65535;      // grid.y / grid.z limit of the prefill launch

// Kv units, tile width and block shape, from the sizes alone.
struct SplitShape {
    int kind = 0, mq = 0;          // SplitKind; several queries per sequence
    int nslices = 0, GS = 0, NT = 0, U = 0;
    int warps = 0, stages = 0;
    int64_t max_pages = 0;         // pages of the longest possible sequence
    int64_t P_max = 0;             // pages over all (sequence, kv unit) segments, at most
    size_t stage_bytes = 0, lens_bytes = 0, smem = 0;
    size_t q_bytes = 0;            // per warp: query rows outside the ring (tiles that reread them)
};
// Warps per block of the tiles that reread their query rows (several queries
// per sequence, or two n-tiles): as many as the shared memory holds, at most
// 12 (three warps per SM sub-partition at up to 170 registers a thread).
constexpr int kQsMaxWarps = 12;
// kind: kSplitFma (one query head per kv unit) or kSplitMma; nq > 0 selects
// the multi-query tile (nq queries x g heads, tensor cores). Returns false
// when the sizes do not fit (page count over 32 bits, shared memory over the
// limit).
bool split_shape(int kind, int nq, int B, int Hq, int Hkv, int D, int block_size, int max_blocks,
                 int max_seq_len, SplitShape* s);

// Grid, dynamic tail and workspace carve-up at per_sm resident blocks.
struct SplitGrid {
    int blocks = 0, NW = 0;        // grid size, warps in the grid
    int dyn_permille = 0, dyn_pages = 0;
    int64_t ranges = 0;            // partial records: static ranges + dynamic pieces
    int merge_wpr = 1;             // warps per output row in the merge kernel (1 .. 32)
    size_t meta_bytes = 0, ml_bytes = 0, acc_bytes = 0;
    size_t cnt_bytes = 0;          // segment counters of the fused merge (0 without it)
    size_t workspace_bytes() const { return meta_bytes + ml_bytes + acc_bytes + cnt_bytes; }
};
// rows: output rows the merge writes (B * Hq, or T * Hq with several queries
// per sequence). dynamic = false plans static ranges only (the fewest
// partials); max_blocks > 0 caps the grid (fewer warps, fewer partials);
// force_permille >= 0 (with force_pages >= 1) replaces the automatic choice
// of the dynamic tail, for any tile (a test and benchmark hook).
SplitGrid split_grid(const SplitShape& s, int B, int D, int block_size, int64_t rows, int num_sms,
                     int per_sm, bool dynamic = true, int max_blocks = 0,
                     int force_permille = -1, int force_pages = 0);

// Copies the planned fields (shape, grid, tail) into a.
void set_split_plan(SplitArgs* a, const SplitShape& s, const SplitGrid& gr);

// View a [NB][Hkv][BS][D] bf16 pool as a 3-D tensor (D, BS, rows = NB*Hkv)
// whose boxes are [64 columns][BS rows][1 page] with the 128-byte swizzle.
bool encode_pool_map(CUtensorMap* map, const void* pool, int rows, int D, int BS);

struct MergeArgs {
    int* ws_meta;
    const float* ws_acc;
    const float* ws_ml;
    void* out;
    int B, Hq, g, GS, nslices, U, D;
    int out_bf16;
    int wpr;   // warps per output row: 1, 2, 4, 8, 16 or 32 (more for more partials per row)
    int rows;  // output rows: B * Hq, or T * Hq with several queries per sequence
    const int32_t* q_start;  // several queries per sequence (see SplitArgs), else null
};
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream);

struct SimpleArgs {
    const void* q;
    const void* kpool;
    const void* vpool;
    const int32_t* tables;
    const int32_t* seq_lens;
    void* out;
    int* err;
    int B, Hq, Hkv, D, BS, max_blocks, num_blocks, max_seq_len;
    float scale_log2;
    int kv_bf16, out_bf16;
};
cudaError_t launch_simple(const SimpleArgs& a, cudaStream_t stream);

struct AppendArgs {
    const void* k_new;
    const void* v_new;
    void* kpool;
    void* vpool;
    const int32_t* tables;
    const int32_t* cache_lens;
    int B, Hkv, D, BS, max_blocks, num_blocks, elem_bytes;
    int pos_offset = 0;  // position = cache_lens[b] - pos_offset (1 when given seq_lens)
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);

struct CopyArgs {
    void* kpool;
    void* vpool;
    const int32_t* src;
    const int32_t* dst;
    int n, num_blocks;
    int64_t block_bytes;  // bytes of one block of one pool (multiple of 16)
};
cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t stream);
// Read and clear the append error word of the current device (synchronous).
cudaError_t read_append_error(int* err);
// Device address of that word on the current device.
cudaError_t append_error_address(int** p);

// Tensor map of the prefill's query rows q [T][Hq][128] bf16: one box is one
// 64-column half of a query tile (Qb queries x g heads, 128-byte swizzle).
bool encode_query_map(CUtensorMap* map, const void* q, int T, int Hq, int g, int Qb);

// Causal paged multi-query attention on the tensor cores. Calls whose
// sequences all fit one query tile, or with at most three waves of tiles,
// run the one-tile kernel (pa_prefill_1t.cu), the others the two-tile
// kernel. splits > 1 (one-tile kernel only) cuts every tile's key range into
// that many blocks whose partials go to part (prefill_split_bytes) and are
// merged by a second kernel.
cudaError_t launch_prefill(const CUtensorMap& kmap, const CUtensorMap& vmap, const void* q,
                           int num_q, const int32_t* q_start, const int32_t* tables,
                           const int32_t* seq_lens, void* out, int* err, int B, int Hq, int Hkv,
                           int max_blocks, int num_blocks, int max_seq_len, int max_q,
                           float scale_log2, int out_bf16, int block_size, cudaStream_t stream,
                           float* part = nullptr, int splits = 1, int zero_invalid = 0);
cudaError_t launch_prefill_one_tile(const CUtensorMap& kmap, const CUtensorMap& vmap, const void* q,
                                    int num_q, const int32_t* q_start, const int32_t* tables,
                                    const int32_t* seq_lens, void* out, int* err, int B, int Hq,
                                    int Hkv, int max_blocks, int num_blocks, int max_seq_len,
                                    int max_q, float scale_log2, int out_bf16, int block_size,
                                    cudaStream_t stream, float* part, int splits,
                                    int zero_invalid);
// Key splits for a one-tile call (1: none) and the partial bytes they need;
// nq = min(max_q, num_queries).
int prefill_split_count(int B, int Hq, int Hkv, int64_t nq, int max_seq_len, int num_sms);
size_t prefill_split_bytes(int B, int Hq, int Hkv, int64_t nq, int splits);

}  // namespace pa
