// Host side of the C ABI declared in include/pa.h: argument validation, kernel
// selection, split planning, workspace ownership and launches.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "pa.h"
#include "pa_internal.h"

namespace {

using pa::SplitLaunch;

constexpr int kDefaultWarps = 3;           // warps per block of the split kernels
constexpr int kMqWarps = 5;                // ... with 9-16 multi-query columns (two blocks per SM)
constexpr int kDefaultStages = 1;          // pipeline stages per warp
constexpr int kDynPermille = 150;          // share of the page stream scheduled dynamically
constexpr int kDynMinPages = 1024;         // ... when a sequence may have this many pages
constexpr int kDynPiecePages = 16;         // ... in pieces of this many pages
constexpr int kDynShortPermille = 250;     // ... on the one-head path with shorter sequences
constexpr int kDynMidPages = 256;          // multi-head units, sequences of 256 .. 1023 pages:
constexpr int kDynMidPiecePages = 8;       // ... the same share in pieces of this many pages
constexpr int kDynMidMaxRows = 2048;       // ... while the merge has at most this many rows
constexpr int kMergeRowsPerSm = 16;        // rows one SM merges at once with 4 warps per row
constexpr int kMinPagesPerWarp = 4;
constexpr int kHeadSlice = 16;             // query heads per kv unit on the tensor-core path

struct MapKey {
    const void* ptr = nullptr;
    int rows = 0, D = 0, BS = 0;
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && rows == o.rows && D == o.D && BS == o.BS;
    }
};

struct OccKey {
    int kind, D, BS, NT, warps;
    size_t smem;
    int blocks_per_sm;
    int mq;
    int fused;
    int append;
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

std::atomic<int> g_wait_probe{0};
std::atomic<int> g_prefill_kernel{PA_PREFILL_AUTO};

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev) {
        if (dev >= 0 && cudaGetDevice(&prev) == cudaSuccess && prev != dev) cudaSetDevice(dev);
        else prev = -1;
    }
    ~DeviceGuard() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

}  // namespace

namespace pa {

int wait_probe() { return g_wait_probe.load(std::memory_order_relaxed); }
int prefill_kernel_choice() { return g_prefill_kernel.load(std::memory_order_relaxed); }

bool encode_pool_map(CUtensorMap* map, const void* pool, int rows, int D, int BS) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(BS),
                          static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(BS) * D * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BS), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_query_map(CUtensorMap* map, const void* q, int T, int Hq, int g, int Qb) {
    // q [T][Hq][D = 128] bf16 as (D, Hq, T); one box = one 64-column half of a
    // query tile: Qb queries x the g heads of a kv head, rows in (query, head)
    // order, 128-byte swizzle (the K-major layout of the tile's MMA operand).
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(T)};
    cuuint64_t strides[2] = {128 * 2, static_cast<cuuint64_t>(Hq) * 128 * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(Qb)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool split_shape(int kind, int nq, int B, int Hq, int Hkv, int D, int block_size, int max_blocks,
                 int max_seq_len, SplitShape* out) {
    SplitShape s;
    const int g = Hq / Hkv;
    s.kind = kind;
    s.mq = nq > 0 ? 1 : 0;
    if (kind == kSplitFma) {
        s.nslices = g;  // one query head per kv unit
        s.GS = 1;
    } else if (s.mq) {
        s.nslices = 1;  // one tile: nq queries x g heads of the kv head
        s.GS = nq * g;
        s.NT = (s.GS + 7) / 8;
    } else {
        s.nslices = (g + kHeadSlice - 1) / kHeadSlice;
        s.GS = (g + s.nslices - 1) / s.nslices;
        s.NT = (s.GS + 7) / 8;
    }
    s.U = Hkv * s.nslices;
    s.max_pages = (static_cast<int64_t>(std::min(max_seq_len, max_blocks * block_size)) +
                   block_size - 1) / block_size;
    s.P_max = static_cast<int64_t>(B) * s.U * s.max_pages;
    if (s.P_max > INT32_MAX) return false;

    s.lens_bytes = round_up(static_cast<size_t>(2 * B + 1) * 4u, 1024);
    // Many warps with one stage each: a warp waits for its chunk while the other
    // warps of the SM compute, so bytes in flight scale with the warp count.
    s.stages = kDefaultStages;
    if (s.mq) {
        // Several queries per sequence: the query rows at a padded pitch in
        // the stage after K and V (reread at every chunk; one stage per warp
        // keeps a segment's rows in place), two blocks of five warps per SM
        // at 16 columns, three warps a block below. The per-warp row region
        // of the two-n-tile decode below measured slower for this kernel
        // (its launch bound then caps registers at 170 instead of 204).
        s.stages = 1;
        s.stage_bytes = round_up(2u * kChunkTokens * D * 2u +
                                     static_cast<size_t>(s.GS) * mq_q_pitch(D), 1024);
        s.q_bytes = 0;
        s.warps = s.NT == 2 ? kMqWarps : kDefaultWarps;
    } else if (s.NT == 2) {
        // One query, two n-tiles (9-16 query heads per kv head): the query
        // rows are reread at every chunk from a region of their own per warp
        // at a padded pitch, so that a stage is just a chunk's K and V and
        // wastes nothing to the 1 KiB rounding. One stage per warp: a
        // segment's rows stay in place until it ends. As many warps as the
        // shared memory holds, in one block per SM: 11 at D = 128 (20.3 KB a
        // warp), 12 at D = 64.
        s.stages = 1;
        s.stage_bytes = round_up(2u * kChunkTokens * D * 2u, 1024);
        s.q_bytes = round_up(static_cast<size_t>(s.GS) * mq_q_pitch(D), 16);
        const size_t per_warp = s.stage_bytes + s.q_bytes + 8 + 16;  // ring, rows, barrier, record
        const size_t fixed = 1024 + s.lens_bytes + 16 + 16;         // alignment, arrays, padding, probe
        if (fixed >= kSmemLimit) return false;
        s.warps = static_cast<int>(std::min<size_t>(kQsMaxWarps, (kSmemLimit - fixed) / per_warp));
        if (s.warps < 1) return false;
    } else {
        // K and V of a chunk, then the segment's query rows (read once per
        // segment): 3 warps per block, up to 4 blocks per SM.
        s.stage_bytes = round_up(2u * kChunkTokens * D * 2u + static_cast<size_t>(s.GS) * D * 2u,
                                 1024);
        s.q_bytes = 0;
        s.warps = kDefaultWarps;
    }
    // ring, mbarriers (8 B each, padded to 16 B), per-stage range records (16 B
    // each), the wait-probe mbarrier (16 B), the query-row regions
    s.smem = 1024 + s.lens_bytes + static_cast<size_t>(s.warps) * s.stages * s.stage_bytes +
             round_up(static_cast<size_t>(s.warps) * s.stages * 8, 16) +
             static_cast<size_t>(s.warps) * s.stages * 16 + 16 +
             static_cast<size_t>(s.warps) * s.q_bytes;
    if (s.smem > kSmemLimit) return false;
    *out = s;
    return true;
}

SplitGrid split_grid(const SplitShape& s, int B, int D, int block_size, int64_t rows, int num_sms,
                     int per_sm, bool dynamic, int max_blocks, int force_permille,
                     int force_pages) {
    SplitGrid gr;
    const int64_t need = (s.P_max + static_cast<int64_t>(s.warps) * kMinPagesPerWarp - 1) /
                         (static_cast<int64_t>(s.warps) * kMinPagesPerWarp);
    int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
    if (max_blocks > 0) cap = std::min<int64_t>(cap, max_blocks);
    gr.blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(need, cap)));
    gr.NW = gr.blocks * s.warps;
    // Dynamic tail: part of the page stream handed out in pieces through an
    // atomic counter, so that warps whose pages arrive early take more of the
    // end; its partials are merged with four warps per row. Measured (whole
    // decode call, or step):
    //  * one query per sequence, sequences up to 1024 pages or more: 15 % in
    //    16-page pieces; Llama-3-8B GQA batches of 64 / 96 / 128 / 192 / 256
    //    long sequences ran 2-5 % faster with it (DRAM-saturating kernels
    //    finish unevenly without it). 16 pages beat 8 and 32 on both the GQA
    //    batch (block size 16) and the 128k-token one (block size 32).
    //  * several query heads per kv unit, sequences of 256 .. 1023 pages, at
    //    most 2048 merge rows: 15 % in 8-page pieces (the kernel still drops
    //    the tail when the batch has fewer than 8 pieces per warp). Uniform
    //    GQA batches, decode device time (graph replay, us): 32 x 8192 tokens
    //    159.7-159.9 vs 166.3-167.0 without, 64 x 4096 159.3-159.4 vs
    //    163.3-163.5, 32 x 4096 87.4-87.8 vs 90.0 (with the merge widths
    //    below), 8-16 sequences 0.6-2 % faster. The mixed shared-prefix batch
    //    (8192 rows) stays without a tail.
    //  * one query head per kv unit with shorter sequences: a quarter of the
    //    stream in 64-token pieces (one-head partials stay cheap), while the
    //    merge of all rows fits in one wave; Llama-7B MHA (1024 rows) step
    //    97.4-97.5 us against 98.4-98.5 with half and 101.8 with none (same
    //    box; 15 % and 35 % 97.7-97.9). Wider partials with shorter sequences
    //    gain nothing (mixed shared prefix, 4 heads: 142 vs 141 us split, and
    //    a slower merge).
    //  * tiles of two n-tiles (9-16 columns), several queries per sequence
    //    included: none. Those kernels (ten warps per SM, DRAM about 84 %)
    //    finish evenly without it, and it only adds partials: four queries
    //    per sequence of the GQA batch, split 335.8 vs 335.6-339.7 us and a
    //    merge of 30-34 instead of 16 us; 16 query heads per kv head
    //    (Llama-3-405B's grouping), split 281.7 us either way, step 290.7-
    //    290.9 us without against 303.3-304.0 with.
    const bool merge_fits = rows <= static_cast<int64_t>(num_sms) * kMergeRowsPerSm;
    gr.dyn_permille = 0;
    gr.dyn_pages = kDynPiecePages;
    if (dynamic && !s.mq && s.NT <= 1) {
        if (s.max_pages >= kDynMinPages) {
            gr.dyn_permille = kDynPermille;
        } else if (s.GS > 1 && s.max_pages >= kDynMidPages && rows <= kDynMidMaxRows) {
            gr.dyn_permille = kDynPermille;
            gr.dyn_pages = kDynMidPiecePages;
        } else if (s.GS == 1 && merge_fits) {
            gr.dyn_permille = kDynShortPermille;
            gr.dyn_pages = 64 / block_size;
        }
    }
    if (dynamic && force_permille >= 0) {
        gr.dyn_permille = force_permille;
        gr.dyn_pages = force_pages;
    }
    const int64_t max_pieces = s.P_max * gr.dyn_permille / 1000 / gr.dyn_pages + 1;
    gr.ranges = static_cast<int64_t>(gr.NW) + max_pieces;
    // Warps per output row in the merge kernel, from the partials per kv unit
    // (static ranges + dynamic pieces, on average). Eight when the kv units
    // have ~16 partials or more and eight warps per row still fit in one wave
    // (at most 8 rows per SM), so that a warp folds its share in one batch of
    // loads instead of several in turn; four with a dynamic tail or ~4
    // partials or more (the Llama-3-8B GQA step measured 4 against 2 and 8);
    // one otherwise. Against one warp per row without a tail, decode device
    // time (graph replay, us): one GQA sequence of 2,048 / 8,192 tokens 9.8 /
    // 12.9 vs 15.4 / 32.7, 8 sequences 17.2 / 49.4 vs 22.4 / 56.1, 16
    // sequences 31.8 / 89.0 vs 34.5 / 92.5; 128k-token context 615.8 vs 621.0.
    // Rows of 64 or 128 partials or more (one or two very long sequences)
    // take 16 or 32 warps while the rows still fit one wave at 64 warps per
    // SM.
    const int64_t units = static_cast<int64_t>(B) * s.U;
    if (rows * 32 <= 64LL * num_sms && gr.ranges >= 128 * units) gr.merge_wpr = 32;
    else if (rows * 16 <= 64LL * num_sms && gr.ranges >= 64 * units) gr.merge_wpr = 16;
    else if (rows <= 8LL * num_sms && gr.ranges >= 16 * units) gr.merge_wpr = 8;
    else if (gr.dyn_permille > 0 || gr.ranges >= 4 * units) gr.merge_wpr = 4;
    else gr.merge_wpr = 1;
    gr.meta_bytes = round_up(static_cast<size_t>(kMetaHeader + B + 1) * 4u, 256);
    gr.ml_bytes = round_up(static_cast<size_t>(2) * gr.ranges * s.GS * 2 * 4u, 256);
    gr.acc_bytes = round_up(static_cast<size_t>(2) * gr.ranges * s.GS * D * 4u, 256);
    return gr;
}

void set_split_plan(SplitArgs* a, const SplitShape& s, const SplitGrid& gr) {
    a->GS = s.GS;
    a->nslices = s.nslices;
    a->U = s.U;
    a->stages = s.stages;
    a->stage_bytes = static_cast<int>(s.stage_bytes);
    a->lens_bytes = static_cast<int>(s.lens_bytes);
    a->q_bytes = static_cast<int>(s.q_bytes);
    a->dyn_permille = gr.dyn_permille;
    a->dyn_pages = gr.dyn_pages;
}

}  // namespace pa

struct pa_plan {
    int device = -1;
    int num_sms = 0;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    int* err = nullptr;
    int forced_path = PA_PATH_AUTO;
    int sched_permille = -1, sched_pages = 0;  // forced dynamic tail (pa_plan_set_schedule)
    int merge_mode = PA_MERGE_AUTO;             // pa_plan_set_merge
    int last_fused = 0;
    size_t cnt_clean = 0;  // bytes at the end of the workspace known to be zero
    int last_path = 0, last_blocks = 0, last_warps = 0;
    cudaEvent_t ev_start = nullptr, ev_stop = nullptr;
    MapKey kkey, vkey;
    CUtensorMap kmap, vmap;
    std::vector<OccKey> occ;
};

extern "C" {

const char* pa_status_str(pa_status s) {
    switch (s) {
        case PA_OK: return "ok";
        case PA_ERR_NULL: return "a required pointer is NULL";
        case PA_ERR_SHAPE: return "sizes out of range or inconsistent";
        case PA_ERR_DTYPE: return "unsupported element type or path";
        case PA_ERR_BLOCK_SIZE: return "block_size must be 16 or 32";
        case PA_ERR_WORKSPACE: return "workspace too small";
        case PA_ERR_CUDA: return "a CUDA call failed";
        case PA_ERR_BOUNDS: return "a length or table entry was out of range on the device";
        case PA_ERR_ALIGN: return "a tensor is not 16-byte aligned";
        case PA_ERR_NO_BLOCKS: return "the block pool has too few free blocks";
    }
    return "unknown status";
}

pa_status pa_append_kv(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                       const int32_t* block_tables, int max_blocks, const int32_t* cache_lens,
                       int B, int Hkv, int D, int block_size, int num_blocks, pa_dtype kv_dtype,
                       struct CUstream_st* stream) {
    if (!k_new || !v_new || !k_pool || !v_pool || !block_tables || !cache_lens) return PA_ERR_NULL;
    if (kv_dtype != PA_F32 && kv_dtype != PA_BF16) return PA_ERR_DTYPE;
    if (block_size != 16 && block_size != 32) return PA_ERR_BLOCK_SIZE;
    if (B < 0 || Hkv < 1 || (D != 64 && D != 128) || num_blocks < 1 || max_blocks < 1)
        return PA_ERR_SHAPE;
    if (static_cast<int64_t>(max_blocks) * block_size > INT32_MAX) return PA_ERR_SHAPE;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
        return PA_ERR_ALIGN;
    if (B == 0) return PA_OK;
    pa::AppendArgs a{k_new, v_new, k_pool, v_pool, block_tables, cache_lens,
                     B, Hkv, D, block_size, max_blocks, num_blocks,
                     kv_dtype == PA_F32 ? 4 : 2};
    return pa::launch_append(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

namespace {

// The decode of pa_decode, with q_start != null (T query rows, at most nq per
// sequence) of pa_decode_multi, and with k_new != null of pa_append_decode
// (the step's new rows appended at position seq_lens[b] - 1 first).
pa_status decode_impl(const void* q, const int32_t* q_start, int T, int nq, const void* k_pool,
                      const void* v_pool, const int32_t* block_tables, int max_blocks,
                      const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int block_size,
                      int num_blocks, int max_seq_len, float scale, pa_dtype kv_dtype, void* out,
                      pa_dtype out_dtype, pa_plan** plan_inout, struct CUstream_st* stream_,
                      const void* k_new = nullptr, const void* v_new = nullptr) {
    if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out || !plan_inout)
        return PA_ERR_NULL;
    if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PA_ERR_ALIGN;
    if ((kv_dtype != PA_F32 && kv_dtype != PA_BF16) || (out_dtype != PA_F32 && out_dtype != PA_BF16))
        return PA_ERR_DTYPE;
    if (block_size != 16 && block_size != 32) return PA_ERR_BLOCK_SIZE;
    if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || (D != 64 && D != 128) || num_blocks < 1 ||
        max_blocks < 1 || max_seq_len < 1 || !std::isfinite(scale) || B > pa::kMaxBatch)
        return PA_ERR_SHAPE;
    if (static_cast<int64_t>(num_blocks) * Hkv > INT32_MAX ||
        static_cast<int64_t>(max_blocks) * block_size > INT32_MAX)
        return PA_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return PA_ERR_ALIGN;
    // Several queries per sequence: up to 16 (query, head) columns per kv
    // head run on the split decode's tensor-core tiles (the pages streamed
    // once for all of them); more run on the prefill kernel's tcgen05 tiles
    // (128-row query tiles, D = 128, Hq / Hkv dividing 128). bf16 pools.
    bool via_prefill = false;
    if (q_start) {
        if (kv_dtype != PA_BF16) return PA_ERR_DTYPE;
        if (T < 0 || nq < 1) return PA_ERR_SHAPE;
        if (static_cast<int64_t>(nq) * (Hq / Hkv) > 16) {
            const int gq = Hq / Hkv;
            if (D != 128 || gq > 128 || 128 % gq != 0 || max_blocks > 16384 ||
                Hkv > pa::kMaxGridYZ)
                return PA_ERR_SHAPE;
            via_prefill = true;
        }
    }
    if (static_cast<int64_t>(q_start ? T : B) * Hq > pa::kMaxRows) return PA_ERR_SHAPE;
    if (q_start && T == 0) return PA_OK;
    if (B == 0) return PA_OK;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

    // Everything that depends on the arguments alone is checked before a plan
    // exists, so that an argument error never creates one.
    const int g = Hq / Hkv;
    int path = q_start ? PA_PATH_MMA : (*plan_inout ? (*plan_inout)->forced_path : PA_PATH_AUTO);
    // bf16 pools run on the tensor-core tile for every group size, one query
    // head per kv head included (one real column of eight: with the dynamic
    // tail it measured 94.9-95.0 us against 96.2 us for the CUDA-core path on
    // the Llama-7B MHA workload; PA_PATH_FMA still selects the latter).
    if (path == PA_PATH_AUTO) path = kv_dtype == PA_F32 ? PA_PATH_SIMPLE : PA_PATH_MMA;
    if (kv_dtype == PA_F32 && path != PA_PATH_SIMPLE) return PA_ERR_DTYPE;
    if (path == PA_PATH_SIMPLE && max_seq_len > PA_SIMPLE_MAX_SEQ_LEN) return PA_ERR_SHAPE;
    const float scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    pa::SplitShape sh;
    if (path != PA_PATH_SIMPLE && !via_prefill &&
        !pa::split_shape(path == PA_PATH_FMA ? pa::kSplitFma : pa::kSplitMma, q_start ? nq : 0, B,
                         Hq, Hkv, D, block_size, max_blocks, max_seq_len, &sh))
        return PA_ERR_SHAPE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    pa_plan* plan = *plan_inout;
    if (!plan) {
        plan = new pa_plan();
        plan->device = dev;
        if (cudaDeviceGetAttribute(&plan->num_sms, cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess ||
            cudaMalloc(reinterpret_cast<void**>(&plan->err), 256) != cudaSuccess ||
            cudaMemset(plan->err, 0, 256) != cudaSuccess) {
            if (plan->err) cudaFree(plan->err);
            delete plan;
            return PA_ERR_CUDA;
        }
        *plan_inout = plan;
    }
    if (plan->device != dev) return PA_ERR_CUDA;  // a plan belongs to one device

    if (via_prefill) {
        CUtensorMap kmap, vmap;
        if (!pa::encode_pool_map(&kmap, k_pool, num_blocks * Hkv, D, block_size) ||
            !pa::encode_pool_map(&vmap, v_pool, num_blocks * Hkv, D, block_size))
            return PA_ERR_CUDA;
        // A small call (fewer one-tile blocks than SMs) splits every tile's
        // key range over several blocks; their partials live in the plan's
        // workspace after its first 64 bytes, which hold the split decode's
        // counters (zero between calls, left untouched here).
        const int64_t nqq = std::min<int64_t>(nq, T);
        const int splits = pa::prefill_split_count(B, Hq, Hkv, nqq, max_seq_len, plan->num_sms);
        float* part = nullptr;
        if (splits > 1) {
            const size_t need = 64 + pa::prefill_split_bytes(B, Hq, Hkv, nqq, splits);
            if (plan->ws_bytes < need) {
                if (plan->ws) cudaFree(plan->ws);
                plan->ws = nullptr;
                plan->ws_bytes = 0;
                if (cudaMalloc(&plan->ws, need) != cudaSuccess) return PA_ERR_CUDA;
                if (cudaMemset(plan->ws, 0, need) != cudaSuccess) return PA_ERR_CUDA;
                plan->ws_bytes = need;
                plan->cnt_clean = need;
            }
            part = reinterpret_cast<float*>(static_cast<char*>(plan->ws) + 64);
            plan->cnt_clean = std::min(plan->cnt_clean, plan->ws_bytes - need);
        }
        if (plan->ev_start) cudaEventRecord(plan->ev_start, stream);
        const cudaError_t e = pa::launch_prefill(kmap, vmap, q, T, q_start, block_tables, seq_lens,
                                                 out, plan->err, B, Hq, Hkv, max_blocks,
                                                 num_blocks, max_seq_len, nq, scale_log2,
                                                 out_dtype == PA_BF16, block_size, stream, part,
                                                 splits, /*zero_invalid=*/1);
        if (plan->ev_stop) cudaEventRecord(plan->ev_stop, stream);
        plan->last_path = PA_PATH_PREFILL;
        plan->last_blocks = 0;
        plan->last_warps = 0;
        return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }

    // The append as its own kernel, for the paths that do not fuse it: the
    // step's rows at position seq_lens[b] - 1, before the decode reads them.
    auto append_first = [&]() -> cudaError_t {
        pa::AppendArgs ap{k_new, v_new, const_cast<void*>(k_pool), const_cast<void*>(v_pool),
                          block_tables, seq_lens, B, Hkv, D, block_size, max_blocks, num_blocks,
                          kv_dtype == PA_F32 ? 4 : 2};
        ap.pos_offset = 1;
        return pa::launch_append(ap, stream);
    };

    if (path == PA_PATH_SIMPLE) {
        if (k_new && append_first() != cudaSuccess) return PA_ERR_CUDA;
        pa::SimpleArgs a{q, k_pool, v_pool, block_tables, seq_lens, out, plan->err,
                         B, Hq, Hkv, D, block_size, max_blocks, num_blocks, max_seq_len,
                         scale_log2, kv_dtype == PA_BF16, out_dtype == PA_BF16};
        if (plan->ev_start) cudaEventRecord(plan->ev_start, stream);
        const cudaError_t e = pa::launch_simple(a, stream);
        if (plan->ev_stop) cudaEventRecord(plan->ev_stop, stream);
        plan->last_path = PA_PATH_SIMPLE;
        plan->last_blocks = (B * Hq + 3) / 4;
        plan->last_warps = B * Hq;
        return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }

    // Split paths (bf16 pools).
    SplitLaunch L{sh.kind, D, block_size, sh.NT, sh.warps, 0, sh.smem};
    L.mq = sh.mq;
    // The fused merge serves one query per sequence on one n-tile.
    const bool can_fuse = !q_start && sh.kind == pa::kSplitMma && sh.NT == 1 && sh.warps == 3;
    L.fused = can_fuse && plan->merge_mode == PA_MERGE_FUSED ? 1 : 0;
    if (plan->merge_mode == PA_MERGE_FUSED && !can_fuse) return PA_ERR_SHAPE;
    // The append rides in the split kernel on the one-n-tile tensor-core
    // tiles (up to 8 query heads per kv head) with one stage per warp and the
    // merge kernel; elsewhere it runs first on its own. With two n-tiles the
    // fused kernel measured slower than the two launches (Llama-3-405B
    // grouping: step 283.5 vs 280.2 us), so those shapes take the append
    // kernel.
    L.append = k_new && !q_start && !L.fused && sh.kind == pa::kSplitMma && sh.NT == 1 &&
                       sh.stages == 1 ? 1 : 0;
    int per_sm = 0;
    for (const OccKey& o : plan->occ) {
        if (o.kind == L.kind && o.D == D && o.BS == block_size && o.NT == L.NT &&
            o.warps == L.warps && o.smem == L.smem && o.mq == L.mq && o.fused == L.fused &&
            o.append == L.append)
            per_sm = o.blocks_per_sm;
    }
    if (per_sm == 0) {
        cudaError_t e;
        per_sm = pa::split_blocks_per_sm(L, &e);
        if (e != cudaSuccess || per_sm < 1) return PA_ERR_CUDA;
        plan->occ.push_back(OccKey{L.kind, D, block_size, L.NT, L.warps, L.smem, per_sm, L.mq,
                                   L.fused, L.append});
    }
    pa::SplitGrid gr = pa::split_grid(sh, B, D, block_size,
                                      static_cast<int64_t>(q_start ? T : B) * Hq,
                                      plan->num_sms, per_sm, true, 0,
                                      plan->sched_permille, plan->sched_pages);
    if (L.fused) gr.cnt_bytes = round_up(static_cast<size_t>(B) * sh.U * 4u, 256);
    L.blocks = gr.blocks;

    // Workspace: metadata, partial (m, l), partial value sums.
    const size_t need_ws = gr.workspace_bytes();
    if (plan->ws_bytes < need_ws) {
        if (plan->ws) cudaFree(plan->ws);
        plan->ws = nullptr;
        plan->ws_bytes = 0;
        if (cudaMalloc(&plan->ws, need_ws) != cudaSuccess) return PA_ERR_CUDA;
        if (cudaMemset(plan->ws, 0, need_ws) != cudaSuccess) return PA_ERR_CUDA;  // piece counter = 0
        plan->ws_bytes = need_ws;
        plan->cnt_clean = need_ws;
    }
    char* ws = static_cast<char*>(plan->ws);
    int* meta = reinterpret_cast<int*>(ws);
    float* ml = reinterpret_cast<float*>(ws + gr.meta_bytes);
    float* acc = reinterpret_cast<float*>(ws + gr.meta_bytes + gr.ml_bytes);
    // The segment counters of the fused merge sit at the end of the
    // workspace. A fused call leaves them zero; the plan tracks how many bytes
    // at the end are known to be zero (all of a fresh workspace, less what
    // any call's partials have overwritten) and clears the counters when a
    // call needs more than that.
    int* cnt = nullptr;
    if (L.fused) {
        cnt = reinterpret_cast<int*>(ws + plan->ws_bytes - gr.cnt_bytes);
        if (plan->cnt_clean < gr.cnt_bytes) {
            if (cudaMemsetAsync(cnt, 0, gr.cnt_bytes, stream) != cudaSuccess) return PA_ERR_CUDA;
            plan->cnt_clean = gr.cnt_bytes;
        }
    }
    plan->cnt_clean = std::min(plan->cnt_clean,
                               plan->ws_bytes - (gr.meta_bytes + gr.ml_bytes + gr.acc_bytes));

    const int rows = num_blocks * Hkv;
    MapKey kk{k_pool, rows, D, block_size}, vk{v_pool, rows, D, block_size};
    if (!(plan->kkey == kk)) {
        if (!pa::encode_pool_map(&plan->kmap, k_pool, rows, D, block_size)) {
            plan->kkey = MapKey{};
            return PA_ERR_CUDA;
        }
        plan->kkey = kk;
    }
    if (!(plan->vkey == vk)) {
        if (!pa::encode_pool_map(&plan->vmap, v_pool, rows, D, block_size)) {
            plan->vkey = MapKey{};
            return PA_ERR_CUDA;
        }
        plan->vkey = vk;
    }

    pa::SplitArgs a{};
    a.q = static_cast<const uint16_t*>(q);
    a.tables = block_tables;
    a.seq_lens = seq_lens;
    a.out = out;
    a.ws_acc = acc;
    a.ws_ml = ml;
    a.ws_meta = meta;
    a.err = plan->err;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.g = g;
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    a.max_seq_len = max_seq_len;
    a.scale_log2 = scale_log2;
    a.out_bf16 = out_dtype == PA_BF16;
    pa::set_split_plan(&a, sh, gr);
    a.q_start = q_start;
    a.nq = nq;
    a.num_q = T;
    a.probe_wait = pa::wait_probe();
    a.ws_cnt = cnt;
    if (L.append) {
        a.k_new = static_cast<const uint16_t*>(k_new);
        a.v_new = static_cast<const uint16_t*>(v_new);
        a.kpool_w = static_cast<uint16_t*>(const_cast<void*>(k_pool));
        a.vpool_w = static_cast<uint16_t*>(const_cast<void*>(v_pool));
    } else if (k_new && append_first() != cudaSuccess) {
        return PA_ERR_CUDA;
    }

    if (plan->ev_start) cudaEventRecord(plan->ev_start, stream);
    cudaError_t e = pa::launch_split(L, plan->kmap, plan->vmap, a, stream);
    if (plan->ev_stop) cudaEventRecord(plan->ev_stop, stream);
    if (e != cudaSuccess) return PA_ERR_CUDA;
    plan->last_fused = L.fused;
    if (!L.fused) {
        pa::MergeArgs m{meta, acc, ml, out, B, Hq, g, sh.GS, sh.nslices, sh.U, D,
                        out_dtype == PA_BF16, gr.merge_wpr, (q_start ? T : B) * Hq,
                        q_start};
        e = pa::launch_merge(m, stream);
    }
    plan->last_path = path;
    plan->last_blocks = L.blocks;
    plan->last_warps = gr.NW;
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

pa_status pa_decode(const void* q, const void* k_pool, const void* v_pool,
                    const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, int B,
                    int Hq, int Hkv, int D, int block_size, int num_blocks, int max_seq_len,
                    float scale, pa_dtype kv_dtype, void* out, pa_dtype out_dtype,
                    pa_plan** plan_inout, struct CUstream_st* stream) {
    return decode_impl(q, nullptr, B, 1, k_pool, v_pool, block_tables, max_blocks, seq_lens, B,
                       Hq, Hkv, D, block_size, num_blocks, max_seq_len, scale, kv_dtype, out,
                       out_dtype, plan_inout, stream);
}

pa_status pa_append_decode(const void* q, const void* k_new, const void* v_new, void* k_pool,
                           void* v_pool, const int32_t* block_tables, int max_blocks,
                           const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int block_size,
                           int num_blocks, int max_seq_len, float scale, pa_dtype kv_dtype,
                           void* out, pa_dtype out_dtype, pa_plan** plan_inout,
                           struct CUstream_st* stream) {
    if (!k_new || !v_new) return PA_ERR_NULL;
    return decode_impl(q, nullptr, B, 1, k_pool, v_pool, block_tables, max_blocks, seq_lens, B,
                       Hq, Hkv, D, block_size, num_blocks, max_seq_len, scale, kv_dtype, out,
                       out_dtype, plan_inout, stream, k_new, v_new);
}

pa_status pa_decode_multi(const void* q, const int32_t* q_start, int num_queries, int max_q,
                          const void* k_pool, const void* v_pool, const int32_t* block_tables,
                          int max_blocks, const int32_t* seq_lens, int B, int Hq, int Hkv, int D,
                          int block_size, int num_blocks, int max_seq_len, float scale,
                          pa_dtype kv_dtype, void* out, pa_dtype out_dtype, pa_plan** plan_inout,
                          struct CUstream_st* stream) {
    if (!q_start) return PA_ERR_NULL;
    return decode_impl(q, q_start, num_queries, max_q, k_pool, v_pool, block_tables, max_blocks,
                       seq_lens, B, Hq, Hkv, D, block_size, num_blocks, max_seq_len, scale, kv_dtype,
                       out, out_dtype, plan_inout, stream);
}

pa_status pa_copy_blocks(void* k_pool, void* v_pool, const int32_t* copy_src,
                         const int32_t* copy_dst, int n, int Hkv, int D, int block_size,
                         int num_blocks, pa_dtype kv_dtype, struct CUstream_st* stream) {
    if (!k_pool || !v_pool || (n > 0 && (!copy_src || !copy_dst))) return PA_ERR_NULL;
    if (kv_dtype != PA_F32 && kv_dtype != PA_BF16) return PA_ERR_DTYPE;
    if (block_size != 16 && block_size != 32) return PA_ERR_BLOCK_SIZE;
    if (n < 0 || n > (1 << 24) || Hkv < 1 || (D != 64 && D != 128) || num_blocks < 1)
        return PA_ERR_SHAPE;
    if (!aligned16(k_pool) || !aligned16(v_pool)) return PA_ERR_ALIGN;
    if (n == 0) return PA_OK;
    pa::CopyArgs a{k_pool, v_pool, copy_src, copy_dst, n, num_blocks,
                   static_cast<int64_t>(Hkv) * block_size * D * (kv_dtype == PA_F32 ? 4 : 2)};
    return pa::launch_copy_blocks(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_prefill(const void* q, const int32_t* q_start, int num_queries, const void* k_pool,
                     const void* v_pool, const int32_t* block_tables, int max_blocks,
                     const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int block_size,
                     int num_blocks, int max_q, int max_seq_len, float scale, pa_dtype kv_dtype,
                     void* out, pa_dtype out_dtype, int* device_error,
                     struct CUstream_st* stream) {
    if (!q || !q_start || !k_pool || !v_pool || !block_tables || !seq_lens || !out)
        return PA_ERR_NULL;
    if (kv_dtype != PA_BF16 || (out_dtype != PA_F32 && out_dtype != PA_BF16)) return PA_ERR_DTYPE;
    if (block_size != 16 && block_size != 32) return PA_ERR_BLOCK_SIZE;
    if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D != 128 || num_blocks < 1 ||
        max_blocks < 1 || max_blocks > 16384 || max_q < 1 || max_seq_len < 1 ||
        !std::isfinite(scale) || num_queries < 0 || B > pa::kMaxGridYZ || Hkv > pa::kMaxGridYZ)
        return PA_ERR_SHAPE;
    const int g = Hq / Hkv;
    if (g > 128 || 128 % g != 0) return PA_ERR_SHAPE;  // a block holds 128 / g whole queries
    if (static_cast<int64_t>(num_blocks) * Hkv > INT32_MAX ||
        static_cast<int64_t>(max_blocks) * block_size > INT32_MAX)
        return PA_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return PA_ERR_ALIGN;
    if (B == 0 || num_queries == 0) return PA_OK;
    CUtensorMap kmap, vmap;
    if (!pa::encode_pool_map(&kmap, k_pool, num_blocks * Hkv, D, block_size) ||
        !pa::encode_pool_map(&vmap, v_pool, num_blocks * Hkv, D, block_size))
        return PA_ERR_CUDA;
    int* err = device_error;
    if (!err && pa::append_error_address(&err) != cudaSuccess) return PA_ERR_CUDA;
    const float scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    return pa::launch_prefill(kmap, vmap, q, num_queries, q_start, block_tables, seq_lens, out,
                              err, B, Hq, Hkv, max_blocks, num_blocks, max_seq_len, max_q, scale_log2,
                              out_dtype == PA_BF16, block_size,
                              reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_free(pa_plan* plan) {
    if (!plan) return PA_OK;
    DeviceGuard guard(plan->device);
    pa_status st = PA_OK;
    if (plan->ws && cudaFree(plan->ws) != cudaSuccess) st = PA_ERR_CUDA;
    if (plan->err && cudaFree(plan->err) != cudaSuccess) st = PA_ERR_CUDA;
    delete plan;
    return st;
}

pa_status pa_last_device_error(pa_plan* plan, int* err) {
    if (!err) return PA_ERR_NULL;
    *err = 0;
    if (!plan) {
        if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
        return pa::read_append_error(err) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
    DeviceGuard guard(plan->device);
    if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, plan->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(plan->err, 0, sizeof(int)) != cudaSuccess)
        return PA_ERR_CUDA;
    *err = v;
    return PA_OK;
}

pa_status pa_plan_set_path(pa_plan* plan, int path) {
    if (!plan) return PA_ERR_NULL;
    if (path < PA_PATH_AUTO || path > PA_PATH_MMA) return PA_ERR_SHAPE;
    plan->forced_path = path;
    return PA_OK;
}

pa_status pa_plan_set_merge(pa_plan* plan, int mode) {
    if (!plan) return PA_ERR_NULL;
    if (mode < PA_MERGE_AUTO || mode > PA_MERGE_FUSED) return PA_ERR_SHAPE;
    plan->merge_mode = mode;
    return PA_OK;
}

pa_status pa_debug_set_wait_probe(int enable) {
    g_wait_probe.store(enable ? 1 : 0, std::memory_order_relaxed);
    return PA_OK;
}

pa_status pa_debug_set_prefill_kernel(int which) {
    if (which != PA_PREFILL_AUTO && which != PA_PREFILL_ONE_TILE && which != PA_PREFILL_TWO_TILE)
        return PA_ERR_SHAPE;
    g_prefill_kernel.store(which, std::memory_order_relaxed);
    return PA_OK;
}

pa_status pa_plan_set_schedule(pa_plan* plan, int dyn_permille, int dyn_pages) {
    if (!plan) return PA_ERR_NULL;
    if (dyn_permille < 0) {
        plan->sched_permille = -1;
        plan->sched_pages = 0;
        return PA_OK;
    }
    if (dyn_permille > 500 || dyn_pages < 1 || dyn_pages > 4096) return PA_ERR_SHAPE;
    plan->sched_permille = dyn_permille;
    plan->sched_pages = dyn_pages;
    return PA_OK;
}

pa_status pa_plan_info(const pa_plan* plan, int* path, int* blocks, int* warps) {
    if (!plan) return PA_ERR_NULL;
    if (path) *path = plan->last_path;
    if (blocks) *blocks = plan->last_blocks;
    if (warps) *warps = plan->last_warps;
    return PA_OK;
}

pa_status pa_plan_set_split_events(pa_plan* plan, struct CUevent_st* start,
                                   struct CUevent_st* stop) {
    if (!plan) return PA_ERR_NULL;
    if ((start == nullptr) != (stop == nullptr)) return PA_ERR_NULL;
    plan->ev_start = reinterpret_cast<cudaEvent_t>(start);
    plan->ev_stop = reinterpret_cast<cudaEvent_t>(stop);
    return PA_OK;
}

}  // extern "C"
