// Paged multi-query attention on the tcgen05 tensor cores, for calls whose
// sequences all fit one query tile (at most 128 / g queries each: the
// speculative verification of a few drafted tokens, short chunks).
//
// It computes what prefill_kernel in pa_prefill.cu computes: query i of
// sequence b, at position L_b - n_b + i, attends causally to the tokens up to
// its position through the block table ("FlashAttention vs PagedAttention",
// "How prefill and decode change the diagnosis"; exact attention as in
// "39 · PagedAttention" §1-§2). That kernel keeps two query tiles per block so
// that one tile's softmax runs while the tensor core works on the other; with
// one tile per sequence and kv head its second tile is empty, and every
// chunk then waits for its own softmax. Here a block holds one tile and
// instead keeps three score buffers in tensor memory beside O (3 x 128 + 128
// = all 512 columns): S(c) goes to buffer c % 3, and S(c + 3) is issued right
// after PV(c), which reads P(c) from that buffer (one thread's products run
// in issue order). The scores of the next chunks are therefore ready while a
// softmax runs.
//
// Warps:
//   * 16 and 18 (producers): tiled bulk tensor copies of 128-token K and V
//     chunks through the block table into 3-stage K and V rings, the table
//     entries of a chunk loaded one chunk ahead; the K warp first copies the
//     query tile (the tensor map over q of the two-tile kernel);
//   * 17 (MMA): one thread issues S(c) = Q K(c)^T and O (+)= P(c) V(c), both
//     M = 128, N = 128, K = 128, with P read from tensor memory;
//   * 0-7 and 8-15 (softmax, two groups taking the even and the odd chunks,
//     two threads per row on 64 scores each): the reference max of chunk c is
//     handed to the group of chunk c + 1 through shared memory (an mbarrier
//     per chunk parity). It is raised only when a chunk exceeds it by more
//     than 2^8; the group that raises it rescales O after the previous value
//     product is done. Each group keeps its own part of the row sum; at the
//     end both bring theirs to the final reference max and add them through
//     shared memory, and each group normalises and stores half of O's columns.
// V rows past the last token of the final chunk are zeroed before its value
// product. Blocks are ordered longest sequence first.
//
// Key split (a small call with a workspace, from pa_decode_multi): grid.x
// holds tiles x splits blocks, and split s of a tile takes its chunks
// s * ceil(nc / splits) onward. The pipeline counts the block's own chunks;
// pages and the causal mask use the sequence's. Each block writes its O
// unnormalised with every row's reference max and row sum, and
// prefill_split_merge_kernel combines the splits of each row.
//
// Every mbarrier wait is bounded. A role that gives up raises a shared abort
// flag (and PA_DEVERR_TIMEOUT); the others see it in their own waits. Before
// the block leaves, each producer waits (bounded) for its copies in flight,
// the MMA thread for its products, and the block frees its tensor memory.
#include <cuda_bf16.h>

#include <algorithm>

#include "pa.h"
#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "pa_tc.cuh"

namespace pa {
namespace {

constexpr int kRows = 128;      // M: query rows per tile (one tile per block)
constexpr int kChunk = 128;     // tokens per K/V chunk
constexpr int kD = 128;         // head dimension
constexpr int kStagesK = 3;     // K ring depth
constexpr int kStagesV = 3;     // V ring depth
constexpr int kSbuf = 3;        // score buffers in tensor memory (chunk c uses c % 3)
constexpr int kGroupThreads = 2 * kRows;            // softmax threads of a group: two per row
constexpr int kSoftmaxThreads = 2 * kGroupThreads;   // two groups, alternate chunks
constexpr int kWarpLoad = kSoftmaxThreads / 32;     // warp 16: K copies
constexpr int kWarpMma = kWarpLoad + 1;             // warp 17
constexpr int kWarpLoadV = kWarpMma + 1;            // warp 18: V copies
constexpr int kThreads = kSoftmaxThreads + 96;
constexpr int kSortMax = 256;   // sequences ordered by length up to this batch size
constexpr uint32_t kTmemCols = 512;
// Tensor-memory columns: score buffer j (128; P over its first 64), then O (128).
__host__ __device__ constexpr uint32_t col_s(int j) { return 128u * j; }
constexpr uint32_t kColO = 128u * kSbuf;
static_assert(kColO + 128 <= kTmemCols, "tensor-memory columns");
constexpr float kRescaleLog2 = 8.f;  // raise the reference max only beyond 2^8

// Shared-memory layout (byte offsets from a 1024-aligned base).
constexpr uint32_t kTileQ = 32768;                    // 2 halves x 128 rows x 128 B
constexpr uint32_t kHalfKV = kChunk * 128;            // one 64-column half of a chunk
constexpr uint32_t kStageKV = 2 * kHalfKV;            // 2 halves x 128 rows x 128 B
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileQ;
constexpr uint32_t kOffV = kOffK + kStagesK * kStageKV;
constexpr uint32_t kOffBar = kOffV + kStagesV * kStageKV;
// mbarriers (8 bytes each) and slots, at kOffBar + ...
constexpr uint32_t kBarKFull = 0;                     // [kStagesK]
constexpr uint32_t kBarKEmpty = kBarKFull + 8 * kStagesK;
constexpr uint32_t kBarVFull = kBarKEmpty + 8 * kStagesK;  // [kStagesV]
constexpr uint32_t kBarVEmpty = kBarVFull + 8 * kStagesV;
constexpr uint32_t kBarS = kBarVEmpty + 8 * kStagesV; // [kSbuf] scores of a chunk ready
constexpr uint32_t kBarP = kBarS + 8 * kSbuf;         // [kSbuf] P of a chunk stored, 256 arrivals
constexpr uint32_t kBarPV = kBarP + 8 * kSbuf;        // [kSbuf] the chunk's value product done
constexpr uint32_t kBarM = kBarPV + 8 * kSbuf;        // [2] a chunk's reference max published
constexpr uint32_t kBarO = kBarM + 16;                // the last value product done
constexpr uint32_t kBarDrain = kBarO + 8;
constexpr uint32_t kBarProbe = kBarDrain + 8;         // nothing completes it (wait-expiry probe)
constexpr uint32_t kBarQ = kBarProbe + 8;             // the block's query tile has landed
constexpr uint32_t kSlotTmem = kBarQ + 8;
constexpr uint32_t kSlotAbort = kSlotTmem + 4;
constexpr uint32_t kSlotSeq = kSlotAbort + 4;
// One 1 KB area, used in turn for: the lengths of the ordering (prologue),
// the published reference max [2][kRows] (chunk loop), the row sums of the
// two groups [2][kRows] (epilogue, after a barrier of both groups).
constexpr uint32_t kOffLens = kOffBar + 256;
constexpr uint32_t kOffM = kOffLens;
constexpr uint32_t kOffL = kOffLens;
constexpr uint32_t kSmemBytes = 1024 + kOffLens + 4 * kSortMax;
static_assert(4 * kSortMax >= 2 * 4 * kRows, "shared area");
static_assert(kSlotSeq + 4 <= 256, "barrier area overlaps the max array");
static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0, "swizzle atoms");
static_assert(kSmemBytes <= 227 * 1024 && 2 * kSmemBytes > 228 * 1024,
              "one block per SM: it holds all 512 tensor-memory columns");

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kRows, kChunk, false, false);
constexpr uint32_t kIdescO = tc::idesc_bf16_f32(kRows, kD, false, true);  // B (V) MN-major

struct PrefillArgs {
    const uint16_t* q;        // [T][Hq][D] bf16
    const int32_t* q_start;   // [B + 1]
    const int32_t* tables;
    const int32_t* seq_lens;
    void* out;                // [T][Hq][D]
    int* err;
    int B, Hq, Hkv, g, Qb;    // Qb = queries per tile = 128 / g
    int num_q;                // rows of q and out
    int max_blocks, num_blocks, max_seq_len;
    float scale_log2;
    int out_bf16;
    int probe_wait;           // 1: the MMA thread's first wait expires (a test hook)
    int max_q;                // bound on every sequence's query count
    int zero_invalid;         // 1: an invalid sequence's rows get zeros (multi-query calls)
    // Key split: grid.x = tiles x splits, block x takes split x % splits of
    // tile x / splits. With splits > 1 every block writes a partial instead
    // of output rows: O unnormalised [num_parts][kRows][kD] at part, then
    // (reference max, row sum) [num_parts][kRows][2]; the merge kernel below
    // combines them.
    int splits, tiles;
    int num_parts;            // B * Hkv * tiles * splits
    float* part;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

template <int ND>
__device__ __forceinline__ void write_row(const PrefillArgs& a, size_t row, const float (&v)[ND],
                                          float inv, int d0) {
    if (a.out_bf16) {
        uint16_t* o = static_cast<uint16_t*>(a.out) + row * kD + d0;
#pragma unroll
        for (int i = 0; i < ND; i += 8) {
            uint4 w;
            w.x = pack_bf16x2(v[i] * inv, v[i + 1] * inv);
            w.y = pack_bf16x2(v[i + 2] * inv, v[i + 3] * inv);
            w.z = pack_bf16x2(v[i + 4] * inv, v[i + 5] * inv);
            w.w = pack_bf16x2(v[i + 6] * inv, v[i + 7] * inv);
            *reinterpret_cast<uint4*>(o + i) = w;
        }
    } else {
        float* o = static_cast<float*>(a.out) + row * kD + d0;
#pragma unroll
        for (int i = 0; i < ND; i += 4)
            *reinterpret_cast<float4*>(o + i) =
                make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv, v[i + 3] * inv);
    }
}

// Bounded wait that also gives up when another role raised the abort flag.
__device__ __forceinline__ bool wait_role(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
}

// Zeroes output rows [r0, r1) x query heads [h0, h0 + g) (an invalid
// sequence of a multi-query call), the block's threads in turn.
__device__ void zero_rows(const PrefillArgs& a, int64_t r0, int64_t r1, int h0, int tid) {
    const int64_t per_row = static_cast<int64_t>(a.g) * kD;
    const int64_t total = (r1 - r0) * per_row;
    for (int64_t i = tid; i < total; i += kThreads) {
        const int64_t r = r0 + i / per_row, e = i - (i / per_row) * per_row;
        const size_t idx = (static_cast<size_t>(r) * a.Hq + h0) * kD + static_cast<size_t>(e);
        if (a.out_bf16) static_cast<uint16_t*>(a.out)[idx] = 0;
        else static_cast<float*>(a.out)[idx] = 0.f;
    }
}

template <int BS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_one_tile_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const __grid_constant__ CUtensorMap qmap, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t bars = base + kOffBar;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kOffBar + kSlotAbort);
    int* seq_slot = reinterpret_cast<int*>(gbase + kOffBar + kSlotSeq);

    // The sequence of this block: blockIdx.z is its rank by length (longest
    // first, ties by index) when the batch is small enough to rank here.
    int b = blockIdx.z;
    if (a.B <= kSortMax) {
        int* lens = reinterpret_cast<int*>(gbase + kOffLens);
        for (int i = tid; i < a.B; i += kThreads) lens[i] = a.seq_lens[i];
        __syncthreads();
        for (int i = tid; i < a.B; i += kThreads) {
            const int li = lens[i];
            int r = 0;
            for (int j = 0; j < a.B; ++j) {
                const int lj = lens[j];
                r += (lj > li) || (lj == li && j < i);
            }
            if (r == static_cast<int>(blockIdx.z)) *seq_slot = i;
        }
        __syncthreads();
        b = *seq_slot;
    }
    const int h = blockIdx.y;
    const int L = a.seq_lens[b];
    const int limit = min(a.max_seq_len, a.max_blocks * BS);
    {
        const int64_t qs64 = a.q_start[b], n64 = static_cast<int64_t>(a.q_start[b + 1]) - qs64;
        if (n64 < 1 || n64 > a.max_q || L < n64 || L > limit || qs64 < 0 || qs64 + n64 > a.num_q) {
            if (blockIdx.x == 0 && h == 0 && tid == 0) atomicOr(a.err, kErrSeqLen);
            // The rows inside the arrays get zeros in a multi-query call and
            // are left untouched otherwise.
            if (a.zero_invalid && blockIdx.x == 0)
                zero_rows(a, qs64 > 0 ? qs64 : 0,
                          n64 > 0 ? (qs64 + n64 < a.num_q ? qs64 + n64 : a.num_q) : 0, h * a.g, tid);
            return;
        }
    }
    const int qs = a.q_start[b];
    const int n = a.q_start[b + 1] - qs;
    const int split = blockIdx.x % a.splits, tile = blockIdx.x / a.splits;
    const int q0 = tile * a.Qb;
    if (q0 >= n) return;
    const int nq = min(a.Qb, n - q0);
    const int ntok = L - n + q0 + nq;  // tokens the tile's last row sees
    const int nc = (ntok + kChunk - 1) / kChunk;
    const int nb = (ntok + BS - 1) / BS;
    const int32_t* table = a.tables + static_cast<size_t>(b) * a.max_blocks;
    // This block's chunks: c_beg .. c_beg + nk - 1, its split of the key range.
    // Pipeline stages, score buffers, barrier phases and the softmax groups
    // count k = c - c_beg; pages and the causal mask use the chunk index c.
    const int per = (nc + a.splits - 1) / a.splits;
    const int c_beg = min(nc, split * per);
    const int nk = min(nc, c_beg + per) - c_beg;
    const bool partial = a.splits > 1;
    const size_t pidx = ((static_cast<size_t>(b) * a.Hkv + h) * a.tiles + tile) * a.splits + split;
    float* part_o = partial ? a.part + pidx * kRows * kD : nullptr;
    float* part_ml = partial ? a.part + static_cast<size_t>(a.num_parts) * kRows * kD + pidx * kRows * 2
                             : nullptr;
    if (nk == 0) {  // a split past a short sequence's end: an empty partial
        if (tid < kRows) {
            part_ml[2 * tid] = -INFINITY;
            part_ml[2 * tid + 1] = 0.f;
        }
        return;
    }

    // This thread's query row (softmax warps): group G (warps 0-7 take the
    // even chunks, warps 8-15 the odd ones), row r of the tile, and which
    // half of the row's 128 columns it holds. The 8 warps of a group cover
    // the tile's 128 tensor-memory lanes in 16-lane groups, each warp within
    // its lane quarter (32 * (warp % 4) + 0 or 16); threads i and i + 16 of
    // a warp share a row.
    const int grp = (tid / kGroupThreads) & 1;
    const int quarter = warp & 3, sub16 = (warp >> 2) & 1, half = lane >> 4;
    const int row = 32 * quarter + 16 * sub16 + (lane & 15);
    const bool softmax = tid < kSoftmaxThreads;
    const int qi = row / a.g, qj = row - qi * a.g;
    const bool row_valid = softmax && qi < nq;
    const size_t out_row = (static_cast<size_t>(qs) + q0 + qi) * a.Hq + h * a.g + qj;

    // The block's barriers, set up before the table check so that the copy
    // warps can start as soon as it has passed.
    if (tid == 0) {
        for (int s = 0; s < kStagesK; ++s) {
            mbar_init(bars + kBarKFull + 8 * s, 1);
            mbar_init(bars + kBarKEmpty + 8 * s, 1);
        }
        for (int s = 0; s < kStagesV; ++s) {
            mbar_init(bars + kBarVFull + 8 * s, 1);
            mbar_init(bars + kBarVEmpty + 8 * s, 1);
        }
        for (int j = 0; j < kSbuf; ++j) {
            mbar_init(bars + kBarS + 8 * j, 1);
            mbar_init(bars + kBarP + 8 * j, kGroupThreads);
            mbar_init(bars + kBarPV + 8 * j, 1);
        }
        for (int j = 0; j < 2; ++j) mbar_init(bars + kBarM + 8 * j, kGroupThreads);
        mbar_init(bars + kBarO, 1);
        mbar_init(bars + kBarDrain, 1);
        mbar_init(bars + kBarProbe, 1);
        mbar_init(bars + kBarQ, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    // The table entries this block reads, validated once.
    bool bad = false;
    for (int i = tid; i < nb; i += kThreads) {
        const int p = table[i];
        bad |= p < 0 || p >= a.num_blocks;
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0) atomicOr(a.err, kErrTable);
        if (row_valid && grp == 0) {
            float z[kD / 2] = {};
            write_row<kD / 2>(a, out_row, z, 0.f, 64 * half);
        }
        if (partial && tid < kRows) part_ml[2 * tid] = NAN;  // the merge writes zeros too
        return;
    }
    // The copy warps go straight to work. The softmax warps and the MMA warp
    // meet on a named barrier of their own once the tensor memory is
    // allocated.
    uint32_t tmem = 0;
    if (warp != kWarpLoad && warp != kWarpLoadV) {
        if (warp == kWarpMma) {
            tc::alloc(bars + kSlotTmem, kTmemCols);
            tc::relinquish();
        }
        tc::fence_before_sync();
        asm volatile("bar.sync 1, %0;" ::"n"(kSoftmaxThreads + 32) : "memory");
        tc::fence_after_sync();
        tmem = *reinterpret_cast<volatile uint32_t*>(gbase + kOffBar + kSlotTmem);
    }

    if (warp == kWarpLoad || warp == kWarpLoadV) {
        // ------------------------------------------------------------ producers (K, V)
        if (lane == 0) {
            const bool is_k = warp == kWarpLoad;
            const int nst = is_k ? kStagesK : kStagesV;
            const uint32_t full = bars + (is_k ? kBarKFull : kBarVFull);
            const uint32_t empty = bars + (is_k ? kBarKEmpty : kBarVEmpty);
            const uint32_t ring = base + (is_k ? kOffK : kOffV);
            const CUtensorMap* map = is_k ? &kmap : &vmap;
            const uint64_t policy = policy_evict_first();
            if (is_k) {
                // The query tile, in the swizzled K-major layout of the score
                // products' A operand: one box per 64-column half, rows in
                // (query, head) order. Rows past the tile's queries hold other
                // rows of q or zeros; the softmax masks them by predicate.
                mbar_arrive_expect_tx(bars + kBarQ, kTileQ);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
                    tma_load_3d(base + kOffQ + hf * 16384, &qmap, hf * 64, h * a.g, qs + q0, bars + kBarQ,
                                policy);
            }
            // The table entries of a chunk are loaded one chunk ahead, so
            // that their latency overlaps the wait for a free stage instead
            // of preceding every page's copy.
            constexpr int kPages = kChunk / BS;
            int pg[kPages];
            auto load_pages = [&](int c) {
#pragma unroll
                for (int j = 0; j < kPages; ++j) {
                    const int p = c * kPages + j;
                    pg[j] = p < nb ? table[p] : 0;
                }
            };
            load_pages(c_beg);
            int issued = 0;
            for (int k = 0; k < nk; ++k) {
                const int c = c_beg + k;
                const int s = k % nst;
                if (k >= nst && !wait_role(empty + 8 * s, ((k / nst) - 1) & 1, abort_flag, a.err)) break;
                // One chunk (its pages, both 64-column halves) into the stage.
                const int np = min(kPages, nb - c * kPages);
                const uint32_t bar = full + 8 * s, stage = ring + s * kStageKV;
                mbar_arrive_expect_tx(bar, static_cast<uint32_t>(np) * BS * kD * 2);
#pragma unroll
                for (int j = 0; j < kPages; ++j) {
                    if (j < np) {
                        const int r = pg[j] * a.Hkv + h;
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf)
                            tma_load_3d(stage + hf * kHalfKV + j * BS * 128, map, hf * 64, 0, r, bar, policy);
                    }
                }
                issued = k + 1;
                load_pages(c + 1);
            }
            // Copies still in flight land before the block leaves: the last
            // chunk issued on each stage (its phase is then final; earlier
            // chunks of a stage were consumed before it was reissued). Without
            // an abort the consumers have waited for them already.
            for (int k = max(0, issued - nst); k < issued; ++k)
                mbar_wait_bounded(full + 8 * (k % nst), (k / nst) & 1, kWaitLimitNs);
            if (is_k) mbar_wait_bounded(bars + kBarQ, 0, kWaitLimitNs);  // the query tile too
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            // Descriptor low words of every shared-memory operand, built once;
            // all share the high word (SBO = 1024, 128-byte swizzle).
            const uint32_t hi = static_cast<uint32_t>(tc::smem_desc(base, 16, 1024) >> 32);
            const uint32_t lo_q = tc::desc_lo(base + kOffQ, 16);
            const uint32_t lo_k = tc::desc_lo(base + kOffK, 16);
            const uint32_t lo_v = tc::desc_lo(base + kOffV, kHalfKV);
            // (The MMA thread counts the block's own chunks, 0 .. nk - 1.)
            // S(c) = Q K(c)^T into score buffer c % kSbuf; its completion frees
            // the K stage.
            auto issue_s = [&](int c) {
                const uint32_t b0 = lo_k + (c % kStagesK) * (kStageKV >> 4);
                const uint32_t d = tmem + col_s(c % kSbuf);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t da = (kk >> 2) * (16384 >> 4) + (kk & 3) * 2;
                    const uint32_t db = (kk >> 2) * (kHalfKV >> 4) + (kk & 3) * 2;
                    tc::mma_bf16_lo(d, lo_q + da, b0 + db, hi, kIdescS, kk > 0);
                }
                tc::commit(bars + kBarS + 8 * (c % kSbuf));
                tc::commit(bars + kBarKEmpty + 8 * (c % kStagesK));
            };
            // O (+)= P(c) V(c), P read from the chunk's score buffer; its
            // completion frees the V stage.
            auto issue_pv = [&](int c) {
                const uint32_t b0 = lo_v + (c % kStagesV) * (kStageKV >> 4);
                const uint32_t pa = tmem + col_s(c % kSbuf);
#pragma unroll
                for (int kk = 0; kk < kChunk / 16; ++kk)   // 16 tokens = 8 columns of P
                    tc::mma_bf16_ts(tmem + kColO, pa + kk * 8, b0 + kk * (2048 >> 4), hi, kIdescO,
                                    c > 0 || kk > 0);
                tc::commit(bars + kBarVEmpty + 8 * (c % kStagesV));
                tc::commit(bars + kBarPV + 8 * (c % kSbuf));
            };
            bool ok;
            if (a.probe_wait) {
                // The wait-expiry probe: a bounded wait on a barrier nothing
                // completes, then the abort every other role follows.
                mbar_wait_bounded(bars + kBarProbe, 0, kProbeLimitNs);
                *abort_flag = 1;
                atomicOr(a.err, kErrTimeout);
                ok = false;
            } else {
                ok = wait_role(bars + kBarQ, 0, abort_flag, a.err);
            }
            // The first score products, as their K chunks land.
            for (int c = 0; c < min(kSbuf, nk) && ok; ++c) {
                ok = wait_role(bars + kBarKFull + 8 * (c % kStagesK), (c / kStagesK) & 1, abort_flag, a.err);
                if (!ok) break;
                tc::fence_after_sync();
                issue_s(c);
            }
            // Then per chunk: its value product once P(c) is stored, and the
            // score product kSbuf chunks ahead into the buffer P(c) leaves.
            // One thread's products run in issue order, so S(c + kSbuf)
            // overwrites P(c) only after PV(c) has read it.
            for (int c = 0; c < nk && ok; ++c) {
                ok = wait_role(bars + kBarP + 8 * (c % kSbuf), (c / kSbuf) & 1, abort_flag, a.err) &&
                     wait_role(bars + kBarVFull + 8 * (c % kStagesV), (c / kStagesV) & 1, abort_flag, a.err);
                if (!ok) break;
                tc::fence_after_sync();
                issue_pv(c);
                const int c3 = c + kSbuf;
                if (c3 < nk) {
                    ok = wait_role(bars + kBarKFull + 8 * (c3 % kStagesK), (c3 / kStagesK) & 1, abort_flag,
                                   a.err);
                    if (!ok) break;
                    tc::fence_after_sync();
                    issue_s(c3);
                }
            }
            if (ok) tc::commit(bars + kBarO);
            if (*abort_flag) {
                tc::commit(bars + kBarDrain);
                mbar_wait_bounded(bars + kBarDrain, 0, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax (group grp)
        // Group grp takes the chunks c = grp, grp + 2, ... Two threads per
        // row: thread half hf holds the row's scores of tokens 64hf .. 64hf +
        // 63 of each chunk and writes their probabilities to P columns 32hf ..
        // 32hf + 31 of the chunk's score buffer; the row maximum is joined
        // with the partner thread (lane ^ 16). The reference max of chunk c
        // is published in shared memory for the group that takes chunk c + 1.
        const uint32_t lane_base = static_cast<uint32_t>(32 * quarter + 16 * sub16) << 16;
        const uint32_t o_addr = tmem + lane_base + kColO;
        const int pos_r = L - n + q0 + qi;  // last token this row sees
        float* mpub = reinterpret_cast<float*>(gbase + kOffM);
        float m_l = -INFINITY, l = 0.f;  // this thread's part of the row sum, in units of 2^m_l
        bool ok = true;
        for (int k = grp; k < nk; k += 2) {
            const int c = c_beg + k;  // the chunk of the sequence (k: of this block)
            const int j = k % kSbuf;
            const uint32_t s_addr = tmem + lane_base + col_s(j);
            ok = __all_sync(0xffffffffu, wait_role(bars + kBarS + 8 * j, (k / kSbuf) & 1, abort_flag, a.err));
            if (!ok) break;
            tc::fence_after_sync();
            float sv[kChunk / 2];
            tc::ld16x2_32<64>(s_addr, *reinterpret_cast<float(*)[32]>(sv));
            tc::ld16x2_32<64>(s_addr + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
            tc::wait_ld();
            // Causal mask by predicate; the warp skips it when no row needs it.
            const int tok0 = c * kChunk + 64 * half;
            if (!__all_sync(0xffffffffu, row_valid && c * kChunk + kChunk - 1 <= pos_r)) {
#pragma unroll
                for (int i = 0; i < kChunk / 2; ++i)
                    sv[i] = (row_valid && tok0 + i <= pos_r) ? sv[i] : -INFINITY;
            }
            // Row max: three-input max over pairs, four short chains, then the
            // partner's half.
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < kChunk / 4; ++i) mq[i & 3] = max3(mq[i & 3], sv[2 * i], sv[2 * i + 1]);
            float mx = max3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            mx *= a.scale_log2;  // scale > 0, so this is the max of the scaled scores
            // The reference max of chunk c - 1, from the other group; raise it
            // only when this chunk exceeds it by > 2^8.
            float mprev = -INFINITY;
            if (k > 0) {
                ok = __all_sync(0xffffffffu, wait_role(bars + kBarM + 8 * ((k - 1) & 1), ((k - 1) >> 1) & 1,
                                                       abort_flag, a.err));
                if (!ok) break;
                mprev = mpub[((k - 1) & 1) * kRows + row];
            }
            const float mc = mx > mprev + kRescaleLog2 ? mx : mprev;
            if (half == 0) mpub[(k & 1) * kRows + row] = mc;
            mbar_arrive(bars + kBarM + 8 * (k & 1));
            if (mc != m_l) {
                l = l > 0.f ? l * fast_exp2(m_l - mc) : 0.f;
                m_l = mc;
            }
            const float m_use = mc == -INFINITY ? 0.f : mc;
            // P = 2^(s * scale - m) (bf16 pairs) over P columns 32hf .. 32hf + 31
            // of this row; the arguments and the partial row sum two at a time.
            const uint64_t sc2 = f32x2(a.scale_log2, a.scale_log2), nm2 = f32x2(-m_use, -m_use);
            uint64_t ps2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t pw[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float2 x = f32x2_split(
                        fma_f32x2(f32x2(sv[32 * h2 + 2 * i], sv[32 * h2 + 2 * i + 1]), sc2, nm2));
                    const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
                    ps2[i & 1] = add_f32x2(ps2[i & 1], f32x2(p0, p1));
                    pw[i] = pack_bf16x2(p0, p1);
                }
                tc::st16x2_16u<32>(s_addr + 16 * h2, pw);
            }
            {
                const float2 s0 = f32x2_split(ps2[0]), s1 = f32x2_split(ps2[1]);
                l += (s0.x + s0.y) + (s1.x + s1.y);
            }
            // O holds the products of chunks < c in units of 2^mprev: rescale
            // this row's half once PV(c - 1) is done (PV(c) waits for this P).
            // The parity wait is unambiguous: the barrier of buffer (c-1) % 3
            // last completed for PV(c - 4), which was done before S(c - 1)
            // (issued after it) was, and this group has seen chunk c - 1's max.
            if (k > 0 && __any_sync(0xffffffffu, mc != mprev)) {
                const int jp = (k - 1) % kSbuf;
                ok = __all_sync(0xffffffffu, wait_role(bars + kBarPV + 8 * jp, ((k - 1) / kSbuf) & 1,
                                                       abort_flag, a.err));
                if (!ok) break;
                tc::fence_after_sync();
                const float alpha = mc != mprev ? fast_exp2(mprev - mc) : 1.f;
#pragma unroll
                for (int piece = 0; piece < 2; ++piece) {
                    float o[32];
                    tc::ld16x2_32<64>(o_addr + 32 * piece, o);
                    tc::wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tc::st16x2_32<64>(o_addr + 32 * piece, o);
                }
            }
            // Final chunk: zero the V rows past the last token before its
            // value product. The stage's previous chunk (c - 3) was consumed by
            // PV(c - 3), issued before S(c), so this parity wait is unambiguous.
            if (c == nc - 1) {
                const int valid = ntok - c * kChunk;
                ok = __all_sync(0xffffffffu, wait_role(bars + kBarVFull + 8 * (k % kStagesV),
                                                       (k / kStagesV) & 1, abort_flag, a.err));
                if (!ok) break;
                if (valid < kChunk) {
                    const uint32_t vst = base + kOffV + (k % kStagesV) * kStageKV;
                    for (int idx = tid % kGroupThreads; idx < (kChunk - valid) * 16; idx += kGroupThreads) {
                        const int r = valid + (idx >> 4), hf = (idx >> 3) & 1, ch = idx & 7;
                        st_shared_v4(vst + hf * kHalfKV + r * 128 + ch * 16, make_uint4(0, 0, 0, 0));
                    }
                }
                fence_proxy_async_smem();
            }
            tc::wait_st();
            tc::fence_before_sync();
            mbar_arrive(bars + kBarP + 8 * j);
        }
        // Epilogue. The final reference max is the block's last chunk's; both
        // groups bring their row sums to it and add them through shared memory
        // (the area of the published max, reused after a barrier of both
        // groups).
        bool fine = ok && __all_sync(0xffffffffu, wait_role(bars + kBarM + 8 * ((nk - 1) & 1),
                                                             ((nk - 1) >> 1) & 1, abort_flag, a.err));
        const float mfin = fine ? mpub[((nk - 1) & 1) * kRows + row] : 0.f;
        if (fine && mfin != m_l) l = l > 0.f ? l * fast_exp2(m_l - mfin) : 0.f;
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        asm volatile("bar.sync 2, %0;" ::"n"(kSoftmaxThreads) : "memory");
        float* lsum = reinterpret_cast<float*>(gbase + kOffL);
        if (half == 0) lsum[grp * kRows + row] = l;
        asm volatile("bar.sync 2, %0;" ::"n"(kSoftmaxThreads) : "memory");
        const float lt = l + lsum[(grp ^ 1) * kRows + row];
        fine = fine && !*abort_flag;
        if (fine) {
            fine = __all_sync(0xffffffffu, wait_role(bars + kBarO, 0, abort_flag, a.err));
            if (fine) {
                // Each group takes 32 of the row's 64 columns per thread half:
                // columns 64hf + 32grp .. + 31. Without a split it normalises
                // and writes them; with one it stores them unnormalised in the
                // block's partial, with the row's (reference max, row sum).
                tc::fence_after_sync();
                float o[32];
                tc::ld16x2_32<64>(o_addr + 32 * grp, o);
                tc::wait_ld();
                if (!partial) {
                    const float inv = (row_valid && lt > 0.f) ? 1.f / lt : 0.f;
                    if (row_valid) write_row<32>(a, out_row, o, inv, 64 * half + 32 * grp);
                } else if (row_valid) {
                    float* dst = part_o + static_cast<size_t>(row) * kD + 64 * half + 32 * grp;
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(dst + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
                    if (grp == 0 && half == 0) {
                        part_ml[2 * row] = mfin;
                        part_ml[2 * row + 1] = lt;
                    }
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        tc::fence_after_sync();
        tc::dealloc(tmem, kTmemCols);
    }
}

// Combines the partials of a split call: one warp per output row (query,
// head), lane l on columns 4l .. 4l + 3. The two-partial rule of
// "39 · PagedAttention" §3 over the splits: m = max_s m_s, l = sum_s l_s
// 2^(m_s - m), o = sum_s O_s 2^(m_s - m) / l (maxima in the log2 domain); a
// split with m_s = -inf saw no token of the row and is skipped, a NaN m_s
// (a bad table entry) makes the row zeros. Rows of invalid sequences get
// zeros (only multi-query calls split).
struct SplitMergeArgs {
    const float* part;
    int num_parts;
    const int32_t* q_start;
    const int32_t* seq_lens;
    void* out;
    int out_bf16;
    int B, Hq, Hkv, g, Qb, tiles, splits, num_q, limit, max_q;
};

__global__ void __launch_bounds__(256) prefill_split_merge_kernel(const SplitMergeArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t R = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (R >= static_cast<int64_t>(a.num_q) * a.Hq) return;
    const int t = static_cast<int>(R / a.Hq), hq = static_cast<int>(R - static_cast<int64_t>(t) * a.Hq);
    int lo = 0, hi = a.B - 1;  // the sequence whose query rows hold t
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.q_start[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const size_t o0 = static_cast<size_t>(R) * kD + 4 * lane;
    const int64_t qs64 = a.q_start[b], n64 = static_cast<int64_t>(a.q_start[b + 1]) - qs64;
    const int L = a.seq_lens[b];
    if (n64 < 1 || n64 > a.max_q || L < n64 || L > a.limit || qs64 < 0 || qs64 + n64 > a.num_q ||
        t < qs64 || t >= qs64 + n64) {
        // An invalid sequence (the split blocks wrote no partial for it): zeros.
        if (a.out_bf16) *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + o0) = make_uint2(0, 0);
        else *reinterpret_cast<float4*>(static_cast<float*>(a.out) + o0) = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    const int qs = static_cast<int>(qs64);
    const int i = t - qs, tile = i / a.Qb;  // i < min(max_q, num_q): tile < tiles
    const int h = hq / a.g, r = (i - tile * a.Qb) * a.g + (hq - h * a.g);
    const size_t p0 = ((static_cast<size_t>(b) * a.Hkv + h) * a.tiles + tile) * a.splits;
    const float* ml = a.part + static_cast<size_t>(a.num_parts) * kRows * kD;
    float M = -INFINITY;
    bool poison = false;
    for (int sp = 0; sp < a.splits; ++sp) {
        const float m = ml[((p0 + sp) * kRows + r) * 2];
        poison |= m != m;
        M = fmaxf(M, m);
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float lsum = 0.f;
    if (!poison && M != -INFINITY) {
        for (int sp = 0; sp < a.splits; ++sp) {
            const size_t pr = (p0 + sp) * kRows + r;
            const float m = ml[pr * 2];
            if (m == -INFINITY) continue;
            const float w = fast_exp2(m - M);
            lsum = fmaf(ml[pr * 2 + 1], w, lsum);
            const float4 o = *reinterpret_cast<const float4*>(a.part + pr * kD + 4 * lane);
            acc[0] = fmaf(o.x, w, acc[0]);
            acc[1] = fmaf(o.y, w, acc[1]);
            acc[2] = fmaf(o.z, w, acc[2]);
            acc[3] = fmaf(o.w, w, acc[3]);
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    if (a.out_bf16) {
        uint2 w;
        w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + o0) = w;
    } else {
        *reinterpret_cast<float4*>(static_cast<float*>(a.out) + o0) =
            make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    }
}

}  // namespace

int prefill_split_count(int B, int Hq, int Hkv, int64_t nq, int max_seq_len, int num_sms) {
    // A small call (fewer tile blocks than SMs) splits every tile's key range
    // into as many pieces as fill the SMs once, each of at least two chunks.
    const int qb = kRows / (Hq / Hkv);
    const int64_t tiles = (nq + qb - 1) / qb;
    const int64_t blocks = tiles * Hkv * B;
    if (blocks <= 0 || blocks >= num_sms) return 1;
    const int64_t chunks = (static_cast<int64_t>(max_seq_len) + kChunk - 1) / kChunk;
    const int64_t s = std::min<int64_t>({num_sms / blocks, chunks / 2, 32});
    return static_cast<int>(std::max<int64_t>(1, s));
}

size_t prefill_split_bytes(int B, int Hq, int Hkv, int64_t nq, int splits) {
    const int qb = kRows / (Hq / Hkv);
    const int64_t tiles = (nq + qb - 1) / qb;
    const size_t parts = static_cast<size_t>(tiles) * Hkv * B * splits;
    return parts * kRows * (kD + 2) * sizeof(float);
}

cudaError_t launch_prefill_one_tile(const CUtensorMap& kmap, const CUtensorMap& vmap, const void* q,
                                    int num_q, const int32_t* q_start, const int32_t* tables,
                                    const int32_t* seq_lens, void* out, int* err, int B, int Hq,
                                    int Hkv, int max_blocks, int num_blocks, int max_seq_len,
                                    int max_q, float scale_log2, int out_bf16, int block_size,
                                    cudaStream_t stream, float* part, int splits,
                                    int zero_invalid) {
    PrefillArgs a{};
    a.q = static_cast<const uint16_t*>(q);
    a.q_start = q_start;
    a.tables = tables;
    a.seq_lens = seq_lens;
    a.out = out;
    a.err = err;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.g = Hq / Hkv;
    a.Qb = kRows / a.g;
    a.num_q = num_q;
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    a.max_seq_len = max_seq_len;
    a.scale_log2 = scale_log2;
    a.out_bf16 = out_bf16;
    a.probe_wait = wait_probe();
    a.max_q = max_q;
    a.zero_invalid = zero_invalid;
    if (B > kMaxGridYZ || Hkv > kMaxGridYZ) return cudaErrorInvalidValue;  // checked by the callers
    // No sequence has more queries than the call has rows.
    const int64_t nq = std::min<int64_t>(max_q, num_q);
    if (splits < 1 || (splits > 1 && !part)) return cudaErrorInvalidValue;
    const int64_t tiles = (nq + a.Qb - 1) / a.Qb;
    a.splits = splits;
    a.tiles = static_cast<int>(tiles);
    a.num_parts = static_cast<int>(tiles * Hkv * B * splits);
    a.part = splits > 1 ? part : nullptr;
    dim3 grid(static_cast<unsigned>(tiles * splits), Hkv, B);
    CUtensorMap qmap;
    if (!encode_query_map(&qmap, q, num_q, Hq, a.g, a.Qb)) return cudaErrorInvalidValue;
    auto kern = block_size == 16 ? prefill_one_tile_kernel<16> : prefill_one_tile_kernel<32>;
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, kSmemBytes, stream>>>(kmap, vmap, qmap, a);
    e = cudaGetLastError();
    if (e != cudaSuccess || splits == 1) return e;
    SplitMergeArgs m{part, a.num_parts, q_start, seq_lens, out, out_bf16, B, Hq, Hkv, a.g, a.Qb,
                     a.tiles, splits, num_q, std::min(max_seq_len, max_blocks * block_size), max_q};
    const int64_t rows = static_cast<int64_t>(num_q) * Hq;
    prefill_split_merge_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(m);
    return cudaGetLastError();
}

}  // namespace pa
