// Paged multi-query attention (chunked prefill, speculative verification) on
// the tcgen05 tensor cores.
//
// The newest n_b tokens of sequence b are queries at once; query i at position
// pos = L_b - n_b + i attends causally to tokens t <= pos read through the
// block table ("FlashAttention vs PagedAttention", "How prefill and decode
// change the diagnosis"; exact attention as in "39 · PagedAttention" §1-§2).
// Here the query side is a real dense contraction: a query tile holds 128
// rows = (128 / g) queries x the g query heads of one kv head, so every K/V
// chunk is read once for all of them.
//
// One block = two query tiles of the same (sequence, kv head) that share the
// K/V stream, with specialised warps:
//   * warps 16 and 18 (producers): tiled bulk tensor copies of 128-token K
//     and V chunks (whole pages, through the block table) into a 2-stage K
//     ring and a 3-stage V ring, each stream on its own warp so that a wait
//     for a free V stage never holds back the next K; the K warp first
//     copies the block's query tiles (a tensor map over q whose box is one
//     64-column half of a tile, rows in (query, head) order, landing in the
//     swizzled K-major layout the score products read), so that the
//     prologue holds no query rows in registers and the first chunk is on
//     its way as soon as the table check has passed;
//   * warp 17 (MMA): one thread issues S_t = Q_t K^T (M=128, N=128, K=128,
//     both operands in shared memory) into tensor memory and
//     O_t += P_t V (M=128, N=128, K=128) with P_t read from tensor memory and
//     V read MN-major straight from the page layout, for both tiles t, and
//     signals completion through tcgen05.commit on mbarriers;
//   * warps 0-7 / 8-15 (softmax, two warpgroups per tile, two threads per
//     row, each on 64 of the row's 128 scores, tensor memory read in the
//     16-lane 16x32bx2 shape so that the partner threads sit in one warp):
//     load the scores from tensor memory, scale (log2 domain), mask causally
//     by predicate, join the row maximum with the partner (one shuffle), run
//     the online softmax and store the bf16 probabilities P_t over the first
//     64 columns of the same scores (the A operand of the PV product); at the
//     end, read the row of O_t and normalise it. A full tile with bf16
//     output is staged in the tile's query buffer (the same swizzled box
//     layout the query copy used) and leaves by two tiled bulk tensor
//     stores; a partial tile or float output is stored by the threads.
// The MMA thread issues PV_0(c), S_0(c+1), PV_1(c), S_1(c+1), ...: one
// thread's products run in issue order, so S_t(c+1) overwrites P_t(c) only
// after PV_t(c) has read it, and its completion (one commit covers every
// earlier product) also tells the softmax that PV_t(c) is done. While one
// warpgroup exponentiates, the tensor core works on the other tile, so the
// two tiles take turns. Keeping P out of shared memory leaves the shared
// memory bandwidth to the S operands, V and the incoming copies.
// The running maximum is raised only when a chunk's maximum exceeds it by
// more than 2^8 (any fixed reference gives the same quotient acc / l; this
// one keeps every probability below 256): the accumulator rows in tensor
// memory are then rescaled, otherwise left.
// V rows past the last token of the final chunk are zeroed before the
// product so that slots beyond the sequence never reach a sum. Blocks are
// ordered longest sequence first so that the long ones do not form the tail.
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

constexpr int kRows = 128;      // M: query rows per tile
constexpr int kChunk = 128;     // tokens per K/V chunk
constexpr int kD = 128;         // head dimension
constexpr int kStagesK = 2;     // K ring depth
constexpr int kStagesV = 3;     // V ring depth (PV waits on V last)
constexpr int kTileThreads = 2 * kRows;            // softmax threads of a tile: two per row
constexpr int kSoftmaxThreads = 2 * kTileThreads;   // two tiles
constexpr int kWarpLoad = kSoftmaxThreads / 32;     // warp 16: K copies
constexpr int kWarpMma = kWarpLoad + 1;             // warp 17
constexpr int kWarpLoadV = kWarpMma + 1;            // warp 18: V copies
constexpr int kThreads = kSoftmaxThreads + 96;
constexpr int kSortMax = 256;   // sequences ordered by length up to this batch size
constexpr uint32_t kTmemCols = 512;
// Tensor-memory columns: S of tile t (128; P_t over its first 64), then O of tile t (128).
__host__ __device__ constexpr uint32_t col_s(int t) { return 128u * t; }
__host__ __device__ constexpr uint32_t col_o(int t) { return 256u + 128u * t; }
constexpr float kRescaleLog2 = 8.f;  // raise the reference max only beyond 2^8

// Shared-memory layout (byte offsets from a 1024-aligned base).
constexpr uint32_t kTileQ = 32768;                    // 2 halves x 128 rows x 128 B
constexpr uint32_t kHalfKV = kChunk * 128;            // one 64-column half of a chunk
constexpr uint32_t kStageKV = 2 * kHalfKV;            // 2 halves x 128 rows x 128 B
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + 2 * kTileQ;
constexpr uint32_t kOffV = kOffK + kStagesK * kStageKV;
constexpr uint32_t kOffBar = kOffV + kStagesV * kStageKV;
// mbarriers (8 bytes each) and slots, at kOffBar + ...
constexpr uint32_t kBarKFull = 0;                     // [kStagesK]
constexpr uint32_t kBarKEmpty = kBarKFull + 8 * kStagesK;
constexpr uint32_t kBarVFull = kBarKEmpty + 8 * kStagesK;  // [kStagesV]
constexpr uint32_t kBarVEmpty = kBarVFull + 8 * kStagesV;
constexpr uint32_t kBarS = kBarVEmpty + 8 * kStagesV; // [tile]
constexpr uint32_t kBarP = kBarS + 16;                // [tile], 128 arrivals each
constexpr uint32_t kBarO = kBarP + 16;                // [tile]
constexpr uint32_t kBarDrain = kBarO + 16;
constexpr uint32_t kSlotTmem = kBarDrain + 8;
constexpr uint32_t kSlotAbort = kSlotTmem + 4;
constexpr uint32_t kSlotSeq = kSlotAbort + 4;
constexpr uint32_t kBarProbe = kSlotSeq + 8;          // nothing completes it (wait-expiry probe)
constexpr uint32_t kBarQ = kBarProbe + 8;             // the block's query tiles have landed
constexpr uint32_t kOffLens = kOffBar + 256;          // [kSortMax] lengths, for the ordering
constexpr uint32_t kSmemBytes = 1024 + kOffLens + 4 * kSortMax;
static_assert(kBarQ % 8 == 0 && kBarQ + 8 <= kOffLens - kOffBar,
              "barrier area overlaps the length array");
static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0, "swizzle atoms");
static_assert(kSmemBytes <= 227 * 1024 && 2 * kSmemBytes > 228 * 1024,
              "one block per SM: it holds all 512 tensor-memory columns");

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kRows, kChunk, false, false);
constexpr uint32_t kIdescO = tc::idesc_bf16_f32(kRows, kD, false, true);  // A from tensor memory

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
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Named barrier over `count` threads that also returns the AND of `pred`
// over them.
__device__ __forceinline__ bool bar_red_and(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Tiled tensor copy shared -> global (3-D box), tracked as a bulk async group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(src)
                 : "memory");
}

// Close the bulk group and wait until its copies have read shared memory.
__device__ __forceinline__ void bulk_commit_and_wait_read() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
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

template <int BS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                   const PrefillArgs a) {
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
    const int q0 = blockIdx.x * 2 * a.Qb;
    if (q0 >= n) return;
    const int nq0 = min(a.Qb, n - q0);
    const int nq1 = max(0, min(a.Qb, n - q0 - a.Qb));
    const bool two = nq1 > 0;
    const int ntok = L - n + q0 + (two ? a.Qb + nq1 : nq0);  // tokens the last row sees
    const int nc = (ntok + kChunk - 1) / kChunk;
    const int nb = (ntok + BS - 1) / BS;
    const int32_t* table = a.tables + static_cast<size_t>(b) * a.max_blocks;

    // This thread's query row (softmax warps): tile t, row r of the tile, and
    // which half of the row's 128 columns it holds. The 8 warps of a tile
    // cover the tile's 128 tensor-memory lanes in 16-lane groups, each warp
    // within its lane quarter (32 * (warp % 4) + 0 or 16); threads i and
    // i + 16 of a warp share a row.
    const int t = tid / kTileThreads;
    const int quarter = warp & 3, sub16 = (warp >> 2) & 1, half = lane >> 4;
    const int row = 32 * quarter + 16 * sub16 + (lane & 15);
    const bool softmax = tid < kSoftmaxThreads;
    const int qi = row / a.g, qj = row - qi * a.g;
    const bool row_valid = softmax && qi < (t == 0 ? nq0 : nq1);
    const size_t out_row = (static_cast<size_t>(qs) + q0 + t * a.Qb + qi) * a.Hq + h * a.g + qj;

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
        for (int u = 0; u < 2; ++u) {
            mbar_init(bars + kBarS + 8 * u, 1);
            mbar_init(bars + kBarP + 8 * u, kTileThreads);
            mbar_init(bars + kBarO + 8 * u, 1);
        }
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
        if (row_valid) {
            float z[kD / 2] = {};
            write_row<kD / 2>(a, out_row, z, 0.f, 64 * half);
        }
        return;
    }
    // The copy warps go straight to work (the query tiles arrive by tiled
    // bulk copies with the first chunk, see below). The softmax warps and the
    // MMA warp meet on a named barrier of their own once the tensor memory
    // is allocated.
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
                // The query tiles, in the swizzled K-major layout of the score
                // products' A operand: one box per 64-column half, rows in
                // (query, head) order. Rows past the tile's queries hold other
                // rows of q or zeros; the softmax masks them by predicate.
                mbar_arrive_expect_tx(bars + kBarQ, (two ? 2u : 1u) * kTileQ);
                for (int u = 0; u < (two ? 2 : 1); ++u)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf)
                        tma_load_3d(base + kOffQ + u * kTileQ + hf * 16384, &qmap, hf * 64, h * a.g,
                                    qs + q0 + u * a.Qb, bars + kBarQ, policy);
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
            load_pages(0);
            int issued = 0;
            for (int c = 0; c < nc; ++c) {
                const int s = c % nst;
                if (c >= nst && !wait_role(empty + 8 * s, ((c / nst) - 1) & 1, abort_flag, a.err)) break;
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
                issued = c + 1;
                load_pages(c + 1);
            }
            // Copies still in flight land before the block leaves: the last
            // chunk issued on each stage (its phase is then final; earlier
            // chunks of a stage were consumed before it was reissued). Without
            // an abort the consumers have waited for them already.
            for (int c = max(0, issued - nst); c < issued; ++c)
                mbar_wait_bounded(full + 8 * (c % nst), (c / nst) & 1, kWaitLimitNs);
            if (is_k) mbar_wait_bounded(bars + kBarQ, 0, kWaitLimitNs);  // the query tiles too
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
            auto issue_s = [&](int u, int c) {
                const uint32_t a0 = lo_q + u * (kTileQ >> 4);
                const uint32_t b0 = lo_k + (c % kStagesK) * (kStageKV >> 4);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t da = (kk >> 2) * (16384 >> 4) + (kk & 3) * 2;
                    const uint32_t db = (kk >> 2) * (kHalfKV >> 4) + (kk & 3) * 2;
                    tc::mma_bf16_lo(tmem + col_s(u), a0 + da, b0 + db, hi, kIdescS, kk > 0);
                }
                tc::commit(bars + kBarS + 8 * u);
            };
            auto issue_pv = [&](int u, int c) {
                const uint32_t b0 = lo_v + (c % kStagesV) * (kStageKV >> 4);
#pragma unroll
                for (int kk = 0; kk < kChunk / 16; ++kk)   // 16 tokens = 8 columns of P
                    tc::mma_bf16_ts(tmem + col_o(u), tmem + col_s(u) + kk * 8, b0 + kk * (2048 >> 4), hi,
                                    kIdescO, c > 0 || kk > 0);
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
                ok = wait_role(bars + kBarQ, 0, abort_flag, a.err) &&
                     wait_role(bars + kBarKFull, 0, abort_flag, a.err);
            }
            if (ok) {
                tc::fence_after_sync();
                issue_s(0, 0);
                if (two) issue_s(1, 0);
                tc::commit(bars + kBarKEmpty);  // K stage of chunk 0 free once both S are done
            }
            for (int c = 0; c < nc && ok; ++c) {
                const int c1 = c + 1;
                ok = wait_role(bars + kBarP, c & 1, abort_flag, a.err) &&
                     wait_role(bars + kBarVFull + 8 * (c % kStagesV), (c / kStagesV) & 1, abort_flag, a.err);
                if (!ok) break;
                tc::fence_after_sync();
                issue_pv(0, c);
                if (c1 < nc) {
                    ok = wait_role(bars + kBarKFull + 8 * (c1 % kStagesK), (c1 / kStagesK) & 1,
                                   abort_flag, a.err);
                    if (!ok) break;
                    tc::fence_after_sync();
                    issue_s(0, c1);  // after PV_0(c) in issue order: P_0(c) is read first
                    if (!two) tc::commit(bars + kBarKEmpty + 8 * (c1 % kStagesK));
                }
                if (two) {
                    ok = wait_role(bars + kBarP + 8, c & 1, abort_flag, a.err);
                    if (!ok) break;
                    tc::fence_after_sync();
                    issue_pv(1, c);
                }
                // The V stage of chunk c is free once these products are done.
                tc::commit(bars + kBarVEmpty + 8 * (c % kStagesV));
                if (two && c1 < nc) {
                    issue_s(1, c1);
                    tc::commit(bars + kBarKEmpty + 8 * (c1 % kStagesK));
                }
            }
            if (ok) {
                tc::commit(bars + kBarO);
                if (two) tc::commit(bars + kBarO + 8);
            }
            if (*abort_flag) {
                tc::commit(bars + kBarDrain);
                mbar_wait_bounded(bars + kBarDrain, 0, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else if (t == 0 || two) {
        // ------------------------------------------------------------ softmax (tile t)
        // Two threads per row: thread half h holds the row's scores of tokens
        // 64h .. 64h + 63 of each chunk and writes their probabilities to P
        // columns 32h .. 32h + 31; the row maximum and, at the end, the row
        // sum are joined with the partner thread (lane ^ 16).
        const uint32_t lane_base = static_cast<uint32_t>(32 * quarter + 16 * sub16) << 16;
        const uint32_t s_addr = tmem + lane_base + col_s(t);
        const uint32_t o_addr = tmem + lane_base + col_o(t);
        const int pos_r = L - n + q0 + t * a.Qb + qi;  // last token this row sees
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int c = 0; c < nc; ++c) {
            // S_t(c) done; its commit also covers PV_t(c-1).
            ok = __all_sync(0xffffffffu, wait_role(bars + kBarS + 8 * t, c & 1, abort_flag, a.err));
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
            // Raise the reference max only when the chunk exceeds it by > 2^8.
            float alpha = 1.f;
            if (mx > m + kRescaleLog2) {
                alpha = fast_exp2(m - mx);  // 0 while m is still -inf
                m = mx;
                l *= alpha;
            }
            const float m_use = m == -INFINITY ? 0.f : m;
            // P = 2^(s * scale - m) (bf16 pairs) over P columns 32h .. 32h + 31
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
            // Rescale this row's half of O_t if the reference max moved (PV_t(c-1) is done).
            if (c > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
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
            // Final chunk: tile 0 zeroes the V rows past the last token (both
            // tiles' products run after tile 0 has published its P).
            if (t == 0 && c == nc - 1) {
                const int valid = ntok - c * kChunk;
                // V of this chunk arrives on its own barrier.
                ok = __all_sync(0xffffffffu, wait_role(bars + kBarVFull + 8 * (c % kStagesV),
                                                       (c / kStagesV) & 1, abort_flag, a.err));
                if (!ok) break;
                if (valid < kChunk) {
                    const uint32_t vst = base + kOffV + (c % kStagesV) * kStageKV;
                    for (int idx = tid; idx < (kChunk - valid) * 16; idx += kTileThreads) {
                        const int r = valid + (idx >> 4), hf = (idx >> 3) & 1, ch = idx & 7;
                        st_shared_v4(vst + hf * kHalfKV + r * 128 + ch * 16, make_uint4(0, 0, 0, 0));
                    }
                }
                fence_proxy_async_smem();
            }
            tc::wait_st();
            tc::fence_before_sync();
            mbar_arrive(bars + kBarP + 8 * t);
        }
        // Epilogue. A full tile with bf16 output goes out by tiled bulk
        // tensor copies: each thread normalises its half row of O_t into the
        // tile's query buffer (free once every product is done; a half row
        // is one 128-byte row of a 64-column box, 16-byte chunk c at
        // c ^ (row % 8)), then one thread stores both boxes. A partial tile
        // (a box would cover rows of the next sequence) or float output is
        // written by the threads directly.
        const bool tma_out = a.out_bf16 && (t == 0 ? nq0 : nq1) == a.Qb;
        const uint32_t qbuf = base + kOffQ + t * kTileQ;
        bool fine = ok && __all_sync(0xffffffffu, wait_role(bars + kBarO + 8 * t, 0, abort_flag, a.err));
        if (fine) {
            tc::fence_after_sync();
            if (tma_out) fence_proxy_async_smem();  // the buffer was last used by the copies and products
            const float lt = l + __shfl_xor_sync(0xffffffffu, l, 16);
            const float inv = (row_valid && lt > 0.f) ? 1.f / lt : 0.f;
            const uint32_t srow = qbuf + half * 16384 + row * 128;
#pragma unroll
            for (int piece = 0; piece < 2; ++piece) {
                float o[32];
                tc::ld16x2_32<64>(o_addr + 32 * piece, o);
                tc::wait_ld();
                if (tma_out) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint4 w = make_uint4(pack_bf16x2(o[8 * k] * inv, o[8 * k + 1] * inv),
                                                   pack_bf16x2(o[8 * k + 2] * inv, o[8 * k + 3] * inv),
                                                   pack_bf16x2(o[8 * k + 4] * inv, o[8 * k + 5] * inv),
                                                   pack_bf16x2(o[8 * k + 6] * inv, o[8 * k + 7] * inv));
                        st_shared_v4(srow + (((4 * piece + k) ^ (row & 7)) << 4), w);
                    }
                } else if (row_valid) {
                    write_row<32>(a, out_row, o, inv, 64 * half + 32 * piece);
                }
            }
        }
        if (tma_out) {
            fence_proxy_async_smem();  // this thread's rows, visible to the tensor copy
            // Every thread of the tile meets here; the copy runs only if all
            // of them staged their rows.
            if (bar_red_and(2 + t, kTileThreads, fine) && tid == t * kTileThreads) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
                    tma_store_3d(&omap, qbuf + hf * 16384, hf * 64, h * a.g, qs + q0 + t * a.Qb);
                bulk_commit_and_wait_read();
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

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& kmap, const CUtensorMap& vmap, const void* q,
                           int num_q, const int32_t* q_start, const int32_t* tables,
                           const int32_t* seq_lens, void* out, int* err, int B, int Hq, int Hkv,
                           int max_blocks, int num_blocks, int max_seq_len, int max_q,
                           float scale_log2, int out_bf16, int block_size, cudaStream_t stream,
                           float* part, int splits, int zero_invalid) {
    // The one-tile kernel overlaps a tile's softmax with its own next score
    // products (~2,100 cycles per 128-token chunk and tile); this kernel
    // alternates two tiles (~3,100 cycles per chunk for both), which halves
    // the K/V bytes each SM takes in per row. The one-tile kernel runs when
    // every sequence fits one tile (this kernel's second tile would be
    // empty) or when its grid is at most three waves of blocks, where a
    // block's chunk time, not the SMs' intake, sets the call's time. Prefill
    // workload (16 sequences), us: 33 / 48 / 64 / 96 queries per sequence
    // 117 / 116 / 106 / 131 against 197 / 192 / 150 / 148; 128 queries (four
    // waves) 170 against 150 on this kernel, which then stays.
    {
        const int64_t nq = std::min<int64_t>(max_q, num_q);
        const int qb = kRows / (Hq / Hkv);
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cudaErrorInvalidValue;
        const int64_t blocks1 = (nq + qb - 1) / qb * static_cast<int64_t>(Hkv) * B;
        const int force = prefill_kernel_choice();  // a test may pin either kernel
        if (force == PA_PREFILL_ONE_TILE ||
            (force == PA_PREFILL_AUTO && (nq <= qb || blocks1 <= 3LL * sms)))
            return launch_prefill_one_tile(kmap, vmap, q, num_q, q_start, tables, seq_lens, out, err,
                                           B, Hq, Hkv, max_blocks, num_blocks, max_seq_len, max_q,
                                           scale_log2, out_bf16, block_size, stream, part,
                                           splits, zero_invalid);
    }
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
    dim3 grid(static_cast<unsigned>((nq + 2 * a.Qb - 1) / (2 * a.Qb)), Hkv, B);
    CUtensorMap qmap, omap;
    if (!encode_query_map(&qmap, q, num_q, Hq, a.g, a.Qb)) return cudaErrorInvalidValue;
    // bf16 output has q's shape, so the same box describes the output tiles.
    if (out_bf16) {
        if (!encode_query_map(&omap, out, num_q, Hq, a.g, a.Qb)) return cudaErrorInvalidValue;
    } else {
        omap = qmap;  // not used: float output is written by the threads
    }
    auto kern = block_size == 16 ? prefill_kernel<16> : prefill_kernel<32>;
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, kSmemBytes, stream>>>(kmap, vmap, qmap, omap, a);
    return cudaGetLastError();
}

}  // namespace pa
