// Paged multi-query attention (chunked prefill, speculative verification) on
// the tcgen05 tensor cores.
//
// The newest n_b tokens of sequence b are queries at once; query i at position
// pos = L_b - n_b + i attends causally to tokens t <= pos read through the
// block table ("FlashAttention vs PagedAttention", "How prefill and decode
// change the diagnosis"; exact attention as in "39 · PagedAttention" §1-§2).
// Here the query side is a real dense contraction: one block takes 128 rows =
// (128 / g) queries x the g query heads of one kv head, so every K/V chunk is
// read once for all of them.
//
// Per block: the 128 x 128 query tile is written to shared memory in the
// 128-byte-swizzled K-major layout; K and V chunks of 64 tokens (whole pages)
// arrive by tiled bulk tensor copies into a two-stage ring. For each chunk one
// thread issues S = Q K^T (M=128, N=64, K=128: eight k16 MMAs) into tensor
// memory; every thread then owns one row: it loads its 64 scores from TMEM,
// applies the scale (log2 domain), the causal mask by predicate and the online
// softmax, writes its bf16 probabilities into a swizzled P tile (over the
// chunk's consumed K stage), rescales its
// row of the TMEM accumulator when the running max moved, and one thread
// issues O += P V (M=128, N=128, K=64, V read MN-major). Rows past the last
// valid token of the final chunk are zeroed in V before the product so that
// slots beyond the sequence never reach a sum. Every mbarrier wait is bounded;
// on expiry the block reports PA_DEVERR_TIMEOUT, waits for its copies and
// MMAs in flight (bounded), frees its tensor memory and returns.
#include <cuda_bf16.h>

#include "pa.h"
#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "pa_tc.cuh"

namespace pa {
namespace {

constexpr int kRows = 128;    // M: query rows per block
constexpr int kChunk = 64;    // tokens per K/V chunk
constexpr int kD = 128;       // head dimension
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;   // scores: 64 columns
constexpr uint32_t kColO = 64;  // output accumulator: 128 columns

// Shared-memory layout (byte offsets from a 1024-aligned base).
// The probabilities of chunk c (128 rows x 128 B) are written over chunk c's
// K stage, which is free once S = Q K^T has completed; that keeps a block at
// ~97 KB so that two blocks share an SM.
constexpr uint32_t kOffQ = 0;                       // 2 halves x 128 rows x 128 B
constexpr uint32_t kOffK = 32768;                   // 2 stages x 2 halves x 64 rows x 128 B
constexpr uint32_t kOffV = kOffK + 2 * 16384;
constexpr uint32_t kOffBar = kOffV + 2 * 16384;     // 4 mbarriers + TMEM address slot
constexpr uint32_t kOffTable = kOffBar + 64;        // the sequence's physical block ids

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kRows, kChunk, false, false);
constexpr uint32_t kIdescO = tc::idesc_bf16_f32(kRows, kD, false, true);

struct PrefillArgs {
    const uint16_t* q;        // [T][Hq][D] bf16
    const int32_t* q_start;   // [B + 1]
    const int32_t* tables;
    const int32_t* seq_lens;
    void* out;                // [T][Hq][D]
    int* err;
    int B, Hq, Hkv, g, Qb;    // Qb = queries per block = 128 / g
    int max_blocks, num_blocks, max_seq_len;
    float scale_log2;
    int out_bf16;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void write_row(const PrefillArgs& a, size_t row, const float* v, float inv,
                                          int d0, int nd) {
    if (a.out_bf16) {
        uint16_t* o = static_cast<uint16_t*>(a.out) + row * kD + d0;
        for (int i = 0; i < nd; i += 2)
            *reinterpret_cast<uint32_t*>(o + i) = pack_bf16x2(v[i] * inv, v[i + 1] * inv);
    } else {
        float* o = static_cast<float*>(a.out) + row * kD + d0;
        for (int i = 0; i < nd; ++i) o[i] = v[i] * inv;
    }
}

template <int BS>
__global__ void __launch_bounds__(128, 2)
    prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    int32_t* tbl = reinterpret_cast<int32_t*>(gbase + kOffTable);
    const uint32_t bar_kv0 = base + kOffBar, bar_s = base + kOffBar + 16, bar_pv = base + kOffBar + 24;
    const uint32_t tmem_slot = base + kOffBar + 32;

    const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int qs = a.q_start[b];
    const int n = a.q_start[b + 1] - qs;
    const int L = a.seq_lens[b];
    const int limit = min(a.max_seq_len, a.max_blocks * BS);
    const int q0 = qb * a.Qb;
    if (n < 1 || L < n || L > limit) {
        if (qb == 0 && h == 0 && tid == 0) atomicOr(a.err, kErrSeqLen);
        return;  // rows of an invalid sequence are left untouched
    }
    if (q0 >= n) return;
    const int nq = min(a.Qb, n - q0);
    const int ntok = L - n + q0 + nq;           // tokens any row of this block may see
    const int nc = (ntok + kChunk - 1) / kChunk;
    const int nb = (ntok + BS - 1) / BS;

    // The table row of this sequence, validated once.
    bool bad = false;
    for (int i = tid; i < nb; i += blockDim.x) {
        const int p = a.tables[static_cast<size_t>(b) * a.max_blocks + i];
        tbl[i] = p;
        bad |= p < 0 || p >= a.num_blocks;
    }
    const int row = tid;                         // this thread's query row
    const int qi = row / a.g, qj = row - qi * a.g;
    const bool row_valid = qi < nq;
    const size_t out_row = (static_cast<size_t>(qs) + q0 + qi) * a.Hq + h * a.g + qj;
    if (__syncthreads_or(bad)) {
        if (tid == 0) atomicOr(a.err, kErrTable);
        if (row_valid) {
            float z[kD] = {};
            write_row(a, out_row, z, 0.f, 0, kD);
        }
        return;
    }
    if (tid == 0) {
        mbar_init(bar_kv0, 1);
        mbar_init(bar_kv0 + 8, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_pv, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tc::alloc(tmem_slot, kTmemCols);
        tc::relinquish();
    }
    // Query rows -> swizzled K-major tile (two 64-column halves).
    {
        const uint16_t* src = a.q + out_row * kD;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const uint4 w = row_valid ? *reinterpret_cast<const uint4*>(src + c * 8)
                                      : make_uint4(0, 0, 0, 0);
            const int half = c >> 3, cc = c & 7;
            st_shared_v4(base + kOffQ + half * 16384 + row * 128 + ((cc ^ (row & 7)) << 4), w);
        }
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + kOffBar + 32);
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint64_t policy = policy_evict_first();

    auto issue_kv = [&](int c, int s) {
        if (tid != 0) return;
        const int p0 = c * (kChunk / BS);
        const int np = min(kChunk / BS, nb - p0);
        const uint32_t bar = bar_kv0 + 8 * s;
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(np) * BS * kD * 2 * 2);
        const uint32_t kst = base + kOffK + s * 16384, vst = base + kOffV + s * 16384;
        for (int j = 0; j < np; ++j) {
            const int r = tbl[p0 + j] * a.Hkv + h;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint32_t off = half * 8192 + j * BS * 128;
                tma_load_3d(kst + off, &kmap, half * 64, 0, r, bar, policy);
                tma_load_3d(vst + off, &vmap, half * 64, 0, r, bar, policy);
            }
        }
    };
    // Bounded wait by every thread; false if any thread gave up.
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
        const bool ok = mbar_wait_bounded(bar, parity, kWaitLimitNs);
        return !__syncthreads_or(!ok);
    };
    uint32_t ph_kv = 0, ph_s = 0, ph_pv = 0;
    int kv_issued = 0, kv_done = 0, s_issued = 0, s_done = 0, pv_issued = 0, pv_done = 0;
    auto bail = [&]() {
        if (tid == 0) {
            atomicOr(a.err, kErrTimeout);
            // Bounded waits for this block's copies and MMAs still in flight.
            for (int k = kv_done; k < kv_issued; ++k)
                mbar_wait_bounded(bar_kv0 + 8 * (k & 1), (ph_kv >> (k & 1)) & 1u, kWaitLimitNs);
            if (s_issued > s_done) mbar_wait_bounded(bar_s, ph_s, kWaitLimitNs);
            if (pv_issued > pv_done) mbar_wait_bounded(bar_pv, ph_pv, kWaitLimitNs);
        }
        tc::fence_before_sync();
        __syncthreads();
        if (warp == 0) tc::dealloc(tmem, kTmemCols);
    };

    issue_kv(0, 0);
    kv_issued = 1;
    const int pos_r = L - n + q0 + qi;
    float m = -INFINITY, l = 0.f;
    for (int c = 0; c < nc; ++c) {
        const int s = c & 1;
        if (!wait_all(bar_kv0 + 8 * s, (ph_kv >> s) & 1u)) { bail(); return; }
        ph_kv ^= 1u << s;
        ++kv_done;
        // S = Q K^T into TMEM columns [0, 64).
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t kst = base + kOffK + s * 16384;
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
                const uint32_t half = kk >> 2, off = (kk & 3) * 32;
                const uint64_t ad = tc::smem_desc(base + kOffQ + half * 16384 + off, 16, 1024);
                const uint64_t bd = tc::smem_desc(kst + half * 8192 + off, 16, 1024);
                tc::mma_bf16(tmem + kColS, ad, bd, kIdescS, kk > 0);
            }
            tc::commit(bar_s);
        }
        ++s_issued;
        if (!wait_all(bar_s, ph_s)) { bail(); return; }
        ph_s ^= 1u;
        ++s_done;
        tc::fence_after_sync();
        float sv[64];
        {
            float t0[32], t1[32];
            tc::ld32(tmem + lane_base + kColS, t0);
            tc::ld32(tmem + lane_base + kColS + 32, t1);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                sv[i] = t0[i];
                sv[32 + i] = t1[i];
            }
        }
        // Scale, causal mask by predicate, online softmax (this thread's row).
        const int t0 = c * kChunk;
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            const float v = (row_valid && t0 + i <= pos_r) ? sv[i] * a.scale_log2 : -INFINITY;
            sv[i] = v;
            mx = fmaxf(mx, v);
        }
        const float m_new = fmaxf(m, mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = fast_exp2(m - m_use);
        uint32_t pw[32];
        float psum = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            pw[i] = pack_bf16x2(fast_exp2(sv[2 * i] - m_use), fast_exp2(sv[2 * i + 1] - m_use));
            psum += bf16_lo(pw[i]) + bf16_hi(pw[i]);
        }
        l = l * alpha + psum;
        m = m_new;
        // The previous P V must be done before P and O are touched again.
        if (c > 0) {
            if (!wait_all(bar_pv, ph_pv)) { bail(); return; }
            ph_pv ^= 1u;
            ++pv_done;
            tc::fence_after_sync();
        }
        if (c + 1 < nc) {
            issue_kv(c + 1, s ^ 1);
            ++kv_issued;
        }
        // P row -> swizzled K-major tile in this chunk's (consumed) K stage.
        const uint32_t pst = base + kOffK + s * 16384;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
            st_shared_v4(pst + row * 128 + ((ch ^ (row & 7)) << 4),
                         make_uint4(pw[4 * ch], pw[4 * ch + 1], pw[4 * ch + 2], pw[4 * ch + 3]));
        // Rescale this row of the TMEM accumulator if its max moved.
        if (c > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int piece = 0; piece < kD / 32; ++piece) {
                float o[32];
                tc::ld32(tmem + lane_base + kColO + piece * 32, o);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] *= alpha;
                tc::st32(tmem + lane_base + kColO + piece * 32, o);
            }
            tc::wait_st();
        }
        // Final chunk: zero the V rows past the last token any row may see.
        const int valid = min(kChunk, ntok - t0);
        if (valid < kChunk) {
            const uint32_t vst = base + kOffV + s * 16384;
            for (int idx = tid; idx < (kChunk - valid) * 16; idx += blockDim.x) {
                const int r = valid + (idx >> 4), half = (idx >> 3) & 1, ch = idx & 7;
                st_shared_v4(vst + half * 8192 + r * 128 + ch * 16, make_uint4(0, 0, 0, 0));
            }
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        // O += P V into TMEM columns [64, 192).
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t vst = base + kOffV + s * 16384;
#pragma unroll
            for (int kk = 0; kk < kChunk / 16; ++kk) {
                const uint64_t ad = tc::smem_desc(pst + kk * 32, 16, 1024);
                const uint64_t bd = tc::smem_desc(vst + kk * 2048, 8192, 1024);
                tc::mma_bf16(tmem + kColO, ad, bd, kIdescO, c > 0 || kk > 0);
            }
            tc::commit(bar_pv);
        }
        ++pv_issued;
    }
    if (!wait_all(bar_pv, ph_pv)) { bail(); return; }
    tc::fence_after_sync();
    const float inv = (row_valid && l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
    for (int piece = 0; piece < kD / 32; ++piece) {
        float o[32];
        tc::ld32(tmem + lane_base + kColO + piece * 32, o);
        tc::wait_ld();
        if (row_valid) write_row(a, out_row, o, inv, piece * 32, 32);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& kmap, const CUtensorMap& vmap, const void* q,
                           const int32_t* q_start, const int32_t* tables, const int32_t* seq_lens,
                           void* out, int* err, int B, int Hq, int Hkv, int max_blocks,
                           int num_blocks, int max_seq_len, int max_q, float scale_log2,
                           int out_bf16, int block_size, cudaStream_t stream) {
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
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    a.max_seq_len = max_seq_len;
    a.scale_log2 = scale_log2;
    a.out_bf16 = out_bf16;
    const size_t smem = 1024 + kOffTable + static_cast<size_t>(max_blocks) * 4;
    dim3 grid((max_q + a.Qb - 1) / a.Qb, Hkv, B);
    auto kern = block_size == 16 ? prefill_kernel<16> : prefill_kernel<32>;
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, 128, smem, stream>>>(kmap, vmap, a);
    return cudaGetLastError();
}

}  // namespace pa
