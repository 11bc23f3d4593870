// PagedEviction page scores on the device.
//
// Pith review of arXiv 2509.04377 (PagedEviction), "Core claim" and "What
// carries the argument": a token's importance is S = ||V||_2 / ||K||_2 of its
// cached value and key; a page's importance is the mean of S over its tokens;
// when the most recent page has just filled (L % block_size == 0) the page
// with the lowest mean is the one evicted. K and V of a token are taken over
// all kv heads together (one block table serves every head, so a page is
// evicted for all heads at once); ||K|| = 0 gives S = +inf; every full page is
// a candidate and ties go to the lowest logical page.
//
// The scan reads every attended K and V element once: it is HBM-bound like
// the decode, and is built the same way (balanced page ranges per warp of a
// persistent grid, per-warp bulk-copy pipelines on mbarriers, no block-level
// synchronisation after the prologue). A second small kernel picks each
// sequence's victim.
#include <algorithm>
#include <cmath>

#include "pa.h"
#include "pa_internal.h"
#include "pa_split.cuh"

namespace pa {
namespace {

struct ScoreArgs {
    const void* kpool;
    const void* vpool;
    const int32_t* tables;
    const int32_t* seq_lens;
    float* scores;
    int32_t* victims;  // victims[0] is also the score kernel's piece counter (zeroed before it)
    int* err;
    int B, Hkv, D, max_blocks, num_blocks, max_seq_len;
    int stages, stage_bytes, lens_bytes;
    int probe_wait;    // 1: the first pipeline wait of each warp expires (a test hook)
};

// Dynamic tail of the score kernel: the last 15 % of the page list in pieces
// of 2 logical pages (all kv heads of a page stay with one warp, so a piece
// leaves nothing to merge), claimed through a counter by whichever warp is
// free, so that warps whose pages arrive early take more of the end.
constexpr int kScoreDynPermille = 150;
constexpr int kScoreDynPages = 2;

__device__ __forceinline__ void sts_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void report(int* err, int bit) {
    if (err) atomicOr(err, bit);
}

template <typename T>
__device__ __forceinline__ float sumsq16(const uint4 w);
template <>
__device__ __forceinline__ float sumsq16<uint16_t>(const uint4 w) {
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
    float s0 = 0.f, s1 = 0.f;  // two chains for instruction-level parallelism
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = bf16_lo(x[i]), b = bf16_hi(x[i]);
        s0 = fmaf(a, a, s0);
        s1 = fmaf(b, b, s1);
    }
    return s0 + s1;
}
template <>
__device__ __forceinline__ float sumsq16<float>(const uint4 w) {
    const float a = __uint_as_float(w.x), b = __uint_as_float(w.y), c = __uint_as_float(w.z),
                d = __uint_as_float(w.w);
    return fmaf(a, a, fmaf(b, b, fmaf(c, c, d * d)));
}

// Score kernel: persistent blocks of kWarps warps; the flattened page list is
// cut into equal static ranges, one per warp, followed by small pieces that
// free warps claim (as in the split decode). A warp streams its pages head by
// head through a ring of shared-memory stages: one stage = the K and V pages
// of one (block, kv head), each a contiguous run moved by a 1-D bulk copy
// that completes on the stage's mbarrier, with the stage's page index
// recorded beside it. Lane (half, token)
// sums the squares of its half row, rotating the 16-byte column order by the
// token so that the eight rows a quarter-warp reads hit different banks; after
// the last head of a page the halves are joined, the token ratios formed and
// averaged, and lane 0 writes the page score.
constexpr int kScoreWarps = 8;

template <int BS, typename T>
__global__ void __launch_bounds__(kScoreWarps * 32, 1) page_score_kernel(const ScoreArgs a) {
    constexpr int TPL = BS / 16;  // tokens per lane
    extern __shared__ uint8_t smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 127u) & ~127u;
    int* pre = reinterpret_cast<int*>(smem_raw + (base - raw));
    int* len = pre + (a.B + 1);
    const uint32_t ring0 = base + a.lens_bytes;
    const uint32_t bars0 = ring0 + kScoreWarps * a.stages * a.stage_bytes;
    // After the barriers and page records: an mbarrier that nothing completes
    // (the wait-expiry probe's first wait).
    const uint32_t probe_bar = bars0 + kScoreWarps * a.stages * 12;
    if (threadIdx.x == 0 && a.probe_wait) {
        mbar_init(probe_bar, 1);
        fence_barrier_init();
    }
    const int limit = min(a.max_seq_len, a.max_blocks * BS);
    split::scan_lengths<BS>(a.seq_lens, a.B, limit, pre, len, a.err);

    const int P = pre[a.B];
    const int NW = gridDim.x * kScoreWarps;
    // Static ranges over the first part of the page list, then pieces of qd
    // pages (none for small lists, whose static ranges are already short).
    const int qd = kScoreDynPages;
    const int Dp = (P >= 8 * NW * qd)
                       ? (static_cast<int>(static_cast<long long>(P) * kScoreDynPermille / 1000) / qd) * qd
                       : 0;
    const int A = P - Dp, nd = Dp / qd;
    const int per = (A + NW - 1) / NW;
    const int gw = blockIdx.x * kScoreWarps + warp;
    const int S = a.stages, H = a.Hkv;
    const uint32_t my_bars = bars0 + warp * S * 8;
    const uint32_t my_xs = bars0 + kScoreWarps * S * 8 + warp * S * 4;  // page of each stage
    const uint32_t my_ring = ring0 + warp * S * a.stage_bytes;

    // Issue range [ix, ix1): the warp's static range, then claimed pieces.
    int ix = min(gw * per, A), ix1 = min(gw * per + per, A);
    auto claim = [&]() -> bool {  // warp-collective
        int j = 0;
        if (lane == 0) j = atomicAdd(a.victims, 1);
        j = __shfl_sync(0xffffffffu, j, 0);
        if (j >= nd) return false;
        ix = A + j * qd;
        ix1 = min(ix + qd, P);
        return true;
    };
    if (ix >= ix1 && !claim()) return;
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(my_bars + 8 * s, 1);
        fence_barrier_init();
    }
    __syncwarp();
    const uint32_t row_bytes = a.D * sizeof(T);
    const uint32_t page_bytes = BS * row_bytes;  // one pool, one (block, head)

    // Page x -> (sequence, logical page).
    auto locate = [&](int x, int& b, int& p) {
        int lo = 0, hi = a.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pre[mid] <= x) lo = mid; else hi = mid - 1;
        }
        b = lo;
        p = x - pre[lo];
    };
    int ib, ip, ih = 0;  // issue cursor: page ix = (ib, ip), head ih
    locate(ix, ib, ip);
    int iphys = a.tables[static_cast<int64_t>(ib) * a.max_blocks + ip];
    uint32_t badmask = 0, phase = 0;
    int n_issued = 0;
    bool issue_done = false;

    auto issue = [&](int s) {  // warp-collective
        const bool bad = iphys < 0 || iphys >= a.num_blocks;
        badmask = bad ? (badmask | (1u << s)) : (badmask & ~(1u << s));
        if (lane == 0) {
            const uint32_t bar = my_bars + 8 * s;
            const uint32_t stg = my_ring + s * a.stage_bytes;
            sts_u32(my_xs + 4 * s, static_cast<uint32_t>(ix));  // released by the arrive below
            if (bad) {
                mbar_arrive(bar);
            } else {
                const int64_t off = (static_cast<int64_t>(iphys) * H + ih) * page_bytes;
                mbar_arrive_expect_tx(bar, 2 * page_bytes);
                bulk_load(stg, static_cast<const char*>(a.kpool) + off, page_bytes, bar);
                bulk_load(stg + page_bytes, static_cast<const char*>(a.vpool) + off, page_bytes, bar);
            }
        }
        ++n_issued;
        if (++ih < H) return;
        ih = 0;
        if (++ix == ix1) {
            if (!claim()) {
                issue_done = true;
                return;
            }
            locate(ix, ib, ip);
        } else if (++ip == pre[ib + 1] - pre[ib]) {
            locate(ix, ib, ip);
        }
        iphys = a.tables[static_cast<int64_t>(ib) * a.max_blocks + ip];
    };
    for (int s = 0; s < S && !issue_done; ++s) issue(s);

    const int hh = lane >> 4, tl = lane & 15;
    const int CH = row_bytes / 32;  // 16-byte columns in half a row
    int cb = 0, cp = 0;
    float kk[TPL], vv[TPL];
    bool poison = false;
    int s = 0, n_done = 0;
    while (n_done < n_issued) {
        const int h = n_done % H;  // every page issues its H heads in a row
        const uint32_t bar = my_bars + 8 * s;
        const uint32_t stg = my_ring + s * a.stage_bytes;
        const bool ready = (a.probe_wait && n_done == 0)
                               ? mbar_wait_bounded(probe_bar, 0, kProbeLimitNs)
                               : mbar_wait_bounded(bar, (phase >> s) & 1u, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, ready)) {
            if (lane == 0) report(a.err, kErrTimeout);
            for (int j = n_done; j < n_issued; ++j) {
                const int sj = j % S;
                mbar_wait_bounded(my_bars + 8 * sj, (phase >> sj) & 1u, kWaitLimitNs);
            }
            return;
        }
        phase ^= 1u << s;
        if (h == 0) {
            locate(static_cast<int>(lds_u32(my_xs + 4 * s)), cb, cp);
#pragma unroll
            for (int j = 0; j < TPL; ++j) kk[j] = vv[j] = 0.f;
            poison = false;
        }
        const int n = min(BS, len[cb] - cp * BS);
        if ((badmask >> s) & 1u) {
            poison = true;
        } else {
#pragma unroll
            for (int j = 0; j < TPL; ++j) {
                const int t = tl + 16 * j;
                if (t < n) {
                    for (int c = 0; c < CH; ++c) {
                        const int col = hh * CH + (c + t) % CH;
                        kk[j] += sumsq16<T>(lds_u128(stg + t * row_bytes + col * 16));
                        vv[j] += sumsq16<T>(lds_u128(stg + page_bytes + t * row_bytes + col * 16));
                    }
                }
            }
        }
        __syncwarp();
        if (!issue_done) {
            fence_proxy_async_smem();
            issue(s);
        }
        if (h == H - 1) {
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < TPL; ++j) {
                const float k2 = kk[j] + __shfl_xor_sync(0xffffffffu, kk[j], 16);
                const float v2 = vv[j] + __shfl_xor_sync(0xffffffffu, vv[j], 16);
                const int t = tl + 16 * j;
                if (hh == 0 && t < n) sum += k2 > 0.f ? sqrtf(v2) / sqrtf(k2) : INFINITY;
            }
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            if (lane == 0) {
                float* out = a.scores + static_cast<int64_t>(cb) * a.max_blocks + cp;
                if (poison) {
                    report(a.err, kErrTable);
                    *out = __int_as_float(0x7fc00000);
                } else {
                    *out = sum / static_cast<float>(n);
                }
            }
        }
        ++n_done;
        if (++s == S) s = 0;
    }
}

// One warp per sequence: the lowest-scoring full page when L % BS == 0.
__global__ void __launch_bounds__(128) victim_kernel(const ScoreArgs a, int BS) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (b >= a.B) return;
    const int L = a.seq_lens[b];
    const int limit = min(a.max_seq_len, a.max_blocks * BS);
    int32_t victim = -1;
    if (L >= 1 && L <= limit && L % BS == 0) {
        const int nb = L / BS;
        float best = INFINITY;
        int best_p = 0x7fffffff;
        bool nan = false;
        for (int p = lane; p < nb; p += 32) {
            const float s = a.scores[static_cast<int64_t>(b) * a.max_blocks + p];
            nan |= s != s;
            if (s < best || (s == best && p < best_p)) {
                best = s;
                best_p = p;
            }
        }
        nan = __any_sync(0xffffffffu, nan);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float os = __shfl_xor_sync(0xffffffffu, best, off);
            const int op = __shfl_xor_sync(0xffffffffu, best_p, off);
            if (os < best || (os == best && op < best_p)) {
                best = os;
                best_p = op;
            }
        }
        // All pages scoring +inf: the lowest page; a NaN score (bad entry): none.
        victim = nan ? -1 : (best_p == 0x7fffffff ? 0 : best_p);
    }
    if (lane == 0) a.victims[b] = victim;
}

template <int BS>
cudaError_t launch_scores(ScoreArgs a, bool bf16, int num_sms, cudaStream_t stream) {
    const int esize = bf16 ? 2 : 4;
    a.stage_bytes = 2 * BS * a.D * esize;               // K and V page of one (block, head)
    a.lens_bytes = static_cast<int>((static_cast<size_t>(2 * a.B + 1) * 4 + 127) / 128 * 128);
    a.stages = std::max(1, std::min(8, (192 * 1024) / (kScoreWarps * a.stage_bytes)));
    const size_t smem = 128 + a.lens_bytes + static_cast<size_t>(kScoreWarps) * a.stages * a.stage_bytes +
                        static_cast<size_t>(kScoreWarps) * a.stages * (8 + 4) + 8;
    a.probe_wait = wait_probe();
    auto kern = bf16 ? page_score_kernel<BS, uint16_t> : page_score_kernel<BS, float>;
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reinterpret_cast<const void*>(kern),
                                                      kScoreWarps * 32, smem);
    if (e != cudaSuccess) return e;
    const int64_t max_pages = static_cast<int64_t>(a.B) *
                              ((std::min(a.max_seq_len, a.max_blocks * BS) + BS - 1) / BS);
    const int64_t need = (max_pages + kScoreWarps * 4 - 1) / (kScoreWarps * 4);
    const int blocks = static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>(need, static_cast<int64_t>(std::max(per_sm, 1)) * num_sms)));
    // victims[0] counts the claimed pieces during the score kernel; the victim
    // kernel overwrites it afterwards.
    e = cudaMemsetAsync(a.victims, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    kern<<<blocks, kScoreWarps * 32, smem, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    victim_kernel<<<(a.B + 3) / 4, 128, 0, stream>>>(a, BS);
    return cudaGetLastError();
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_page_scores(const void* k_pool, const void* v_pool,
                                    const int32_t* block_tables, int max_blocks,
                                    const int32_t* seq_lens, int B, int Hkv, int D,
                                    int block_size, int num_blocks, int max_seq_len,
                                    pa_dtype kv_dtype, float* scores, int32_t* victims,
                                    int* device_error, struct CUstream_st* stream) {
    if (!k_pool || !v_pool || !block_tables || !seq_lens || !scores || !victims)
        return PA_ERR_NULL;
    if (kv_dtype != PA_F32 && kv_dtype != PA_BF16) return PA_ERR_DTYPE;
    if (block_size != 16 && block_size != 32) return PA_ERR_BLOCK_SIZE;
    if (B < 0 || B > 8192 || Hkv < 1 || (D != 64 && D != 128) || num_blocks < 1 ||
        max_blocks < 1 || max_seq_len < 1)
        return PA_ERR_SHAPE;
    if (static_cast<int64_t>(max_blocks) * block_size > INT32_MAX ||
        static_cast<int64_t>(B) * max_blocks > INT32_MAX)
        return PA_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool)) & 15u)
        return PA_ERR_ALIGN;
    if (B == 0) return PA_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PA_ERR_CUDA;
    pa::ScoreArgs a{k_pool, v_pool, block_tables, seq_lens, scores, victims, device_error,
                    B, Hkv, D, max_blocks, num_blocks, max_seq_len, 0, 0, 0, 0};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool bf16 = kv_dtype == PA_BF16;
    const cudaError_t e = block_size == 16 ? pa::launch_scores<16>(a, bf16, sms, s)
                                           : pa::launch_scores<32>(a, bf16, sms, s);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
