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
// the decode. Blocks of a persistent grid walk the flattened (sequence, page)
// list with a stride, so work is balanced whatever the length mix; each page
// of each kv head is read with 16-byte vector loads, the squares of a token
// row are reduced by shuffles, the per-token sums over heads are gathered in
// shared memory, and one warp turns them into the page's mean. A second small
// kernel picks each sequence's victim.
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
    int32_t* victims;
    int* err;
    int B, Hkv, D, max_blocks, num_blocks, max_seq_len;
};

__device__ __forceinline__ void report(int* err, int bit) {
    if (err) atomicOr(err, bit);
}

template <typename T>
__device__ __forceinline__ float sumsq16(const uint4 w);
template <>
__device__ __forceinline__ float sumsq16<uint16_t>(const uint4 w) {
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = bf16_lo(x[i]), b = bf16_hi(x[i]);
        s = fmaf(a, a, s);
        s = fmaf(b, b, s);
    }
    return s;
}
template <>
__device__ __forceinline__ float sumsq16<float>(const uint4 w) {
    const float a = __uint_as_float(w.x), b = __uint_as_float(w.y), c = __uint_as_float(w.z),
                d = __uint_as_float(w.w);
    return fmaf(a, a, fmaf(b, b, fmaf(c, c, d * d)));
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <int BS, typename T>
__global__ void __launch_bounds__(256) page_score_kernel(const ScoreArgs a) {
    extern __shared__ int smem_i[];
    __shared__ float tok_kk[32], tok_vv[32];
    int* pre = smem_i;
    int* len = pre + (a.B + 1);
    const int tid = threadIdx.x, lane = tid & 31;
    const int limit = min(a.max_seq_len, a.max_blocks * BS);
    split::scan_lengths<BS>(a.seq_lens, a.B, limit, pre, len, a.err);
    const int total = pre[a.B];
    const int cpr = a.D * static_cast<int>(sizeof(T)) / 16;  // 16-byte chunks per token row
    const int per_head = BS * cpr;
    const int64_t row_bytes = static_cast<int64_t>(a.D) * sizeof(T);
    for (int x = blockIdx.x; x < total; x += gridDim.x) {
        int lo = 0, hi = a.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pre[mid] <= x) lo = mid; else hi = mid - 1;
        }
        const int b = lo, p = x - pre[b];
        const int phys = a.tables[static_cast<int64_t>(b) * a.max_blocks + p];
        float* out = a.scores + static_cast<int64_t>(b) * a.max_blocks + p;
        if (phys < 0 || phys >= a.num_blocks) {
            if (tid == 0) {
                report(a.err, kErrTable);
                *out = __int_as_float(0x7fc00000);
            }
            continue;  // uniform across the block
        }
        const int n = min(BS, len[b] - p * BS);
        if (tid < 32) {
            tok_kk[tid] = 0.f;
            tok_vv[tid] = 0.f;
        }
        __syncthreads();
        const char* kbase = static_cast<const char*>(a.kpool) + static_cast<int64_t>(phys) * a.Hkv * BS * row_bytes;
        const char* vbase = static_cast<const char*>(a.vpool) + static_cast<int64_t>(phys) * a.Hkv * BS * row_bytes;
        const int nchunks = a.Hkv * per_head;
#pragma unroll 4
        for (int c = tid; c < nchunks; c += blockDim.x) {
            const int h = c / per_head, r = c - h * per_head;
            const int t = r / cpr;
            float kk = 0.f, vv = 0.f;
            if (t < n) {
                const int64_t off = (static_cast<int64_t>(h) * BS) * row_bytes + static_cast<int64_t>(r) * 16;
                kk = sumsq16<T>(ld_stream(kbase + off));
                vv = sumsq16<T>(ld_stream(vbase + off));
            }
            // Lanes c .. c+cpr-1 hold one token row (cpr is a power of two <= 32
            // and blockDim.x a multiple of 32, so a row never straddles warps).
            for (int off = 1; off < cpr; off <<= 1) {
                kk += __shfl_xor_sync(0xffffffffu, kk, off);
                vv += __shfl_xor_sync(0xffffffffu, vv, off);
            }
            if ((lane & (cpr - 1)) == 0 && t < n) {
                atomicAdd(&tok_kk[t], kk);
                atomicAdd(&tok_vv[t], vv);
            }
        }
        __syncthreads();
        if (tid < 32) {
            float s = 0.f;
            if (tid < n) {
                const float kk = tok_kk[tid], vv = tok_vv[tid];
                s = kk > 0.f ? sqrtf(vv) / sqrtf(kk) : INFINITY;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            if (tid == 0) *out = s / static_cast<float>(n);
        }
        __syncthreads();
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
cudaError_t launch_scores(const ScoreArgs& a, bool bf16, int num_sms, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(2 * a.B + 1) * 4;
    auto kern = bf16 ? page_score_kernel<BS, uint16_t> : page_score_kernel<BS, float>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    const int64_t max_pages = static_cast<int64_t>(a.B) *
                              ((std::min(a.max_seq_len, a.max_blocks * BS) + BS - 1) / BS);
    const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(max_pages, 8ll * num_sms)));
    kern<<<blocks, 256, smem, stream>>>(a);
    cudaError_t e = cudaGetLastError();
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
                    B, Hkv, D, max_blocks, num_blocks, max_seq_len};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool bf16 = kv_dtype == PA_BF16;
    const cudaError_t e = block_size == 16 ? pa::launch_scores<16>(a, bf16, sms, s)
                                           : pa::launch_scores<32>(a, bf16, sms, s);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
