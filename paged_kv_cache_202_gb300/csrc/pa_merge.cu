// Merge of split partials: for every (sequence, query head) whose segment was
// cut across warps, combine the partials (m_i, l_i, acc_i) with
//   m = max_i m_i,  l = sum_i l_i 2^(m_i - m),  o = sum_i acc_i 2^(m_i - m) / l
// -- the two-partial rule of "39 · PagedAttention" §3 applied left to right,
// with the value sums rescaled by the same factors; the maxima are in the log2
// domain of the split kernel. Rows of invalid sequences are written as zeros,
// rows whose partial carries the poison marker (NaN max, a bad table entry)
// too. Segments finished inside one range were already written by the split
// kernel and are skipped. The merge also resets the split kernel's
// dynamic-piece counter for the next call.
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

// WPR warps per (sequence, query head) row, 8 / WPR rows per block of 8
// warps. The warps of a row split its partials (warp w folds every WPR-th
// one, with its loads unrolled so that several are in flight), then the
// row's first warp folds the warps' results. Lane l owns elements
// [l * D/32, (l+1) * D/32) of the row. Many warps per row pay off when
// dynamic pieces cut long segments into many partials; one warp per row is
// cheaper otherwise.
template <int D, int WPR>
__global__ void __launch_bounds__(256) merge_kernel(const MergeArgs a) {
    constexpr int DPL = D / 32;
    constexpr int kMergeWarps = WPR;
    constexpr int kRowsPerBlock = 8 / WPR;
    __shared__ float sm_m[8], sm_l[8];
    __shared__ float sm_acc[8][D];
    const int lane = threadIdx.x & 31;
    const int gwarp = threadIdx.x >> 5;
    const int warp = gwarp % WPR;            // warp within the row
    const int slotw = gwarp - warp;          // first warp of the row in this block
    const int row = blockIdx.x * kRowsPerBlock + gwarp / WPR;
    if (row >= a.B * a.Hq) return;
    const int b = row / a.Hq, hq = row - b * a.Hq;
    const int* pre = a.ws_meta + kMetaHeader;
    const int per = a.ws_meta[1], NW = a.ws_meta[2], A = a.ws_meta[4], qd = a.ws_meta[5];
    if (row == 0 && threadIdx.x == 0) a.ws_meta[3] = 0;  // dynamic-piece counter, for the next call
    const int nb = pre[b + 1] - pre[b];
    const int d0 = lane * DPL;
    const size_t orow = static_cast<size_t>(row) * D + d0;

    auto store = [&](const float (&v)[DPL]) {
        if (a.out_bf16) {
            uint16_t* o = static_cast<uint16_t*>(a.out) + orow;
            if constexpr (DPL == 4) {
                uint2 w;
                w.x = pack_bf16x2(v[0], v[1]);
                w.y = pack_bf16x2(v[2], v[3]);
                *reinterpret_cast<uint2*>(o) = w;
            } else {
                *reinterpret_cast<uint32_t*>(o) = pack_bf16x2(v[0], v[1]);
            }
        } else {
            float* o = static_cast<float*>(a.out) + orow;
#pragma unroll
            for (int i = 0; i < DPL; ++i) o[i] = v[i];
        }
    };

    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
    if (nb == 0) {
        if (warp == 0) store(acc);
        return;
    }
    const int kvh = hq / a.g, hr = hq - kvh * a.g;
    const int slice = hr / a.GS, j = hr - slice * a.GS;
    const int u = kvh * a.nslices + slice;
    const int sb = a.U * pre[b] + u * nb;
    // Range of page x: static ranges of `per` pages up to A, then pieces of qd.
    auto range_of = [&](int x) { return x < A ? x / per : NW + (x - A) / qd; };
    const int rf = range_of(sb), rl = range_of(sb + nb - 1);
    if (rf == rl) return;  // finished inside one range by the split kernel

    // Ranges rf .. rl that hold part of the segment: the tail slot of rf, then
    // the head slots of the others (empty static ranges past A hold nothing).
    auto holds = [&](int r) { return r >= NW || static_cast<long long>(r) * per < A; };
    auto slot_of = [&](int r) { return r == rf ? r * 2 + 1 : r * 2; };
    // Pass 1: the row maximum (and poison) over all partials.
    float m = -INFINITY;
    bool poison = false;
    for (int r = rf + warp * 32 + lane; r <= rl; r += kMergeWarps * 32) {
        if (!holds(r)) continue;
        const float mi = a.ws_ml[(static_cast<size_t>(slot_of(r)) * a.GS + j) * 2];
        poison |= mi != mi;
        m = fmaxf(m, mi);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    poison = __any_sync(0xffffffffu, poison);
    if constexpr (WPR > 1) {
        if (lane == 0) {
            sm_m[slotw + warp] = m;
            sm_l[slotw + warp] = poison ? 1.f : 0.f;
        }
        __syncthreads();
        m = sm_m[slotw];
        poison = false;
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) {
            m = fmaxf(m, sm_m[slotw + w]);
            poison |= sm_l[slotw + w] != 0.f;
        }
    }
    if (poison) {
        if (warp == 0) store(acc);
        return;
    }
    if constexpr (WPR > 1) __syncthreads();
    // Pass 2: this warp's share of l and acc, rescaled to the row maximum.
    float l = 0.f;
#pragma unroll 4
    for (int r = rf + warp; r <= rl; r += kMergeWarps) {
        if (!holds(r)) continue;
        const size_t base = static_cast<size_t>(slot_of(r)) * a.GS + j;
        const float f = fast_exp2(a.ws_ml[base * 2] - m);
        l = fmaf(a.ws_ml[base * 2 + 1], f, l);
        const float* src = a.ws_acc + base * D + d0;
        if constexpr (DPL == 4) {
            const float4 v = *reinterpret_cast<const float4*>(src);
            acc[0] = fmaf(v.x, f, acc[0]);
            acc[1] = fmaf(v.y, f, acc[1]);
            acc[2] = fmaf(v.z, f, acc[2]);
            acc[3] = fmaf(v.w, f, acc[3]);
        } else {
            const float2 v = *reinterpret_cast<const float2*>(src);
            acc[0] = fmaf(v.x, f, acc[0]);
            acc[1] = fmaf(v.y, f, acc[1]);
        }
    }
    if constexpr (WPR == 1) {  // every lane folded every partial: l is already the row's
        const float inv = 1.f / l;
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] *= inv;
        store(acc);
    } else {
        if (lane == 0) sm_l[slotw + warp] = l;
#pragma unroll
        for (int i = 0; i < DPL; ++i) sm_acc[slotw + warp][d0 + i] = acc[i];
        __syncthreads();
        if (warp != 0) return;
        float lt = 0.f;
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) lt += sm_l[slotw + w];
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kMergeWarps; ++w) v += sm_acc[slotw + w][d0 + i];
            acc[i] = v / lt;
        }
        store(acc);
    }
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
    const int rows = a.B * a.Hq;
    if (rows == 0) return cudaSuccess;
    const bool wide = a.wide;
    const int blocks = wide ? rows : (rows + 7) / 8;
    if (a.D == 128) {
        if (wide) merge_kernel<128, 8><<<blocks, 256, 0, stream>>>(a);
        else merge_kernel<128, 1><<<blocks, 256, 0, stream>>>(a);
    } else if (a.D == 64) {
        if (wide) merge_kernel<64, 8><<<blocks, 256, 0, stream>>>(a);
        else merge_kernel<64, 1><<<blocks, 256, 0, stream>>>(a);
    }
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace pa
