// Merge of split partials: for every (sequence, query head) whose segment was
// cut across warps, combine the partials (m_i, l_i, acc_i) with
//   m = max_i m_i,  l = sum_i l_i 2^(m_i - m),  o = sum_i acc_i 2^(m_i - m) / l
// -- the two-partial rule of "39 · PagedAttention" §3 applied left to right,
// with the value sums rescaled by the same factors; the maxima are in the log2
// domain of the split kernel. Rows of invalid sequences are written as zeros,
// rows whose partial carries the poison marker (NaN max, a bad table entry)
// too. Segments finished inside one warp were already written by the split
// kernel and are skipped.
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

template <int D>
__global__ void __launch_bounds__(128) merge_kernel(const MergeArgs a) {
    constexpr int DPL = D / 32;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= a.B * a.Hq) return;
    const int b = row / a.Hq, hq = row - b * a.Hq;
    const int* pre = a.ws_meta + kMetaHeader;
    const int per = a.ws_meta[1];
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
        store(acc);
        return;
    }
    const int kvh = hq / a.g, r = hq - kvh * a.g;
    const int slice = r / a.GS, j = r - slice * a.GS;
    const int u = kvh * a.nslices + slice;
    const int sb = a.U * pre[b] + u * nb;
    const int wf = sb / per, wl = (sb + nb - 1) / per;
    if (wf == wl) return;

    // Slot of piece i (i = 0 .. wl-wf): the tail slot of warp wf, then the
    // head slots of warps wf+1 .. wl.
    auto slot_of = [&](int i) { return i == 0 ? wf * 2 + 1 : (wf + i) * 2; };
    const int n = wl - wf + 1;
    float m = -INFINITY;
    bool poison = false;
    for (int i = 0; i < n; ++i) {
        const float mi = a.ws_ml[(static_cast<size_t>(slot_of(i)) * a.GS + j) * 2];
        poison |= mi != mi;
        m = fmaxf(m, mi);
    }
    if (poison) {
        store(acc);
        return;
    }
    float l = 0.f;
    for (int i = 0; i < n; ++i) {
        const size_t base = static_cast<size_t>(slot_of(i)) * a.GS + j;
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
    const float inv = 1.f / l;
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] *= inv;
    store(acc);
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
    const int rows = a.B * a.Hq;
    if (rows == 0) return cudaSuccess;
    const int warps = 4;
    const int blocks = (rows + warps - 1) / warps;
    if (a.D == 128)
        merge_kernel<128><<<blocks, warps * 32, 0, stream>>>(a);
    else if (a.D == 64)
        merge_kernel<64><<<blocks, warps * 32, 0, stream>>>(a);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace pa
