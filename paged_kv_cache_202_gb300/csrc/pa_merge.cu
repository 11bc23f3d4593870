// Merge of split partials: for every (sequence, query head) whose segment was
// cut across warps, combine the partials (m_i, l_i, acc_i) with
//   m = max_i m_i,  l = sum_i l_i 2^(m_i - m),  o = sum_i acc_i 2^(m_i - m) / l
// -- the two-partial rule of "39 · PagedAttention" §3, applied to batches of
// partials against a running maximum, with the value sums rescaled by the
// same factors; the maxima are in the log2 domain of the split kernel. Rows of invalid sequences are written as zeros,
// rows whose partial carries the poison marker (NaN max, a bad table entry)
// too. Segments finished inside one range were already written by the split
// kernel and are skipped. The merge also resets the split kernel's
// dynamic-piece counter for the next call.
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

// WPR warps per (sequence, query head) row; a block has max(8, WPR) warps
// and max(8, WPR) / WPR rows. Warp w of a row folds partials rf + w, rf + w + WPR, ... in batches
// of kBatch: the loads of a whole batch are issued before any is used, then
// the batch is folded into the warp's running (m, l, acc) with one rescale.
// The warps of a row then combine their results through shared memory, on a
// named barrier of their own, so rows of one block may leave at different
// points. Lane l owns elements [l * D/32, (l+1) * D/32) of the row.
// Launched as a programmatic dependent of the split kernel: it waits for the
// split kernel's completion before reading anything.
// Batches of 4 keep the kernel at 55 registers, four blocks per SM (8 took 73
// registers and three blocks; the Llama-3-8B GQA step was 1 us longer).
template <int D, int WPR>
__global__ void __launch_bounds__(32 * (WPR > 8 ? WPR : 8)) merge_kernel(const MergeArgs a) {
    constexpr int DPL = D / 32;
    constexpr int kBatch = 4;
    constexpr int kWarps = WPR > 8 ? WPR : 8;
    constexpr int kRowsPerBlock = kWarps / WPR;
    __shared__ float sm_m[kWarps], sm_l[kWarps];
    __shared__ int sm_poison[kWarps];
    __shared__ float sm_acc[WPR > 1 ? kWarps : 1][D];
    const int lane = threadIdx.x & 31;
    const int gwarp = threadIdx.x >> 5;
    const int warp = gwarp % WPR;            // warp within the row
    const int slotw = gwarp - warp;          // first warp of the row in this block
    const int row = blockIdx.x * kRowsPerBlock + gwarp / WPR;
    // Barrier over the WPR warps of this row only: named barrier 1 + the row's
    // index in the block (barrier 0 is the block's), ids kept immediate.
    auto row_sync = [&] {
        const int rb = gwarp / WPR;
        if (rb == 0) asm volatile("bar.sync 1, %0;" ::"n"(WPR * 32) : "memory");
        if constexpr (kRowsPerBlock > 1) {
            if (rb == 1) asm volatile("bar.sync 2, %0;" ::"n"(WPR * 32) : "memory");
        }
        if constexpr (kRowsPerBlock > 2) {
            if (rb == 2) asm volatile("bar.sync 3, %0;" ::"n"(WPR * 32) : "memory");
            if (rb == 3) asm volatile("bar.sync 4, %0;" ::"n"(WPR * 32) : "memory");
        }
    };
    griddep_wait();  // the split kernel's partials and metadata
    if (row >= a.rows) return;
    // Row -> (sequence b, query head hq, column j of the kv unit's partials).
    int b, hq, qcol = 0;
    if (a.q_start) {  // several queries per sequence: row = t * Hq + hq
        const int t = row / a.Hq;
        hq = row - t * a.Hq;
        int lo = 0, hi = a.B - 1;  // the sequence whose query rows hold t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.q_start[mid] <= t) lo = mid; else hi = mid - 1;
        }
        b = lo;
        qcol = (t - a.q_start[b]) * a.g;  // column of query (t - q_start[b]), head 0
    } else {
        b = row / a.Hq;
        hq = row - b * a.Hq;
    }
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
    const int slice = hr / a.GS, j = qcol + hr - slice * a.GS;
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

    // This warp's partials, folded with a running maximum m (log2 domain).
    float m = -INFINITY, l = 0.f;
    bool poison = false;
    for (int r0 = rf + warp; r0 <= rl; r0 += kBatch * WPR) {
        float mi[kBatch], li[kBatch], v[kBatch][DPL];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int r = r0 + k * WPR;
            mi[k] = -INFINITY;
            li[k] = 0.f;
#pragma unroll
            for (int i = 0; i < DPL; ++i) v[k][i] = 0.f;
            if (r <= rl && holds(r)) {
                const size_t base = static_cast<size_t>(slot_of(r)) * a.GS + j;
                mi[k] = a.ws_ml[base * 2];
                li[k] = a.ws_ml[base * 2 + 1];
                const float* src = a.ws_acc + base * D + d0;
                if constexpr (DPL == 4) {
                    const float4 t = *reinterpret_cast<const float4*>(src);
                    v[k][0] = t.x; v[k][1] = t.y; v[k][2] = t.z; v[k][3] = t.w;
                } else {
                    const float2 t = *reinterpret_cast<const float2*>(src);
                    v[k][0] = t.x; v[k][1] = t.y;
                }
            }
        }
        float mb = m;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            poison |= mi[k] != mi[k];   // the split kernel's poison marker
            mb = fmaxf(mb, mi[k]);      // fmaxf passes over NaN
        }
        if (mb == -INFINITY) continue;  // nothing of the segment in this batch
        const float fo = fast_exp2(m - mb);   // 0 while m is still -inf
        l *= fo;
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] *= fo;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const float f = fast_exp2(mi[k] - mb);  // 0 for the empty entries
            l = fmaf(li[k], f, l);
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[i] = fmaf(v[k][i], f, acc[i]);
        }
        m = mb;
    }

    if constexpr (WPR == 1) {
        if (poison) {
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
        } else {
            const float inv = 1.f / l;
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[i] *= inv;
        }
        store(acc);
    } else {
        if (lane == 0) {
            sm_m[slotw + warp] = m;
            sm_l[slotw + warp] = l;
            sm_poison[slotw + warp] = poison ? 1 : 0;
        }
#pragma unroll
        for (int i = 0; i < DPL; ++i) sm_acc[slotw + warp][d0 + i] = acc[i];
        row_sync();
        if (warp != 0) return;
        float M = -INFINITY;
        bool bad = false;
#pragma unroll
        for (int w = 0; w < WPR; ++w) {
            M = fmaxf(M, sm_m[slotw + w]);
            bad |= sm_poison[slotw + w] != 0;
        }
        if (bad || M == -INFINITY) {
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
            store(acc);
            return;
        }
        float f[WPR];
        float lt = 0.f;
#pragma unroll
        for (int w = 0; w < WPR; ++w) {
            f[w] = fast_exp2(sm_m[slotw + w] - M);  // 0 for a warp that held nothing
            lt = fmaf(sm_l[slotw + w], f[w], lt);
        }
        const float inv = 1.f / lt;
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < WPR; ++w) t = fmaf(sm_acc[slotw + w][d0 + i], f[w], t);
            acc[i] = t * inv;
        }
        store(acc);
    }
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
    const int rows = a.rows;
    if (rows == 0) return cudaSuccess;
    // The plan chooses the warps per row from the partials per row.
    const int wpr = a.wpr;
    if (wpr != 1 && wpr != 2 && wpr != 4 && wpr != 8 && wpr != 16 && wpr != 32)
        return cudaErrorInvalidValue;
    const int warps = wpr > 8 ? wpr : 8;
    const int rows_per_block = warps / wpr;
    void (*fn)(MergeArgs) = nullptr;
    if (a.D == 128) {
        fn = wpr == 1 ? merge_kernel<128, 1> : wpr == 2 ? merge_kernel<128, 2>
           : wpr == 4 ? merge_kernel<128, 4> : wpr == 8 ? merge_kernel<128, 8>
           : wpr == 16 ? merge_kernel<128, 16> : merge_kernel<128, 32>;
    } else if (a.D == 64) {
        fn = wpr == 1 ? merge_kernel<64, 1> : wpr == 2 ? merge_kernel<64, 2>
           : wpr == 4 ? merge_kernel<64, 4> : wpr == 8 ? merge_kernel<64, 8>
           : wpr == 16 ? merge_kernel<64, 16> : merge_kernel<64, 32>;
    }
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((rows + rows_per_block - 1) / rows_per_block);
    cfg.blockDim = dim3(32 * warps);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, a);
}

}  // namespace pa
