// Simple paged decode: one warp per (sequence, query head), no split, plain
// loads. It walks the logical blocks in order through the block table and
// folds each token into a running (m, l, acc) -- the online form of one
// softmax over all scores ("39 · PagedAttention" §2-§3). It serves float32
// pools and any shape the staged kernels do not take; for bf16 it is a
// slower cross-check of the staged kernels.
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

template <typename T>
__device__ __forceinline__ float load_elem(const T* p, size_t i);
template <>
__device__ __forceinline__ float load_elem<float>(const float* p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float load_elem<uint16_t>(const uint16_t* p, size_t i) {
    return __uint_as_float(static_cast<uint32_t>(p[i]) << 16);
}

template <typename T, int D>
__global__ void __launch_bounds__(128) simple_kernel(const SimpleArgs a) {
    constexpr int DPL = D / 32;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= a.B * a.Hq) return;
    const int b = row / a.Hq, h = row - b * a.Hq;
    const int j = h / (a.Hq / a.Hkv);
    const T* q = static_cast<const T*>(a.q);
    const T* kp = static_cast<const T*>(a.kpool);
    const T* vp = static_cast<const T*>(a.vpool);
    const int L = a.seq_lens[b];
    const int limit = min(a.max_seq_len, a.max_blocks * a.BS);
    float qf[DPL], acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
        qf[i] = load_elem(q, static_cast<size_t>(row) * D + lane + 32 * i);
        acc[i] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    bool poison = false;
    if (L < 1 || L > limit) {
        if (lane == 0 && h == 0) atomicOr(a.err, kErrSeqLen);
        poison = true;
    } else {
        const int nb = (L + a.BS - 1) / a.BS;
        for (int blk = 0; blk < nb && !poison; ++blk) {
            const int phys = a.tables[static_cast<size_t>(b) * a.max_blocks + blk];
            if (phys < 0 || phys >= a.num_blocks) {
                if (lane == 0) atomicOr(a.err, kErrTable);
                poison = true;
                break;
            }
            const int n = min(a.BS, L - blk * a.BS);
            for (int t = 0; t < n; ++t) {
                const size_t base = ((static_cast<size_t>(phys) * a.Hkv + j) * a.BS + t) * D;
                float dot = 0.f;
#pragma unroll
                for (int i = 0; i < DPL; ++i) dot = fmaf(qf[i], load_elem(kp, base + lane + 32 * i), dot);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
                const float s2 = dot * a.scale_log2;
                const float m_new = fmaxf(m, s2);
                const float alpha = fast_exp2(m - m_new);
                const float p = fast_exp2(s2 - m_new);
                l = l * alpha + p;
#pragma unroll
                for (int i = 0; i < DPL; ++i)
                    acc[i] = fmaf(p, load_elem(vp, base + lane + 32 * i), acc[i] * alpha);
                m = m_new;
            }
        }
    }
    const float inv = poison ? 0.f : 1.f / l;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
        const float v = poison ? 0.f : acc[i] * inv;
        const size_t o = static_cast<size_t>(row) * D + lane + 32 * i;
        if (a.out_bf16)
            static_cast<uint16_t*>(a.out)[o] = f32_to_bf16_bits(v);
        else
            static_cast<float*>(a.out)[o] = v;
    }
}

}  // namespace

cudaError_t launch_simple(const SimpleArgs& a, cudaStream_t stream) {
    const int rows = a.B * a.Hq;
    if (rows == 0) return cudaSuccess;
    const int warps = 4;
    const int blocks = (rows + warps - 1) / warps;
    if (a.kv_bf16) {
        if (a.D == 128) simple_kernel<uint16_t, 128><<<blocks, warps * 32, 0, stream>>>(a);
        else if (a.D == 64) simple_kernel<uint16_t, 64><<<blocks, warps * 32, 0, stream>>>(a);
        else return cudaErrorInvalidValue;
    } else {
        if (a.D == 128) simple_kernel<float, 128><<<blocks, warps * 32, 0, stream>>>(a);
        else if (a.D == 64) simple_kernel<float, 64><<<blocks, warps * 32, 0, stream>>>(a);
        else return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace pa
