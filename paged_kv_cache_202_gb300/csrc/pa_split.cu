// Instantiations and launch of the split paged decode kernels.
#include "pa_split.cuh"

namespace pa {
namespace split {

template <int D, int BS>
__global__ void __launch_bounds__(256, 1)
    fma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const SplitArgs a) {
    split_body<D, BS, FmaState<D, kChunkTokens>>(&kmap, &vmap, a);
}

// Two n-tiles (9-16 query heads per kv head) read their query fragments
// from shared memory at every chunk, as the multi-query kernel does, and run
// one block of up to twelve warps per SM (as many as the shared memory holds).
template <int D, int BS, int NT>
__global__ void __launch_bounds__(NT == 2 ? 32 * kQsMaxWarps : 256, 1)
    mma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const SplitArgs a) {
    split_body<D, BS, MmaState<D, kChunkTokens, NT, NT == 2>>(&kmap, &vmap, a);
}

// The one-n-tile kernel with the step's append fused in (pa_append_decode).
template <int D, int BS>
__global__ void __launch_bounds__(256, 1)
    mma_append_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const SplitArgs a) {
    split_body<D, BS, MmaState<D, kChunkTokens, 1, false>, false, false, true>(&kmap, &vmap, a);
}

// One n-tile with the fused merge: the warp that writes a segment's last
// partial folds them, so no merge kernel follows. Three warps a block and
// four blocks an SM, as the plain kernel runs: at most 170 registers a thread.
template <int D, int BS>
__global__ void __launch_bounds__(96, 4)
    mma_fused_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const SplitArgs a) {
    split_body<D, BS, MmaState<D, kChunkTokens, 1, false>, false, true>(&kmap, &vmap, a);
}

// Several queries per sequence (speculative verification) on the same tiles,
// query fragments read from the stage's query rows at every chunk; at most
// 204 registers a thread, so that two blocks of five warps fit an SM.
template <int D, int BS, int NT>
__global__ void __launch_bounds__(160, 2)
    mma_mq_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const SplitArgs a) {
    split_body<D, BS, MmaState<D, kChunkTokens, NT, true>, true>(&kmap, &vmap, a);
}

using KernelFn = void (*)(CUtensorMap, CUtensorMap, SplitArgs);

KernelFn select(const SplitLaunch& L) {
#define PA_CASE(D_, BS_)                                                        \
    if (L.D == D_ && L.BS == BS_) {                                             \
        if (L.mq) {                                                             \
            if (L.kind == kSplitMma && L.NT == 1) return mma_mq_kernel<D_, BS_, 1>; \
            if (L.kind == kSplitMma && L.NT == 2) return mma_mq_kernel<D_, BS_, 2>; \
            return nullptr;                                                     \
        }                                                                       \
        if (L.fused) {                                                          \
            if (L.kind == kSplitMma && L.NT == 1 && L.warps == 3)              \
                return mma_fused_kernel<D_, BS_>;                               \
            return nullptr;                                                     \
        }                                                                       \
        if (L.append) {                                                         \
            if (L.kind == kSplitMma && L.NT == 1) return mma_append_kernel<D_, BS_>; \
            return nullptr;                                                     \
        }                                                                       \
        if (L.kind == kSplitFma) return fma_kernel<D_, BS_>;                    \
        if (L.kind == kSplitMma && L.NT == 1) return mma_kernel<D_, BS_, 1>;    \
        if (L.kind == kSplitMma && L.NT == 2) return mma_kernel<D_, BS_, 2>;    \
    }
    PA_CASE(128, 16)
    PA_CASE(128, 32)
    PA_CASE(64, 16)
    PA_CASE(64, 32)
#undef PA_CASE
    return nullptr;
}

}  // namespace split

int split_blocks_per_sm(const SplitLaunch& L, cudaError_t* status) {
    split::KernelFn fn = split::select(L);
    if (!fn) {
        *status = cudaErrorInvalidValue;
        return 0;
    }
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L.smem));
    if (e != cudaSuccess) {
        *status = e;
        return 0;
    }
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, reinterpret_cast<const void*>(fn),
                                                      L.warps * 32, L.smem);
    *status = e;
    return e == cudaSuccess ? n : 0;
}

cudaError_t launch_split(const SplitLaunch& L, const CUtensorMap& kmap, const CUtensorMap& vmap,
                         const SplitArgs& a, cudaStream_t stream) {
    split::KernelFn fn = split::select(L);
    if (!fn) return cudaErrorInvalidValue;
    // Programmatic dependent launch: the kernel waits for its predecessor at
    // griddep_wait(), so its launch can overlap the predecessor's drain.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.blocks);
    cfg.blockDim = dim3(L.warps * 32);
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, kmap, vmap, a);
}

}  // namespace pa
