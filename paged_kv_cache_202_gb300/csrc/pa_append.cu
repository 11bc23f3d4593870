// KV append: the step's new key/value rows go to slot cache_len % BS of the
// physical block that the table names for logical block cache_len / BS -- the
// only partly filled block of the sequence ("PagedAttention: The Cache Was
// Storing Nothing" §1 and §2.2). A raw 16-byte-vector copy, bit-exact.
#include <algorithm>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

__device__ int g_append_error;  // library-wide word of append and block copies (per device)

// blockIdx.x = sequence; each thread moves one 16-byte vector of the
// sequence's new K and V rows (blockIdx.y picks the group of 256 vectors).
// The vector's load does not depend on where it goes, so it is issued first
// and its latency overlaps the two dependent index loads (cache length, then
// table entry). Launched as a programmatic dependent of whatever the stream
// ran before (the previous step's merge, typically): its launch overlaps that
// kernel's run, and it waits for its completion before touching memory.
__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a) {
    griddep_wait();               // the stream's previous kernel has completed
    griddep_launch_dependents();  // a following decode may start launching
    const int b = blockIdx.x;
    const int row_bytes = a.D * a.elem_bytes;
    const int chunks = row_bytes / 16;        // 16-byte vectors per head row
    const int per_pool = a.Hkv * chunks;
    const int i = blockIdx.y * blockDim.x + threadIdx.x;
    const bool mine = i < 2 * per_pool;
    const int which = i / per_pool;           // 0 = K, 1 = V
    const int r = i - which * per_pool;
    const int h = r / chunks, c = r - h * chunks;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (mine) {
        const char* src = static_cast<const char*>(which ? a.v_new : a.k_new) +
                          (static_cast<size_t>(b) * a.Hkv + h) * row_bytes + c * 16;
        w = *reinterpret_cast<const uint4*>(src);
    }
    const int pos = a.cache_lens[b] - a.pos_offset;
    if (pos < 0 || pos >= a.max_blocks * a.BS) {
        if (threadIdx.x == 0) atomicOr(&g_append_error, kErrCacheLen);
        return;
    }
    const int phys = a.tables[static_cast<size_t>(b) * a.max_blocks + pos / a.BS];
    if (phys < 0 || phys >= a.num_blocks) {
        if (threadIdx.x == 0) atomicOr(&g_append_error, kErrTable);
        return;
    }
    if (mine) {
        char* dst = static_cast<char*>(which ? a.vpool : a.kpool) +
                    ((static_cast<size_t>(phys) * a.Hkv + h) * a.BS + pos % a.BS) * row_bytes +
                    c * 16;
        *reinterpret_cast<uint4*>(dst) = w;
    }
}

// Block copies: blockIdx.x = copy pair, blockIdx.y = pool (0 = K, 1 = V).
// Each thread issues kVec 16-byte loads before storing any of them, so a
// block moves in about one memory round trip.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const CopyArgs a) {
    constexpr int kVec = 8;
    const int i = blockIdx.x;
    const int32_t s = a.src[i], d = a.dst[i];
    if (s < 0 || s >= a.num_blocks || d < 0 || d >= a.num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(&g_append_error, kErrCopy);
        return;
    }
    char* pool = static_cast<char*>(blockIdx.y ? a.vpool : a.kpool);
    const uint4* src = reinterpret_cast<const uint4*>(pool + static_cast<int64_t>(s) * a.block_bytes);
    uint4* dst = reinterpret_cast<uint4*>(pool + static_cast<int64_t>(d) * a.block_bytes);
    const int64_t nvec = a.block_bytes / 16;
    for (int64_t base = 0; base < nvec; base += kVec * blockDim.x) {
        uint4 w[kVec];
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
            const int64_t v = base + k * blockDim.x + threadIdx.x;
            if (v < nvec) w[k] = src[v];
        }
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
            const int64_t v = base + k * blockDim.x + threadIdx.x;
            if (v < nvec) dst[v] = w[k];
        }
    }
}

}  // namespace

cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t stream) {
    if (a.n == 0) return cudaSuccess;
    dim3 grid(a.n, 2);
    copy_blocks_kernel<<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    const int per_seq = 2 * a.Hkv * (a.D * a.elem_bytes / 16);  // 16-byte vectors
    const int threads = per_seq >= 256 ? 256 : ((per_seq + 31) / 32) * 32;
    const int groups = (per_seq + threads - 1) / threads;
    if (groups > 65535) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.B, groups);
    cfg.blockDim = dim3(threads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, append_kernel, a);
}

cudaError_t read_append_error(int* err) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_append_error, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_append_error, &zero, sizeof(int));
    *err = v;
    return e;
}

}  // namespace pa

namespace pa {
cudaError_t append_error_address(int** p) {
    return cudaGetSymbolAddress(reinterpret_cast<void**>(p), g_append_error);
}
}  // namespace pa
