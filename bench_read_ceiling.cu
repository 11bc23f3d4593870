// Read-only HBM ceiling of one GPU, for the decode kernel's roofline context.
//
// The decode step only reads the KV pools (a few MB of partials aside), while
// the copy peak it is quoted against moves half its bytes as writes. This
// program times, over the same number of bytes as one decode of the
// Llama-3-8B GQA workload (2.2 GB), three ways of moving them:
//   - a device-to-device copy (read + write bytes counted, like the copy peak),
//   - a grid-stride streaming read of 16-byte vectors (no writes),
//   - whole 4 KB pages read in a random permutation, one page per warp, the
//     access pattern of a paged pool whose pages sit anywhere in memory.
// Each variant: 3 untimed launches, then `reps` launches timed one by one with
// CUDA events; one JSON line with the median and best of each goes to stdout.
// Every load stays inside the buffer: the streaming loop only issues a batch
// whose last address is below the end, and a page load's index is below
// (page + 1) * 256 sixteen-byte vectors with page < pages.
//
// Usage: read_ceiling [pages (default 538112 = 2.204 GB)] [reps (default 30)]
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <random>
#include <string>
#include <vector>

#define CK(x)                                                                              \
    do {                                                                                   \
        cudaError_t e_ = (x);                                                              \
        if (e_ != cudaSuccess) {                                                           \
            fprintf(stderr, "CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
            exit(1);                                                                       \
        }                                                                                  \
    } while (0)

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// The loaded words are folded into one value that is compared with a
// constant, so no load can be dropped; the sink is written only on a match.
template <int UNR>
__global__ void stream_read(const uint4* __restrict__ p, size_t n16, unsigned long long* sink) {
    uint32_t acc = 0;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + (UNR - 1) * stride < n16; i += UNR * stride) {
        uint4 v[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) v[u] = ld_stream(p + i + u * stride);
#pragma unroll
        for (int u = 0; u < UNR; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    for (; i < n16; i += stride) {
        const uint4 v = ld_stream(p + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    if (acc == 0x9e3779b9u) atomicAdd(sink, 1ull);
}

__global__ void page_read(const uint4* __restrict__ p, const int* __restrict__ perm, int pages,
                          unsigned long long* sink) {
    uint32_t acc = 0;
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int i = warp; i < pages; i += warps) {
        const uint4* page = p + static_cast<size_t>(perm[i]) * 256;
        uint4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = ld_stream(page + k * 32 + lane);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
    }
    if (acc == 0x9e3779b9u) atomicAdd(sink, 1ull);
}

struct Result {
    std::string name;
    double bytes, med_us, best_us;
};

template <class F>
static Result timeit(const char* name, double bytes, int reps, F launch) {
    cudaEvent_t a, b;
    CK(cudaEventCreate(&a));
    CK(cudaEventCreate(&b));
    for (int i = 0; i < 3; ++i) launch();
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
    std::vector<float> ms;
    for (int r = 0; r < reps; ++r) {
        CK(cudaEventRecord(a));
        launch();
        CK(cudaEventRecord(b));
        CK(cudaEventSynchronize(b));
        float t;
        CK(cudaEventElapsedTime(&t, a, b));
        ms.push_back(t);
    }
    CK(cudaGetLastError());
    std::sort(ms.begin(), ms.end());
    CK(cudaEventDestroy(a));
    CK(cudaEventDestroy(b));
    return {name, bytes, ms[reps / 2] * 1e3, ms[0] * 1e3};
}

int main(int argc, char** argv) {
    const int pages = argc > 1 ? atoi(argv[1]) : 538112;
    const int reps = argc > 2 ? std::max(3, atoi(argv[2])) : 30;
    if (pages <= 0) return 2;
    const size_t bytes = static_cast<size_t>(pages) * 4096;
    const size_t n16 = bytes / 16;
    uint4 *src, *dst;
    unsigned long long* sink;
    int* dperm;
    CK(cudaMalloc(&src, bytes));
    CK(cudaMalloc(&dst, bytes));
    CK(cudaMalloc(&sink, 8));
    CK(cudaMalloc(&dperm, pages * sizeof(int)));
    CK(cudaMemset(src, 0x5a, bytes));
    CK(cudaMemset(sink, 0, 8));
    std::vector<int> perm(pages);
    for (int i = 0; i < pages; ++i) perm[i] = i;
    std::mt19937 rng(7);
    std::shuffle(perm.begin(), perm.end(), rng);
    CK(cudaMemcpy(dperm, perm.data(), pages * sizeof(int), cudaMemcpyHostToDevice));
    int sms;
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));

    std::vector<Result> res;
    res.push_back(timeit("copy_d2d", 2.0 * bytes, reps, [&] {
        CK(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice));
    }));
    const int shapes[][2] = {{2, 512}, {4, 256}, {8, 256}};
    for (const auto& s : shapes) {
        const std::string nm = "stream_" + std::to_string(s[0]) + "x" + std::to_string(s[1]);
        res.push_back(timeit(nm.c_str(), static_cast<double>(bytes), reps, [&] {
            stream_read<8><<<s[0] * sms, s[1]>>>(src, n16, sink);
        }));
    }
    const int pshapes[][2] = {{4, 512}, {8, 256}};
    for (const auto& s : pshapes) {
        const std::string nm = "pages_" + std::to_string(s[0]) + "x" + std::to_string(s[1]);
        res.push_back(timeit(nm.c_str(), static_cast<double>(bytes), reps, [&] {
            page_read<<<s[0] * sms, s[1]>>>(src, dperm, pages, sink);
        }));
    }
    CK(cudaDeviceSynchronize());

    printf("{\"bytes\": %zu, \"sms\": %d, \"reps\": %d, \"results\": [", bytes, sms, reps);
    for (size_t i = 0; i < res.size(); ++i) {
        const Result& r = res[i];
        printf("%s{\"name\": \"%s\", \"bytes\": %.0f, \"median_us\": %.2f, \"best_us\": %.2f, "
               "\"median_gbs\": %.1f, \"best_gbs\": %.1f}",
               i ? ", " : "", r.name.c_str(), r.bytes, r.med_us, r.best_us,
               r.bytes / (r.med_us * 1e3), r.bytes / (r.best_us * 1e3));
    }
    printf("]}\n");
    CK(cudaFree(src));
    CK(cudaFree(dst));
    CK(cudaFree(sink));
    CK(cudaFree(dperm));
    return 0;
}
