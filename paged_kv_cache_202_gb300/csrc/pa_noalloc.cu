// pa_decode_noalloc: the split paged decode with a fixed, library-owned
// scratch area instead of a plan workspace, for callers that must not have a
// library allocate device memory.
//
// Some callers own every byte of device memory themselves: a serving engine
// that has reserved the HBM it does not need for weights as its KV block pool
// and budgets it exactly, or a plugin host that hands a kernel only its input
// and output tensors. A cudaMalloc inside such a call takes memory outside
// that budget, and cudaMalloc / cudaFree also synchronise the device, which
// stalls the caller's other streams. This entry point therefore allocates
// nothing: the split partials and metadata live in one file-scope device
// array of kNoAllocScratchBytes that every GPU loading this library holds
// until the process exits.
//
// Scratch rules. All calls share the one array and it keeps the last call's
// contents; everything a call reads from it is written earlier in the same
// call (the only word that must start at zero, the fallback error word, is
// cleared by each call). Calls whose kernels overlap on the GPU (different
// streams without ordering) race on the array: serialise them. A call whose
// dynamic-tail partials would not fit runs on static ranges alone, and if
// those do not fit either, on fewer blocks; only a call whose partials would
// not fit for one block returns PA_ERR_WORKSPACE, before any launch.
//
// Set-up. The device address of the array is looked up per device with
// cudaGetSymbolAddress, on the first call made while that device is current,
// and kept once the lookup succeeds (a failed lookup, say during a stream
// capture or before the device has a context, is retried by the next call);
// host code never passes the array's host-side name to a kernel. The array
// itself is reserved on a device when the library's device code is loaded
// there, which with lazy module loading (the CUDA default) can be that first
// call: make one warm-up call at start-up, before sizing the KV pool from the
// free memory and before any stream capture.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

#include "pa.h"
#include "pa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

}  // namespace

// The shared scratch array (16 MiB on every device that loads the library).
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

namespace {

struct DeviceScratch {
    std::mutex mu;
    void* ptr = nullptr;  // set once a lookup has succeeded
};
DeviceScratch g_scratch[kMaxDevices];

// Device address of the scratch array on device `dev` (the current device).
// Only a successful lookup is kept; a failed one is retried by the next call.
void* scratch_address(int dev, cudaError_t* status) {
    if (dev < 0 || dev >= kMaxDevices) {
        *status = cudaErrorInvalidDevice;
        return nullptr;
    }
    DeviceScratch& d = g_scratch[dev];
    std::lock_guard<std::mutex> lk(d.mu);
    *status = cudaSuccess;
    if (!d.ptr) {
        void* p = nullptr;
        *status = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (*status == cudaSuccess) d.ptr = p;
    }
    return d.ptr;
}

struct OccEntry {
    int dev, kind, D, BS, NT, warps;
    size_t smem;
    int blocks_per_sm;
};
std::mutex g_occ_mutex;
std::vector<OccEntry> g_occ;

int blocks_per_sm(int dev, const pa::SplitLaunch& L, cudaError_t* status) {
    {
        std::lock_guard<std::mutex> lk(g_occ_mutex);
        for (const OccEntry& o : g_occ)
            if (o.dev == dev && o.kind == L.kind && o.D == L.D && o.BS == L.BS && o.NT == L.NT &&
                o.warps == L.warps && o.smem == L.smem) {
                *status = cudaSuccess;
                return o.blocks_per_sm;
            }
    }
    const int n = pa::split_blocks_per_sm(L, status);
    if (*status == cudaSuccess && n > 0) {
        std::lock_guard<std::mutex> lk(g_occ_mutex);
        g_occ.push_back(OccEntry{dev, L.kind, L.D, L.BS, L.NT, L.warps, L.smem, n});
    }
    return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" pa_status pa_decode_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                       const int32_t* block_tables, int max_blocks,
                                       const int32_t* seq_lens, int B, int Hq, int Hkv, int D,
                                       int block_size, int num_blocks, int max_seq_len,
                                       float scale, pa_dtype kv_dtype, void* out,
                                       pa_dtype out_dtype, int* device_error,
                                       struct CUstream_st* stream_) {
    if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out) return PA_ERR_NULL;
    if (kv_dtype != PA_BF16 || (out_dtype != PA_F32 && out_dtype != PA_BF16)) return PA_ERR_DTYPE;
    if (block_size != 16 && block_size != 32) return PA_ERR_BLOCK_SIZE;
    if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || (D != 64 && D != 128) || num_blocks < 1 ||
        max_blocks < 1 || max_seq_len < 1 || !std::isfinite(scale) || B > pa::kMaxBatch)
        return PA_ERR_SHAPE;
    if (static_cast<int64_t>(num_blocks) * Hkv > INT32_MAX ||
        static_cast<int64_t>(max_blocks) * block_size > INT32_MAX ||
        static_cast<int64_t>(B) * Hq > pa::kMaxRows)
        return PA_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return PA_ERR_ALIGN;
    if (B == 0) return PA_OK;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

    // Same planning as pa_decode's automatic choice (the tensor-core tiles),
    // at the default block shape and dynamic tail.
    const int g = Hq / Hkv;
    pa::SplitShape sh;
    if (!pa::split_shape(pa::kSplitMma, 0, B, Hq, Hkv, D, block_size, max_blocks, max_seq_len,
                         &sh))
        return PA_ERR_SHAPE;

    int dev = 0, num_sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PA_ERR_CUDA;
    cudaError_t st;
    char* scratch = static_cast<char*>(scratch_address(dev, &st));
    if (!scratch) return PA_ERR_CUDA;

    pa::SplitLaunch L{sh.kind, D, block_size, sh.NT, sh.warps, 0, sh.smem};
    const int per_sm = blocks_per_sm(dev, L, &st);
    if (st != cudaSuccess || per_sm < 1) return PA_ERR_CUDA;
    // Scratch layout: fallback error word, then the workspace (metadata,
    // partial (m, l), partial sums). A dynamic tail adds partials; when they
    // do not fit, the call runs on static ranges alone, and when those do not
    // fit either, on as many blocks as the scratch holds partials for.
    const size_t err_bytes = 256;
    const int64_t out_rows = static_cast<int64_t>(B) * Hq;
    auto fits = [&](const pa::SplitGrid& g) {
        return err_bytes + g.workspace_bytes() <= kNoAllocScratchBytes;
    };
    pa::SplitGrid gr = pa::split_grid(sh, B, D, block_size, out_rows, num_sms, per_sm);
    if (!fits(gr)) gr = pa::split_grid(sh, B, D, block_size, out_rows, num_sms, per_sm, false);
    if (!fits(gr)) {
        // The largest grid whose static-range partials fit, found with the
        // planner itself: the workspace grows with the block count.
        int lo = 1, hi = gr.blocks;
        while (lo < hi) {
            const int mid = lo + (hi - lo + 1) / 2;
            if (fits(pa::split_grid(sh, B, D, block_size, out_rows, num_sms, per_sm, false, mid)))
                lo = mid;
            else
                hi = mid - 1;
        }
        gr = pa::split_grid(sh, B, D, block_size, out_rows, num_sms, per_sm, false, lo);
    }
    if (!fits(gr)) return PA_ERR_WORKSPACE;
    L.blocks = gr.blocks;
    int* err = reinterpret_cast<int*>(scratch);
    int* meta = reinterpret_cast<int*>(scratch + err_bytes);
    float* ml = reinterpret_cast<float*>(scratch + err_bytes + gr.meta_bytes);
    float* acc = reinterpret_cast<float*>(scratch + err_bytes + gr.meta_bytes + gr.ml_bytes);
    if (!device_error) {
        if (cudaMemsetAsync(err, 0, sizeof(int), stream) != cudaSuccess) return PA_ERR_CUDA;
        device_error = err;
    }
    // The split kernel's dynamic-piece counter must start at zero.
    if (cudaMemsetAsync(meta + 3, 0, sizeof(int), stream) != cudaSuccess) return PA_ERR_CUDA;

    CUtensorMap kmap, vmap;
    const int rows = num_blocks * Hkv;
    if (!pa::encode_pool_map(&kmap, k_pool, rows, D, block_size) ||
        !pa::encode_pool_map(&vmap, v_pool, rows, D, block_size))
        return PA_ERR_CUDA;

    pa::SplitArgs a{};
    a.q = static_cast<const uint16_t*>(q);
    a.tables = block_tables;
    a.seq_lens = seq_lens;
    a.out = out;
    a.ws_acc = acc;
    a.ws_ml = ml;
    a.ws_meta = meta;
    a.err = device_error;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.g = g;
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    a.max_seq_len = max_seq_len;
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    a.out_bf16 = out_dtype == PA_BF16;
    pa::set_split_plan(&a, sh, gr);
    a.probe_wait = pa::wait_probe();
    if (pa::launch_split(L, kmap, vmap, a, stream) != cudaSuccess) return PA_ERR_CUDA;
    pa::MergeArgs m{meta, acc, ml, out, B, Hq, g, sh.GS, sh.nslices, sh.U, D,
                    out_dtype == PA_BF16, gr.merge_wpr, B * Hq, nullptr};
    return pa::launch_merge(m, stream) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
