// decode_noalloc.cu -- batched decode for callers that cannot allocate device memory.
//
// attn_decode_batched needs a caller-provided workspace.  Some callers cannot
// call cudaMalloc (or any allocator) at the point where they decode: code that
// runs inside a framework's memory arena without access to it, plugin hosts
// that forbid allocation after start-up, or real-time loops that must never
// block in the allocator.  attn_decode_batched_noalloc serves them: it runs
// the same split-KV decode, with its scratch taken from a fixed array in this
// library's own device memory instead of a caller buffer.
//
// The array lives as long as the library is loaded, on every GPU that loads
// it.  Its device address is looked up on the first call made with a device
// current, and again whenever that device's context has changed since (for
// instance after cudaDeviceReset); make that first call before any stream
// capture.  Every call shares the one array: calls that overlap on the GPU
// (two streams, or two host threads on one device) race on it and give wrong
// results.
#include <cuda.h>

#include <cstdint>
#include <mutex>

#include "rkv_internal.cuh"
#include "rkv_launch.h"

namespace rkv {

// Largest workspace the allocation-free entry point can serve (4 MiB).
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Unique id of the current context (0 if none or unknown).  Ids are never reused within a
// process, unlike context handles, so a context created after a reset never matches an old entry.
static unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_decode_scratch for the current device (nullptr on failure), cached
// per device together with the id of the context it was resolved in.
static void* scratch_device_address(cudaError_t* err) {
    constexpr int kMaxDevices = 64;
    struct Entry {
        unsigned long long ctx_id;
        void* ptr;
    };
    static Entry cached[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = current_context_id();
    if (id != 0 && cached[dev].ptr && cached[dev].ctx_id == id) {
        *err = cudaSuccess;
        return cached[dev].ptr;
    }
    void* p = nullptr;   // resolving also makes the device's primary context current
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) {
        *err = e;
        return nullptr;
    }
    cached[dev] = Entry{current_context_id(), p};
    *err = cudaSuccess;
    return p;
}

}  // namespace rkv

using namespace rkv;

extern "C" rkv_status attn_decode_batched_noalloc(const float* q, const float* k_cache, const float* v_cache,
                                                  float* o, int M, int n_heads, int n_kv_heads, int head_dim,
                                                  int max_len, const int* seq_lens, float scale,
                                                  cudaStream_t stream) {
    const char* op = "attn_decode_batched_noalloc";
    if (M == 0) return attn_decode_batched(q, k_cache, v_cache, o, M, n_heads, n_kv_heads, head_dim, max_len,
                                           seq_lens, scale, nullptr, 0, stream);
    const size_t need = attn_decode_workspace_bytes(M, n_heads, n_kv_heads, head_dim, max_len);
    if (need == 0)   // invalid sizes: let the regular entry point produce its precise message
        return attn_decode_batched(q, k_cache, v_cache, o, M, n_heads, n_kv_heads, head_dim, max_len, seq_lens,
                                   scale, nullptr, 0, stream);
    if (need > kNoAllocScratchBytes)
        return set_error(RKV_ERR_UNSUPPORTED,
                         "%s: these sizes need %zu bytes of scratch but the built-in array holds %zu; "
                         "use attn_decode_batched with a caller workspace",
                         op, need, kNoAllocScratchBytes);
    cudaError_t e;
    void* scratch = scratch_device_address(&e);
    if (!scratch)
        return set_error(RKV_ERR_LAUNCH, "%s: cannot resolve the scratch array's device address: %s", op,
                         cudaGetErrorString(e));
    // The completion tickets at the head of the workspace must start at zero.  The kernel
    // leaves them zero, but a call that stopped early would not, so clear them every time.
    const size_t ticket_bytes = ((size_t)M * n_kv_heads * 4 + 255) / 256 * 256;
    e = cudaMemsetAsync(scratch, 0, ticket_bytes, stream);
    if (e != cudaSuccess)
        return set_error(RKV_ERR_LAUNCH, "%s: clearing the scratch tickets failed: %s", op, cudaGetErrorString(e));
    return attn_decode_batched(q, k_cache, v_cache, o, M, n_heads, n_kv_heads, head_dim, max_len, seq_lens,
                               scale, scratch, kNoAllocScratchBytes, stream);
}
