// rkv_abi.cu -- the C ABI: host-side validation, error reporting and dispatch.
//
// Validation follows the pages' pattern of rejecting bad geometry before any
// device work (trueno-gpu attention.rs: InvalidParameter on size mismatch and
// on pos >= max_seq_len; trustformers-core attention.rs: checked_len overflow
// checks and PitchedCopy::validate).  Nothing here allocates or synchronises.
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <initializer_list>

#include "rkv_internal.cuh"
#include "rkv_launch.h"

namespace rkv {

static thread_local char g_msg[512] = "";

rkv_status set_error(rkv_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

rkv_status check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return set_error(RKV_ERR_LAUNCH, "%s: %s", what, cudaGetErrorString(e));
    return RKV_OK;
}

// One flag word per device, in this module's device memory.
static __device__ unsigned int g_device_flags;

static unsigned int* device_flags_ptr() {
    constexpr int kMaxDevices = 64;
    static unsigned int* cached[kMaxDevices] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (!cached[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_flags) != cudaSuccess) return nullptr;
        cached[dev] = static_cast<unsigned int*>(p);
    }
    return cached[dev];
}

int sm_count() {
    constexpr int kMaxDevices = 64;
    static int cached[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

// ------------------------------------------------------------- validation
static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

static bool head_dim_supported(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

// Element count of a tensor with the given dims, false if it (or its byte size) overflows int64.
static bool elems(int64_t& out, std::initializer_list<int64_t> dims) {
    int64_t acc = 4;   // bytes per element: the byte size must fit as well
    for (int64_t d : dims) {
        if (d < 0) return false;
        if (d != 0 && acc > INT64_MAX / d) return false;
        acc *= d;
    }
    out = acc / 4;
    return true;
}

static rkv_status resolve_scale(float scale, int head_dim, float& out, const char* op) {
    if (!std::isfinite(scale) || scale < 0.0f)
        return set_error(RKV_ERR_INVALID_ARG,
                         "%s: scale must be finite and >= 0 (0 selects 1/sqrt(head_dim)), got %g", op,
                         (double)scale);
    out = scale == 0.0f ? 1.0f / std::sqrt((float)head_dim) : scale;
    return RKV_OK;
}

static rkv_status check_heads(int n_heads, int n_kv_heads, int head_dim, const char* op) {
    if (n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0)
        return set_error(RKV_ERR_INVALID_ARG,
                         "%s: n_heads, n_kv_heads and head_dim must be > 0 (got %d, %d, %d)", op, n_heads,
                         n_kv_heads, head_dim);
    if (n_heads % n_kv_heads != 0)
        return set_error(RKV_ERR_INVALID_ARG, "%s: n_heads (%d) must be a multiple of n_kv_heads (%d)", op,
                         n_heads, n_kv_heads);
    if (!head_dim_supported(head_dim))
        return set_error(RKV_ERR_UNSUPPORTED, "%s: head_dim %d not supported (16, 32, 64 or 128)", op,
                         head_dim);
    return RKV_OK;
}

}  // namespace rkv

using namespace rkv;

extern "C" {

int rkv_version(void) { return (0 << 16) | 1; }

const char* rkv_status_string(rkv_status s) {
    switch (s) {
        case RKV_OK: return "ok";
        case RKV_ERR_INVALID_ARG: return "invalid argument";
        case RKV_ERR_UNSUPPORTED: return "unsupported";
        case RKV_ERR_LAUNCH: return "CUDA launch or runtime error";
        case RKV_ERR_DEVICE: return "device-side condition";
    }
    return "unknown status";
}

const char* rkv_last_error(void) { return g_msg; }

rkv_status rkv_read_device_flags(unsigned int* flags, int clear, cudaStream_t stream) {
    g_msg[0] = 0;
    if (!flags) return set_error(RKV_ERR_INVALID_ARG, "rkv_read_device_flags: flags is NULL");
    unsigned int* dptr = device_flags_ptr();
    if (!dptr) return set_error(RKV_ERR_LAUNCH, "rkv_read_device_flags: no device flag word");
    cudaError_t e = cudaMemcpyAsync(flags, dptr, sizeof(unsigned int), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(dptr, 0, sizeof(unsigned int), stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return set_error(RKV_ERR_LAUNCH, "rkv_read_device_flags: %s", cudaGetErrorString(e));
    return RKV_OK;
}

// One warp waits, through the kernels' own bounded-wait helper, on a barrier whose first phase
// nothing completes.
__global__ void wait_check_kernel(uint64_t limit_ns, unsigned int* flags) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    (void)mbar_wait(smem_addr(&bar), 0u, &abort_flag, flags, limit_ns);
}

rkv_status rkv_check_wait_timeout(unsigned int limit_us, cudaStream_t stream) {
    g_msg[0] = 0;
    if (limit_us == 0u || limit_us > 1000000u)
        return set_error(RKV_ERR_INVALID_ARG, "rkv_check_wait_timeout: limit_us must be in [1, 1000000], got %u",
                         limit_us);
    unsigned int* flags = device_flags_ptr();
    if (!flags) return set_error(RKV_ERR_LAUNCH, "rkv_check_wait_timeout: no device flag word");
    wait_check_kernel<<<1, 32, 0, stream>>>((uint64_t)limit_us * 1000ull, flags);
    return check_launch("rkv_check_wait_timeout");
}

// Each element: ours = the prefill's operand rounding with the 13 bits the tensor core drops
// cleared; ref = the hardware conversion to TF32 with round-to-nearest, ties away.
__global__ void tf32_round_check_kernel(const uint32_t* __restrict__ x, uint32_t* __restrict__ ours,
                                        uint32_t* __restrict__ ref, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const uint32_t b = x[i];
        ours[i] = tf32_round_bits(b) & 0xFFFFE000u;
        uint32_t r;
        asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(__uint_as_float(b)));
        ref[i] = r;
    }
}

rkv_status rkv_check_tf32_round(const unsigned int* x, unsigned int* ours, unsigned int* ref, int n,
                                cudaStream_t stream) {
    const char* op = "rkv_check_tf32_round";
    g_msg[0] = 0;
    if (n < 0) return set_error(RKV_ERR_INVALID_ARG, "%s: n must be >= 0, got %d", op, n);
    if (n == 0) return RKV_OK;
    if (!x || !ours || !ref) return set_error(RKV_ERR_INVALID_ARG, "%s: x, ours and ref must be non-NULL", op);
    if (!aligned(x, 4) || !aligned(ours, 4) || !aligned(ref, 4))
        return set_error(RKV_ERR_INVALID_ARG, "%s: x, ours and ref must be 4-byte aligned", op);
    const int blocks = (int)(((int64_t)n + 255) / 256 < 4096 ? ((int64_t)n + 255) / 256 : 4096);
    tf32_round_check_kernel<<<blocks, 256, 0, stream>>>(x, ours, ref, n);
    return check_launch(op);
}

rkv_status attn_prefill(const float* q, const float* k, const float* v, float* o, int batch, int seq_len,
                        int n_heads, int n_kv_heads, int head_dim, int causal, const int* seq_lens,
                        float scale, cudaStream_t stream) {
    const char* op = "attn_prefill";
    g_msg[0] = 0;
    if (batch < 0 || seq_len < 0)
        return set_error(RKV_ERR_INVALID_ARG, "%s: batch (%d) and seq_len (%d) must be >= 0", op, batch,
                         seq_len);
    rkv_status st = check_heads(n_heads, n_kv_heads, head_dim, op);
    if (st != RKV_OK) return st;
    float sc;
    if ((st = resolve_scale(scale, head_dim, sc, op)) != RKV_OK) return st;
    if (batch == 0 || seq_len == 0) return RKV_OK;
    if (!q || !k || !v || !o) return set_error(RKV_ERR_INVALID_ARG, "%s: q, k, v and o must be non-NULL", op);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(seq_lens, 4))
        return set_error(RKV_ERR_INVALID_ARG, "%s: q, k, v and o must be 16-byte aligned", op);
    int64_t nq, nkv;
    if (!elems(nq, {batch, seq_len, n_heads, head_dim}) || !elems(nkv, {batch, seq_len, n_kv_heads, head_dim}))
        return set_error(RKV_ERR_INVALID_ARG, "%s: tensor sizes overflow int64", op);
    // Tensor-copy descriptor limits: strides below 2^40 bytes, grid.y (batch*heads) below 2^16.
    if ((int64_t)seq_len * n_kv_heads * head_dim * 4 >= (int64_t(1) << 40) ||
        (int64_t)batch * n_heads > 65535)
        return set_error(RKV_ERR_UNSUPPORTED, "%s: batch*n_heads (%lld) or row stride beyond the kernel's limits",
                         op, (long long)batch * n_heads);
    if ((const void*)o == (const void*)q || (const void*)o == (const void*)k || (const void*)o == (const void*)v)
        return set_error(RKV_ERR_INVALID_ARG, "%s: o must not alias q, k or v", op);
    PrefillArgs a{q, k, v, o, batch, seq_len, n_heads, n_kv_heads, head_dim, causal != 0, seq_lens, sc,
                  device_flags_ptr(), op, false, 0, nullptr, nullptr, nullptr, 0};
    if (!a.flags) return set_error(RKV_ERR_LAUNCH, "%s: device flag word unavailable", op);
    return launch_prefill(a, stream);
}

rkv_status attn_prefill_fill_cache(const float* q, const float* k, const float* v, float* o, int batch,
                                   int seq_len, int n_heads, int n_kv_heads, int head_dim, int causal, float scale,
                                   float* k_cache, float* v_cache, int max_len, cudaStream_t stream) {
    const char* op = "attn_prefill_fill_cache";
    g_msg[0] = 0;
    if (batch < 0 || batch > kDecodeMaxSeqs)
        return set_error(RKV_ERR_INVALID_ARG, "%s: batch must be in [0, %d], got %d", op, kDecodeMaxSeqs, batch);
    if (seq_len < 0) return set_error(RKV_ERR_INVALID_ARG, "%s: seq_len must be >= 0, got %d", op, seq_len);
    rkv_status st = check_heads(n_heads, n_kv_heads, head_dim, op);
    if (st != RKV_OK) return st;
    if (max_len <= 0) return set_error(RKV_ERR_INVALID_ARG, "%s: max_len must be > 0, got %d", op, max_len);
    if (seq_len > max_len)
        return set_error(RKV_ERR_INVALID_ARG, "%s: seq_len (%d) exceeds max_len (%d)", op, seq_len, max_len);
    float sc;
    if ((st = resolve_scale(scale, head_dim, sc, op)) != RKV_OK) return st;
    if (batch == 0 || seq_len == 0) return RKV_OK;
    if (!q || !k || !v || !o || !k_cache || !v_cache)
        return set_error(RKV_ERR_INVALID_ARG, "%s: q, k, v, o and the caches must be non-NULL", op);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16))
        return set_error(RKV_ERR_INVALID_ARG, "%s: q, k, v, o and the caches must be 16-byte aligned", op);
    int64_t nq, nkv, nc;
    if (!elems(nq, {batch, seq_len, n_heads, head_dim}) || !elems(nkv, {batch, seq_len, n_kv_heads, head_dim}) ||
        !elems(nc, {batch, n_kv_heads, max_len, head_dim}))
        return set_error(RKV_ERR_INVALID_ARG, "%s: tensor sizes overflow int64", op);
    if ((int64_t)seq_len * n_kv_heads * head_dim * 4 >= (int64_t(1) << 40) ||
        (int64_t)max_len * head_dim * 4 >= (int64_t(1) << 40))
        return set_error(RKV_ERR_UNSUPPORTED, "%s: row stride beyond the kernel's limits", op);
    const void* outs[3] = {o, k_cache, v_cache};
    const void* ins[3] = {q, k, v};
    for (const void* w : outs)
        for (const void* r : ins)
            if (w == r) return set_error(RKV_ERR_INVALID_ARG, "%s: o and the caches must not alias q, k or v", op);
    if ((const void*)o == (const void*)k_cache || (const void*)o == (const void*)v_cache || k_cache == v_cache)
        return set_error(RKV_ERR_INVALID_ARG, "%s: o, k_cache and v_cache must be distinct", op);
    PrefillArgs a{q, k, v, o, batch, seq_len, n_heads, n_kv_heads, head_dim, causal != 0, nullptr, sc,
                  device_flags_ptr(), op, false, 0, nullptr, k_cache, v_cache, max_len};
    if (!a.flags) return set_error(RKV_ERR_LAUNCH, "%s: device flag word unavailable", op);
    return launch_prefill(a, stream);
}

rkv_status attn_prefill_chunked(const float* q, const float* k_cache, const float* v_cache, float* o, int M,
                                int T, int n_heads, int n_kv_heads, int head_dim, int max_len, int causal,
                                const int* start_pos, const int* q_lens, float scale, cudaStream_t stream) {
    const char* op = "attn_prefill_chunked";
    g_msg[0] = 0;
    if (M < 0 || M > kDecodeMaxSeqs)
        return set_error(RKV_ERR_INVALID_ARG, "%s: M must be in [0, %d], got %d", op, kDecodeMaxSeqs, M);
    if (T < 0) return set_error(RKV_ERR_INVALID_ARG, "%s: T must be >= 0, got %d", op, T);
    rkv_status st = check_heads(n_heads, n_kv_heads, head_dim, op);
    if (st != RKV_OK) return st;
    if (max_len <= 0) return set_error(RKV_ERR_INVALID_ARG, "%s: max_len must be > 0, got %d", op, max_len);
    if (T > max_len) return set_error(RKV_ERR_INVALID_ARG, "%s: T (%d) exceeds max_len (%d)", op, T, max_len);
    float sc;
    if ((st = resolve_scale(scale, head_dim, sc, op)) != RKV_OK) return st;
    if (M == 0 || T == 0) return RKV_OK;
    if (!q || !k_cache || !v_cache || !o || !start_pos)
        return set_error(RKV_ERR_INVALID_ARG, "%s: q, caches, o and start_pos must be non-NULL", op);
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) ||
        !aligned(start_pos, 4) || !aligned(q_lens, 4))
        return set_error(RKV_ERR_INVALID_ARG, "%s: q, caches and o must be 16-byte aligned", op);
    int64_t nq, nc;
    if (!elems(nq, {M, T, n_heads, head_dim}) || !elems(nc, {M, n_kv_heads, max_len, head_dim}))
        return set_error(RKV_ERR_INVALID_ARG, "%s: tensor sizes overflow int64", op);
    if ((int64_t)max_len * head_dim * 4 >= (int64_t(1) << 40))
        return set_error(RKV_ERR_UNSUPPORTED, "%s: cache stride beyond the kernel's limits", op);
    if ((const void*)o == (const void*)q || (const void*)o == (const void*)k_cache ||
        (const void*)o == (const void*)v_cache)
        return set_error(RKV_ERR_INVALID_ARG, "%s: o must not alias q or the caches", op);
    PrefillArgs a{q, k_cache, v_cache, o, M, T, n_heads, n_kv_heads, head_dim, causal != 0, q_lens, sc,
                  device_flags_ptr(), op, true, max_len, start_pos, nullptr, nullptr, 0};
    if (!a.flags) return set_error(RKV_ERR_LAUNCH, "%s: device flag word unavailable", op);
    return launch_prefill(a, stream);
}

size_t attn_decode_workspace_bytes(int M, int n_heads, int n_kv_heads, int head_dim, int max_len) {
    if (M <= 0 || M > kDecodeMaxSeqs || n_heads <= 0 || n_kv_heads <= 0 || max_len <= 0 ||
        n_heads % n_kv_heads != 0 || !head_dim_supported(head_dim) || (int64_t)M * n_kv_heads > kDecodeTicketSlots)
        return 0;
    return decode_workspace_bytes(M, n_heads, n_kv_heads, head_dim);
}

// Batched decode over either the batched cache (k_cache/v_cache) or per-sequence caches
// (k_ptrs/v_ptrs, device arrays of M pointers).
static rkv_status decode_entry(const char* op, const float* q, const float* k_cache, const float* v_cache,
                               const float* const* k_ptrs, const float* const* v_ptrs, float* o, int M, int n_heads,
                               int n_kv_heads, int head_dim, int max_len, const int* seq_lens, float scale,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream,
                               const float* k_new = nullptr, const float* v_new = nullptr) {
    g_msg[0] = 0;
    if (M < 0 || M > kDecodeMaxSeqs)
        return set_error(RKV_ERR_INVALID_ARG, "%s: M must be in [0, %d], got %d", op, kDecodeMaxSeqs, M);
    rkv_status st = check_heads(n_heads, n_kv_heads, head_dim, op);
    if (st != RKV_OK) return st;
    if (max_len <= 0) return set_error(RKV_ERR_INVALID_ARG, "%s: max_len must be > 0, got %d", op, max_len);
    float sc;
    if ((st = resolve_scale(scale, head_dim, sc, op)) != RKV_OK) return st;
    if (M == 0) return RKV_OK;
    if (!decode_group_supported(n_heads / n_kv_heads))
        return set_error(RKV_ERR_UNSUPPORTED, "%s: n_heads/n_kv_heads = %d not supported (1, 2, 4 or 8)", op,
                         n_heads / n_kv_heads);
    if ((int64_t)M * n_kv_heads > kDecodeTicketSlots)
        return set_error(RKV_ERR_UNSUPPORTED, "%s: M * n_kv_heads = %lld exceeds the %d workspace tickets", op,
                         (long long)M * n_kv_heads, kDecodeTicketSlots);
    const bool ptrs = k_ptrs || v_ptrs;
    if (!q || !o || !seq_lens || !workspace || (ptrs ? (!k_ptrs || !v_ptrs) : (!k_cache || !v_cache)))
        return set_error(RKV_ERR_INVALID_ARG, "%s: q, caches, o, seq_lens and workspace must be non-NULL", op);
    if (!aligned(q, 16) || !aligned(o, 16) || !aligned(workspace, 256) || !aligned(seq_lens, 4) ||
        (ptrs ? (!aligned(k_ptrs, 8) || !aligned(v_ptrs, 8)) : (!aligned(k_cache, 16) || !aligned(v_cache, 16))))
        return set_error(RKV_ERR_INVALID_ARG,
                         "%s: q, caches and o must be 16-byte aligned, workspace 256-byte aligned", op);
    int64_t nc;
    if (!elems(nc, {M, n_kv_heads, max_len, head_dim}))
        return set_error(RKV_ERR_INVALID_ARG, "%s: cache size overflows int64", op);
    const size_t need = decode_workspace_bytes(M, n_heads, n_kv_heads, head_dim);
    if (workspace_bytes < need)
        return set_error(RKV_ERR_INVALID_ARG, "%s: workspace of %zu bytes is below the %zu required", op,
                         workspace_bytes, need);
    DecodeArgs a{q, k_cache, v_cache, o, M, n_heads, n_kv_heads, head_dim, max_len, seq_lens, sc,
                 workspace, device_flags_ptr(), k_ptrs, v_ptrs, k_new, v_new};
    if (!a.flags) return set_error(RKV_ERR_LAUNCH, "%s: device flag word unavailable", op);
    return launch_decode(a, stream);
}

rkv_status attn_decode_batched(const float* q, const float* k_cache, const float* v_cache, float* o, int M,
                               int n_heads, int n_kv_heads, int head_dim, int max_len, const int* seq_lens,
                               float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return decode_entry("attn_decode_batched", q, k_cache, v_cache, nullptr, nullptr, o, M, n_heads, n_kv_heads,
                        head_dim, max_len, seq_lens, scale, workspace, workspace_bytes, stream);
}

rkv_status attn_decode_append(const float* q, const float* k_new, const float* v_new, float* k_cache, float* v_cache,
                              float* o, int M, int n_heads, int n_kv_heads, int head_dim, int max_len,
                              const int* seq_lens, float scale, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
    const char* op = "attn_decode_append";
    if (M > 0 && M <= kDecodeMaxSeqs) {
        g_msg[0] = 0;
        if (!k_new || !v_new)
            return set_error(RKV_ERR_INVALID_ARG, "%s: k_new and v_new must be non-NULL", op);
        if (!aligned(k_new, 16) || !aligned(v_new, 16))
            return set_error(RKV_ERR_INVALID_ARG, "%s: k_new and v_new must be 16-byte aligned", op);
        const void* ins[3] = {q, k_new, v_new};
        for (const void* w : {(const void*)k_cache, (const void*)v_cache, (const void*)o})
            for (const void* r : ins)
                if (w && w == r) return set_error(RKV_ERR_INVALID_ARG, "%s: outputs must not alias the inputs", op);
        if (k_cache && k_cache == v_cache)
            return set_error(RKV_ERR_INVALID_ARG, "%s: k_cache and v_cache must be distinct", op);
    }
    return decode_entry(op, q, k_cache, v_cache, nullptr, nullptr, o, M, n_heads, n_kv_heads, head_dim, max_len,
                        seq_lens, scale, workspace, workspace_bytes, stream, k_new, v_new);
}

rkv_status attn_decode_batched_ptrs(const float* q, const float* const* k_ptrs, const float* const* v_ptrs, float* o,
                                    int M, int n_heads, int n_kv_heads, int head_dim, int max_len,
                                    const int* seq_lens, float scale, void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream) {
    return decode_entry("attn_decode_batched_ptrs", q, nullptr, nullptr, k_ptrs, v_ptrs, o, M, n_heads, n_kv_heads,
                        head_dim, max_len, seq_lens, scale, workspace, workspace_bytes, stream);
}

rkv_status kv_append_rope(float* q, float* k_new, const float* v_new, float* k_cache, float* v_cache, int M, int T,
                          int n_heads, int n_kv_heads, int head_dim, int max_len, const int* start_pos,
                          int rotary_ndims, float theta, int* overflow, cudaStream_t stream) {
    const char* op = "kv_append_rope";
    g_msg[0] = 0;
    if (M < 0 || M > kDecodeMaxSeqs)
        return set_error(RKV_ERR_INVALID_ARG, "%s: M must be in [0, %d], got %d", op, kDecodeMaxSeqs, M);
    if (T < 0) return set_error(RKV_ERR_INVALID_ARG, "%s: T must be >= 0, got %d", op, T);
    rkv_status st = check_heads(n_heads, n_kv_heads, head_dim, op);
    if (st != RKV_OK) return st;
    if (max_len <= 0) return set_error(RKV_ERR_INVALID_ARG, "%s: max_len must be > 0, got %d", op, max_len);
    if (T > max_len) return set_error(RKV_ERR_INVALID_ARG, "%s: T (%d) exceeds max_len (%d)", op, T, max_len);
    if (rotary_ndims <= 0 || rotary_ndims > head_dim || rotary_ndims % 2 != 0)
        return set_error(RKV_ERR_INVALID_ARG, "%s: rotary_ndims must be even and in (0, head_dim], got %d", op,
                         rotary_ndims);
    if (rotary_ndims % 8 != 0)
        return set_error(RKV_ERR_UNSUPPORTED, "%s: rotary_ndims must be a multiple of 8, got %d", op, rotary_ndims);
    if (!std::isfinite(theta) || theta <= 0.0f)
        return set_error(RKV_ERR_INVALID_ARG, "%s: theta must be finite and > 0, got %g", op, (double)theta);
    if (M == 0 || T == 0) return RKV_OK;
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !start_pos)
        return set_error(RKV_ERR_INVALID_ARG, "%s: q, new rows, caches and start_pos must be non-NULL", op);
    if (!aligned(q, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(start_pos, 4) || !aligned(overflow, 4))
        return set_error(RKV_ERR_INVALID_ARG, "%s: rows and caches must be 16-byte aligned", op);
    int64_t nq, nn, nc;
    if (!elems(nq, {M, T, n_heads, head_dim}) || !elems(nn, {M, T, n_kv_heads, head_dim}) ||
        !elems(nc, {M, n_kv_heads, max_len, head_dim}))
        return set_error(RKV_ERR_INVALID_ARG, "%s: tensor sizes overflow int64", op);
    const void* bufs[5] = {q, k_new, v_new, k_cache, v_cache};
    for (int i = 0; i < 5; ++i)
        for (int j = i + 1; j < 5; ++j)
            if (bufs[i] == bufs[j]) return set_error(RKV_ERR_INVALID_ARG, "%s: the five tensors must be distinct", op);
    unsigned int* flags = device_flags_ptr();
    if (!flags) return set_error(RKV_ERR_LAUNCH, "%s: device flag word unavailable", op);
    return launch_rope_append(q, k_new, v_new, k_cache, v_cache, M, T, n_heads, n_kv_heads, head_dim, max_len,
                              start_pos, rotary_ndims, (double)theta, overflow, flags, stream);
}

// Append into either the batched cache or per-sequence caches (k_ptrs/v_ptrs, device arrays).
static rkv_status scatter_entry(const char* op, const float* k_new, const float* v_new, float* k_cache,
                                float* v_cache, float* const* k_ptrs, float* const* v_ptrs, int M, int T,
                                int n_kv_heads, int head_dim, int max_len, const int* start_pos, int* overflow,
                                cudaStream_t stream) {
    g_msg[0] = 0;
    if (M < 0 || M > kDecodeMaxSeqs)
        return set_error(RKV_ERR_INVALID_ARG, "%s: M must be in [0, %d], got %d", op, kDecodeMaxSeqs, M);
    if (T < 0) return set_error(RKV_ERR_INVALID_ARG, "%s: T must be >= 0, got %d", op, T);
    if (n_kv_heads <= 0 || max_len <= 0)
        return set_error(RKV_ERR_INVALID_ARG, "%s: n_kv_heads and max_len must be > 0", op);
    if (!head_dim_supported(head_dim))
        return set_error(RKV_ERR_UNSUPPORTED, "%s: head_dim %d not supported (16, 32, 64 or 128)", op,
                         head_dim);
    if (T > max_len) return set_error(RKV_ERR_INVALID_ARG, "%s: T (%d) exceeds max_len (%d)", op, T, max_len);
    if (M == 0 || T == 0) return RKV_OK;
    const bool ptrs = k_ptrs || v_ptrs;
    if (!k_new || !v_new || !start_pos || (ptrs ? (!k_ptrs || !v_ptrs) : (!k_cache || !v_cache)))
        return set_error(RKV_ERR_INVALID_ARG, "%s: new rows, caches and start_pos must be non-NULL", op);
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(start_pos, 4) || !aligned(overflow, 4) ||
        (ptrs ? (!aligned(k_ptrs, 8) || !aligned(v_ptrs, 8)) : (!aligned(k_cache, 16) || !aligned(v_cache, 16))))
        return set_error(RKV_ERR_INVALID_ARG, "%s: rows and caches must be 16-byte aligned", op);
    int64_t nn, nc;
    if (!elems(nn, {M, T, n_kv_heads, head_dim}) || !elems(nc, {M, n_kv_heads, max_len, head_dim}))
        return set_error(RKV_ERR_INVALID_ARG, "%s: tensor sizes overflow int64", op);
    unsigned int* flags = device_flags_ptr();
    if (!flags) return set_error(RKV_ERR_LAUNCH, "%s: device flag word unavailable", op);
    return launch_scatter(k_new, v_new, k_cache, v_cache, M, T, n_kv_heads, head_dim, max_len, start_pos,
                          overflow, flags, stream, k_ptrs, v_ptrs);
}

rkv_status kv_cache_scatter(const float* k_new, const float* v_new, float* k_cache, float* v_cache, int M,
                            int T, int n_kv_heads, int head_dim, int max_len, const int* start_pos,
                            int* overflow, cudaStream_t stream) {
    return scatter_entry("kv_cache_scatter", k_new, v_new, k_cache, v_cache, nullptr, nullptr, M, T, n_kv_heads,
                         head_dim, max_len, start_pos, overflow, stream);
}

rkv_status kv_cache_scatter_ptrs(const float* k_new, const float* v_new, float* const* k_ptrs, float* const* v_ptrs,
                                 int M, int T, int n_kv_heads, int head_dim, int max_len, const int* start_pos,
                                 int* overflow, cudaStream_t stream) {
    return scatter_entry("kv_cache_scatter_ptrs", k_new, v_new, nullptr, nullptr, k_ptrs, v_ptrs, M, T, n_kv_heads,
                         head_dim, max_len, start_pos, overflow, stream);
}

}  // extern "C"
