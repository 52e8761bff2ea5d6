// kv_scatter.cu -- append new K/V rows into the resident batched cache.
//
//   cache[m, kh, start_pos[m] + t, :] = new[m, t, kh*D : (kh+1)*D]
//
// trueno-gpu 0.4.11, src/memory/resident/attention.rs, fn kv_cache_scatter_gpu
// writes one interleaved [n_heads*head_dim] row into a head-first cache with one
// block per head and one thread per element.  Here one launch covers every
// sequence, token, kv head, and both K and V: grid.y = sequence, grid.x = chunks
// of tokens, 16-byte vector loads/stores, and positions come from device memory
// so the bounds check moves on chip (skipped tokens are counted).
#include "rkv_internal.cuh"
#include "rkv_launch.h"

namespace rkv {

constexpr int kScatterThreads = 256;
constexpr int kScatterElemsPerBlock = 2048;   // float4 elements per tensor per block

template <int D4>
__global__ void __launch_bounds__(kScatterThreads)
kv_scatter_kernel(const float4* __restrict__ k_new, const float4* __restrict__ v_new,
                  float4* __restrict__ k_cache, float4* __restrict__ v_cache, int T, int Hk, int Lmax,
                  int tokens_per_block, const int* __restrict__ start_pos, int* __restrict__ overflow,
                  unsigned int* __restrict__ flags, float* const* __restrict__ k_ptrs,
                  float* const* __restrict__ v_ptrs) {
    const int m = blockIdx.y;
    const int t0 = blockIdx.x * tokens_per_block;
    const int n_tok = min(tokens_per_block, T - t0);
    if (n_tok <= 0) return;
    const int p0 = __ldg(start_pos + m);
    const int row4 = Hk * D4;                         // float4 elements per token
    const int total = n_tok * row4;
    const int64_t src_base = ((int64_t)m * T + t0) * row4;
    // the sequence's cache: a slice of the batched cache, or its own allocation (pointer arrays);
    // a null or misaligned base is never written -- the sequence's tokens are skipped
    float4* kc = k_ptrs ? reinterpret_cast<float4*>(k_ptrs[m]) : k_cache + (int64_t)m * Hk * Lmax * D4;
    float4* vc = v_ptrs ? reinterpret_cast<float4*>(v_ptrs[m]) : v_cache + (int64_t)m * Hk * Lmax * D4;
    if (!kc || !vc || ((reinterpret_cast<uintptr_t>(kc) | reinterpret_cast<uintptr_t>(vc)) & 15u)) {
        if (threadIdx.x == 0) atomicOr(flags, RKV_FLAG_BAD_POINTER);
        return;
    }

    if (threadIdx.x < n_tok) {                        // per-token bounds accounting
        const int64_t pos = (int64_t)p0 + t0 + threadIdx.x;
        if (pos < 0 || pos >= Lmax) {
            if (overflow) atomicAdd(overflow, 1);
            if (p0 < 0) atomicOr(flags, RKV_FLAG_NEGATIVE_INPUT);
        }
    }

#pragma unroll 4
    for (int idx = threadIdx.x; idx < total; idx += kScatterThreads) {
        const int j = idx / row4;                     // token within the block
        const int rem = idx - j * row4;
        const int kh = rem / D4;
        const int d4 = rem - kh * D4;
        const int64_t pos = (int64_t)p0 + t0 + j;
        if (pos < 0 || pos >= Lmax) continue;
        const int64_t dst = ((int64_t)kh * Lmax + pos) * D4 + d4;
        if (!in_bounds(src_base + idx, (int64_t)gridDim.y * T * row4, flags) ||
            !in_bounds(dst, (int64_t)Hk * Lmax * D4, flags))
            continue;
        const float4 kv = __ldcs(k_new + src_base + idx);
        const float4 vv = __ldcs(v_new + src_base + idx);
        __stcs(kc + dst, kv);          // streaming stores: the cache is far larger than L2
        __stcs(vc + dst, vv);
    }
}

// Cache fill of whole sequences at positions 0..S-1, one persistent CTA per SM (grid-stride over
// every float4 of K and V).  It is launched as a programmatic dependent of the prefill: its CTAs
// start beside the prefill's (256 threads and a few registers fit in what a prefill CTA leaves
// free), read the same inputs the prefill reads and write rows nothing else touches; the final
// griddepcontrol.wait keeps it from completing before the prefill, so later work in the stream
// is ordered after both.
template <int D4>
__global__ void __launch_bounds__(kScatterThreads)
kv_fill_kernel(const float4* __restrict__ k, const float4* __restrict__ v, float4* __restrict__ k_cache,
               float4* __restrict__ v_cache, int S, int Hk, int Lmax, int64_t total, unsigned int* __restrict__ flags) {
    const int row4 = Hk * D4;                         // float4 elements per token
#pragma unroll 4
    for (int64_t idx = (int64_t)blockIdx.x * kScatterThreads + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * kScatterThreads) {
        const int64_t tok = idx / row4;               // b * S + t
        const int rem = (int)(idx - tok * row4);
        const int kh = rem / D4, d4 = rem - kh * D4;
        const int64_t b = tok / S, t = tok - b * S;
        const int64_t dst = ((b * Hk + kh) * Lmax + t) * D4 + d4;
        if (!in_bounds(dst, total / ((int64_t)S * row4) * Hk * Lmax * D4, flags)) continue;
        __stcs(k_cache + dst, __ldg(k + idx));
        __stcs(v_cache + dst, __ldg(v + idx));
    }
    griddep_wait();
}

rkv_status launch_fill_dependent(const float* k, const float* v, float* k_cache, float* v_cache, int B, int S,
                                 int Hk, int D, int Lmax, unsigned int* flags, cudaStream_t stream) {
    const int sms = sm_count();
    if (sms <= 0) return set_error(RKV_ERR_LAUNCH, "attn_prefill_fill_cache: cannot query the SM count");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sms);
    cfg.blockDim = dim3(kScatterThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int64_t total = (int64_t)B * S * Hk * (D / 4);
    auto k4 = reinterpret_cast<const float4*>(k);
    auto v4 = reinterpret_cast<const float4*>(v);
    auto kc = reinterpret_cast<float4*>(k_cache);
    auto vc = reinterpret_cast<float4*>(v_cache);
    cudaError_t e;
    switch (D) {
        case 16: e = cudaLaunchKernelEx(&cfg, kv_fill_kernel<4>, k4, v4, kc, vc, S, Hk, Lmax, total, flags); break;
        case 32: e = cudaLaunchKernelEx(&cfg, kv_fill_kernel<8>, k4, v4, kc, vc, S, Hk, Lmax, total, flags); break;
        case 64: e = cudaLaunchKernelEx(&cfg, kv_fill_kernel<16>, k4, v4, kc, vc, S, Hk, Lmax, total, flags); break;
        case 128: e = cudaLaunchKernelEx(&cfg, kv_fill_kernel<32>, k4, v4, kc, vc, S, Hk, Lmax, total, flags); break;
        default: return set_error(RKV_ERR_UNSUPPORTED, "attn_prefill_fill_cache: head_dim %d", D);
    }
    if (e != cudaSuccess)
        return set_error(RKV_ERR_LAUNCH, "attn_prefill_fill_cache: fill launch: %s", cudaGetErrorString(e));
    return check_launch("attn_prefill_fill_cache");
}

rkv_status launch_scatter(const float* k_new, const float* v_new, float* k_cache, float* v_cache, int M,
                          int T, int Hk, int D, int Lmax, const int* start_pos, int* overflow,
                          unsigned int* flags, cudaStream_t stream, float* const* k_ptrs, float* const* v_ptrs) {
    const int row4 = Hk * (D / 4);
    int tok = kScatterElemsPerBlock / row4;
    if (tok < 1) tok = 1;
    if (tok > kScatterThreads) tok = kScatterThreads;   // one accounting thread per token
    const dim3 grid((unsigned)((T + tok - 1) / tok), (unsigned)M);
    const dim3 block(kScatterThreads);
    auto k4 = reinterpret_cast<const float4*>(k_new);
    auto v4 = reinterpret_cast<const float4*>(v_new);
    auto kc = reinterpret_cast<float4*>(k_cache);
    auto vc = reinterpret_cast<float4*>(v_cache);
    switch (D) {
        case 16: kv_scatter_kernel<4><<<grid, block, 0, stream>>>(k4, v4, kc, vc, T, Hk, Lmax, tok, start_pos, overflow, flags, k_ptrs, v_ptrs); break;
        case 32: kv_scatter_kernel<8><<<grid, block, 0, stream>>>(k4, v4, kc, vc, T, Hk, Lmax, tok, start_pos, overflow, flags, k_ptrs, v_ptrs); break;
        case 64: kv_scatter_kernel<16><<<grid, block, 0, stream>>>(k4, v4, kc, vc, T, Hk, Lmax, tok, start_pos, overflow, flags, k_ptrs, v_ptrs); break;
        case 128: kv_scatter_kernel<32><<<grid, block, 0, stream>>>(k4, v4, kc, vc, T, Hk, Lmax, tok, start_pos, overflow, flags, k_ptrs, v_ptrs); break;
        default: return set_error(RKV_ERR_UNSUPPORTED, "kv_cache_scatter: head_dim %d", D);
    }
    return check_launch("kv_cache_scatter");
}

}  // namespace rkv
