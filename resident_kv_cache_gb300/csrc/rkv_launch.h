// rkv_launch.h -- internal launcher interface between the C ABI and the kernels.
#pragma once

#include <cstddef>

#include "../../include/rkv_attn.h"

namespace rkv {

// Batched decode handles at most 32 sequences (realizar
// cache_from_cache_from_kv_cache.rs, fn init_batched_kv_cache_gpu).
constexpr int kDecodeMaxSeqs = 32;

// The decode workspace starts with a fixed block of completion tickets, one int per
// (sequence, kv head) at index m * n_kv_heads + kh, whatever the call's sizes; the partial
// records follow it.  A workspace sized for the largest call therefore serves calls of any
// sizes without clearing (each call leaves its tickets zero).
constexpr int kDecodeTicketSlots = RKV_DECODE_TICKET_BYTES / 4;
static_assert(RKV_DECODE_TICKET_BYTES % 256 == 0, "records start 256-byte aligned");

struct PrefillArgs {
    const float* q;
    const float* k;        // interleaved [B, S, Hk*D], or the cache [B, Hk, max_len, D] (kv_cache)
    const float* v;
    float* o;
    int B, S, H, Hk, D;
    bool causal;
    const int* seq_lens;   // device valid query rows, may be NULL
    float scale;           // resolved (never 0)
    unsigned int* flags;   // device flag word
    const char* op;        // entry point name for messages
    bool kv_cache;         // K/V read from the cache: query i sits at key position start_pos + i
    int max_len;           // cache capacity (kv_cache)
    const int* start_pos;  // device int32[B] (kv_cache)
    float* k_cache_out;    // non-NULL: also write K/V rows 0..S-1 into these caches [B, Hk, fill_max_len, D]
    float* v_cache_out;
    int fill_max_len;
};

struct DecodeArgs {
    const float* q;
    const float* k_cache;
    const float* v_cache;
    float* o;
    int M, H, Hk, D, Lmax;
    const int* seq_lens;
    float scale;
    void* workspace;
    unsigned int* flags;
    const float* const* k_ptrs = nullptr;   // device float*[M]: per-sequence caches [Hk, Lmax, D]
    const float* const* v_ptrs = nullptr;   // (then k_cache / v_cache are unused)
    const float* k_new = nullptr;           // non-NULL: append [M, Hk*D] rows at len-1 first (fused)
    const float* v_new = nullptr;
};

rkv_status launch_prefill(const PrefillArgs& a, cudaStream_t stream);
// The CTA-pair prefill (prefill_pair.cu): head_dim 128 and an even number of query heads per kv
// head.
bool prefill_pair_supported(const PrefillArgs& a);
rkv_status launch_prefill_pair(const PrefillArgs& a, bool guard, cudaStream_t stream);

bool decode_group_supported(int group);
size_t decode_workspace_bytes(int M, int H, int Hk, int D);
rkv_status launch_decode(const DecodeArgs& a, cudaStream_t stream);

rkv_status launch_scatter(const float* k_new, const float* v_new, float* k_cache, float* v_cache, int M,
                          int T, int Hk, int D, int Lmax, const int* start_pos, int* overflow,
                          unsigned int* flags, cudaStream_t stream, float* const* k_ptrs = nullptr,
                          float* const* v_ptrs = nullptr);

// RoPE prologue: q and the new K rows rotated in place at start_pos[m] + t, K (rotated) and V
// written into the cache (rope_append.cu).  rotary_ndims: multiple of 8, at most head_dim.
constexpr int kRopeMaxPairs = 64;
rkv_status launch_rope_append(float* q, float* k_new, const float* v_new, float* k_cache, float* v_cache, int M, int T,
                              int H, int Hk, int D, int Lmax, const int* start_pos, int rotary_ndims, double theta,
                              int* overflow, unsigned int* flags, cudaStream_t stream);

// Cache fill of rows 0..S-1 (K and V [B, S, Hk*D] -> caches [B, Hk, Lmax, D]) launched as a
// programmatic dependent of the kernel just enqueued on `stream`: it may start while that kernel
// runs, and completes only after it.
rkv_status launch_fill_dependent(const float* k, const float* v, float* k_cache, float* v_cache, int B, int S,
                                 int Hk, int D, int Lmax, unsigned int* flags, cudaStream_t stream);

}  // namespace rkv
