// prefill_simt.cu -- first correct prefill: one lane group per query row, f32 FMA.
//
// Semantics: trueno-gpu 0.4.11 src/memory/resident/attention.rs,
// fn batched_multihead_attention_optimized (interleaved [seq, n_heads*head_dim]
// in and out, scale 1/sqrt(head_dim)) and trustformers-core 0.2.0
// src/gpu_ops/cuda/oxicuda/attention.rs, fn attention_prefill_gpu_to_gpu
// (causal: query i sees keys 0..=i).  Heads are read in place, no score matrix
// is stored: D/4 lanes share one query row, each holding a float4 of q and of
// the output accumulator, and the softmax is online in base 2.
#include "rkv_internal.cuh"
#include "rkv_launch.h"

namespace rkv {

constexpr int kSimtWarps = 4;
constexpr float kSimtLog2e = 1.4426950408889634f;

template <int D>
__global__ void __launch_bounds__(kSimtWarps * 32)
prefill_simt_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                    float* __restrict__ o, int S, int H, int Hk, bool causal, const int* __restrict__ seq_lens,
                    float scale_log2, unsigned int* __restrict__ flags) {
    constexpr int LPR = D / 4, RPW = 32 / LPR;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int seg = lane % LPR;
    const int i = blockIdx.x * (kSimtWarps * RPW) + warp * RPW + lane / LPR;
    const int bh = blockIdx.y;
    const int b = bh / H, h = bh % H, g = h / (H / Hk);
    int len = S;
    if (seq_lens) {
        len = __ldg(seq_lens + b);
        if (len > S) { len = S; if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(flags, RKV_FLAG_LEN_CLAMPED); }
        if (len < 0) { len = 0; if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(flags, RKV_FLAG_NEGATIVE_INPUT); }
    }
    const int nkeys = (i < S && i < len) ? (causal ? i + 1 : len) : 0;
    int wmax = nkeys;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, off));

    const int64_t q_row = (int64_t)H * D, kv_row = (int64_t)Hk * D;
    float4 qv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < S) {
        qv = __ldg(reinterpret_cast<const float4*>(q + ((int64_t)b * S + i) * q_row + (int64_t)h * D) + seg);
        qv.x *= scale_log2; qv.y *= scale_log2; qv.z *= scale_log2; qv.w *= scale_log2;
    }
    const float4* kb = reinterpret_cast<const float4*>(k + (int64_t)b * S * kv_row + (int64_t)g * D) + seg;
    const float4* vb = reinterpret_cast<const float4*>(v + (int64_t)b * S * kv_row + (int64_t)g * D) + seg;
    const int64_t stride4 = kv_row / 4;

    float mrun = -INFINITY, lrun = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < wmax; ++j) {
        const int jj = j < len ? j : 0;                 // stay in bounds for finished rows
        const float4 kv = __ldg(kb + jj * stride4);
        float s = qv.x * kv.x + qv.y * kv.y + qv.z * kv.z + qv.w * kv.w;
#pragma unroll
        for (int off = LPR / 2; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (j < nkeys) {
            const float mnew = fmaxf(mrun, s);
            const float alpha = fast_exp2(mrun - mnew);
            const float p = fast_exp2(s - mnew);
            const float4 vv = __ldg(vb + jj * stride4);
            lrun = lrun * alpha + p;
            acc.x = acc.x * alpha + p * vv.x;
            acc.y = acc.y * alpha + p * vv.y;
            acc.z = acc.z * alpha + p * vv.z;
            acc.w = acc.w * alpha + p * vv.w;
            mrun = mnew;
        }
    }
    if (i < S) {
        const float inv = lrun > 0.f ? 1.0f / lrun : 0.f;
        float4 r = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        reinterpret_cast<float4*>(o + ((int64_t)b * S + i) * q_row + (int64_t)h * D)[seg] = r;
    }
}

rkv_status launch_prefill_simt(const PrefillArgs& a, cudaStream_t stream) {
    const int rpw = 32 / (a.D / 4);
    const dim3 grid((unsigned)((a.S + kSimtWarps * rpw - 1) / (kSimtWarps * rpw)), (unsigned)(a.B * a.H));
    const dim3 block(kSimtWarps * 32);
    const float sl2 = a.scale * kSimtLog2e;
    switch (a.D) {
        case 16: prefill_simt_kernel<16><<<grid, block, 0, stream>>>(a.q, a.k, a.v, a.o, a.S, a.H, a.Hk, a.causal, a.seq_lens, sl2, a.flags); break;
        case 32: prefill_simt_kernel<32><<<grid, block, 0, stream>>>(a.q, a.k, a.v, a.o, a.S, a.H, a.Hk, a.causal, a.seq_lens, sl2, a.flags); break;
        case 64: prefill_simt_kernel<64><<<grid, block, 0, stream>>>(a.q, a.k, a.v, a.o, a.S, a.H, a.Hk, a.causal, a.seq_lens, sl2, a.flags); break;
        case 128: prefill_simt_kernel<128><<<grid, block, 0, stream>>>(a.q, a.k, a.v, a.o, a.S, a.H, a.Hk, a.causal, a.seq_lens, sl2, a.flags); break;
        default: return set_error(RKV_ERR_UNSUPPORTED, "attn_prefill: head_dim %d", a.D);
    }
    return check_launch("attn_prefill");
}

}  // namespace rkv
