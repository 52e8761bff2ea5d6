// rope_append.cu -- rotary position embedding fused with the KV append.
//
// GPT-NeoX half-split RoPE (trustformers-core 0.2.0 src/gpu_ops/cuda/oxicuda/attention.rs,
// fn rope_neox_gpu_to_gpu: partial rotation of the first rotary_ndims dims of each head at an
// absolute position offset; realizar 0.8.5 src/cuda/executor/cache_from_cache_from_kv_cache.rs,
// fn apply_rope_to_buffer: pair (i, i + half), frequency theta^(-2i/dim), x1' = x1 cos - x2 sin,
// x2' = x1 sin + x2 cos).  The pages run it as separate passes (trustformers pads `offset`
// leading rows to reach an offset); here one launch rotates q and the new K rows in place at
// their own positions (start_pos[m] + t) and writes the rotated K and the V rows into the cache,
// so the prologue of a decode step (or of a prefill) is a single pass over its rows.
//
// Angles: the host passes each frequency in double; per (token, pair) the kernel forms
// position * frequency and reduces it mod 2*pi in double (a few double operations, once per
// token and pair, shared by every head through shared memory), then takes sincosf of the
// reduced angle.  A float angle would be off by ~position * 2^-24 radians.
#include <cmath>

#include "rkv_internal.cuh"
#include "rkv_launch.h"

namespace rkv {

constexpr int kRopeThreads = 256;
constexpr int kRopeTokensPerBlock = 4;

struct RopeFreqs {
    double f[kRopeMaxPairs];   // theta^(-2i / rotary_ndims), i < rotary_ndims / 2
};

template <int D4>
__global__ void __launch_bounds__(kRopeThreads)
rope_append_kernel(float4* __restrict__ q, float4* __restrict__ k_new, const float4* __restrict__ v_new,
                   float4* __restrict__ k_cache, float4* __restrict__ v_cache, int T, int H, int Hk, int Lmax,
                   const int* __restrict__ start_pos, int r, const RopeFreqs freqs, int* __restrict__ overflow,
                   unsigned int* __restrict__ flags) {
    __shared__ float2 cs[kRopeTokensPerBlock][kRopeMaxPairs];   // (cos, sin) per token and pair
    const int m = blockIdx.y;
    const int t0 = blockIdx.x * kRopeTokensPerBlock;
    const int n_tok = min(kRopeTokensPerBlock, T - t0);
    if (n_tok <= 0) return;
    const int p0 = __ldg(start_pos + m);
    if (p0 < 0 && threadIdx.x == 0) atomicOr(flags, RKV_FLAG_NEGATIVE_INPUT);
    const int half = r / 2;
    constexpr double kTwoPi = 6.283185307179586476925286766559;
    for (int idx = threadIdx.x; idx < n_tok * half; idx += kRopeThreads) {
        const int j = idx / half, i = idx - j * half;
        const int64_t pos = max((int64_t)p0 + t0 + j, (int64_t)0);   // rotation position (never negative)
        const double a = (double)pos * freqs.f[i];
        const double red = fma(-rint(a * (1.0 / kTwoPi)), kTwoPi, a);  // in [-pi, pi]
        float s, c;
        sincosf((float)red, &s, &c);
        cs[j][i] = make_float2(c, s);
    }
    __syncthreads();
    if (threadIdx.x < n_tok) {                        // cache bounds accounting, once per token
        const int64_t pos = (int64_t)p0 + t0 + threadIdx.x;
        if ((pos < 0 || pos >= Lmax) && overflow) atomicAdd(overflow, 1);
    }
    const int h4 = half / 4;                          // float4 pairs per head
    const int units = (H + Hk) * h4 + Hk * D4;        // per token: q/k rotations, then k tail + v rows
    for (int idx = threadIdx.x; idx < n_tok * units; idx += kRopeThreads) {
        const int j = idx / units;
        int u = idx - j * units;
        const int t = t0 + j;
        const int64_t pos = (int64_t)p0 + t;
        const bool in_cache = pos >= 0 && pos < Lmax;
        if (u < (H + Hk) * h4) {                      // rotate one float4 pair of q or k
            const int head = u / h4, c4 = u - head * h4;
            const bool is_q = head < H;
            const int hh = is_q ? head : head - H;
            const int64_t roff = is_q ? ((int64_t)m * T + t) * H * D4 + (int64_t)hh * D4
                                      : ((int64_t)m * T + t) * Hk * D4 + (int64_t)hh * D4;
            if (!in_bounds(roff + c4 + h4, (int64_t)gridDim.y * T * (is_q ? H : Hk) * D4, flags)) continue;
            float4* row = (is_q ? q : k_new) + roff;
            const float4 x1 = row[c4], x2 = row[c4 + h4];
            const float2 a0 = cs[j][4 * c4], a1 = cs[j][4 * c4 + 1], a2 = cs[j][4 * c4 + 2], a3 = cs[j][4 * c4 + 3];
            const float4 y1 = make_float4(x1.x * a0.x - x2.x * a0.y, x1.y * a1.x - x2.y * a1.y,
                                          x1.z * a2.x - x2.z * a2.y, x1.w * a3.x - x2.w * a3.y);
            const float4 y2 = make_float4(x1.x * a0.y + x2.x * a0.x, x1.y * a1.y + x2.y * a1.x,
                                          x1.z * a2.y + x2.z * a2.x, x1.w * a3.y + x2.w * a3.x);
            row[c4] = y1;
            row[c4 + h4] = y2;
            if (!is_q && in_cache &&
                in_bounds((((int64_t)m * Hk + hh) * Lmax + pos) * D4 + c4 + h4, (int64_t)gridDim.y * Hk * Lmax * D4, flags)) {
                float4* dst = k_cache + (((int64_t)m * Hk + hh) * Lmax + pos) * D4;
                dst[c4] = y1;
                dst[c4 + h4] = y2;
            }
        } else if (in_cache) {                        // k dims past rotary_ndims, and v: plain copies
            u -= (H + Hk) * h4;
            const int hh = u / D4, c4 = u - hh * D4;
            const int64_t src = ((int64_t)m * T + t) * Hk * D4 + (int64_t)hh * D4 + c4;
            const int64_t dst = (((int64_t)m * Hk + hh) * Lmax + pos) * D4 + c4;
            if (!in_bounds(src, (int64_t)gridDim.y * T * Hk * D4, flags) ||
                !in_bounds(dst, (int64_t)gridDim.y * Hk * Lmax * D4, flags))
                continue;
            if (c4 >= 2 * h4) k_cache[dst] = k_new[src];   // tail of k (not rotated)
            v_cache[dst] = __ldg(v_new + src);
        }
    }
}

rkv_status launch_rope_append(float* q, float* k_new, const float* v_new, float* k_cache, float* v_cache, int M, int T,
                              int H, int Hk, int D, int Lmax, const int* start_pos, int rotary_ndims, double theta,
                              int* overflow, unsigned int* flags, cudaStream_t stream) {
    RopeFreqs fr;
    const int half = rotary_ndims / 2;
    for (int i = 0; i < kRopeMaxPairs; ++i)
        fr.f[i] = i < half ? std::pow(theta, -2.0 * (double)i / (double)rotary_ndims) : 0.0;
    const dim3 grid((unsigned)((T + kRopeTokensPerBlock - 1) / kRopeTokensPerBlock), (unsigned)M);
    auto q4 = reinterpret_cast<float4*>(q);
    auto k4 = reinterpret_cast<float4*>(k_new);
    auto v4 = reinterpret_cast<const float4*>(v_new);
    auto kc = reinterpret_cast<float4*>(k_cache);
    auto vc = reinterpret_cast<float4*>(v_cache);
    switch (D) {
        case 16: rope_append_kernel<4><<<grid, kRopeThreads, 0, stream>>>(q4, k4, v4, kc, vc, T, H, Hk, Lmax, start_pos, rotary_ndims, fr, overflow, flags); break;
        case 32: rope_append_kernel<8><<<grid, kRopeThreads, 0, stream>>>(q4, k4, v4, kc, vc, T, H, Hk, Lmax, start_pos, rotary_ndims, fr, overflow, flags); break;
        case 64: rope_append_kernel<16><<<grid, kRopeThreads, 0, stream>>>(q4, k4, v4, kc, vc, T, H, Hk, Lmax, start_pos, rotary_ndims, fr, overflow, flags); break;
        case 128: rope_append_kernel<32><<<grid, kRopeThreads, 0, stream>>>(q4, k4, v4, kc, vc, T, H, Hk, Lmax, start_pos, rotary_ndims, fr, overflow, flags); break;
        default: return set_error(RKV_ERR_UNSUPPORTED, "kv_append_rope: head_dim %d", D);
    }
    return check_launch("kv_append_rope");
}

}  // namespace rkv
